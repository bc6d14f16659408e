"""Pins for the oracle's planner ``plan_ref``.

The fused tiling is pinned by an independent characterisation that determines it
uniquely (greedy, maximal tiles), checked exhaustively over small segment lists and on
seeded random ones; a worked example is derived by hand from the rule.
"""
import itertools

import numpy as np
import pytest

from oracle import BM, merge_segments, plan_ref, row_adapter_ids


def _check_characterisation(off, ids, T, bm=BM):
    fused, shrink = plan_ref(off, ids, T, bm)
    rid = row_adapter_ids(off, ids, T)
    # (i) contiguous cover of [0, T) in order
    pos = 0
    for (row0, n, tid) in fused:
        assert row0 == pos and 1 <= n <= bm
        pos += n
        nz = set(int(a) for a in rid[row0:row0 + n] if a != 0)
        # (iii) at most one nonzero id, and the tile's id is it (0 if none)
        assert len(nz) <= 1
        assert tid == (nz.pop() if nz else 0)
        # (iv) maximal: a short tile that does not end the batch stops only at an adapter change
        if n < bm and row0 + n < T:
            nxt = int(rid[row0 + n])
            assert tid != 0 and nxt != 0 and nxt != tid
    assert pos == T
    # shrink tiles: the fused tiles with a nonzero id, stably ordered by id
    want = sorted([f for f in fused if f[2] != 0], key=lambda f: f[2])
    assert shrink == want
    # every adapter row is in exactly one shrink tile
    cover = np.zeros(T, dtype=int)
    for (row0, n, tid) in shrink:
        cover[row0:row0 + n] += 1
    assert np.all(cover[rid != 0] == 1)
    return fused, shrink


LENGTHS = (0, 1, 2, 127, 128, 129, 255, 300)


@pytest.mark.parametrize("nseg", [1, 2, 3])
def test_plan_ref_exhaustive_small(nseg):
    for lens in itertools.product(LENGTHS, repeat=nseg):
        T = sum(lens)
        off = [0]
        for n in lens:
            off.append(off[-1] + n)
        for ids in itertools.product((0, 1, 2), repeat=nseg):
            _check_characterisation(off, list(ids), T)


def test_plan_ref_exhaustive_four_segments_short_lengths():
    for lens in itertools.product((0, 1, 3, 64), repeat=4):
        T = sum(lens)
        off = [0]
        for n in lens:
            off.append(off[-1] + n)
        for ids in itertools.product((0, 1, 2), repeat=4):
            _check_characterisation(off, list(ids), T, bm=16)


@pytest.mark.parametrize("seed", range(20))
def test_plan_ref_random(seed):
    rng = np.random.default_rng(seed)
    nseg = int(rng.integers(1, 40))
    lens = rng.integers(0, 400, nseg)
    off = [0] + np.cumsum(lens).tolist()
    ids = rng.integers(0, 5, nseg).tolist()
    _check_characterisation(off, ids, int(off[-1]))


def test_plan_ref_worked_example_sweep_batch():
    # base 300, A1 400, base 362, A1 333, base 362, A1 291 (2048 rows). Only one adapter,
    # so no cut ever happens at an id change: tiles are rows [128k, 128k+128).
    # Adapter rows: [300,700), [1062,1395), [1757,2048). Tile k holds adapter rows for
    # k = 2..5 (256..767), 8..10 (1024..1407) and 13..15 (1664..2047).
    off = [0, 300, 700, 1062, 1395, 1757, 2048]
    ids = [0, 1, 0, 1, 0, 1]
    fused, shrink = plan_ref(off, ids, 2048)
    want_ids = [0, 0, 1, 1, 1, 1, 0, 0, 1, 1, 1, 0, 0, 1, 1, 1]
    assert fused == [(128 * k, 128, want_ids[k]) for k in range(16)]
    assert shrink == [(128 * k, 128, 1) for k in range(16) if want_ids[k]]


def test_plan_ref_worked_example_mixed_batch():
    # 6 x 8 base rows, then 4096 rows of adapter 1: the base rows share the first tile
    # with 80 adapter rows; the last tile holds 4144 - 32*128 = 48 rows.
    off = [0, 8, 16, 24, 32, 40, 48, 4144]
    ids = [0] * 6 + [1]
    fused, shrink = plan_ref(off, ids, 4144)
    assert len(fused) == 33
    assert fused[0] == (0, 128, 1) and fused[-1] == (4096, 48, 1)
    assert shrink == fused


def test_plan_ref_worked_example_adapter_change_cuts():
    # A1 10 rows, base 5, A2 10, A2 3 (merged), base 200. The base rows 10-14 stay in
    # adapter 1's tile; the first adapter-2 row (15) starts a new tile, which then runs
    # 128 rows into the trailing base rows; the rest is one base-only tile.
    off = [0, 10, 15, 25, 28, 228]
    ids = [1, 0, 2, 2, 0]
    fused, shrink = plan_ref(off, ids, 228)
    assert fused == [(0, 15, 1), (15, 128, 2), (143, 85, 0)]
    assert shrink == [(0, 15, 1), (15, 128, 2)]


def test_merge_segments():
    off, ids = merge_segments([0, 0, 5, 5, 9, 12], [1, 1, 2, 1, 1])
    assert (off, ids) == ([0, 12], [1])
    off, ids = merge_segments([0, 3, 3, 7, 10], [0, 2, 0, 1])
    assert (off, ids) == ([0, 7, 10], [0, 1])
    assert merge_segments([0, 0], [3]) == ([0], [])


def test_plan_ref_empty_batch():
    assert plan_ref([0], [], 0) == ([], [])
    assert plan_ref([0, 0, 0], [1, 0], 0) == ([], [])


def _mutant_plan_no_adapter_cut(off, ids, T, bm=BM):
    # planted mistake: never cut at an adapter change (two adapters can share a tile)
    rid = row_adapter_ids(off, ids, T)
    fused = []
    for row0 in range(0, T, bm):
        n = min(bm, T - row0)
        nz = [int(a) for a in rid[row0:row0 + n] if a != 0]
        fused.append((row0, n, nz[0] if nz else 0))
    return fused, sorted([f for f in fused if f[2]], key=lambda f: f[2])


def _mutant_plan_cut_at_every_change(off, ids, T, bm=BM):
    # planted mistake: base rows never share a tile with adapter rows (wasteful, not greedy)
    rid = row_adapter_ids(off, ids, T)
    fused = []
    row0 = 0
    for t in range(1, T + 1):
        if t == T or rid[t] != rid[row0] or t - row0 == bm:
            fused.append((row0, t - row0, int(rid[row0])))
            row0 = t
    return fused, sorted([f for f in fused if f[2]], key=lambda f: f[2])


@pytest.mark.parametrize("mutant", [_mutant_plan_no_adapter_cut, _mutant_plan_cut_at_every_change])
def test_characterisation_rejects_planner_mutants(mutant, monkeypatch):
    import oracle
    off, ids, T = [0, 10, 15, 25, 28, 228], [1, 0, 2, 2, 0], 228
    monkeypatch.setitem(globals(), "plan_ref", mutant)
    with pytest.raises(AssertionError):
        _check_characterisation(off, ids, T)
    assert oracle.plan_ref is not mutant

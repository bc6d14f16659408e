"""The C-ABI library builds, loads without a GPU and exports what include/*.h declares;
its planner equals the oracle's bit for bit; its host-side checks reject bad arguments.
No compute call here needs a GPU."""
import glob
import itertools
import os
import re

import numpy as np
import pytest

from oracle import plan_ref

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"\b(lora_linear_\w+)\s*\(", src))
    return names


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("lora_linear_create", "lora_linear_forward", "lora_linear_destroy", "lora_linear_plan"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import ctypes
    for name in sorted(_declared()):
        assert hasattr(lib, name), name
        assert ctypes.cast(getattr(lib, name), ctypes.c_void_p).value


def test_binding_declares_every_export(lib):
    from mixed_lora_projection_gb300 import _lib
    assert set(_lib.SIGNATURES) == _declared()


def test_error_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6, 7):
        assert lib.lora_linear_error_string(code)


# --------------------------------------------------------------------------- planner parity

def _lib_plan(off, ids, T):
    from mixed_lora_projection_gb300.lora_linear import plan
    return plan(off, ids, T)


LENGTHS = (0, 1, 2, 127, 128, 129, 255, 300)


@pytest.mark.parametrize("nseg", [1, 2, 3])
def test_planner_equals_plan_ref_exhaustive(lib, nseg):
    for lens in itertools.product(LENGTHS, repeat=nseg):
        off = [0] + np.cumsum(lens).tolist()
        for ids in itertools.product((0, 1, 2), repeat=nseg):
            T = off[-1]
            assert _lib_plan(off, ids, T) == plan_ref(off, list(ids), T)


def test_planner_equals_plan_ref_four_segments(lib):
    # four segments over the tile-boundary lengths, every id pattern over 0..2
    lens4 = (0, 1, 127, 128, 129, 300)
    for lens in itertools.product(lens4, repeat=4):
        off = [0] + np.cumsum(lens).tolist()
        for ids in itertools.product((0, 1, 2), repeat=4):
            assert _lib_plan(off, ids, off[-1]) == plan_ref(off, list(ids), off[-1])


def test_planner_equals_plan_ref_every_length(lib):
    # one segment of every length 0..300 and two segments on a 7-row grid of lengths, ids 0..2
    for n in range(301):
        for a in (0, 1, 2):
            assert _lib_plan([0, n], [a], n) == plan_ref([0, n], [a], n)
    for l0 in range(0, 301, 7):
        for l1 in range(0, 301, 7):
            off = [0, l0, l0 + l1]
            for ids in itertools.product((0, 1, 2), repeat=2):
                assert _lib_plan(off, ids, off[-1]) == plan_ref(off, list(ids), off[-1])


@pytest.mark.parametrize("seed", range(30))
def test_planner_equals_plan_ref_random(lib, seed):
    rng = np.random.default_rng(1000 + seed)
    nseg = int(rng.integers(1, 64))
    lens = rng.integers(0, int(rng.choice([4, 64, 400, 3000])), nseg)
    off = [0] + np.cumsum(lens).tolist()
    ids = rng.integers(0, int(rng.integers(1, 6)), nseg).tolist()
    T = int(off[-1])
    assert _lib_plan(off, ids, T) == plan_ref(off, ids, T)


def test_planner_workloads(lib):
    from mixed_lora_projection_gb300.synth import WORKLOADS
    for w in WORKLOADS.values():
        assert _lib_plan(w.seg_offsets, w.seg_ids, w.T) == plan_ref(list(w.seg_offsets), list(w.seg_ids), w.T)


@pytest.mark.parametrize("off,ids,T", [([0, 5], [0], 6), ([1, 6], [0], 6), ([0, 4, 3, 6], [0, 1, 0], 6),
                                       ([0, 6], [-1], 6)])
def test_planner_rejects_bad_segments(lib, off, ids, T):
    from mixed_lora_projection_gb300.lora_linear import LoraError
    with pytest.raises(LoraError):
        _lib_plan(off, ids, T)


# --------------------------------------------------------------------------- host-side checks

def _v(**kw):
    from mixed_lora_projection_gb300.lora_linear import validate
    base = dict(d_in=256, d_out=512, rank=16, max_tokens=64, max_segments=4, x_ptr=0x10000000, T=64,
                seg_offsets=[0, 32, 64], seg_ids=[0, 1], w_ptr=0x20000000, a_ptrs=[0x30000000],
                b_ptrs=[0x40000000], scales=[1.0], y_ptr=0x50000000)
    base.update(kw)
    return validate(**base)


def test_validate_accepts_good_arguments(lib):
    assert _v() == 0
    assert _v(T=0, seg_offsets=[0], seg_ids=[]) == 0
    assert _v(T=0, seg_offsets=[0, 0], seg_ids=[1]) == 0
    # unnamed adapters may be NULL
    assert _v(a_ptrs=[0x30000000, None], b_ptrs=[0x40000000, None], scales=[1.0, 1.0]) == 0


@pytest.mark.parametrize("kw", [
    dict(d_in=250), dict(d_out=0), dict(rank=4), dict(rank=264), dict(rank=12),
    dict(max_tokens=0), dict(T=65), dict(T=-1),
    dict(max_tokens=(1 << 24) + 1), dict(max_segments=(1 << 20) + 1), dict(max_tokens=2**31 - 1),
    dict(d_in=(1 << 20) + 8), dict(d_out=(1 << 20) + 8),
    dict(seg_offsets=[0, 32, 63]), dict(seg_offsets=[1, 32, 64]), dict(seg_offsets=[0, 40, 32, 64], seg_ids=[0, 1, 0]),
    dict(seg_ids=[0, 2]), dict(seg_ids=[-1, 1]),
    dict(seg_offsets=[0, 8, 16, 32, 48, 64], seg_ids=[0, 1, 0, 1, 0]),   # n_seg > max_segments
    dict(x_ptr=0x10000008), dict(y_ptr=0x50000004), dict(w_ptr=0x20000002), dict(a_ptrs=[0x30000001]),
    dict(x_ptr=0), dict(y_ptr=0), dict(a_ptrs=[None]), dict(b_ptrs=[None]),
    dict(scales=[float("nan")]), dict(scales=[float("inf")]),
    dict(y_ptr=0x10000000 + 64 * 256 * 2 - 16),                         # y overlaps x
    dict(y_ptr=0x20000000),                                              # y overlaps W
    dict(a_ptrs=[0x50000000 + 32]),                                      # y overlaps A_1
])
def test_validate_rejects(lib, kw):
    assert _v(**kw) == -1


def test_create_without_a_gpu_reports_no_device(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    import ctypes
    h = ctypes.c_void_p()
    assert lib.lora_linear_create(ctypes.byref(h), 256, 512, 16, 64, 4, 0) == -6
    assert not h.value
    assert lib.lora_linear_destroy(None) == 0


# --------------------------------------------------------------------------- host logic

# the launch-shape model's choices for the configured workloads on a 152-SM GB300 (SM pairs
# with 256 columns for the prefills and mixed batches, grouped column tiles for the prefills,
# single CTAs with 240 columns for the decode batch, token-column units of 256 features for the
# near-ridge batch, the sweep's widths)
SHAPES = {
    "prefill_16k": (2, 256, 2), "prefill_32k": (2, 256, 2), "mixed_batch": (2, 256, 1),
    "mixed_8x300": (2, 256, 1), "prefix_tail_1552": (2, 256, 1), "mixed_decode": (1, 240, None),
    "mixed_near_ridge": (2, 256, 3), "sweep_qkv": (2, 224, None), "sweep_o": (2, 288, None),
    "sweep_gate_up": (2, 256, None), "sweep_down": (2, 288, None),
}
# K halves chosen by a handle of max_tokens = the workload's rows: none of the configured
# workloads (their batches are past the small-batch path, or their K is 5,120)
K_SPLITS = {"sweep_o": 1, "sweep_down": 1, "sweep_qkv": 1, "sweep_gate_up": 1, "prefill_16k": 1, "prefill_32k": 1,
            "mixed_batch": 1, "mixed_decode": 1, "mixed_near_ridge": 1, "mixed_8x300": 1, "prefix_tail_1552": 1,
            "tiny": 1}


@pytest.mark.parametrize("name", sorted(SHAPES))
def test_launch_shape_model_choices(lib, name):
    from mixed_lora_projection_gb300 import launch_shape
    from mixed_lora_projection_gb300.synth import WORKLOADS
    w = WORKLOADS[name]
    s = launch_shape(w.d_in, w.d_out, w.rank, 152, w.T, w.seg_offsets, w.seg_ids)
    cluster, tile_n, order = SHAPES[name]
    assert (s["cluster"], s["tile_n"]) == (cluster, tile_n), s
    if order is not None:
        assert s["unit_order"] == order, s
    # work units: every fused group crosses every column tile once (token-column units: one group
    # of every row); one shrink unit per group of adapter tiles
    n_tiles = -(-w.T // 128)
    groups = 1 if s["unit_order"] == 3 else -(-n_tiles // cluster)
    assert s["fused_units"] >= groups * -(-w.d_out // tile_n) - 1
    assert (s["shrink_units"] == 0) == (w.adapter_rows == 0)
    assert s["bk"] == 64 and 2 <= s["stages"] <= 16


@pytest.mark.parametrize("name", sorted(K_SPLITS))
def test_k_split_choices(lib, name):
    from mixed_lora_projection_gb300 import k_split, launch_shape
    from mixed_lora_projection_gb300.synth import WORKLOADS
    w = WORKLOADS[name]
    ks = k_split(w.d_in, w.d_out, w.rank, w.T, 152)
    assert ks == K_SPLITS[name]
    # with halves every block is two units: the shape model's unit counts are even
    s = launch_shape(w.d_in, w.d_out, w.rank, 152, w.T, w.seg_offsets, w.seg_ids)
    if ks == 2:
        assert s["fused_units"] % 2 == 0 and s["shrink_units"] % 2 == 0 and s["tile_n"] == 256


def test_k_split_rule(lib):
    from mixed_lora_projection_gb300 import LoraError, k_split, launch_shape
    # decode-sized handles on narrow projections with long K split in halves (o 6,144 and down
    # 17,408 -> 5,120); K of 5,120 never does, nor do handles whose batches pass the small-batch
    # path; quarters only when asked for
    for d_in in (6144, 17408):
        for T in (1, 8, 48, 128, 129, 200, 384):
            assert k_split(d_in, 5120, 256, T, 152) == 2, (d_in, T)
        for T in (385, 2048, 32768):
            assert k_split(d_in, 5120, 256, T, 152) == 1, (d_in, T)
    for d_out in (5120, 12288, 34816):
        assert k_split(5120, d_out, 256, 48, 152) == 1
    assert k_split(6080, 5120, 256, 48, 152) == 1        # 95 K-steps of 64
    # a split handle's units come in pairs
    s = launch_shape(6144, 5120, 256, 152, 48, [0, 48], [0])
    assert s["fused_units"] % 2 == 0 and s["fused_units"] >= 2 * (5120 // s["tile_n"])
    with pytest.raises(LoraError):
        k_split(6144, 5120, 256, 48, 1)          # fewer than 2 SMs
    with pytest.raises(LoraError):
        k_split(6144, 5120, 300, 48, 152)        # rank above 256


def test_token_column_rule(lib):
    from mixed_lora_projection_gb300 import launch_shape

    def order(d_in, d_out, T, off, ids, sms=152):
        return launch_shape(d_in, d_out, 256, sms, T, off, ids)["unit_order"]
    # gate_up batches of 129 to 448 rows with one adapter (or none) take token-column units:
    # 256 output features of an SM pair for every row, 136 units
    for T in (129, 160, 200, 256, 300, 348, 400, 448):
        for off, ids in (((0, 48, T), (0, 1)), ((0, T), (0,)), ((0, T), (1,))):
            s = launch_shape(5120, 34816, 256, 152, T, off, ids)
            assert s["unit_order"] == 3 and s["cluster"] == 2 and s["tile_n"] == 256, (T, ids)
            assert s["fused_units"] == 136 and s["shrink_units"] == (0 if ids == (0,) else -(-(-(-T // 128)) // 2))
    # not: one tile (a decode step), more than 448 rows (four nearly full row tiles on SM pairs;
    # only on request, up to 512), two adapters, a base-only tile next to an adapter tile, handles
    # that split K (o and down up to 384 rows), 20 units on 76 SM pairs (o and down past 384 rows),
    # qkv's 300- and 348-row base batches (row tiles measured faster)
    assert order(5120, 34816, 48, (0, 48), (0,)) != 3
    assert order(5120, 34816, 512, (0, 512), (0,)) != 3 and order(5120, 34816, 513, (0, 513), (0,)) != 3
    assert order(5120, 34816, 300, (0, 100, 300), (1, 2)) != 3
    assert order(5120, 34816, 300, (0, 128, 300), (0, 1)) != 3
    for d_in in (6144, 17408):
        for T in (200, 348, 400, 512):
            assert order(d_in, 5120, T, (0, 48, T), (0, 1)) != 3, (d_in, T)
    assert order(5120, 12288, 300, (0, 300), (0,)) != 3 and order(5120, 12288, 348, (0, 348), (0,)) != 3
    assert order(5120, 12288, 400, (0, 400), (0,)) == 3 and order(5120, 12288, 448, (0, 48, 448), (0, 1)) == 3


def test_wide_tile_rule(lib):
    from mixed_lora_projection_gb300 import launch_shape

    def shape(d_in, d_out, T, off, ids):
        s = launch_shape(d_in, d_out, 256, 152, T, off, ids)
        return s["cluster"], s["tile_n"]
    # o and down (K of 96 and 272 steps of 64) with half their rows on an adapter, where 256-column
    # units leave the last wave of 76 SM pairs at most half full, take wide row tiles (the shapes
    # measured): 1,024 rows (80 units + shrink, 8% of a second wave), 2,048 rows (17% of a third)
    # -> 288 columns; 2,176 rows (43%) -> 320; 1,024 rows also without adapter rows or all on one
    for d_in in (6144, 17408):
        for T, tn in ((1024, 288), (2048, 288), (2176, 320)):
            assert shape(d_in, 5120, T, (0, T // 2, T), (0, 1)) == (2, tn), (d_in, T)
        for off, ids in (((0, 1024), (0,)), ((0, 1024), (1,))):
            assert shape(d_in, 5120, 1024, off, ids) == (2, 288), (d_in, ids)
    # not: a last wave more than half full (3,456 base rows: 68%), K of 80 steps (qkv, gate_up,
    # the 16k prefill's 5,120 -> 5,120), decode-sized batches (single CTAs)
    for d_in in (6144, 17408):
        assert shape(d_in, 5120, 3456, (0, 3456), (0,))[1] <= 256
        assert shape(d_in, 5120, 48, (0, 48), (0,))[0] == 1
    for d_out in (12288, 34816, 5120):
        for T in (1024, 2048, 2176, 4096, 16384):
            assert shape(5120, d_out, T, (0, T // 2, T), (0, 1))[1] <= 256, (d_out, T)


def test_launch_shape_of_an_empty_batch_and_bad_arguments(lib):
    from mixed_lora_projection_gb300 import LoraError, launch_shape
    assert launch_shape(256, 512, 16, 152, 0, [0], [])["fused_units"] == 0
    with pytest.raises(LoraError):
        launch_shape(256, 512, 16, 1, 64, [0, 64], [0])           # fewer than 2 SMs
    with pytest.raises(LoraError):
        launch_shape(250, 512, 16, 152, 64, [0, 64], [0])         # d_in not a multiple of 8
    with pytest.raises(LoraError):
        launch_shape(256, 512, 16, 152, 64, [0, 60], [0])         # segments do not span T


@pytest.mark.parametrize("T", [0, 1, 127, 2047, 2048, 2049, 4144, 9999, 16384, 32768, 100000, 1 << 24])
def test_host_chunk_schedule(lib, T):
    # the host-buffer path's row chunks: cover [0, T] in order, at most 16 (its event ring),
    # interior bounds on 128-row tiles, one chunk below 2,048 rows, and no chunk at either end
    # larger than the chunks in the middle (the copy-in before the first kernel and the
    # copy-out after the last one overlap nothing)
    from mixed_lora_projection_gb300 import host_chunks
    b = host_chunks(T)
    assert b[0] == 0 and b[-1] == T
    n = len(b) - 1
    assert 1 <= n <= 16
    if T < 2048:
        assert n == 1
        return
    sizes = [b[i + 1] - b[i] for i in range(n)]
    assert all(x > 0 for x in sizes)
    assert all(v % 128 == 0 for v in b[1:-1])
    mid = max(sizes)
    assert sizes[0] <= mid and sizes[-1] <= mid
    assert sizes[0] < mid and sizes[-1] <= mid   # a ramp at the start


# the 4-bit kernel's shape: two feature tiles per unit for a decode batch (one token tile, no
# adapter rows); token groups fastest where the packed base exceeds 32 MB and X fits in 64 MB;
# one group of three tiles for the near-ridge batch (128 + 128 + 92 rows)
W4_SHAPES = {
    # name: (output columns per unit, unit order, token groups)
    "prefill_16k": (128, 0, 64), "mixed_batch": (128, 1, 17), "mixed_8x300": (128, 1, 10),
    "prefix_tail_1552": (128, 1, 7), "mixed_near_ridge": (128, 0, 1), "mixed_decode": (256, 0, 1),
    "prefill_32k": (128, 0, 128),
}


@pytest.mark.parametrize("name", sorted(W4_SHAPES))
def test_w4_launch_shape_choices(lib, name):
    from mixed_lora_projection_gb300 import launch_shape
    from mixed_lora_projection_gb300.synth import WORKLOADS
    w = WORKLOADS[name]
    s = launch_shape(w.d_in, w.d_out, w.rank, 152, w.T, w.seg_offsets, w.seg_ids, w4=True)
    cols, order, groups = W4_SHAPES[name]
    assert (s["cluster"], s["tile_n"], s["unit_order"]) == (1, cols, order), s
    assert s["fused_units"] == groups * -(-w.d_out // cols)
    assert (s["shrink_units"] == 0) == (w.adapter_rows == 0)


def test_w4_decode_shapes_fill_the_gpu(lib):
    # 48-row decode batches on the 4-bit base: gate_up keeps two feature tiles per unit (136 units),
    # qkv runs one tile per unit (96 units), o and down one tile per unit with K in 3 parts (40 x 3
    # units) on a decode-sized handle; a handle for more than 128 rows never splits
    from mixed_lora_projection_gb300 import launch_shape
    from mixed_lora_projection_gb300.synth import WORKLOADS
    want = {"decode_gate_up": (256, 136), "decode_qkv": (128, 96), "decode_o": (128, 120), "decode_down": (128, 120)}
    for name, (cols, units) in want.items():
        w = WORKLOADS[name]
        s = launch_shape(w.d_in, w.d_out, w.rank, 152, w.T, w.seg_offsets, w.seg_ids, w4=True)
        assert (s["tile_n"], s["fused_units"]) == (cols, units), (name, s)
    s = launch_shape(6144, 5120, 256, 152, 129, (0, 129), (0,), w4=True)
    assert s["fused_units"] == 40          # one token group of two tiles, whole K


def test_w4_launch_shape_rejects_d_in_not_multiple_of_128(lib):
    from mixed_lora_projection_gb300 import LoraError, launch_shape
    with pytest.raises(LoraError):
        launch_shape(192, 256, 16, 152, 16, [0, 16], [0], w4=True)

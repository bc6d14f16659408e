"""Token-column units (LORA_OPT_TOKEN_COLUMNS): each unit of an SM pair computes 256 output
features for every token row of the batch (features on the MMA's M, tokens on its N). Checked
against the fp64 oracle and bit for bit against the row-tile units of the same handle (a row's
bits do not depend on the launch shape), over one and two MMAs per K-step, one and two TMEM
accumulators, ragged token counts and feature tails, base-only batches, the expand's wait for
every shrink tile (flags held back, two launches, graph replays), programmatic dependent launch
and a wait that runs out."""
import numpy as np
import pytest
import torch

from mixed_lora_projection_gb300.synth import WORKLOADS, Workload, make_inputs

from gpu_util import TOL, oracle_full, oracle_rows, rel_err, run, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from mixed_lora_projection_gb300 import build
    build.ensure_built()
    return torch.device("cuda", 0)


def _ll(w, max_segments=16):
    from mixed_lora_projection_gb300 import LoraLinear
    return LoraLinear(w.d_in, w.d_out, w.rank, w.T, max_segments, 0)


def _units(ll, T, off, ids):
    return ll.describe(T, off, ids)["n_units"]


def _order(ll, T, off, ids):
    return ll.describe(T, off, ids)["unit_order"]


def _yt_units(w, n_shrink_groups):
    return -(-w.d_out // 256) + n_shrink_groups


# (T, d_in, d_out, r, lengths, ids): one MMA of N = 16 .. 256 per K-step (T <= 256), two
# (T > 256), one accumulator past 256 columns; feature tails (d_out not a multiple of 256);
# K past the last 64-wide step; base rows inside adapter tiles
CASES = [
    (5, 8, 8, 8, [5], [1]),
    (48, 320, 600, 16, [8] * 6, [0] * 6),
    (100, 320, 600, 16, [100], [1]),
    (129, 256, 520, 48, [60, 69], [0, 1]),
    (200, 384, 1000, 32, [200], [1]),
    (256, 320, 776, 256, [256], [1]),
    (257, 200, 264, 24, [257], [0]),
    (300, 520, 264, 24, [48, 252], [0, 1]),
    (348, 1024, 2048, 256, [8] * 6 + [300], [0] * 6 + [1]),
    (400, 192, 776, 64, [100, 300], [0, 1]),
    (511, 136, 1000, 128, [511], [0]),
    (512, 256, 512, 64, [512], [1]),
]


@pytest.mark.parametrize("case", CASES, ids=[f"T{c[0]}_{c[1]}x{c[2]}_r{c[3]}" for c in CASES])
def test_token_columns_match_oracle_and_row_tiles_bitwise(dev, case):
    from mixed_lora_projection_gb300 import _lib as L
    T, d_in, d_out, r, lens, ids = case
    off = [0] + np.cumsum(lens).tolist()
    w = Workload("yt", 31, T, d_in, d_out, r, tuple(off), tuple(ids), scales=(1.25,))
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        ll.set_option(L.OPT_TOKEN_COLUMNS, 2)
        n_yt = _units(ll, T, off, ids)
        assert _order(ll, T, off, ids) == 3
        y = run(ll, inp, off, ids).clone()
        ll.set_option(L.OPT_TOKEN_COLUMNS, 1)
        assert _order(ll, T, off, ids) != 3
        y_rows = run(ll, inp, off, ids)
        torch.cuda.synchronize()
        assert ll.status() == 0
    n_shrink = (-(-T // 128) + 1) // 2 if any(ids) else 0
    assert n_yt == _yt_units(w, n_shrink)
    assert rel_err(y, oracle_full(inp, off, ids)) <= TOL
    assert torch.equal(y, y_rows)


def test_near_ridge_batch_full_size(dev):
    # 48 chat rows + a 300-row decision on gate_up (5,120 -> 34,816): the auto shape takes
    # token-column units; sampled rows against the oracle, every row bitwise against row tiles,
    # and the 48 chat rows bitwise against the same rows alone (single CTAs, row tiles)
    from mixed_lora_projection_gb300 import _lib as L
    w = WORKLOADS["mixed_near_ridge"]
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with _ll(w) as ll:
        assert _order(ll, w.T, off, ids) == 3 and _units(ll, w.T, off, ids) == _yt_units(w, 2)
        y = run(ll, inp, off, ids).clone()
        alone = ll.forward(inp.x[:48], off[:7], ids[:6], inp.w, inp.a, inp.b, inp.scales).clone()
        ll.set_option(L.OPT_TOKEN_COLUMNS, 1)
        y_rows = run(ll, inp, off, ids)
        torch.cuda.synchronize()
        assert ll.status() == 0
    rows = sample_rows(w.T, off, ids, n_random=64)
    assert rel_err(y[torch.as_tensor(rows, device=dev)], oracle_rows(inp, off, ids, rows)) <= TOL
    assert torch.equal(y, y_rows)
    assert torch.equal(y[:48], alone)


@pytest.mark.parametrize("mode", ["publish_delay", "two_launch"])
def test_expand_waits_for_every_shrink_tile(dev, mode):
    # three shrink tiles (two SM-pair groups) feed every token-column unit: with each flag held
    # back 300 us, or with the shrink as its own launch, the output equals the plain call's, for
    # two inputs in turn (an expand that did not wait would read the other input's U rows)
    from mixed_lora_projection_gb300 import _lib as L
    T = 348
    off, ids = [0, 48, 348], [0, 1]
    w = Workload("yt_wait", 32, T, 512, 1024, 64, tuple(off), tuple(ids))
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        ll.set_option(L.OPT_TOKEN_COLUMNS, 2)
        want = []
        for seed in (1, 2):
            g = torch.Generator(device="cpu").manual_seed(seed)
            inp.x.copy_(torch.randn(inp.x.shape, generator=g).to(torch.bfloat16))
            want.append(run(ll, inp, off, ids).clone())
        if mode == "publish_delay":
            ll.set_option(L.OPT_DEBUG_PUBLISH_DELAY_US, 300)
        else:
            ll.set_option(L.OPT_TWO_LAUNCH, 1)
        for seed, ref in zip((1, 2), want):
            g = torch.Generator(device="cpu").manual_seed(seed)
            inp.x.copy_(torch.randn(inp.x.shape, generator=g).to(torch.bfloat16))
            y = run(ll, inp, off, ids)
            torch.cuda.synchronize()
            assert ll.status() == 0
            assert torch.equal(y, ref)
    assert rel_err(want[1], oracle_full(inp, off, ids)) <= TOL


def test_graph_replays_of_token_columns(dev):
    # a captured call with token-column units (adapter rows: cooperative, ready flags) and one
    # without (base rows) replayed three times equal the eager calls
    from mixed_lora_projection_gb300 import _lib as L
    T = 300
    w = Workload("yt_graph", 33, T, 512, 1024, 32, (0, 40, T), (0, 1))
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        ll.set_option(L.OPT_TOKEN_COLUMNS, 2)
        cases = [([0, 40, T], [0, 1]), ([0, T], [0])]
        ref = [run(ll, inp, o, i).clone() for o, i in cases]
        outs = [torch.zeros_like(r) for r in ref]
        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            for (o, i), y in zip(cases, outs):
                run(ll, inp, o, i, y=y)
        torch.cuda.current_stream(dev).wait_stream(s)
        torch.cuda.synchronize()
        for y in outs:
            y.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for (o, i), y in zip(cases, outs):
                run(ll, inp, o, i, y=y)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert all(torch.equal(a, b) for a, b in zip(ref, outs))


def test_programmatic_dependent_launch_with_token_columns(dev):
    # a chain of base-row calls, each reading the previous call's Y, with token-column units
    # and LORA_OPT_PDL: W tiles go to the A stages before the dependency wait; equal to the chain
    # run without it
    from mixed_lora_projection_gb300 import LoraLinear, _lib as L
    T = 300
    wa = Workload("ytp_a", 34, T, 1024, 1536, 16, (0, T), (0,))
    wb = Workload("ytp_b", 35, T, 1536, 1024, 16, (0, T), (0,))
    ia, ib = make_inputs(wa, dev), make_inputs(wb, dev)
    with LoraLinear(1024, 1536, 16, T, 4, 0) as ha, LoraLinear(1536, 1024, 16, T, 4, 0) as hb:
        for h in (ha, hb):
            h.set_option(L.OPT_TOKEN_COLUMNS, 2)

        def chain(pdl):
            for h in (ha, hb):
                h.set_option(L.OPT_PDL, pdl)
            x, outs = ia.x, []
            for i in range(6):
                h, inp = (ha, ia) if i % 2 == 0 else (hb, ib)
                x = h.forward(x, [0, T], [0], inp.w, inp.a, inp.b, inp.scales)
                outs.append(x)
            return outs
        ref = [y.clone() for y in chain(0)]
        got = chain(1)
        torch.cuda.synchronize()
        assert ha.status() == 0 and hb.status() == 0
    assert all(torch.equal(a, b) for a, b in zip(ref, got))


def test_wait_limit_with_token_columns(dev):
    # the load warp never issues: every wait runs out, the call reports LORA_ETIMEOUT, and the
    # next call on the handle is correct
    from mixed_lora_projection_gb300 import _lib as L
    T = 300
    off, ids = [0, 48, T], [0, 1]
    w = Workload("yt_stall", 36, T, 256, 512, 32, tuple(off), tuple(ids))
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        ll.set_option(L.OPT_TOKEN_COLUMNS, 2)
        ll.set_option(L.OPT_WAIT_LIMIT_US, 20000)
        ll.set_option(L.OPT_DEBUG_STALL, 1)
        run(ll, inp, off, ids)
        torch.cuda.synchronize()
        assert ll.status(reset=True) == L.LORA_ETIMEOUT
        ll.set_option(L.OPT_DEBUG_STALL, 0)
        y = run(ll, inp, off, ids)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert rel_err(y, oracle_full(inp, off, ids)) <= TOL


def test_batches_that_rule_out_token_columns(dev):
    # two adapters among the rows, a handle that splits K, or more than 512 rows: the forced
    # option leaves the shape to row tiles, and results stay correct
    from mixed_lora_projection_gb300 import LoraLinear, _lib as L
    off, ids = [0, 100, 300], [1, 2]
    w = Workload("yt_two", 37, 300, 256, 512, 32, tuple(off), tuple(ids), n_adapters=2, scales=(1.0, -0.5))
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        ll.set_option(L.OPT_TOKEN_COLUMNS, 2)
        order = _order(ll, 300, off, ids)
        y = run(ll, inp, off, ids)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert order != 3
    assert rel_err(y, oracle_full(inp, off, ids)) <= TOL
    with LoraLinear(6144, 512, 16, 300, 4, 0) as ll:
        ll.set_option(L.OPT_K_SPLIT, 2)
        ll.set_option(L.OPT_TOKEN_COLUMNS, 2)
        assert _order(ll, 300, [0, 300], [0]) != 3
    with LoraLinear(256, 512, 16, 600, 4, 0) as ll:
        ll.set_option(L.OPT_TOKEN_COLUMNS, 2)
        assert _order(ll, 513, [0, 513], [0]) != 3 and _order(ll, 512, [0, 512], [0]) == 3

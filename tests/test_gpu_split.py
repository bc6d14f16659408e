"""GPU tests of the K parts (LORA_OPT_K_SPLIT = 2 or 4): every shrink and fused block runs as
that many work units over parts of the base K-steps; every part but the last to finish stores
its fp32 sums, the last adds all of them in part order and rounds. Against the fp64 oracle, and bit for bit across
everything that must not change a row's sum on one handle: launch shape, K-step width, unit
order, one launch or two, the batch a row is in, host-buffer chunks, graph replays."""
import numpy as np
import pytest
import torch

from oracle import row_adapter_ids
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


def _ll(w, split=2, max_segments=64):
    from mixed_lora_projection_gb300 import LoraLinear, _lib as L
    ll = LoraLinear(w.d_in, w.d_out, w.rank, max(w.T, 1), max_segments, 0)
    ll.set_option(L.OPT_K_SPLIT, split)
    return ll


def _w(name, T, d_in, d_out, r, lens, ids, seed=31):
    off = [0] + np.cumsum(lens).tolist()
    na = max(1, max(ids))
    return Workload(name, seed, T, d_in, d_out, r, tuple(off), tuple(ids), n_adapters=na,
                    scales=tuple(0.5 + 0.5 * k for k in range(na)))


SMALL = [
    # (T, d_in, d_out, r, lens, ids): odd and even counts of 64-wide K-steps, ragged d_out, one
    # tile, several adapters, empty segments, a batch with no adapter rows
    (64, 1024, 512, 16, [32, 32], [0, 1]),
    (300, 1088, 264, 24, [0, 100, 1, 0, 199], [1, 0, 2, 2, 1]),
    (517, 1152, 1000, 128, [10, 5, 10, 3, 200, 289], [1, 0, 2, 2, 0, 3]),
    (7, 2048, 384, 256, [3, 4], [0, 1]),
    (48, 1280, 640, 32, [8] * 6, [0] * 6),
]


@pytest.mark.parametrize("case", SMALL, ids=[f"T{c[0]}_{c[1]}x{c[2]}" for c in SMALL])
@pytest.mark.parametrize("cluster", [1, 2])
@pytest.mark.parametrize("parts", [2, 4])
def test_parts_match_oracle_and_every_launch_form(dev, case, cluster, parts):
    from mixed_lora_projection_gb300 import _lib as L
    T, d_in, d_out, r, lens, ids = case
    w = _w("split", T, d_in, d_out, r, lens, ids)
    off = list(w.seg_offsets)
    inp = make_inputs(w, dev)
    outs = []
    with _ll(w, split=parts) as ll:
        assert ll.describe(T, off, ids)["n_units"] % parts == 0
        ll.set_option(L.OPT_CLUSTER, cluster if T > 128 else 1)
        outs.append(run(ll, inp, off, ids).clone())
        ll.set_option(L.OPT_TILE_K, 32)                 # 32-wide K stages: the same halves
        outs.append(run(ll, inp, off, ids).clone())
        ll.set_option(L.OPT_TILE_K, 0)
        ll.set_option(L.OPT_TWO_LAUNCH, 1)              # shrink halves in a launch of their own
        outs.append(run(ll, inp, off, ids).clone())
        ll.set_option(L.OPT_TWO_LAUNCH, 0)
        ll.set_option(L.OPT_INLINE_WORK_LIST, 0)        # uploaded work list
        outs.append(run(ll, inp, off, ids).clone())
        ll.set_option(L.OPT_INLINE_WORK_LIST, 1)
        for mode in (1, 2):                             # unit orders
            ll.set_option(L.OPT_RASTER, mode)
            outs.append(run(ll, inp, off, ids).clone())
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert rel_err(outs[0], oracle_full(inp, off, ids)) <= TOL
    for y in outs[1:]:
        assert torch.equal(y, outs[0])


def test_single_ctas_equal_sm_pairs_with_halves(dev):
    from mixed_lora_projection_gb300 import _lib as L
    w = WORKLOADS["sweep_o_multi"]
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        ll.set_option(L.OPT_CLUSTER, 1)
        y1 = run(ll, inp, w.seg_offsets, w.seg_ids).clone()
        ll.set_option(L.OPT_CLUSTER, 2)
        y2 = run(ll, inp, w.seg_offsets, w.seg_ids)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("proj", [("o", 6144), ("down", 17408)])
def test_auto_halves_on_decode_batches_of_long_k_projections(dev, proj):
    # a handle for 48-row batches of the o or down projection chooses K halves by itself; the
    # result matches the oracle, and so does the same batch with whole K
    from mixed_lora_projection_gb300 import LoraLinear, k_split, _lib as L
    name, d_in = proj
    w = _w(f"dec_{name}", 48, d_in, 5120, 256, [8] * 5 + [8], [0, 0, 0, 0, 0, 1])
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    assert k_split(w.d_in, w.d_out, w.rank, w.T, sms) == 2
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with LoraLinear(w.d_in, w.d_out, w.rank, w.T, 16, 0) as ll:
        ys = run(ll, inp, off, ids).clone()
        assert ll.describe(w.T, off, ids)["n_units"] % 2 == 0
        ll.set_option(L.OPT_K_SPLIT, 1)
        yw = run(ll, inp, off, ids)
        torch.cuda.synchronize()
        assert ll.status() == 0
    ref = oracle_full(inp, off, ids)
    assert rel_err(ys, ref) <= TOL
    assert rel_err(yw, ref) <= TOL


@pytest.mark.parametrize("name", ["sweep_o", "sweep_down_multi"])
def test_forced_halves_on_the_sweep_projections(dev, name):
    # 2,048-row batches with halves forced: every sampled row against the oracle
    w = WORKLOADS[name]
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with _ll(w) as ll:
        ys = run(ll, inp, off, ids)
        assert ll.describe(w.T, off, ids)["n_units"] % 2 == 0
        torch.cuda.synchronize()
        assert ll.status() == 0
    rows = sample_rows(w.T, off, ids, n_random=256, seed=41)
    assert rel_err(ys[torch.as_tensor(rows, device=dev)], oracle_rows(inp, off, ids, rows)) <= TOL


def test_rows_do_not_depend_on_the_batch_with_halves(dev):
    # one request's rows alone (a decode-sized batch: single CTAs, narrow tiles) and inside a
    # 2,048-row batch (SM pairs, 256-column tiles): the same halves, the same bits
    w = WORKLOADS["sweep_down_multi"]
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with _ll(w) as ll:
        full = run(ll, inp, off, ids).clone()
        s0, s1 = off[3], off[4]                          # the second adapter request
        alone = ll.forward(inp.x[s0:s1].contiguous(), [0, s1 - s0], [ids[3]], inp.w, inp.a, inp.b, inp.scales)
        dec = ll.forward(inp.x[:48].contiguous(), [0, 48], [ids[0]], inp.w, inp.a, inp.b, inp.scales)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert torch.equal(full[s0:s1], alone)
    assert torch.equal(full[:48], dec)


def test_quarters_in_part_order_whichever_part_ends_last(dev):
    # four parts of K on a 48-row batch of the down projection: every output is ((P0 + P1) + P2) + P3
    # whatever order the parts finish in; repeated calls (different arrival orders) give the same
    # bits, single CTAs and SM pairs too, and the result matches the oracle
    from mixed_lora_projection_gb300 import _lib as L
    w = _w("q_down", 48, 17408, 5120, 64, [8] * 5 + [8], [0, 0, 0, 0, 0, 1])
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with _ll(w, split=4) as ll:
        ys = [run(ll, inp, off, ids).clone() for _ in range(5)]
        ll.set_option(L.OPT_MAX_CTAS, 40)                 # fewer SMs: other arrival orders
        ys.append(run(ll, inp, off, ids).clone())
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert all(torch.equal(y, ys[0]) for y in ys)
    assert rel_err(ys[0], oracle_full(inp, off, ids)) <= TOL


def test_forced_parts_are_clamped_to_short_k(dev):
    # four parts asked for on d_in = 320 (five K-steps of 64): the handle keeps every part at least
    # one K-step long (two parts), and the result matches the oracle
    w = _w("short_k", 100, 320, 256, 16, [50, 50], [0, 1])
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with _ll(w, split=4) as ll:
        assert ll.describe(w.T, off, ids)["n_units"] % 2 == 0
        y = run(ll, inp, off, ids)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert rel_err(y, oracle_full(inp, off, ids)) <= TOL


def test_decode_batch_on_a_narrow_long_k_projection(dev):
    # 48 rows through the o projection (6,144 -> 5,120): with halves every column block is two
    # units, twice as many SMs stream W
    w = _w("dec_o", 48, 6144, 5120, 256, [8] * 6, [0] * 6)
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with _ll(w) as ll:
        y2 = run(ll, inp, off, ids).clone()
        units2 = ll.describe(w.T, off, ids)["n_units"]
        from mixed_lora_projection_gb300 import _lib as L
        ll.set_option(L.OPT_K_SPLIT, 1)
        y1 = run(ll, inp, off, ids)
        torch.cuda.synchronize()
        assert ll.status() == 0
    ref = oracle_full(inp, off, ids)
    assert rel_err(y2, ref) <= TOL and rel_err(y1, ref) <= TOL
    assert units2 % 2 == 0


def test_host_buffers_equal_device_path_with_halves(dev):
    # row chunks from 2,048 rows: every chunk is a call of its own on the same halves
    w = _w("split_host", 4200, 1024, 768, 64, [100, 2000, 100, 2000], [1, 0, 2, 1])
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    x_host = inp.x.cpu().pin_memory()
    y_host = torch.empty((w.T, w.d_out), dtype=torch.bfloat16).pin_memory()
    with _ll(w) as ll:
        y = run(ll, inp, off, ids).clone()
        ll.forward_host(x_host, off, ids, inp.w, inp.a, inp.b, inp.scales, y_host)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert torch.equal(y.cpu(), y_host)
    rows = sample_rows(w.T, off, ids, n_random=128, seed=43)
    assert rel_err(y[torch.as_tensor(rows, device=dev)], oracle_rows(inp, off, ids, rows)) <= TOL


def test_graph_replays_with_halves_and_late_flags(dev):
    # captured and replayed three times with fresh X, the shrink halves publishing 300 us late:
    # the counters and flags are cleared by every launch, so each replay equals an eager call
    from mixed_lora_projection_gb300 import _lib as L
    w = WORKLOADS["sweep_o_multi"]
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with _ll(w) as ll:
        ref = run(ll, inp, off, ids).clone()
        ll.set_option(L.OPT_DEBUG_PUBLISH_DELAY_US, 300)
        y = torch.empty_like(ref)
        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            run(ll, inp, off, ids, y=y)                  # shape cached before capture
        torch.cuda.current_stream(dev).wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            run(ll, inp, off, ids, y=y)
        x0 = inp.x.clone()
        for seed in range(3):
            gen = torch.Generator(device=dev)
            gen.manual_seed(seed)
            inp.x.copy_(torch.randn(inp.x.shape, generator=gen, device=dev).to(torch.bfloat16))
            g.replay()
            torch.cuda.synchronize()
            ll.set_option(L.OPT_DEBUG_PUBLISH_DELAY_US, 0)
            want = run(ll, inp, off, ids).clone()
            torch.cuda.synchronize()
            ll.set_option(L.OPT_DEBUG_PUBLISH_DELAY_US, 300)
            assert torch.equal(y, want), seed
        inp.x.copy_(x0)
        assert ll.status() == 0


def test_halves_report_timeouts_and_the_handle_recovers(dev):
    # the load warp never issues: every wait runs out after 20 ms, the status word reports it,
    # and the next call (counters cleared by the aborted launch) is correct
    from mixed_lora_projection_gb300 import _lib as L
    w = _w("split_stall", 300, 1024, 768, 32, [48, 200, 52], [0, 1, 0])
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with _ll(w) as ll:
        ll.set_option(L.OPT_WAIT_LIMIT_US, 20000)
        ll.set_option(L.OPT_DEBUG_STALL, 1)
        run(ll, inp, off, ids)
        torch.cuda.synchronize()
        assert ll.status(reset=True) == L.LORA_ETIMEOUT
        ll.set_option(L.OPT_DEBUG_STALL, 0)
        ll.set_option(L.OPT_WAIT_LIMIT_US, 4000000)
        y = run(ll, inp, off, ids)
        torch.cuda.synchronize()
        assert ll.status() == L.LORA_OK
    assert rel_err(y, oracle_full(inp, off, ids)) <= TOL


def test_base_rows_with_halves_equal_an_all_base_run(dev):
    w = WORKLOADS["sweep_o_multi"]
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with _ll(w) as ll:
        y = run(ll, inp, off, ids).clone()
        y0 = run(ll, inp, off, [0] * len(ids))
        torch.cuda.synchronize()
        assert ll.status() == 0
    base = torch.as_tensor(row_adapter_ids(off, ids, w.T) == 0, device=dev)
    assert torch.equal(y[base], y0[base])

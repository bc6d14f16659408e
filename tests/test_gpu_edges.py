"""GPU edge cases through the C-ABI: many requests and many adapters (work lists too large for
the kernel parameters, dozens of tensor maps), adapters named out of order and more than once,
unnamed adapters passed as NULL, scale 0 and negative scales, one handle reused for batches of
very different sizes, and rows that give the same bits in any batch."""
import numpy as np
import pytest
import torch

from oracle import row_adapter_ids
from mixed_lora_projection_gb300.synth import Workload, make_inputs

from gpu_util import TOL, oracle_full, oracle_rows, rel_err, run, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from mixed_lora_projection_gb300 import build
    build.ensure_built()
    return torch.device("cuda", 0)


def _ll(d_in, d_out, r, max_tokens, max_segments):
    from mixed_lora_projection_gb300 import LoraLinear
    return LoraLinear(d_in, d_out, r, max_tokens, max_segments, 0)


def test_many_requests_and_adapters(dev):
    # 300 requests (some empty), 40 of 64 adapters named in scattered order and several times
    rng = np.random.default_rng(7)
    n_seg, n_adapters = 300, 64
    lens = rng.integers(0, 41, n_seg)
    lens[rng.integers(0, n_seg, 20)] = 0
    named = rng.choice(np.arange(1, n_adapters + 1), 40, replace=False)
    ids = np.where(rng.random(n_seg) < 0.3, 0, rng.choice(named, n_seg))
    off = [0] + np.cumsum(lens).tolist()
    T = off[-1]
    scales = tuple(float(s) for s in rng.uniform(-2.0, 2.0, n_adapters))
    w = Workload("many", 21, T, 512, 768, 32, tuple(off), tuple(int(i) for i in ids), n_adapters=n_adapters,
                 scales=scales)
    inp = make_inputs(w, dev)
    used = set(int(i) for i in ids if i)
    a_ptrs = [a if (k + 1) in used else None for k, a in enumerate(inp.a)]   # unnamed: NULL
    b_ptrs = [b if (k + 1) in used else None for k, b in enumerate(inp.b)]
    with _ll(512, 768, 32, T, n_seg) as ll:
        y = ll.forward(inp.x, off, list(w.seg_ids), inp.w, a_ptrs, b_ptrs, inp.scales)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert rel_err(y, oracle_full(inp, off, list(w.seg_ids))) <= TOL


def test_scale_zero_gives_base_rows_and_negative_scale_matches_oracle(dev):
    lens, ids = [100, 200, 156], [1, 2, 1]
    off = [0] + np.cumsum(lens).tolist()
    w0 = Workload("s0", 22, off[-1], 384, 640, 64, tuple(off), tuple(ids), n_adapters=2, scales=(0.0, 0.0))
    inp = make_inputs(w0, dev)
    with _ll(384, 640, 64, off[-1], 8) as ll:
        y0 = ll.forward(inp.x, off, ids, inp.w, inp.a, inp.b, [0.0, 0.0]).clone()
        yb = ll.forward(inp.x, off, [0, 0, 0], inp.w, inp.a, inp.b, [0.0, 0.0]).clone()
        yn = ll.forward(inp.x, off, ids, inp.w, inp.a, inp.b, [-1.75, 0.5])
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert torch.equal(y0, yb)                   # s = 0: U = 0, the expand adds exact zeros
    inp.scales = (-1.75, 0.5)
    assert rel_err(yn, oracle_full(inp, off, ids)) <= TOL


def test_one_handle_serves_batches_of_any_size(dev):
    # a handle for up to 4,300 rows serves 1, 130, 4,300, 777, 0 and 48 rows in turn
    d_in, d_out, r = 1024, 1536, 256
    with _ll(d_in, d_out, r, 4300, 16) as ll:
        for i, (T, lens, ids) in enumerate([(1, [1], [1]), (130, [2, 128], [0, 1]),
                                             (4300, [1000, 3000, 300], [1, 0, 2]),
                                             (777, [777], [2]), (0, [], []), (48, [8] * 6, [0] * 6)]):
            off = [0] + np.cumsum(lens).tolist() if lens else [0]
            w = Workload("sizes", 23 + i, max(T, 1), d_in, d_out, r, tuple(off) if lens else (0, 1),
                         tuple(ids) if ids else (0,), n_adapters=2, scales=(1.0, -0.5))
            inp = make_inputs(w, dev)
            if T == 0:
                y = torch.full((1, d_out), 7.0, dtype=torch.bfloat16, device=dev)
                ll.forward(inp.x[:0], [0], [], inp.w, inp.a, inp.b, inp.scales, y=y[:0])
                torch.cuda.synchronize()
                assert torch.all(y == 7.0)
                continue
            y = run(ll, inp, off, ids)
            torch.cuda.synchronize()
            assert ll.status() == 0
            rows = sample_rows(T, off, ids, n_random=64, seed=i) if T > 512 else list(range(T))
            ref = oracle_rows(inp, off, ids, rows)
            assert rel_err(y[torch.as_tensor(rows, device=dev)], ref) <= TOL, T


def test_rows_do_not_depend_on_the_batch_they_are_in(dev):
    # the 48 decode rows of the mixed batch, computed inside the 4,144-row batch (SM pairs,
    # 256-column tiles, next to 4,096 adapter rows) and alone (single CTAs, 240-column tiles):
    # the same bits
    from mixed_lora_projection_gb300 import LoraLinear
    from mixed_lora_projection_gb300.synth import WORKLOADS
    w = WORKLOADS["mixed_batch"]
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with LoraLinear(w.d_in, w.d_out, w.rank, w.T, 16, 0) as ll:
        full = run(ll, inp, off, ids).clone()
        shape_full = ll.describe(w.T, off, ids)
        alone = ll.forward(inp.x[:48], off[:7], ids[:6], inp.w, inp.a, inp.b, inp.scales)
        shape_alone = ll.describe(48, off[:7], ids[:6])
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert shape_full["tile_n"] != shape_alone["tile_n"] or shape_full["grid"] != shape_alone["grid"]
    assert torch.equal(full[:48], alone)


@pytest.mark.parametrize("name", ["prefill_16k", "mixed_batch", "mixed_decode", "mixed_near_ridge",
                                  "sweep_o", "sweep_down"])
def test_host_shape_model_equals_the_device_handle(dev, name):
    # the host-only launch_shape (given the device's SM count) and a device handle's describe
    # name the same shape
    from mixed_lora_projection_gb300 import LoraLinear, launch_shape
    from mixed_lora_projection_gb300.synth import WORKLOADS
    w = WORKLOADS[name]
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    host = launch_shape(w.d_in, w.d_out, w.rank, sms, w.T, w.seg_offsets, w.seg_ids)
    with LoraLinear(w.d_in, w.d_out, w.rank, w.T, 16, 0) as ll:
        d = ll.describe(w.T, w.seg_offsets, w.seg_ids)
    assert d["tile_n"] == host["tile_n"] and d["stages"] == host["stages"]
    assert d["n_units"] == host["fused_units"] + host["shrink_units"]


def test_max_ctas_caps_the_grid_and_changes_no_bit(dev):
    # a launch capped to fewer SMs (SM pairs round down to whole pairs) computes the same bits
    from mixed_lora_projection_gb300 import LoraError, _lib as L
    from mixed_lora_projection_gb300.synth import WORKLOADS
    w = WORKLOADS["sweep_o_multi"]
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with _ll(w.d_in, w.d_out, w.rank, w.T, 16) as ll:
        y0 = run(ll, inp, off, ids).clone()
        ys = []
        for cap in (40, 7):
            ll.set_option(L.OPT_MAX_CTAS, cap)
            assert ll.describe(w.T, off, ids)["grid"] <= cap
            ys.append(run(ll, inp, off, ids).clone())
        for bad in (1, -1):
            with pytest.raises(LoraError):
                ll.set_option(L.OPT_MAX_CTAS, bad)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert all(torch.equal(y, y0) for y in ys)


def test_two_calls_side_by_side_on_disjoint_sm_counts(dev):
    # the near-ridge batch as one call, and as two calls on two streams capped to 100 and 52 SMs
    # (rows 0-255 on SM pairs, the 92-row tail on single CTAs): the same bits
    from mixed_lora_projection_gb300 import LoraLinear, _lib as L
    from mixed_lora_projection_gb300.synth import WORKLOADS
    w = WORKLOADS["mixed_near_ridge"]
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    y = torch.empty((w.T, w.d_out), dtype=torch.bfloat16, device=dev)
    main = torch.cuda.current_stream(dev)
    sa, sb = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    with LoraLinear(w.d_in, w.d_out, w.rank, w.T, 16, 0) as one, \
            LoraLinear(w.d_in, w.d_out, w.rank, 256, 16, 0) as ha, LoraLinear(w.d_in, w.d_out, w.rank, 128, 16, 0) as hb:
        ref = run(one, inp, off, ids).clone()
        ha.set_option(L.OPT_CLUSTER, 2)
        ha.set_option(L.OPT_MAX_CTAS, 100)
        hb.set_option(L.OPT_MAX_CTAS, 52)
        for _ in range(3):
            sa.wait_stream(main)
            sb.wait_stream(main)
            ha.forward(inp.x[:256], off[:7] + [256], ids, inp.w, inp.a, inp.b, inp.scales, y=y[:256], stream=sa)
            hb.forward(inp.x[256:], [0, w.T - 256], [1], inp.w, inp.a, inp.b, inp.scales, y=y[256:], stream=sb)
            main.wait_stream(sa)
            main.wait_stream(sb)
        torch.cuda.synchronize()
        assert ha.status() == 0 and hb.status() == 0
    assert torch.equal(y, ref)

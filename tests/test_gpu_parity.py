"""GPU parity: the CUDA path through the C-ABI against the fp64 oracle on the same seeded
bf16 inputs (max|dY| / max|Y_ref| <= 5e-3), plus bit-exact routing invariants, odd
shapes, guard rows and determinism."""
import numpy as np
import pytest
import torch

from oracle import row_adapter_ids
from mixed_lora_projection_gb300.synth import WORKLOADS, Workload, make_inputs

from gpu_util import TOL, f64, oracle_full, oracle_rows, rel_err, run, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from mixed_lora_projection_gb300 import build
    build.ensure_built()
    return torch.device("cuda", 0)


def _ll(w, max_segments=64, max_tokens=None):
    from mixed_lora_projection_gb300 import LoraLinear
    return LoraLinear(w.d_in, w.d_out, w.rank, max_tokens or max(w.T, 1), max_segments, 0)


# --------------------------------------------------------------------------- layout pins

def test_one_hot_rows_give_columns_of_w_exactly(dev):
    # X row t = e_{k(t)}: every output is a single product W[n,k] * 1, exact in fp32 and bf16
    T, d_in, d_out = 256, 384, 512
    w = Workload("onehot", 9, T, d_in, d_out, 16, (0, T), (0,))
    inp = make_inputs(w, dev)
    k = torch.arange(T, device=dev) * 7 % d_in
    inp.x.zero_()
    inp.x[torch.arange(T, device=dev), k] = 1.0
    with _ll(w) as ll:
        y = run(ll, inp, [0, T], [0])
    torch.cuda.synchronize()
    want = inp.w[:, k].t().contiguous()
    assert torch.equal(y, want)


def test_one_hot_adapter_lands_in_one_column(dev):
    # W = 0, A[j0,k0] = 1, B[n0,j0] = 1, s = 2: Y[t,n] = 2 X[t,k0] at n = n0, else 0
    T, d_in, d_out, r = 200, 256, 384, 32
    w = Workload("onehot_ad", 9, T, d_in, d_out, r, (0, T), (1,), scales=(2.0,))
    inp = make_inputs(w, dev)
    j0, k0, n0 = 5, 77, 301
    inp.w.zero_()
    inp.a[0].zero_(); inp.a[0][j0, k0] = 1.0
    inp.b[0].zero_(); inp.b[0][n0, j0] = 1.0
    with _ll(w) as ll:
        y = run(ll, inp, [0, T], [1])
    torch.cuda.synchronize()
    want = torch.zeros_like(y)
    want[:, n0] = (2.0 * inp.x[:, k0].float()).to(torch.bfloat16)
    assert torch.equal(y, want)


# --------------------------------------------------------------------------- tiny config, full compare

def test_tiny_matches_oracle(dev):
    w = WORKLOADS["tiny"]
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        y = run(ll, inp, w.seg_offsets, w.seg_ids)
    torch.cuda.synchronize()
    ref = oracle_full(inp, list(w.seg_offsets), list(w.seg_ids))
    assert rel_err(y, ref) <= TOL
    # the delta is not negligible: adapter rows differ from base rows by O(1)
    base = oracle_full(inp, list(w.seg_offsets), [0] * len(w.seg_ids))
    assert np.abs(ref[32:] - base[32:]).max() > 0.5


# --------------------------------------------------------------------------- odd shapes

ODD = [
    # (T, d_in, d_out, r, lengths, ids, n_adapters)
    (1, 256, 512, 16, [1], [1], 1),
    (7, 128, 256, 16, [3, 4], [0, 1], 1),
    (127, 192, 320, 32, [127], [1], 1),
    (129, 256, 512, 64, [64, 65], [1, 0], 1),
    (300, 520, 264, 24, [0, 100, 1, 0, 199], [1, 0, 2, 2, 1], 2),
    (517, 136, 1000, 128, [10, 5, 10, 3, 200, 289], [1, 0, 2, 2, 0, 3], 3),
    (1024, 1024, 768, 256, [128, 256, 1, 639], [2, 1, 0, 2], 2),
    (260, 4096, 4096, 256, [260], [0], 1),
    # the smallest legal shapes: every TMA box is larger than its tensor (read as zeros past it)
    (5, 8, 8, 8, [5], [1], 1),
    (3, 64, 24, 8, [1, 2], [1, 0], 1),
]


@pytest.mark.parametrize("case", ODD, ids=[f"T{c[0]}_{c[1]}x{c[2]}_r{c[3]}" for c in ODD])
def test_odd_shapes_match_oracle(dev, case):
    T, d_in, d_out, r, lens, ids, na = case
    off = [0] + np.cumsum(lens).tolist()
    w = Workload("odd", 7, T, d_in, d_out, r, tuple(off), tuple(ids), n_adapters=na,
                 scales=tuple(0.5 + 0.75 * k for k in range(na)))
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        y = run(ll, inp, off, ids)
    torch.cuda.synchronize()
    ref = oracle_full(inp, off, ids)
    assert rel_err(y, ref) <= TOL


@pytest.mark.parametrize("tile_n", [16, 48, 128, 240, 256])
def test_forced_tile_widths_match_oracle(dev, tile_n):
    from mixed_lora_projection_gb300 import _lib as L
    T, d_in, d_out, r = 300, 512, 1008, 32
    off, ids = [0, 100, 180, 300], [1, 0, 1]
    w = Workload("tilen", 8, T, d_in, d_out, r, tuple(off), tuple(ids))
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        ll.set_option(L.OPT_TILE_N, tile_n)
        y = run(ll, inp, off, ids)
    torch.cuda.synchronize()
    assert rel_err(y, oracle_full(inp, off, ids)) <= TOL


# --------------------------------------------------------------------------- bit-exact invariants

def test_base_rows_bit_identical_to_all_base_run(dev):
    w = WORKLOADS["sweep_qkv_multi"]
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with _ll(w) as ll:
        y = run(ll, inp, off, ids)
        y0 = run(ll, inp, off, [0] * len(ids))
    torch.cuda.synchronize()
    base = torch.as_tensor(row_adapter_ids(off, ids, w.T) == 0, device=dev)
    assert torch.equal(y[base], y0[base])
    assert not torch.equal(y[~base], y0[~base])


def test_zero_b_adapter_rows_bit_identical_to_base(dev):
    w = WORKLOADS["sweep_o"]
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    for b in inp.b:
        b.zero_()
    with _ll(w) as ll:
        y = run(ll, inp, off, ids)
        y0 = run(ll, inp, off, [0] * len(ids))
    torch.cuda.synchronize()
    assert torch.equal(y, y0)


@pytest.mark.parametrize("name", ["sweep_qkv_multi", "mixed_near_ridge", "tiny"])
def test_one_launch_equals_two_launches(dev, name):
    # the in-kernel shrink->expand dependency gives exactly the two-launch result
    from mixed_lora_projection_gb300 import _lib as L
    w = WORKLOADS[name]
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        y1 = run(ll, inp, w.seg_offsets, w.seg_ids).clone()
        ll.set_option(L.OPT_TWO_LAUNCH, 1)
        y2 = run(ll, inp, w.seg_offsets, w.seg_ids)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("name", ["tiny", "sweep_qkv_multi", "mixed_near_ridge", "prefill_16k"])
def test_cta_pairs_equal_single_ctas(dev, name):
    # SM pairs (tcgen05 cta_group::2, M = 256: each CTA loads its own 128 A rows and half of the
    # B tile, the even CTA issues the MMAs) compute exactly what single CTAs do
    from mixed_lora_projection_gb300 import _lib as L
    w = WORKLOADS[name]
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        ll.set_option(L.OPT_CLUSTER, 2)
        y2 = run(ll, inp, w.seg_offsets, w.seg_ids).clone()
        ll.set_option(L.OPT_CLUSTER, 1)
        y1 = run(ll, inp, w.seg_offsets, w.seg_ids)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("name", ["tiny", "sweep_down_multi", "mixed_near_ridge", "mixed_decode"])
def test_k_step_32_equals_64(dev, name):
    # 64-byte-swizzled 32-wide K stages issue the same K=16 MMA sequence as 64-wide ones
    from mixed_lora_projection_gb300 import _lib as L
    w = WORKLOADS[name]
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        ll.set_option(L.OPT_TILE_K, 64)
        y64 = run(ll, inp, w.seg_offsets, w.seg_ids).clone()
        ll.set_option(L.OPT_TILE_K, 32)
        y32 = run(ll, inp, w.seg_offsets, w.seg_ids)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert torch.equal(y64, y32)


def test_mixed_base_and_adapter_pairs(dev):
    # SM pairs may combine a base tile with an adapter tile (the base half's expand reads a
    # block of U that is always zero): row tiles base | a1 | a2 | base | a1 (+ base rows) | a3 |
    # base | base give pairs base-first, adapter-first, an a1/a3 pair that cannot form (padded)
    # and a trailing pad
    from mixed_lora_projection_gb300 import _lib as L
    lens, ids = [128, 128, 128, 128, 64, 64, 128, 256], [0, 1, 2, 0, 1, 0, 3, 0]
    off = [0] + np.cumsum(lens).tolist()
    w = Workload("mixpair", 15, off[-1], 512, 768, 64, tuple(off), tuple(ids), n_adapters=3,
                 scales=(0.5, 1.25, 2.0))
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        ll.set_option(L.OPT_CLUSTER, 2)
        y2 = run(ll, inp, off, ids).clone()
        y0 = run(ll, inp, off, [0] * len(ids)).clone()
        ll.set_option(L.OPT_CLUSTER, 1)
        y1 = run(ll, inp, off, ids)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert rel_err(y2, oracle_full(inp, off, ids)) <= TOL
    base = torch.as_tensor(row_adapter_ids(off, ids, w.T) == 0, device=dev)
    assert torch.equal(y2[base], y0[base])
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("cluster", [1, 2])
def test_raster_orders_are_exact(dev, cluster):
    # the order in which units visit row and column tiles (row tiles first, column tiles first,
    # groups of column tiles, groups that do not divide the column-tile count) changes which
    # SM computes a block, never its MMA sequence: all results are identical
    from mixed_lora_projection_gb300 import _lib as L
    lens, ids = [200, 300, 1, 267, 256], [1, 0, 2, 2, 1]
    off = [0] + np.cumsum(lens).tolist()
    w = Workload("raster", 20, off[-1], 384, 1000, 64, tuple(off), tuple(ids), n_adapters=2, scales=(0.5, 1.5))
    inp = make_inputs(w, dev)
    outs = []
    with _ll(w) as ll:
        ll.set_option(L.OPT_CLUSTER, cluster)
        ll.set_option(L.OPT_TILE_N, 128)                      # 8 column tiles
        for mode, group in [(0, 4), (1, 4), (2, 4), (3, 1), (3, 3), (3, 4), (3, 8), (3, 100)]:
            ll.set_option(L.OPT_RASTER, mode)
            ll.set_option(L.OPT_RASTER_GROUP, group)
            outs.append(run(ll, inp, off, ids).clone())
        torch.cuda.synchronize()
        assert ll.status() == 0
    for y in outs[1:]:
        assert torch.equal(y, outs[0])
    assert rel_err(outs[0], oracle_full(inp, off, ids)) <= TOL


@pytest.mark.parametrize("cluster", [1, 2])
@pytest.mark.parametrize("case", [(300, 320, 272, 64), (517, 384, 1000, 128)], ids=["odd_k_steps", "even_k_steps"])
def test_mma_grouping_is_exact(dev, case, cluster):
    # the MMA warp waiting for one or two stages at once issues the same MMA sequence; an odd
    # number of K-steps per unit (5 base + 1 expand) exercises the single-stage tail
    from mixed_lora_projection_gb300 import _lib as L
    T, d_in, d_out, r = case
    lens, ids = [100, 1, 0, 199], [1, 0, 2, 2]
    if T == 517:
        lens, ids = [10, 5, 10, 3, 200, 289], [1, 0, 2, 2, 0, 3]
    off = [0] + np.cumsum(lens).tolist()
    na = max(ids)
    w = Workload("grp", 14, T, d_in, d_out, r, tuple(off), tuple(ids), n_adapters=na, scales=(0.5,) * na)
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        ll.set_option(L.OPT_CLUSTER, cluster)
        ll.set_option(L.OPT_MMA_GROUP, 1)
        y1 = run(ll, inp, off, ids).clone()
        ll.set_option(L.OPT_MMA_GROUP, 2)
        y2 = run(ll, inp, off, ids)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert torch.equal(y1, y2)
    assert rel_err(y2, oracle_full(inp, off, ids)) <= TOL


@pytest.mark.parametrize("name", ["tiny", "sweep_qkv_multi", "mixed_decode", "mixed_near_ridge"])
def test_inline_work_list_equals_uploaded(dev, name):
    # small work lists travel in the kernel parameters; the result equals the uploaded path
    from mixed_lora_projection_gb300 import _lib as L
    w = WORKLOADS[name]
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        y1 = run(ll, inp, w.seg_offsets, w.seg_ids).clone()
        ll.set_option(L.OPT_INLINE_WORK_LIST, 0)
        y2 = run(ll, inp, w.seg_offsets, w.seg_ids)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert torch.equal(y1, y2)


def test_repeated_calls_reuse_flags(dev):
    # many calls in a row on one handle: each launch clears its ready flags, none goes stale
    w = WORKLOADS["sweep_o_multi"]
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        ys = [run(ll, inp, w.seg_offsets, w.seg_ids).clone() for _ in range(20)]
        torch.cuda.synchronize()
        assert ll.status() == 0
    for y in ys[1:]:
        assert torch.equal(y, ys[0])


def test_deterministic(dev):
    w = WORKLOADS["sweep_down"]
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        y1 = run(ll, inp, w.seg_offsets, w.seg_ids).clone()
        y2 = run(ll, inp, w.seg_offsets, w.seg_ids)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


def test_guard_rows_untouched(dev):
    T, d_in, d_out, r, G = 333, 256, 520, 16, 3
    off, ids = [0, 100, 101, 333], [1, 0, 1]
    w = Workload("guard", 6, T, d_in, d_out, r, tuple(off), tuple(ids))
    inp = make_inputs(w, dev)
    full = torch.full((T + 2 * G, d_out), -77.0, dtype=torch.bfloat16, device=dev)
    with _ll(w) as ll:
        run(ll, inp, off, ids, y=full[G:G + T])
    torch.cuda.synchronize()
    assert bool((full[:G] == -77.0).all()) and bool((full[G + T:] == -77.0).all())
    assert rel_err(full[G:G + T], oracle_full(inp, off, ids)) <= TOL


@pytest.mark.parametrize("cluster", [1, 2])
def test_bounded_waits_report_timeout_and_the_handle_recovers(dev, cluster):
    # the load warp never issues: every wait runs out after 20 ms, the kernel returns with
    # the status word set (no hang, no trap), and the next normal call is correct again
    from mixed_lora_projection_gb300 import _lib as L
    w = WORKLOADS["sweep_o"]
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        ll.set_option(L.OPT_CLUSTER, cluster)
        ll.set_option(L.OPT_WAIT_LIMIT_US, 20000)
        ll.set_option(L.OPT_DEBUG_STALL, 1)
        run(ll, inp, w.seg_offsets, w.seg_ids)
        torch.cuda.synchronize()
        assert ll.status(reset=True) == L.LORA_ETIMEOUT
        assert ll.status() == L.LORA_OK
        ll.set_option(L.OPT_DEBUG_STALL, 0)
        ll.set_option(L.OPT_WAIT_LIMIT_US, 4000000)
        y = run(ll, inp, w.seg_offsets, w.seg_ids)
        torch.cuda.synchronize()
        assert ll.status() == L.LORA_OK
    rows = sample_rows(w.T, list(w.seg_offsets), list(w.seg_ids), n_random=64, seed=1)
    ref = oracle_rows(inp, list(w.seg_offsets), list(w.seg_ids), rows)
    assert rel_err(y[torch.as_tensor(rows, device=dev)], ref) <= TOL


def test_empty_batch_launches_nothing(dev):
    w = WORKLOADS["tiny"]
    inp = make_inputs(w, dev)
    with _ll(w) as ll:
        y = torch.empty((0, w.d_out), dtype=torch.bfloat16, device=dev)
        ll.forward(inp.x[:0], [0], [], inp.w, inp.a, inp.b, inp.scales, y=y)
        _, _, launched = ll.timing(1)
        assert launched == 0


def test_invalid_call_leaves_output_untouched(dev):
    from mixed_lora_projection_gb300 import LoraError
    w = WORKLOADS["tiny"]
    inp = make_inputs(w, dev)
    y = torch.full((w.T, w.d_out), 3.0, dtype=torch.bfloat16, device=dev)
    with _ll(w) as ll:
        with pytest.raises(LoraError):
            run(ll, inp, [0, 32, 63], [0, 1], y=y)        # offsets do not end at T
        with pytest.raises(LoraError):
            run(ll, inp, [0, 32, 64], [0, 2], y=y)        # adapter 2 does not exist
        torch.cuda.synchronize()
        assert bool((y == 3.0).all())
        assert ll.timing(1)[2] == 0


@pytest.mark.parametrize("name", ["tiny", "mixed_batch", "sweep_qkv_multi", "prefix_tail_1552", "sweep_down"])
def test_host_buffers_path_matches_device_path(dev, name):
    # the host-buffer entry point pipelines row chunks (from 2,048 rows) over copy and compute
    # streams; each chunk is planned on its own rows, and a row's sums do not depend on the
    # batch it is in, so the result is the device path's bit for bit (sweep_down: the device call
    # runs 288-column wide row tiles, its chunks narrower ones)
    w = WORKLOADS[name]
    inp = make_inputs(w, dev)
    x_host = inp.x.cpu().pin_memory()
    y_host = torch.full((w.T, w.d_out), 5.0, dtype=torch.bfloat16).pin_memory()
    with _ll(w) as ll:
        y = run(ll, inp, w.seg_offsets, w.seg_ids)
        ll.forward_host(x_host, w.seg_offsets, w.seg_ids, inp.w, inp.a, inp.b, inp.scales, y_host)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert torch.equal(y.cpu(), y_host)


# --------------------------------------------------------------------------- full-size workloads

FULL = ["prefill_16k", "mixed_batch", "mixed_decode", "mixed_near_ridge", "prefill_32k", "mixed_8x300",
        "prefix_tail_1552"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload_sampled_rows(dev, name):
    w = WORKLOADS[name]
    inp = make_inputs(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with _ll(w) as ll:
        y = run(ll, inp, off, ids)
    torch.cuda.synchronize()
    rows = sample_rows(w.T, off, ids, n_random=256, seed=w.index)
    ref = oracle_rows(inp, off, ids, rows)
    assert rel_err(y[torch.as_tensor(rows, device=dev)], ref) <= TOL


@pytest.mark.parametrize("proj", ["qkv", "o", "gate_up", "down", "qkv_multi", "down_multi"])
def test_sweep_layer_sampled_rows(dev, proj):
    w = WORKLOADS[f"sweep_{proj}"]
    inp = make_inputs(w, dev, layer=23)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with _ll(w) as ll:
        y = run(ll, inp, off, ids)
    torch.cuda.synchronize()
    rows = sample_rows(w.T, off, ids, n_random=1024, seed=3)
    ref = oracle_rows(inp, off, ids, rows)
    assert rel_err(y[torch.as_tensor(rows, device=dev)], ref) <= TOL


@pytest.mark.parametrize("proj", ["qkv", "o", "gate_up", "down"])
def test_sweep_every_layer_sampled_rows(dev, proj):
    # each of the 24 layers on its own seeded X, W, A and B (layers are not chained): rows
    # [0, 64), every segment boundary +-2, every tile boundary +-1 and 256 seeded random rows
    w = WORKLOADS[f"sweep_{proj}"]
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with _ll(w) as ll:
        for layer in range(24):
            inp = make_inputs(w, dev, layer=layer)
            y = run(ll, inp, off, ids)
            torch.cuda.synchronize()
            assert ll.status() == 0
            rows = sample_rows(w.T, off, ids, n_random=256, seed=100 + layer)
            ref = oracle_rows(inp, off, ids, rows)
            assert rel_err(y[torch.as_tensor(rows, device=dev)], ref) <= TOL, layer

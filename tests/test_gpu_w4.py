"""GPU parity of the 4-bit-base path (lora_linear_w4_repack + lora_linear_forward_w4) against
the fp64 oracle on the same seeded inputs: W[n,k] = q[n,k] * s[k//128, n], adapters in bf16.
The oracle reads the plain layout; the library reads the kernel layout written by its repack."""
import numpy as np
import pytest
import torch

from oracle import bf16_bits_to_f64, lora_linear_w4_fp64, row_adapter_ids, w4_dequantize_fp64, w4_weights_bf16_fp64
from oracle import lora_linear_rows_fp64
from mixed_lora_projection_gb300.synth import WORKLOADS, Workload, bf16_bits, make_inputs, make_w4_base

from gpu_util import TOL, f64, rel_err, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from mixed_lora_projection_gb300 import build
    build.ensure_built()
    return torch.device("cuda", 0)


def _ll(w, max_segments=64):
    from mixed_lora_projection_gb300 import LoraLinear
    return LoraLinear(w.d_in, w.d_out, w.rank, max(w.T, 1), max_segments, 0)


def _kq(q):
    from mixed_lora_projection_gb300 import w4_repack
    return w4_repack(q)


def _kernel_layout_np(q):
    """The kernel layout, restated from the header's description, one word at a time."""
    w = np.ascontiguousarray(q.cpu().numpy()).view(np.uint32).astype(np.uint64)
    out = np.zeros_like(w)
    for j in range(4):
        out |= ((w >> (8 * j)) & 0xF) << (4 * j)           # feature 8c+2j -> nibble j
        out |= ((w >> (8 * j + 4)) & 0xF) << (4 * j + 16)  # feature 8c+2j+1 -> nibble j+4
    out ^= 0x88888888                                      # offset binary q + 8
    return out.astype(np.uint32).view(np.uint8).reshape(q.shape)


def _oracle(inp, q, sc, off, ids, rows=None):
    qn = q.cpu().numpy()
    sb = bf16_bits(sc)
    a64 = [f64(a) for a in inp.a]
    b64 = [f64(b) for b in inp.b]
    if rows is None:
        return lora_linear_w4_fp64(f64(inp.x), off, ids, qn, sb, a64, b64, inp.scales)
    w = w4_weights_bf16_fp64(qn, sb)
    rid = row_adapter_ids(off, ids, inp.x.shape[0])[rows]
    return lora_linear_rows_fp64(f64(inp.x[torch.as_tensor(rows, device=inp.x.device)]), rid, w, a64, b64, inp.scales)


SMALL = [
    # (T, d_in, d_out, r, lengths, ids, n_adapters)
    (64, 256, 512, 16, [32, 32], [0, 1], 1),
    (7, 128, 256, 16, [3, 4], [0, 1], 1),
    (300, 512, 264, 24, [0, 100, 1, 0, 199], [1, 0, 2, 2, 1], 2),
    (517, 384, 1000, 128, [10, 5, 10, 3, 200, 289], [1, 0, 2, 2, 0, 3], 3),
    # decode-sized batches: X boxes as tall as the one token tile (16 .. 128 rows), deeper rings
    (1, 256, 384, 16, [1], [0], 1),
    (33, 384, 640, 16, [33], [1], 1),
    (48, 512, 1000, 32, [8] * 6, [0] * 6, 1),
    (100, 256, 256, 16, [30, 40, 30], [1, 0, 2], 2),
    (128, 256, 512, 16, [128], [0], 1),
    # the smallest legal shapes (d_in one 128-input group, d_out and rank 8)
    (3, 128, 8, 8, [3], [1], 1),
    (2, 128, 16, 8, [2], [0], 1),
]


@pytest.mark.parametrize("case", SMALL, ids=[f"T{c[0]}_{c[1]}x{c[2]}" for c in SMALL])
@pytest.mark.parametrize("cluster", [1, 2])
def test_w4_small_shapes_match_oracle(dev, case, cluster):
    from mixed_lora_projection_gb300 import _lib as L
    T, d_in, d_out, r, lens, ids, na = case
    off = [0] + np.cumsum(lens).tolist()
    w = Workload("w4", 11, T, d_in, d_out, r, tuple(off), tuple(ids), n_adapters=na,
                 scales=tuple(0.5 + 0.75 * k for k in range(na)))
    inp = make_inputs(w, dev)
    q, sc = make_w4_base(w, dev)
    with _ll(w) as ll:
        ll.set_option(L.OPT_CLUSTER, cluster if T > 128 else 1)
        y = ll.forward_w4(inp.x, off, ids, _kq(q), sc, inp.a, inp.b, inp.scales)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert rel_err(y, _oracle(inp, q, sc, off, ids)) <= TOL


def test_w4_dequantisation_is_exact_per_weight(dev):
    # X = I: row k of Y is bf16(column k of W) exactly (one product per output)
    d_in, d_out = 128, 256
    w = Workload("w4eye", 12, d_in, d_in, d_out, 16, (0, d_in), (0,))
    inp = make_inputs(w, dev)
    inp.x.zero_()
    inp.x.fill_diagonal_(1.0)
    q, sc = make_w4_base(w, dev)
    with _ll(w) as ll:
        y = ll.forward_w4(inp.x, [0, d_in], [0], _kq(q), sc, inp.a, inp.b, inp.scales)
    torch.cuda.synchronize()
    wd = w4_dequantize_fp64(q.cpu().numpy(), bf16_bits(sc))          # exact q * s
    want = torch.from_numpy(wd.T.copy()).to(torch.bfloat16)           # rounded once, RNE
    assert torch.equal(y.cpu(), want)
    widened = w4_weights_bf16_fp64(q.cpu().numpy(), bf16_bits(sc))    # the oracle's widening
    assert torch.equal(y.cpu().double(), torch.from_numpy(widened.T.copy()))


@pytest.mark.parametrize("name", ["mixed_decode", "mixed_near_ridge", "sweep_qkv_multi", "prefill_16k"])
def test_w4_full_size_sampled_rows(dev, name):
    w = WORKLOADS[name]
    inp = make_inputs(w, dev)
    q, sc = make_w4_base(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with _ll(w) as ll:
        y = ll.forward_w4(inp.x, off, ids, _kq(q), sc, inp.a, inp.b, inp.scales)
        torch.cuda.synchronize()
        assert ll.status() == 0
    rows = sample_rows(w.T, off, ids, n_random=128, seed=5)
    ref = _oracle(inp, q, sc, off, ids, rows)
    assert rel_err(y[torch.as_tensor(rows, device=dev)], ref) <= TOL


@pytest.mark.parametrize("name", ["mixed_decode", "mixed_near_ridge", "sweep_qkv_multi", "prefill_16k"])
def test_w4_gap_to_exact_dequantisation_within_the_widening_bound(dev, name, record_property):
    """The 4-bit base is widened to bf16 before it meets X (the W4A16 reading). Measured here:
    how far the GPU result sits from the result on the exact weights q * s (no widening), on the
    full-size workloads. Round to nearest even to bf16 (8 significant bits) moves each weight by
    at most half an ulp, 2^-8 of its magnitude, so the widened and exact products differ by at
    most 2^-8 (|X| |W|^T) per element; with the triangle inequality that bounds the GPU's gap to
    the exact result by its gap to the widened result plus that bound."""
    w = WORKLOADS[name]
    inp = make_inputs(w, dev)
    q, sc = make_w4_base(w, dev)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with _ll(w) as ll:
        y = ll.forward_w4(inp.x, off, ids, _kq(q), sc, inp.a, inp.b, inp.scales)
        torch.cuda.synchronize()
        assert ll.status() == 0
    rows = sample_rows(w.T, off, ids, n_random=64, seed=8)
    w_exact = w4_dequantize_fp64(q.cpu().numpy(), bf16_bits(sc))
    w_wide = w4_weights_bf16_fp64(q.cpu().numpy(), bf16_bits(sc))
    x = f64(inp.x[torch.as_tensor(rows, device=dev)])
    rid = row_adapter_ids(off, ids, w.T)[rows]
    a64, b64 = [f64(a) for a in inp.a], [f64(b) for b in inp.b]
    y_exact = lora_linear_rows_fp64(x, rid, w_exact, a64, b64, inp.scales)
    y_wide = lora_linear_rows_fp64(x, rid, w_wide, a64, b64, inp.scales)
    bound = 2.0 ** -8 * (np.abs(x) @ np.abs(w_exact).T)
    # the widening's own effect, in the oracle alone, stays inside its bound element by element
    assert np.all(np.abs(y_wide - y_exact) <= bound * (1 + 1e-9))
    yg = f64(y[torch.as_tensor(rows, device=dev)])
    ref_max = np.max(np.abs(y_exact))
    gap_wide = np.max(np.abs(yg - y_wide)) / np.max(np.abs(y_wide))
    gap_exact = np.max(np.abs(yg - y_exact)) / ref_max
    widening = np.max(np.abs(y_wide - y_exact)) / ref_max
    record_property("gap_to_widened", float(gap_wide))
    record_property("gap_to_exact", float(gap_exact))
    record_property("widening_alone", float(widening))
    print(f"\nw4 {name}: max|dY|/max|Y| to the widened-weight oracle {gap_wide:.3e}, to the exact-weight "
          f"oracle {gap_exact:.3e}; widening alone {widening:.3e}, its bound {np.max(bound) / ref_max:.3e}")
    assert gap_wide <= TOL
    assert gap_exact <= gap_wide * np.max(np.abs(y_wide)) / ref_max + np.max(bound) / ref_max


ROWS = [1, 16, 17, 48, 64, 80, 128]


@pytest.mark.parametrize("T", ROWS)
def test_w4_decode_batches_match_oracle(dev, T):
    # one token tile without adapter rows (two 128-feature tiles per unit, X boxes of the
    # batch's rows); d_out not a multiple of 256
    lens = [T // 2, T - T // 2] if T > 1 else [1]
    off = [0] + np.cumsum(lens).tolist()
    w = Workload("w4dec", 15, T, 640, 1000, 32, tuple(off), tuple([0] * len(lens)))
    inp = make_inputs(w, dev)
    q, sc = make_w4_base(w, dev)
    with _ll(w) as ll:
        y = ll.forward_w4(inp.x, off, [0] * len(lens), _kq(q), sc, inp.a, inp.b, inp.scales)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert rel_err(y, _oracle(inp, q, sc, off, [0] * len(lens))) <= TOL


def test_w4_decode_rows_equal_the_same_rows_in_a_larger_batch(dev):
    # 48 base rows alone (two feature tiles per unit, 48-row X boxes) and as the first rows of
    # a 300-row batch with adapter rows (one feature tile, two token tiles per unit): every
    # output summed in the same K order, the same bits
    lens, ids = [8] * 6 + [252], [0] * 6 + [1]
    off = [0] + np.cumsum(lens).tolist()
    w = Workload("w4inv", 16, off[-1], 1024, 1536, 64, tuple(off), tuple(ids), scales=(0.5,))
    inp = make_inputs(w, dev)
    q, sc = make_w4_base(w, dev)
    kq = _kq(q)
    with _ll(w) as ll:
        full = ll.forward_w4(inp.x, off, ids, kq, sc, inp.a, inp.b, inp.scales).clone()
        alone = ll.forward_w4(inp.x[:48], off[:7], ids[:6], kq, sc, inp.a, inp.b, inp.scales)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert torch.equal(full[:48], alone)


@pytest.mark.parametrize("name", ["mixed_batch", "mixed_8x300"])
def test_w4_unit_orders_are_exact(dev, name):
    # token groups fastest (the default for these: packed gate_up 89 MB, X under 64 MB) and
    # feature tiles fastest run the same sums: the same bits
    from mixed_lora_projection_gb300 import _lib as L
    w = WORKLOADS[name]
    inp = make_inputs(w, dev)
    q, sc = make_w4_base(w, dev)
    kq = _kq(q)
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    with _ll(w) as ll:
        ys = []
        for raster in (1, 2, 0):
            ll.set_option(L.OPT_RASTER, raster)
            ys.append(ll.forward_w4(inp.x, off, ids, kq, sc, inp.a, inp.b, inp.scales).clone())
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert torch.equal(ys[0], ys[1]) and torch.equal(ys[0], ys[2])
    rows = sample_rows(w.T, off, ids, n_random=64, seed=6)
    assert rel_err(ys[0][torch.as_tensor(rows, device=dev)], _oracle(inp, q, sc, off, ids, rows)) <= TOL


@pytest.mark.parametrize("case", [("tiny2", [48, 200, 8], [0, 1, 0]), ("decode", [24, 24], [0, 0])])
def test_w4_bounded_waits_report_timeout_and_the_handle_recovers(dev, case):
    # the load warps never issue: every wait of the shrink launch and of the 4-bit kernel
    # (transposed tile with two token tiles, or two feature tiles for a decode batch) runs out
    # after 20 ms; the kernels return with the status word set, and the next call is correct
    from mixed_lora_projection_gb300 import _lib as L
    _, lens, ids = case
    off = [0] + np.cumsum(lens).tolist()
    w = Workload("w4stall", 17, off[-1], 512, 768, 32, tuple(off), tuple(ids), scales=(0.5,))
    inp = make_inputs(w, dev)
    q, sc = make_w4_base(w, dev)
    kq = _kq(q)
    with _ll(w) as ll:
        ll.set_option(L.OPT_WAIT_LIMIT_US, 20000)
        ll.set_option(L.OPT_DEBUG_STALL, 1)
        ll.forward_w4(inp.x, off, ids, kq, sc, inp.a, inp.b, inp.scales)
        torch.cuda.synchronize()
        assert ll.status(reset=True) == L.LORA_ETIMEOUT
        assert ll.status() == L.LORA_OK
        ll.set_option(L.OPT_DEBUG_STALL, 0)
        ll.set_option(L.OPT_WAIT_LIMIT_US, 4000000)
        y = ll.forward_w4(inp.x, off, ids, kq, sc, inp.a, inp.b, inp.scales)
        torch.cuda.synchronize()
        assert ll.status() == L.LORA_OK
    assert rel_err(y, _oracle(inp, q, sc, off, ids)) <= TOL


def test_w4_rejects_d_in_not_multiple_of_128(dev):
    from mixed_lora_projection_gb300 import LoraError
    w = Workload("w4bad", 13, 16, 192, 256, 16, (0, 16), (0,))
    inp = make_inputs(w, dev)
    q = torch.zeros((256, 96), dtype=torch.uint8, device=dev)
    sc = torch.ones((1, 256), dtype=torch.bfloat16, device=dev)
    with _ll(w) as ll:
        with pytest.raises(LoraError):
            ll.forward_w4(inp.x, [0, 16], [0], q, sc, inp.a, inp.b, inp.scales)


@pytest.mark.parametrize("name", ["tiny", "mixed_batch"])
def test_w4_host_buffers_match_device_path(dev, name):
    # row chunks from 2,048 rows; every row summed as in the device path: the same bits
    w = WORKLOADS[name]
    inp = make_inputs(w, dev)
    q, sc = make_w4_base(w, dev) if w.d_in % 128 == 0 else (None, None)
    x_host = inp.x.cpu().pin_memory()
    y_host = torch.empty((w.T, w.d_out), dtype=torch.bfloat16).pin_memory()
    kq = _kq(q)
    with _ll(w) as ll:
        y = ll.forward_w4(inp.x, w.seg_offsets, w.seg_ids, kq, sc, inp.a, inp.b, inp.scales)
        ll.forward_host_w4(x_host, w.seg_offsets, w.seg_ids, kq, sc, inp.a, inp.b, inp.scales, y_host)
    torch.cuda.synchronize()
    assert torch.equal(y.cpu(), y_host)


def test_w4_repack_layout_bit_exact(dev):
    w = WORKLOADS["sweep_o"]
    q, _ = make_w4_base(w, dev)
    got = _kq(q)
    torch.cuda.synchronize()
    assert np.array_equal(got.cpu().numpy(), _kernel_layout_np(q))
    # in place gives the same bytes
    q2 = q.clone()
    from mixed_lora_projection_gb300 import w4_repack
    w4_repack(q2, q2)
    torch.cuda.synchronize()
    assert torch.equal(q2, got)


def test_w4_repack_rejects_bad_arguments(dev):
    from mixed_lora_projection_gb300 import _lib as L
    lib = L.load()
    buf = torch.zeros(64, dtype=torch.uint8, device=dev)
    p = buf.data_ptr()
    assert lib.lora_linear_w4_repack(p, p, 6, None) == L.LORA_EINVAL        # not whole words
    assert lib.lora_linear_w4_repack(p + 1, p + 1, 8, None) == L.LORA_EINVAL  # misaligned
    assert lib.lora_linear_w4_repack(p, p + 4, 32, None) == L.LORA_EINVAL    # partial overlap
    assert lib.lora_linear_w4_repack(p, p, 0, None) == L.LORA_OK             # nothing to do


# --------------------------------------------------------------------------- K parts (4-bit base)

@pytest.mark.parametrize("parts", [1, 2, 3, 4])
@pytest.mark.parametrize("T", [17, 48, 128])
def test_w4_k_parts_match_oracle(dev, parts, T):
    # decode batches (one token tile, no adapter rows) with the base's K-steps in 1..4 parts
    # (2,048 inputs: 32 K-steps, parts of 8 or more); d_out 520 leaves a feature-tile tail
    from mixed_lora_projection_gb300 import _lib as L
    lens = [T // 2, T - T // 2] if T > 1 else [1]
    off = [0] + np.cumsum(lens).tolist()
    ids = [0] * len(lens)
    w = Workload("w4kp", 18, T, 2048, 520, 32, tuple(off), tuple(ids))
    inp = make_inputs(w, dev)
    q, sc = make_w4_base(w, dev)
    kq = _kq(q)
    with _ll(w) as ll:
        ll.set_option(L.OPT_W4_K_SPLIT, parts)
        y1 = ll.forward_w4(inp.x, off, ids, kq, sc, inp.a, inp.b, inp.scales).clone()
        y2 = ll.forward_w4(inp.x, off, ids, kq, sc, inp.a, inp.b, inp.scales)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert torch.equal(y1, y2)                      # the same sum whichever part finishes last
    assert rel_err(y1, _oracle(inp, q, sc, off, ids)) <= TOL


def test_w4_k_parts_rows_do_not_depend_on_the_batch(dev):
    # a decode-sized handle (at most 128 rows) of a narrow projection splits K by itself; the 48
    # base rows alone and as the first rows of a 100-row batch with adapter rows (an expand on the
    # last part) give the same bits, and the expand rows match the oracle
    from mixed_lora_projection_gb300 import launch_shape
    lens, ids = [8] * 6 + [52], [0] * 6 + [1]
    off = [0] + np.cumsum(lens).tolist()
    w = Workload("w4kpinv", 19, 128, 6144, 1024, 64, tuple(off), tuple(ids), scales=(0.75,))
    inp = make_inputs(w, dev, x_rows=100)
    q, sc = make_w4_base(w, dev)
    kq = _kq(q)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    s = launch_shape(6144, 1024, 64, sms, 100, off, ids, w4=True)
    assert s["fused_units"] == 8 * 4           # 8 one-tile units, K in 4 parts
    with _ll(w) as ll:
        full = ll.forward_w4(inp.x, off, ids, kq, sc, inp.a, inp.b, inp.scales).clone()
        alone = ll.forward_w4(inp.x[:48], off[:7], ids[:6], kq, sc, inp.a, inp.b, inp.scales)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert torch.equal(full[:48], alone)
    assert rel_err(full, _oracle(inp, q, sc, off, ids)) <= TOL


@pytest.mark.parametrize("name", ["decode_o", "decode_down"])
def test_w4_k_parts_full_size_decode(dev, name):
    # the 48-row decode batch of the o and down projections at full size: 40 one-tile units, K
    # in 3 parts (120 units), sampled rows against the oracle
    from mixed_lora_projection_gb300 import launch_shape
    w = WORKLOADS[name]
    off, ids = list(w.seg_offsets), list(w.seg_ids)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    assert launch_shape(w.d_in, w.d_out, w.rank, sms, w.T, off, ids, w4=True)["fused_units"] == 40 * 3
    inp = make_inputs(w, dev)
    q, sc = make_w4_base(w, dev)
    with _ll(w) as ll:
        y = ll.forward_w4(inp.x, off, ids, _kq(q), sc, inp.a, inp.b, inp.scales)
        torch.cuda.synchronize()
        assert ll.status() == 0
    rows = sample_rows(w.T, off, ids, n_random=16, seed=8)
    assert rel_err(y[torch.as_tensor(rows, device=dev)], _oracle(inp, q, sc, off, ids, rows)) <= TOL


def test_w4_k_parts_graph_replays_and_timeout(dev):
    # K parts across CUDA-graph replays (the block counters only grow, so replays need no reset);
    # then every wait running out (20 ms) reports LORA_ETIMEOUT, the status reset also resets the
    # counters, and the next call is correct
    from mixed_lora_projection_gb300 import LoraLinear, _lib as L
    T = 48
    off, ids = [0, 24, 48], [0, 0]
    w = Workload("w4kpg", 20, T, 2048, 768, 16, tuple(off), tuple(ids))
    inp = make_inputs(w, dev)
    q, sc = make_w4_base(w, dev)
    kq = _kq(q)
    with LoraLinear(2048, 768, 16, T, 4, 0) as ll:
        ll.set_option(L.OPT_W4_K_SPLIT, 3)
        ref = ll.forward_w4(inp.x, off, ids, kq, sc, inp.a, inp.b, inp.scales).clone()
        y = torch.zeros_like(ref)
        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(s):
            ll.forward_w4(inp.x, off, ids, kq, sc, inp.a, inp.b, inp.scales, y=y)
        torch.cuda.current_stream(dev).wait_stream(s)
        torch.cuda.synchronize()
        y.zero_()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            ll.forward_w4(inp.x, off, ids, kq, sc, inp.a, inp.b, inp.scales, y=y)
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        assert ll.status() == 0
        assert torch.equal(y, ref)
        ll.set_option(L.OPT_WAIT_LIMIT_US, 20000)
        ll.set_option(L.OPT_DEBUG_STALL, 1)
        ll.forward_w4(inp.x, off, ids, kq, sc, inp.a, inp.b, inp.scales)
        torch.cuda.synchronize()
        assert ll.status(reset=True) == L.LORA_ETIMEOUT
        ll.set_option(L.OPT_DEBUG_STALL, 0)
        ll.set_option(L.OPT_WAIT_LIMIT_US, 4000000)
        y2 = ll.forward_w4(inp.x, off, ids, kq, sc, inp.a, inp.b, inp.scales)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert torch.equal(y2, ref)
    assert rel_err(ref, _oracle(inp, q, sc, off, ids)) <= TOL


def test_w4_k_parts_with_several_token_groups(dev):
    # a decode-sized batch on three adapters and base rows: four planner tiles in two token groups,
    # each block's K in 2 parts with the expand on the last; against the oracle, and repeated calls
    # give the same bits
    from mixed_lora_projection_gb300 import _lib as L
    lens, ids = [20, 30, 10, 40, 20], [1, 2, 0, 3, 1]
    off = [0] + np.cumsum(lens).tolist()
    w = Workload("w4kpg2", 21, off[-1], 2048, 640, 32, tuple(off), tuple(ids), n_adapters=3,
                 scales=(0.5, -1.0, 1.5))
    inp = make_inputs(w, dev)
    q, sc = make_w4_base(w, dev)
    kq = _kq(q)
    with _ll(w) as ll:
        ll.set_option(L.OPT_W4_K_SPLIT, 2)
        y1 = ll.forward_w4(inp.x, off, ids, kq, sc, inp.a, inp.b, inp.scales).clone()
        y2 = ll.forward_w4(inp.x, off, ids, kq, sc, inp.a, inp.b, inp.scales)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert torch.equal(y1, y2)
    assert rel_err(y1, _oracle(inp, q, sc, off, ids)) <= TOL


@pytest.mark.parametrize("case", [([128, 128, 92], [1, 1, 1]), ([50, 78, 128, 60], [0, 1, 2, 3]),
                                  ([128, 100, 28, 40], [0, 2, 2, 0])])
def test_w4_three_token_tiles_in_one_group(dev, case):
    # a batch of three tiles whose last has at most 96 rows runs as one token group (the third
    # tile's rows the B operand of a second MMA, its expand the group's third): against the oracle,
    # and its first 128 rows bitwise equal to the same rows in a batch of their own
    from mixed_lora_projection_gb300 import launch_shape
    lens, ids = case
    off = [0] + np.cumsum(lens).tolist()
    T = off[-1]
    w = Workload("w4t3", 22, T, 1024, 768, 32, tuple(off), tuple(ids), n_adapters=3, scales=(0.5, -1.0, 1.5))
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    assert launch_shape(1024, 768, 32, sms, T, off, ids, w4=True)["fused_units"] == 768 // 128
    inp = make_inputs(w, dev)
    q, sc = make_w4_base(w, dev)
    kq = _kq(q)
    with _ll(w) as ll:
        y = ll.forward_w4(inp.x, off, ids, kq, sc, inp.a, inp.b, inp.scales).clone()
        off1 = [o for o in off if o <= 128] + ([] if 128 in off else [128])   # the first 128 rows
        ids1 = ids[:len(off1) - 1]
        y1 = ll.forward_w4(inp.x[:128], off1, ids1, kq, sc, inp.a, inp.b, inp.scales)
        torch.cuda.synchronize()
        assert ll.status() == 0
    assert rel_err(y, _oracle(inp, q, sc, off, ids)) <= TOL
    assert torch.equal(y[:128], y1)

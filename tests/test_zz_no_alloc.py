"""The allocation-free entry point, lora_linear_forward_noalloc.

It serves callers that cannot call cudaMalloc: a serving engine whose device pools were
reserved at start-up (a raw allocation would fail or fragment them), latency-critical
code where cudaMalloc's device-wide synchronisation would stall other streams, and
plugins whose host forbids allocations after start-up. Its scratch is a fixed array in
the library. Its output must match the fp64 oracle within the tolerance the other GPU tests
use, and, because a row's output does not depend on the launch shape, it must equal the
handle-based entry point bit for bit, call after call. This file is named so that pytest
collects it last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from oracle import max_rel_err
from mixed_lora_projection_gb300.synth import WORKLOADS, Workload, make_inputs

from gpu_util import TOL, f64, oracle_full, oracle_rows, sample_rows

pytestmark = pytest.mark.gpu

MAX_TOKENS, MAX_SEGMENTS = 4096, 64   # LORA_NOALLOC_MAX_TOKENS, LORA_NOALLOC_MAX_SEGMENTS


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from mixed_lora_projection_gb300 import build
    build.ensure_built()
    from mixed_lora_projection_gb300 import _lib
    return _lib.load()


def _noalloc(lib, inp, off, ids, d_in, d_out, rank, y, T=None, stream=None):
    T = inp.x.shape[0] if T is None else T
    o = (C.c_int32 * len(off))(*off)
    i = (C.c_int32 * max(1, len(ids)))(*ids)
    na = len(inp.a)
    A = (C.c_void_p * na)(*[a.data_ptr() for a in inp.a])
    B = (C.c_void_p * na)(*[b.data_ptr() for b in inp.b])
    S = (C.c_float * na)(*inp.scales)
    s = (stream or torch.cuda.current_stream()).cuda_stream
    return lib.lora_linear_forward_noalloc(inp.x.data_ptr(), T, o, i, len(ids), d_in, d_out, rank,
                                           inp.w.data_ptr(), A, B, S, na, y.data_ptr(), C.c_void_p(s))


def _limit_workload():
    """T = 4096 rows (the limit) in 64 segments (the limit) on three adapters with different
    scales, every segment length off the 128-row tile grid, two empty segments, rank 256."""
    rng = np.random.default_rng(77)
    cuts = np.sort(rng.choice(np.arange(1, MAX_TOKENS), MAX_SEGMENTS - 3, replace=False))
    lengths = np.diff(np.concatenate([[0], cuts, [MAX_TOKENS]])).tolist()
    lengths[5:5] = [0]
    lengths[40:40] = [0]
    ids = [int(v) for v in rng.integers(0, 4, MAX_SEGMENTS)]
    off = [0]
    for n in lengths:
        off.append(off[-1] + n)
    assert len(ids) == MAX_SEGMENTS and off[-1] == MAX_TOKENS and set(ids) == {0, 1, 2, 3}
    return Workload("noalloc_limit", 9, MAX_TOKENS, 1024, 1536, 256, tuple(off), tuple(ids),
                    n_adapters=3, scales=(1.0, 0.5, -2.0))


def _handle_forward(w, inp):
    from mixed_lora_projection_gb300 import LoraLinear, _lib as L
    with LoraLinear(w.d_in, w.d_out, w.rank, w.T, len(w.seg_ids), 0) as ll:
        ll.set_option(L.OPT_K_SPLIT, 1)   # whole K per block, as the allocation-free entry point sums
        y = ll.forward(inp.x, w.seg_offsets, w.seg_ids, inp.w, inp.a, inp.b, inp.scales)
        torch.cuda.synchronize()
        assert ll.status() == 0
    return y


@pytest.mark.parametrize("name", ["tiny", "sweep_qkv_multi", "mixed_decode", "noalloc_limit"])
def test_noalloc_matches_oracle_and_handle_entry_point_two_calls_in_a_row(lib, name):
    dev = torch.device("cuda", 0)
    w = _limit_workload() if name == "noalloc_limit" else WORKLOADS[name]
    inp = make_inputs(w, dev)
    y_ref = _handle_forward(w, inp)
    if w.T <= 64:
        ref, rows = oracle_full(inp, list(w.seg_offsets), list(w.seg_ids)), np.arange(w.T)
    else:
        rows = sample_rows(w.T, list(w.seg_offsets), list(w.seg_ids), n_random=128, seed=3)
        ref = oracle_rows(inp, list(w.seg_offsets), list(w.seg_ids), rows)
    for _ in range(2):
        y = torch.full((w.T, w.d_out), float("nan"), dtype=torch.bfloat16, device=dev)
        assert _noalloc(lib, inp, w.seg_offsets, w.seg_ids, w.d_in, w.d_out, w.rank, y) == 0
        torch.cuda.synchronize()
        yr = f64(y)
        assert max_rel_err(yr[rows], ref) <= TOL
        # the same kernels with the same summation order: bit-identical to the handle's output
        assert np.array_equal(yr, f64(y_ref))


def test_noalloc_allocates_nothing(lib):
    """After the first call (which looks up the scratch array on the device), ten calls leave
    the device's free memory exactly where it was."""
    dev = torch.device("cuda", 0)
    w = _limit_workload()   # a work list too large for the kernel parameters: the copied form
    inp = make_inputs(w, dev)
    y = torch.empty((w.T, w.d_out), dtype=torch.bfloat16, device=dev)
    assert _noalloc(lib, inp, w.seg_offsets, w.seg_ids, w.d_in, w.d_out, w.rank, y) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(dev)
    tiny = WORKLOADS["tiny"]   # and one whose work list travels in the kernel parameters
    tin = make_inputs(tiny, dev)
    ty = torch.empty((tiny.T, tiny.d_out), dtype=torch.bfloat16, device=dev)
    for _ in range(5):
        assert _noalloc(lib, inp, w.seg_offsets, w.seg_ids, w.d_in, w.d_out, w.rank, y) == 0
        assert _noalloc(lib, tin, tiny.seg_offsets, tiny.seg_ids, tiny.d_in, tiny.d_out, tiny.rank, ty) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(dev)
    assert free1 == free0


def test_noalloc_rejects_sizes_beyond_its_limits(lib):
    dev = torch.device("cuda", 0)
    tiny = WORKLOADS["tiny"]
    # 4097 rows in one consistent segment: beyond LORA_NOALLOC_MAX_TOKENS
    w = Workload("over_rows", 0, MAX_TOKENS + 1, tiny.d_in, tiny.d_out, tiny.rank, (0, MAX_TOKENS + 1), (1,),
                 b_var=1.0 / 16)
    inp = make_inputs(w, dev)
    y = torch.zeros((w.T, w.d_out), dtype=torch.bfloat16, device=dev)
    assert _noalloc(lib, inp, w.seg_offsets, w.seg_ids, w.d_in, w.d_out, w.rank, y) == -1
    # 65 one-row segments: beyond LORA_NOALLOC_MAX_SEGMENTS
    off = tuple(range(MAX_SEGMENTS + 2))
    w65 = Workload("over_segs", 0, MAX_SEGMENTS + 1, tiny.d_in, tiny.d_out, tiny.rank, off,
                   (0, 1) * (MAX_SEGMENTS // 2) + (0,), b_var=1.0 / 16)
    inp65 = make_inputs(w65, dev)
    y65 = torch.zeros((w65.T, w65.d_out), dtype=torch.bfloat16, device=dev)
    assert _noalloc(lib, inp65, w65.seg_offsets, w65.seg_ids, w65.d_in, w65.d_out, w65.rank, y65) == -1
    # rank above 256
    ti = make_inputs(tiny, dev)
    ty = torch.zeros((tiny.T, tiny.d_out), dtype=torch.bfloat16, device=dev)
    assert _noalloc(lib, ti, tiny.seg_offsets, tiny.seg_ids, tiny.d_in, tiny.d_out, 264, ty) == -1
    torch.cuda.synchronize()
    assert bool((y == 0).all()) and bool((y65 == 0).all()) and bool((ty == 0).all())
    # exactly at the segment limit, with the same rows: accepted
    off64 = tuple(range(MAX_SEGMENTS)) + (MAX_SEGMENTS + 1,)
    ids64 = (0, 1) * (MAX_SEGMENTS // 2)
    assert _noalloc(lib, inp65, off64, ids64, w65.d_in, w65.d_out, w65.rank, y65) == 0
    torch.cuda.synchronize()
    assert bool(torch.isfinite(y65.float()).all())


def test_noalloc_enqueues_nothing_while_capturing(lib):
    dev = torch.device("cuda", 0)
    w = WORKLOADS["tiny"]
    inp = make_inputs(w, dev)
    y = torch.zeros((w.T, w.d_out), dtype=torch.bfloat16, device=dev)
    assert _noalloc(lib, inp, w.seg_offsets, w.seg_ids, w.d_in, w.d_out, w.rank, y) == 0   # set-up first
    torch.cuda.synchronize()
    y.zero_()
    torch.cuda.synchronize()
    marker = torch.zeros(16, device=dev)
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(dev)
    with torch.cuda.graph(g, stream=side):
        marker.fill_(1.0)   # the graph records this, and nothing of the refused call
        rc = _noalloc(lib, inp, w.seg_offsets, w.seg_ids, w.d_in, w.d_out, w.rank, y,
                      stream=torch.cuda.current_stream())
    assert rc == -5   # LORA_EUNSUPPORTED
    g.replay()
    torch.cuda.synchronize()
    assert bool((marker == 1).all()) and bool((y == 0).all())

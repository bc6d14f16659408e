"""The allocation-free entry point, lora_linear_forward_noalloc.

It serves callers that cannot call cudaMalloc: a serving engine whose device pools were
reserved at start-up (a raw allocation would fail or fragment them), latency-critical
code where cudaMalloc's device-wide synchronisation would stall other streams, and
plugins whose host forbids allocations after start-up. Its scratch is a fixed array in
the library, so its output must equal what the handle-based entry point computes, call
after call. This file is named so that pytest collects it last.
"""
import ctypes as C

import pytest
import torch

from oracle import max_rel_err
from mixed_lora_projection_gb300.synth import WORKLOADS, make_inputs

from gpu_util import TOL, f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from mixed_lora_projection_gb300 import build
    build.ensure_built()
    from mixed_lora_projection_gb300 import _lib
    return _lib.load()


def _noalloc(lib, w, inp, y, T=None):
    T = w.T if T is None else T
    off = (C.c_int32 * len(w.seg_offsets))(*w.seg_offsets)
    ids = (C.c_int32 * len(w.seg_ids))(*w.seg_ids)
    na = len(inp.a)
    A = (C.c_void_p * na)(*[a.data_ptr() for a in inp.a])
    B = (C.c_void_p * na)(*[b.data_ptr() for b in inp.b])
    S = (C.c_float * na)(*inp.scales)
    stream = torch.cuda.current_stream().cuda_stream
    return lib.lora_linear_forward_noalloc(inp.x.data_ptr(), T, off, ids, len(w.seg_ids), w.d_in, w.d_out,
                                           w.rank, inp.w.data_ptr(), A, B, S, na, y.data_ptr(),
                                           C.c_void_p(stream))


@pytest.mark.parametrize("name", ["tiny", "sweep_qkv_multi", "mixed_decode"])
def test_noalloc_matches_handle_entry_point_two_calls_in_a_row(lib, name):
    from mixed_lora_projection_gb300 import LoraLinear
    dev = torch.device("cuda", 0)
    w = WORKLOADS[name]
    inp = make_inputs(w, dev)
    with LoraLinear(w.d_in, w.d_out, w.rank, w.T, 64, 0) as ll:
        y_ref = ll.forward(inp.x, w.seg_offsets, w.seg_ids, inp.w, inp.a, inp.b, inp.scales)
        torch.cuda.synchronize()
    for _ in range(2):
        y = torch.full((w.T, w.d_out), float("nan"), dtype=torch.bfloat16, device=dev)
        assert _noalloc(lib, w, inp, y) == 0
        torch.cuda.synchronize()
        assert max_rel_err(f64(y), f64(y_ref)) <= TOL


def test_noalloc_rejects_sizes_beyond_its_limit(lib):
    dev = torch.device("cuda", 0)
    w = WORKLOADS["tiny"]
    inp = make_inputs(w, dev)
    y = torch.zeros((w.T, w.d_out), dtype=torch.bfloat16, device=dev)
    # more rows than LORA_NOALLOC_MAX_TOKENS (4096): rejected before any launch
    assert _noalloc(lib, w, inp, y, T=4097) == -1
    torch.cuda.synchronize()
    assert bool((y == 0).all())

"""Helpers shared by the GPU tests: running the library on seeded inputs and checking
rows against the fp64 oracle."""
from __future__ import annotations

import numpy as np
import torch

from oracle import (bf16_bits_to_f64, lora_linear_fp64, lora_linear_rows_fp64, max_rel_err,
                    plan_ref, row_adapter_ids)
from mixed_lora_projection_gb300.synth import bf16_bits

TOL = 5e-3  # max|Y_gpu - Y_ref| / max|Y_ref| per tensor (bf16 output, fp32 accumulation)


def f64(t: torch.Tensor) -> np.ndarray:
    return bf16_bits_to_f64(bf16_bits(t))


def run(ll, inp, off, ids, y=None):
    return ll.forward(inp.x, off, ids, inp.w, inp.a, inp.b, inp.scales, y=y)


def oracle_full(inp, off, ids):
    return lora_linear_fp64(f64(inp.x), off, ids, f64(inp.w), [f64(a) for a in inp.a],
                            [f64(b) for b in inp.b], inp.scales)


def sample_rows(T, off, ids, n_random=256, seed=0):
    """Rows [0,64), every segment boundary +-2, every planner tile boundary +-1, and
    n_random seeded random rows (rows are independent, so any subset is checkable)."""
    rows = set(range(min(T, 64)))
    for b in off:
        rows.update(range(b - 2, b + 3))
    fused, _ = plan_ref(off, ids, T)
    for (r0, n, _) in fused:
        rows.update((r0 - 1, r0, r0 + 1, r0 + n - 1, r0 + n))
    rng = np.random.default_rng(seed)
    rows.update(rng.integers(0, T, min(n_random, T)).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < T), dtype=np.int64)


def oracle_rows(inp, off, ids, rows, w64=None, a64=None, b64=None):
    T = inp.x.shape[0]
    rid = row_adapter_ids(off, ids, T)[rows]
    x_rows = f64(inp.x[torch.as_tensor(rows, device=inp.x.device)])
    w64 = f64(inp.w) if w64 is None else w64
    a64 = [f64(a) for a in inp.a] if a64 is None else a64
    b64 = [f64(b) for b in inp.b] if b64 is None else b64
    return lora_linear_rows_fp64(x_rows, rid, w64, a64, b64, inp.scales)


def rel_err(y_gpu_rows: torch.Tensor, y_ref: np.ndarray) -> float:
    return max_rel_err(f64(y_gpu_rows), y_ref)

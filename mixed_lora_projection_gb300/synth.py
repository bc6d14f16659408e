"""Seeded synthetic inputs for the shared-base, per-request LoRA projection.

This module only draws random tensors and describes batch layouts; it holds none of the
projection's arithmetic. Tests and the benchmark pass the same tensors to the CUDA path
and to the fp64 oracle, so both sides always see identical bf16 bit patterns.

Workloads stand in for the shapes the source pages run ("Two 27B models on a single
RTX 5090": hidden size 5,120, a rank-256 adapter on the last 24 of 64 layers, decision
prefills of 16k-32k tokens, six chats running at once beside decisions; "Qwen3.8-27B on
one RTX 3090 with patched vLLM + DFlash2": a seven-token draft block verified in one pass,
so eight rows per chat per step). Values are Gaussian:

    X ~ N(0, 1),  W ~ N(0, 1/d_in),  A ~ N(0, 1/d_in),  B ~ N(0, 1/r)

(the second parameter is the variance), drawn in fp32 and rounded to bf16 (round to
nearest even). With these scales the base product and the adapter's delta are each of
order one per output element, so the delta is not lost in the check.

Seeds: 1000 * workload_index + 10 * layer + tensor_index, with tensor_index 0 for X,
1 for W, 2k for A_k and 2k+1 for B_k. The same seed on a different device generator gives
different numbers; every check feeds both sides from one generated copy.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    """One batch layout: sizes, request segments and initialisation scales."""
    name: str
    index: int                      # seed group
    T: int
    d_in: int
    d_out: int
    rank: int
    seg_offsets: tuple
    seg_ids: tuple
    n_adapters: int = 1
    scales: tuple = (1.0,)
    b_var: float | None = None      # variance of B (default 1/rank)
    note: str = ""

    @property
    def adapter_rows(self) -> int:
        return sum(self.seg_offsets[i + 1] - self.seg_offsets[i]
                   for i, a in enumerate(self.seg_ids) if a != 0)

    def useful_flops(self) -> float:
        """2 T d_in d_out for the base plus 2 T_a r (d_in + d_out) for the adapter rows."""
        Ta = self.adapter_rows
        return 2.0 * self.T * self.d_in * self.d_out + 2.0 * Ta * self.rank * (self.d_in + self.d_out)

    def algorithmic_bytes(self) -> float:
        """bf16 bytes of X, W, Y and every adapter named in the batch (read or written once)."""
        used = set(a for a in self.seg_ids if a != 0)
        ab = len(used) * self.rank * (self.d_in + self.d_out)
        return 2.0 * (self.T * self.d_in + self.d_out * self.d_in + self.T * self.d_out + ab)


def _segs(lengths, ids):
    off = [0]
    for n in lengths:
        off.append(off[-1] + n)
    return tuple(off), tuple(ids)


_TINY = Workload("tiny", 0, 64, 256, 512, 16, (0, 32, 64), (0, 1), b_var=1.0 / 16,
                 note="2 segments: rows 0-31 no adapter, rows 32-63 adapter 1")
_PREFILL_16K = Workload("prefill_16k", 1, 16384, 5120, 5120, 256, (0, 16384), (1,),
                        note="one 16k-token decision prefill on adapter 1, 5120->5120")
_mix_off, _mix_ids = _segs([8] * 6 + [4096], [0] * 6 + [1])
_MIXED = Workload("mixed_batch", 2, 4144, 5120, 34816, 256, _mix_off, _mix_ids,
                  note="6 chats x 8 decode/draft rows (no adapter) + 4096-row prefill chunk on adapter 1, gate_up 5120->34816")
_dec_off, _dec_ids = _segs([8] * 6, [0] * 6)
_MIXED_DECODE = Workload("mixed_decode", 2, 48, 5120, 34816, 256, _dec_off, _dec_ids,
                         note="the 48 decode rows of the mixed batch alone (6 chats x 8 rows), gate_up 5120->34816")
_PREFILL_32K = Workload("prefill_32k", 3, 32768, 17408, 5120, 256, (0, 32768), (1,),
                        note="one 32k-token decision prefill on adapter 1, down 17408->5120")
_ridge_off, _ridge_ids = _segs([8] * 6 + [300], [0] * 6 + [1])
_NEAR_RIDGE = Workload("mixed_near_ridge", 5, 348, 5120, 34816, 256, _ridge_off, _ridge_ids,
                       note="48 decode rows + one 300-token decision on adapter 1, gate_up 5120->34816")

_c8_off, _c8_ids = _segs([8] * 6 + [300] * 8, [0] * 6 + [1] * 8)
_CONCURRENT_8 = Workload("mixed_8x300", 6, 2448, 5120, 34816, 256, _c8_off, _c8_ids,
                         note="48 decode rows + eight concurrent 300-token decisions on adapter 1, gate_up 5120->34816")
_tail_off, _tail_ids = _segs([8] * 6 + [1552], [0] * 6 + [1])
_PREFIX_TAIL = Workload("prefix_tail_1552", 7, 1600, 5120, 34816, 256, _tail_off, _tail_ids,
                        note="48 decode rows + a 1,552-row decision tail after a reused prefix on adapter 1, gate_up")

# 2048-row batch of the 24-layer sweep: base 300, A 400, base 362, A 333, base 362, A 291.
SWEEP_LENGTHS = (300, 400, 362, 333, 362, 291)
SWEEP_IDS = (0, 1, 0, 1, 0, 1)
SWEEP_PROJECTIONS = (("qkv", 5120, 12288), ("o", 6144, 5120),
                     ("gate_up", 5120, 34816), ("down", 17408, 5120))
SWEEP_LAYERS = 24


def sweep_workload(proj: str, multi_adapter: bool = False) -> Workload:
    d_in, d_out = {p: (i, o) for p, i, o in SWEEP_PROJECTIONS}[proj]
    ids = (0, 1, 0, 2, 0, 3) if multi_adapter else SWEEP_IDS
    off, ids = _segs(SWEEP_LENGTHS, ids)
    n_ad = 3 if multi_adapter else 1
    return Workload(f"sweep_{proj}" + ("_multi" if multi_adapter else ""), 4, 2048, d_in, d_out, 256,
                    off, ids, n_adapters=n_ad, scales=(1.0,) * n_ad,
                    note="2048-token batch, half adapter rows in 3 segments, half base rows")


def decode_workload(proj: str) -> Workload:
    """One decode step of six chats (8 rows each: a seven-token draft block and one token, no
    adapter) through one projection of the adapted stack."""
    d_in, d_out = {p: (i, o) for p, i, o in SWEEP_PROJECTIONS}[proj]
    off, ids = _segs([8] * 6, [0] * 6)
    return Workload(f"decode_{proj}", 8, 48, d_in, d_out, 256, off, ids,
                    note="6 chats x 8 decode/draft rows (no adapter) through one projection")


WORKLOADS = {w.name: w for w in (_TINY, _PREFILL_16K, _MIXED, _MIXED_DECODE, _PREFILL_32K, _NEAR_RIDGE,
                                  _CONCURRENT_8, _PREFIX_TAIL)}
for _p, _, _ in SWEEP_PROJECTIONS:
    WORKLOADS[f"sweep_{_p}"] = sweep_workload(_p)
    WORKLOADS[f"sweep_{_p}_multi"] = sweep_workload(_p, True)
    WORKLOADS[f"decode_{_p}"] = decode_workload(_p)


def seed_for(w: Workload, tensor_index: int, layer: int = 0, proj_index: int = 0) -> int:
    return 1000 * w.index + 10 * (4 * layer + proj_index) + tensor_index


def _gauss_bf16(shape, var, seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    return (t * math.sqrt(var)).to(torch.bfloat16)


@dataclass
class Inputs:
    x: torch.Tensor                  # [T, d_in] bf16
    w: torch.Tensor                  # [d_out, d_in] bf16
    a: list = field(default_factory=list)   # [r, d_in] bf16 per adapter
    b: list = field(default_factory=list)   # [d_out, r] bf16 per adapter
    scales: tuple = ()


def make_inputs(w: Workload, device="cpu", layer: int = 0, proj_index: int = 0,
                x_rows: int | None = None, with_x: bool = True) -> Inputs:
    """Seeded bf16 tensors for workload ``w`` on ``device``."""
    T = w.T if x_rows is None else x_rows
    b_var = w.b_var if w.b_var is not None else 1.0 / w.rank
    s = lambda k: seed_for(w, k, layer, proj_index)  # noqa: E731
    x = _gauss_bf16((T, w.d_in), 1.0, s(0), device) if with_x else None
    W = _gauss_bf16((w.d_out, w.d_in), 1.0 / w.d_in, s(1), device)
    A = [_gauss_bf16((w.rank, w.d_in), 1.0 / w.d_in, s(2 * k), device) for k in range(1, w.n_adapters + 1)]
    B = [_gauss_bf16((w.d_out, w.rank), b_var, s(2 * k + 1), device) for k in range(1, w.n_adapters + 1)]
    return Inputs(x=x, w=W, a=A, b=B, scales=tuple(w.scales))


def make_w4_base(w: Workload, device="cpu", layer: int = 0, proj_index: int = 0):
    """A seeded 4-bit base for workload ``w``: (qweight uint8 [d_out, d_in/2], scales bf16
    [d_in/128, d_out]). Nibbles are uniform over [-8, 7] (variance 21.25); scales are
    uniform in [0.5, 1.5] x 1/sqrt(21.25 d_in), so W = q s has variance ~1/d_in like the bf16
    base. Seed: the W seed of the workload + 500000."""
    g = torch.Generator(device=device)
    g.manual_seed(int(seed_for(w, 1, layer, proj_index)) + 500000)
    q = torch.randint(0, 256, (w.d_out, w.d_in // 2), generator=g, device=device, dtype=torch.int32).to(torch.uint8)
    s0 = 1.0 / math.sqrt(21.25 * w.d_in)
    s = (torch.rand((w.d_in // 128, w.d_out), generator=g, device=device) + 0.5) * s0
    return q, s.to(torch.bfloat16)


def bf16_bits(t: torch.Tensor):
    """uint16 numpy view of a bf16 tensor's bit patterns (copied to the host)."""
    import numpy as np
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)

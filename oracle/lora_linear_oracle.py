"""fp64 CPU oracle for the shared-base, per-request LoRA projection.

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference arm of ``bench.py`` may import this module. The product path (the C-ABI library
and its Python binding) never imports, links or calls it, and this module imports nothing
from the product package.

What it computes (plain definitions, written out; no blocking, fusion or reordering):

* ``lora_linear_fp64`` -- for every token row t whose request segment names adapter a,
      Y[t,:] = X[t,:] W^T + s_a (X[t,:] A_a^T) B_a^T
  and for every row whose segment names no adapter (id 0), Y[t,:] = X[t,:] W^T.
  Source: "Two 27B models on a single RTX 5090", section 4 (Running Clef inside vLLM):
  a request that names the adapter runs, beside each changed matrix, the adapter's two
  thin matrices and adds their output; every other request in the same batch is served
  from the base weights alone. Section 3 fixes the shapes: W' = W + B.A in each changed
  matrix, so B is [d_out x r] and A is [r x d_in].
* ``lora_linear_merged_fp64`` -- the same rows through the merged weight W + s_a B_a A_a
  (section 3 of the same page: the adapter plus the base equals the fine-tuned matrix).
  Used as an independent pin of the factored path.
* ``plan_ref`` -- the token-segment planner: which 128-row tiles the fused base+expand
  pass and the shrink pass run over. Pure integer logic, row by row.

Arithmetic: every input arrives as the exact bf16 values (``bf16_bits_to_f64``), and all
products and sums are fp64 (numpy float64 matmul) with no intermediate rounding. The
GPU path rounds the shrink output U and the output Y to bf16; the oracle does not. The one
rounding the oracle does take is part of the method: a 4-bit base (W4A16) is widened to the
16-bit activation type, so ``w4_weights_bf16_fp64`` rounds each q * s to bf16 once.

Pins (tests/test_oracle.py, run with ``-m "not gpu"``): brute-force triple loops on tiny
shapes, the merged-weight identity, routing (id-0 rows equal the base product), B = 0 is a
no-op, the delta has rank <= r, closed forms with an identity X and one-hot A/B that fix
orientation and transposition, linearity in s, and planted mistakes (mutants) that each
pin must reject. The planner is pinned by an independent characterisation of its
greedy output, checked exhaustively on small segment lists.

Parity unpinned: how closely an adapter extracted from real checkpoints reproduces the
fine-tuned model (the page reports a median relative difference of 0.6% for another
extraction) -- that needs trained weights and is outside this module.
"""
from __future__ import annotations

import numpy as np

BM = 128  # rows per tile in the planner's output (the tensor-core tile height)


# --------------------------------------------------------------------------- bf16 values

def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact value of each bf16 bit pattern (uint16) as float64.

    bf16 is the upper half of an IEEE binary32: shifting the 16 bits into the high half
    of a 32-bit word gives the float32 with the same value, which float64 holds exactly.
    """
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    f32 = (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return f32.astype(np.float64)


# --------------------------------------------------------------------------- routing

def check_segments(seg_offsets, seg_ids, T: int, n_adapters: int | None = None) -> None:
    """Raise ValueError unless the segments tile [0, T) in order with valid ids."""
    off = [int(v) for v in seg_offsets]
    ids = [int(v) for v in seg_ids]
    if len(off) != len(ids) + 1:
        raise ValueError("seg_offsets must hold one more entry than seg_ids")
    if len(ids) == 0:
        if T != 0:
            raise ValueError("no segments for a non-empty batch")
        return
    if off[0] != 0 or off[-1] != T:
        raise ValueError("segments must start at row 0 and end at row T")
    for i in range(len(ids)):
        if off[i + 1] < off[i]:
            raise ValueError("segment offsets must be nondecreasing")
        if ids[i] < 0 or (n_adapters is not None and ids[i] > n_adapters):
            raise ValueError("adapter id out of range")


def row_adapter_ids(seg_offsets, seg_ids, T: int) -> np.ndarray:
    """Adapter id of every row: 0 = base only, k >= 1 = adapter k (1-based)."""
    check_segments(seg_offsets, seg_ids, T)
    out = np.zeros(T, dtype=np.int64)
    for i, a in enumerate(seg_ids):
        out[int(seg_offsets[i]):int(seg_offsets[i + 1])] = int(a)
    return out


# --------------------------------------------------------------------------- the projection

def lora_linear_fp64(x, seg_offsets, seg_ids, w, a_list, b_list, scales) -> np.ndarray:
    """Y for a batch of request segments, in float64.

    x: [T, d_in]; w: [d_out, d_in]; a_list[k-1]: [r, d_in]; b_list[k-1]: [d_out, r];
    scales[k-1]: s for adapter k. All arrays are float64 holding the exact input values.
    Each segment is one request; rows of a segment with id 0 get the base product only.
    """
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    T = x.shape[0]
    check_segments(seg_offsets, seg_ids, T, len(a_list))
    y = np.zeros((T, w.shape[0]), dtype=np.float64)
    for i, a in enumerate(seg_ids):
        lo, hi = int(seg_offsets[i]), int(seg_offsets[i + 1])
        if hi == lo:
            continue
        xs = x[lo:hi]
        base = xs @ w.T                                   # the shared base weight
        if int(a) == 0:
            y[lo:hi] = base
        else:
            A = np.asarray(a_list[int(a) - 1], dtype=np.float64)
            B = np.asarray(b_list[int(a) - 1], dtype=np.float64)
            s = float(scales[int(a) - 1])
            u = xs @ A.T                                  # first thin matrix: [rows, r]
            y[lo:hi] = base + s * (u @ B.T)               # second thin matrix, added
    return y


def lora_linear_merged_fp64(x, seg_offsets, seg_ids, w, a_list, b_list, scales) -> np.ndarray:
    """Same rows through the merged weight W_a = W + s_a B_a A_a (the fine-tuned matrix)."""
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    T = x.shape[0]
    check_segments(seg_offsets, seg_ids, T, len(a_list))
    y = np.zeros((T, w.shape[0]), dtype=np.float64)
    for i, a in enumerate(seg_ids):
        lo, hi = int(seg_offsets[i]), int(seg_offsets[i + 1])
        if hi == lo:
            continue
        if int(a) == 0:
            w_eff = w
        else:
            A = np.asarray(a_list[int(a) - 1], dtype=np.float64)
            B = np.asarray(b_list[int(a) - 1], dtype=np.float64)
            w_eff = w + float(scales[int(a) - 1]) * (B @ A)
        y[lo:hi] = x[lo:hi] @ w_eff.T
    return y


def lora_linear_rows_fp64(x_rows, row_ids, w, a_list, b_list, scales) -> np.ndarray:
    """Y for an arbitrary set of rows given each row's adapter id (rows are independent).

    Used to check sampled rows of large batches: row i of the result is the row the full
    batch would give to a row equal to x_rows[i] in a segment with id row_ids[i].
    """
    x_rows = np.asarray(x_rows, dtype=np.float64)
    row_ids = np.asarray(row_ids, dtype=np.int64)
    n = x_rows.shape[0]
    # one segment per row: a plain restatement of the routing rule on these rows
    offs = list(range(n + 1))
    return lora_linear_fp64(x_rows, offs, list(row_ids), w, a_list, b_list, scales)


# --------------------------------------------------------------------------- 4-bit base weights

W4_GROUP = 128  # input features per scale group


def w4_dequantize_fp64(qweight, scale_bits) -> np.ndarray:
    """W [d_out, d_in] from 4-bit weights, exactly (float64).

    "Two 27B models on a single RTX 5090", section 4 and "Qwen3.8-27B on one RTX 3090 with
    patched vLLM + DFlash2" (the W4A16 base of the deployment): the base matrix is stored in 4
    bits, the adapter in bf16. Format (a reading, the pages give none): symmetric int4 with
    one bf16 scale per group of 128 consecutive input features of an output row,
        W[n, k] = q[n, k] * s[k // 128, n],   q in [-8, 7] (two's complement nibbles),
    qweight: uint8 [d_out, d_in / 2], byte j of row n holds k = 2j in its low nibble and
    k = 2j + 1 in its high nibble; scale_bits: bf16 bit patterns [d_in / 128, d_out].
    """
    qweight = np.ascontiguousarray(qweight, dtype=np.uint8)
    d_out, half = qweight.shape
    d_in = 2 * half
    lo = (qweight & 0x0F).astype(np.int64)
    hi = (qweight >> 4).astype(np.int64)
    q = np.empty((d_out, d_in), dtype=np.int64)
    q[:, 0::2] = lo
    q[:, 1::2] = hi
    q = np.where(q >= 8, q - 16, q)                      # two's complement nibble
    s = bf16_bits_to_f64(scale_bits)                     # [d_in // 128, d_out]
    if s.shape != (d_in // W4_GROUP, d_out):
        raise ValueError("scales must be [d_in / 128, d_out]")
    return q.astype(np.float64) * np.repeat(s.T, W4_GROUP, axis=1)


def round_to_bf16_fp64(values) -> np.ndarray:
    """Each value rounded to the nearest bf16 (ties to the even significand), as float64.

    Defined for values that binary32 holds exactly (checked): bf16 keeps the upper 16 bits of
    a binary32, so the rounding adds 0x7FFF plus the lowest kept bit to the pattern and drops
    the lower 16 bits (round half to even on the 16 dropped bits).
    """
    v = np.asarray(values, dtype=np.float64)
    f = v.astype(np.float32)
    if not np.array_equal(f.astype(np.float64), v) or not np.all(np.isfinite(f)):
        raise ValueError("values must be finite and exact in binary32")
    bits = f.view(np.uint32).astype(np.uint64)
    bits = (bits + 0x7FFF + ((bits >> 16) & 1)) & 0xFFFF0000
    return bits.astype(np.uint32).view(np.float32).astype(np.float64)


def w4_weights_bf16_fp64(qweight, scale_bits) -> np.ndarray:
    """The 4-bit base widened to the activation type: bf16(q[n, k] * s[k // 128, n]).

    "Qwen3.8-27B on one RTX 3090 with patched vLLM + DFlash2" runs the base as W4A16: 4-bit
    weights, 16-bit activations, so each weight times its group scale is widened to the
    16-bit activation type (bf16 here) before it meets X. q * s has up to 11 significant bits
    (a 4-bit integer times an 8-bit significand), so the widening rounds it once (RNE).
    """
    return round_to_bf16_fp64(w4_dequantize_fp64(qweight, scale_bits))


def lora_linear_w4_fp64(x, seg_offsets, seg_ids, qweight, scale_bits, a_list, b_list, scales) -> np.ndarray:
    """The projection with a 4-bit base: the plain definition on the widened weights."""
    return lora_linear_fp64(x, seg_offsets, seg_ids, w4_weights_bf16_fp64(qweight, scale_bits),
                            a_list, b_list, scales)


# --------------------------------------------------------------------------- the planner

def merge_segments(seg_offsets, seg_ids):
    """Drop empty segments and join neighbours that name the same adapter.

    Returns (offsets, ids) of the merged runs, in row order.
    """
    out_off, out_ids = [], []
    for i, a in enumerate(seg_ids):
        lo, hi = int(seg_offsets[i]), int(seg_offsets[i + 1])
        if hi == lo:
            continue
        if out_ids and out_ids[-1] == int(a):
            out_off[-1] = hi                      # extend the previous run
        else:
            if not out_ids:
                out_off.append(lo)
            out_off.append(hi)
            out_ids.append(int(a))
    if not out_ids:
        return [0], []
    return out_off, out_ids


def plan_ref(seg_offsets, seg_ids, T: int, bm: int = BM):
    """Tiles for the fused base+expand pass and for the shrink pass.

    Fused tiles: walk the rows in order and start a new tile when the current one holds
    ``bm`` rows, or when the next row names an adapter (id != 0) that differs from an
    adapter already in the tile. Rows with id 0 therefore join whatever tile they fall
    into; a tile holds at most one nonzero id, and its id is that id (0 if none).
    Each tile is (row0, nrows, id).

    Shrink tiles: the fused tiles whose id is nonzero, stably ordered by id (so rows of
    one adapter are contiguous in the launch order); the shrink computes U over exactly
    those rows, writing zeros for the id-0 rows that share a tile with adapter rows.
    """
    check_segments(seg_offsets, seg_ids, T)
    ids = row_adapter_ids(seg_offsets, seg_ids, T)
    fused = []
    row0, nrows, tid = 0, 0, 0
    for t in range(T):
        a = int(ids[t])
        cut = nrows == bm or (a != 0 and tid != 0 and a != tid)
        if cut:
            fused.append((row0, nrows, tid))
            row0, nrows, tid = t, 0, 0
        nrows += 1
        if a != 0:
            tid = a
    if nrows:
        fused.append((row0, nrows, tid))
    shrink = sorted([f for f in fused if f[2] != 0], key=lambda f: f[2])  # stable
    return fused, shrink


# --------------------------------------------------------------------------- tolerance

def max_rel_err(y_test, y_ref) -> float:
    """max |y_test - y_ref| / max |y_ref| over the whole tensor (0 for an all-zero ref)."""
    y_test = np.asarray(y_test, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    denom = float(np.max(np.abs(y_ref))) if y_ref.size else 0.0
    num = float(np.max(np.abs(y_test - y_ref))) if y_ref.size else 0.0
    if denom == 0.0:
        return num
    return num / denom

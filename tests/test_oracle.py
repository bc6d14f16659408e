"""Pins for the fp64 oracle: brute force, the merged-weight identity, routing, B = 0,
rank <= r, closed forms that fix orientation, linearity in s, and planted mistakes.

Every check here is independent of the oracle's own code path: brute-force loops, a
different algebraic route (the merged weight), exact closed forms, or structural facts
(rank, linearity). Each mutant below plants one plausible mistake in a copy of the
oracle and must be rejected by at least one pin.
"""
import itertools

import numpy as np
import pytest

from oracle import (bf16_bits_to_f64, lora_linear_fp64, lora_linear_merged_fp64,
                    lora_linear_rows_fp64, max_rel_err, row_adapter_ids)


# --------------------------------------------------------------------------- helpers

def _rand_case(rng, T, d_in, d_out, r, n_ad, n_seg):
    x = rng.standard_normal((T, d_in))
    w = rng.standard_normal((d_out, d_in)) / np.sqrt(d_in)
    A = [rng.standard_normal((r, d_in)) / np.sqrt(d_in) for _ in range(n_ad)]
    B = [rng.standard_normal((d_out, r)) / np.sqrt(r) for _ in range(n_ad)]
    s = [float(v) for v in rng.uniform(0.5, 2.0, n_ad)]
    cuts = sorted(rng.integers(0, T + 1, n_seg - 1).tolist())
    off = [0] + cuts + [T]
    ids = [int(v) for v in rng.integers(0, n_ad + 1, n_seg)]
    return x, off, ids, w, A, B, s


def _brute(x, off, ids, w, A, B, s):
    """Triple loops: Y[t][n] = sum_k x w + [id != 0] s sum_j (sum_k x A) B."""
    T, d_in = len(x), len(x[0])
    d_out = len(w)
    Y = [[0.0] * d_out for _ in range(T)]
    for seg in range(len(ids)):
        a = ids[seg]
        for t in range(off[seg], off[seg + 1]):
            u = []
            if a:
                Aa = A[a - 1]
                for j in range(len(Aa)):
                    acc = 0.0
                    for k in range(d_in):
                        acc += x[t][k] * Aa[j][k]
                    u.append(acc)
            for n in range(d_out):
                acc = 0.0
                for k in range(d_in):
                    acc += x[t][k] * w[n][k]
                if a:
                    Ba = B[a - 1]
                    d = 0.0
                    for j in range(len(u)):
                        d += u[j] * Ba[n][j]
                    acc += s[a - 1] * d
                Y[t][n] = acc
    return np.array(Y)


# --------------------------------------------------------------------------- mutants (planted mistakes)

def _mut_offset_shift(x, off, ids, w, A, B, s):
    off2 = list(off)
    for i in range(1, len(off2) - 1):
        if off2[i] > 0:
            off2[i] -= 1      # every interior boundary one row early
    return lora_linear_fp64(x, off2, ids, w, A, B, s)


def _mut_swap_adapters(x, off, ids, w, A, B, s):
    return lora_linear_fp64(x, off, ids, w, A[::-1], B[::-1], s[::-1])


def _mut_b_transposed(x, off, ids, w, A, B, s):
    return lora_linear_fp64(x, off, ids, w, A, [b.T for b in B], s)


def _mut_no_scale(x, off, ids, w, A, B, s):
    return lora_linear_fp64(x, off, ids, w, A, B, [1.0] * len(s))


def _mut_w_transposed(x, off, ids, w, A, B, s):
    return lora_linear_fp64(x, off, ids, w.T, A, B, s)


def _mut_delta_on_all_rows(x, off, ids, w, A, B, s):
    ids2 = [1 if a == 0 else a for a in ids]
    return lora_linear_fp64(x, off, ids2, w, A, B, s)


MUTANTS = [_mut_offset_shift, _mut_swap_adapters, _mut_b_transposed, _mut_no_scale,
           _mut_w_transposed, _mut_delta_on_all_rows]


def _square_case(rng):
    # square shapes (d_in = d_out = r) so that transposition mistakes give wrong values,
    # not shape errors; two distinct adapters, distinct scales, both ids and id 0 present
    T, d = 9, 6
    x = rng.standard_normal((T, d))
    w = rng.standard_normal((d, d))
    A = [rng.standard_normal((d, d)) for _ in range(2)]
    B = [rng.standard_normal((d, d)) for _ in range(2)]
    s = [0.75, 1.5]
    off, ids = [0, 3, 5, 9], [0, 1, 2]
    return x, off, ids, w, A, B, s


# --------------------------------------------------------------------------- bf16 decoding

def test_bf16_decoding_closed_forms():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0x8000, 0x0001, 0x7F7F, 0x3E80, 0x4049], dtype=np.uint16)
    want = [1.0, -2.0, 0.0, -0.0, 2.0 ** -133, (2 - 2 ** -7) * 2.0 ** 127, 0.25,
            (1 + 0x49 / 128) * 2.0]
    got = bf16_bits_to_f64(bits)
    assert got.tolist() == want


def test_bf16_decoding_matches_float32_upper_half():
    rng = np.random.default_rng(0)
    f = rng.standard_normal(4096).astype(np.float32)
    u32 = f.view(np.uint32) & np.uint32(0xFFFF0000)          # values exactly representable in bf16
    ref = u32.view(np.float32).astype(np.float64)
    got = bf16_bits_to_f64((u32 >> np.uint32(16)).astype(np.uint16))
    assert np.array_equal(got, ref)


# --------------------------------------------------------------------------- brute force

@pytest.mark.parametrize("seed", range(6))
def test_oracle_matches_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    T = int(rng.integers(1, 9))
    case = _rand_case(rng, T, int(rng.integers(1, 33)), int(rng.integers(1, 25)),
                      int(rng.integers(1, 5)), 2, int(rng.integers(1, 5)))
    y = lora_linear_fp64(*case)
    yb = _brute(*[c.tolist() if isinstance(c, np.ndarray) else
                  ([m.tolist() for m in c] if isinstance(c, list) and c and isinstance(c[0], np.ndarray) else c)
                  for c in case])
    assert max_rel_err(y, yb) < 1e-12


def test_brute_force_rejects_every_mutant():
    rng = np.random.default_rng(7)
    case = _square_case(rng)
    as_lists = [c.tolist() if isinstance(c, np.ndarray) else
                ([m.tolist() for m in c] if isinstance(c, list) and c and isinstance(c[0], np.ndarray) else c)
                for c in case]
    yb = _brute(*as_lists)
    assert max_rel_err(lora_linear_fp64(*case), yb) < 1e-12
    for m in MUTANTS:
        assert max_rel_err(m(*case), yb) > 1e-3, m.__name__


# --------------------------------------------------------------------------- merged-weight identity

@pytest.mark.parametrize("shape", [(64, 256, 512, 16, 1, 2), (200, 96, 160, 8, 3, 7), (5, 32, 48, 32, 2, 5)])
def test_factored_equals_merged_weight(shape):
    T, d_in, d_out, r, n_ad, n_seg = shape
    rng = np.random.default_rng(sum(shape))
    case = _rand_case(rng, T, d_in, d_out, r, n_ad, n_seg)
    y = lora_linear_fp64(*case)
    ym = lora_linear_merged_fp64(*case)
    assert max_rel_err(y, ym) < 1e-12


def test_merged_identity_rejects_mutants_that_change_the_delta():
    rng = np.random.default_rng(11)
    case = _square_case(rng)
    ym = lora_linear_merged_fp64(*case)
    for m in (_mut_swap_adapters, _mut_b_transposed, _mut_no_scale, _mut_offset_shift):
        assert max_rel_err(m(*case), ym) > 1e-3, m.__name__


# --------------------------------------------------------------------------- routing

def test_base_rows_equal_base_product_and_adapter_rows_differ():
    rng = np.random.default_rng(3)
    x, off, ids, w, A, B, s = _rand_case(rng, 120, 64, 80, 8, 2, 1)
    off, ids = [0, 30, 31, 70, 70, 120], [0, 1, 0, 2, 1]
    y = lora_linear_fp64(x, off, ids, w, A, B, s)
    ybase = lora_linear_fp64(x, off, [0] * len(ids), w, A, B, s)
    rid = row_adapter_ids(off, ids, 120)
    base_rows = rid == 0
    assert np.array_equal(y[base_rows], ybase[base_rows])
    # every adapter row moved by an O(1) delta
    d = np.abs(y[~base_rows] - ybase[~base_rows]).max(axis=1)
    assert d.min() > 1e-2


def test_segment_order_permutes_rows_only():
    rng = np.random.default_rng(4)
    x, _, _, w, A, B, s = _rand_case(rng, 50, 40, 24, 4, 2, 1)
    off, ids = [0, 10, 35, 50], [1, 0, 2]
    y = lora_linear_fp64(x, off, ids, w, A, B, s)
    perm = np.r_[35:50, 0:10, 10:35]
    y2 = lora_linear_fp64(x[perm], [0, 15, 25, 50], [2, 1, 0], w, A, B, s)
    assert max_rel_err(y2, y[perm]) < 1e-13


def test_rows_helper_matches_batch():
    rng = np.random.default_rng(5)
    x, off, ids, w, A, B, s = _rand_case(rng, 77, 48, 56, 8, 3, 6)
    y = lora_linear_fp64(x, off, ids, w, A, B, s)
    rid = row_adapter_ids(off, ids, 77)
    pick = np.array([0, 1, 17, 40, 76])
    yr = lora_linear_rows_fp64(x[pick], rid[pick], w, A, B, s)
    assert max_rel_err(yr, y[pick]) < 1e-13


# --------------------------------------------------------------------------- B = 0, rank, linearity

def test_zero_b_is_a_no_op():
    rng = np.random.default_rng(6)
    x, off, ids, w, A, B, s = _rand_case(rng, 64, 32, 48, 8, 2, 4)
    Bz = [np.zeros_like(b) for b in B]
    y = lora_linear_fp64(x, off, ids, w, A, Bz, s)
    ybase = lora_linear_fp64(x, off, [0] * len(ids), w, A, B, s)
    assert np.array_equal(y, ybase)


def test_delta_rank_at_most_r():
    rng = np.random.default_rng(8)
    T, d_in, d_out, r = 96, 64, 72, 8
    x, _, _, w, A, B, s = _rand_case(rng, T, d_in, d_out, r, 1, 1)
    off, ids = [0, T], [1]
    delta = lora_linear_fp64(x, off, ids, w, A, B, s) - lora_linear_fp64(x, off, [0], w, A, B, s)
    sv = np.linalg.svd(delta, compute_uv=False)
    assert sv[r] / sv[0] < 1e-12          # nothing beyond rank r
    assert sv[r - 1] / sv[0] > 1e-4       # generic inputs reach rank r


@pytest.mark.parametrize("s_val", [0.5, -1.25, 3.0])
def test_linear_in_scale(s_val):
    rng = np.random.default_rng(9)
    x, off, ids, w, A, B, _ = _rand_case(rng, 40, 32, 24, 4, 1, 1)
    off, ids = [0, 40], [1]
    y0 = lora_linear_fp64(x, off, ids, w, A, B, [0.0])
    y1 = lora_linear_fp64(x, off, ids, w, A, B, [1.0])
    ys = lora_linear_fp64(x, off, ids, w, A, B, [s_val])
    assert max_rel_err(ys - y0, s_val * (y1 - y0)) < 1e-12


# --------------------------------------------------------------------------- closed forms

def test_identity_input_gives_merged_weight_transposed():
    # X = I (T = d_in), every row on adapter 1: row k of Y is column k of W + s B A.
    rng = np.random.default_rng(10)
    d_in, d_out, r = 12, 7, 3
    w = rng.integers(-3, 4, (d_out, d_in)).astype(np.float64)
    A = [rng.integers(-2, 3, (r, d_in)).astype(np.float64)]
    B = [rng.integers(-2, 3, (d_out, r)).astype(np.float64)]
    s = [2.0]
    y = lora_linear_fp64(np.eye(d_in), [0, d_in], [1], w, A, B, s)
    for k in range(d_in):
        for n in range(d_out):
            want = w[n, k] + s[0] * sum(B[0][n, j] * A[0][j, k] for j in range(r))
            assert y[k, n] == want       # small integers: exact in fp64


def test_one_hot_adapter_is_one_outer_product():
    # A[j0, k0] = 1, B[n0, j0] = 1, W = 0: Y[t, n] = s X[t, k0] when n = n0, else 0.
    d, T = 8, 5
    j0, k0, n0, s = 2, 5, 3, 1.75
    rng = np.random.default_rng(12)
    x = rng.standard_normal((T, d))
    A = np.zeros((d, d)); A[j0, k0] = 1.0
    B = np.zeros((d, d)); B[n0, j0] = 1.0
    y = lora_linear_fp64(x, [0, T], [1], np.zeros((d, d)), [A], [B], [s])
    want = np.zeros((T, d)); want[:, n0] = s * x[:, k0]
    assert np.array_equal(y, want)
    # the same closed form rejects a transposed B (the delta lands in the wrong place)
    ym = _mut_b_transposed(x, [0, T], [1], np.zeros((d, d)), [A], [B], [s])
    assert not np.array_equal(ym, want)
    yt = lora_linear_fp64(x, [0, T], [1], np.zeros((d, d)), [A.T], [B.T], [s])
    assert not np.array_equal(yt, want)


def test_w_orientation_closed_form():
    # X row t = e_t: Y[t, n] = W[n, t] on base rows (nn.Linear layout, W is [d_out, d_in]).
    d_in, d_out = 6, 4
    w = np.arange(d_out * d_in, dtype=np.float64).reshape(d_out, d_in)
    y = lora_linear_fp64(np.eye(d_in), [0, d_in], [0], w, [], [], [])
    assert np.array_equal(y, w.T)


# --------------------------------------------------------------------------- validation

@pytest.mark.parametrize("off,ids,T", [([0, 5], [0], 6), ([1, 6], [0], 6), ([0, 4, 3, 6], [0, 1, 0], 6),
                                       ([0, 6], [2], 6), ([0, 6], [-1], 6), ([0, 6], [], 6)])
def test_bad_segments_are_rejected(off, ids, T):
    x = np.zeros((T, 4)); w = np.zeros((4, 4))
    with pytest.raises(ValueError):
        lora_linear_fp64(x, off, ids, w, [np.zeros((2, 4))], [np.zeros((4, 2))], [1.0])


def test_empty_batch():
    y = lora_linear_fp64(np.zeros((0, 4)), [0], [], np.zeros((3, 4)), [], [], [])
    assert y.shape == (0, 3)
    y = lora_linear_fp64(np.zeros((0, 4)), [0, 0], [1], np.zeros((3, 4)),
                         [np.zeros((2, 4))], [np.zeros((3, 2))], [1.0])
    assert y.shape == (0, 3)


def test_tolerance_helper():
    assert max_rel_err([1.0, -2.0], [1.0, -2.0]) == 0.0
    assert abs(max_rel_err([1.0, -2.01], [1.0, -2.0]) - 0.005) < 1e-12
    assert max_rel_err(np.zeros(3), np.zeros(3)) == 0.0


def test_all_small_segment_layouts_route_correctly():
    # exhaustive over 3-segment layouts of a 6-row batch: every row gets its own segment's id
    rng = np.random.default_rng(13)
    x = rng.standard_normal((6, 5)); w = rng.standard_normal((4, 5))
    A = [rng.standard_normal((2, 5)) for _ in range(2)]
    B = [rng.standard_normal((4, 2)) for _ in range(2)]
    s = [1.0, 0.5]
    per_row = {a: lora_linear_fp64(x, [0, 6], [a], w, A, B, s) for a in (0, 1, 2)}
    for c1, c2 in itertools.combinations_with_replacement(range(7), 2):
        for ids in itertools.product((0, 1, 2), repeat=3):
            off = [0, c1, c2, 6]
            y = lora_linear_fp64(x, off, list(ids), w, A, B, s)
            rid = row_adapter_ids(off, ids, 6)
            for t in range(6):
                assert max_rel_err(y[t], per_row[int(rid[t])][t]) < 1e-13

"""Pins for the oracle's 4-bit base-weight decoding (W[n,k] = q[n,k] * s[k//128, n]) and its
widening to bf16 (one round-to-nearest-even of q * s)."""
import numpy as np
import pytest

import torch

from oracle import (W4_GROUP, lora_linear_fp64, lora_linear_w4_fp64, max_rel_err, round_to_bf16_fp64,
                    w4_dequantize_fp64, w4_weights_bf16_fp64)


def _bf16_bits_of(values):
    f = np.asarray(values, dtype=np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)   # values chosen exactly representable


def test_nibble_order_and_sign_closed_form():
    # one row, 128 inputs; byte j holds k=2j (low nibble) and k=2j+1 (high nibble)
    q = np.zeros((1, 64), dtype=np.uint8)
    q[0, 0] = 0x71          # k0 = 1, k1 = 7
    q[0, 1] = 0x8F          # k2 = -1 (0xF), k3 = -8 (0x8)
    q[0, 63] = 0x9E         # k126 = -2 (0xE), k127 = -7 (0x9)
    s = _bf16_bits_of([[0.5]])
    w = w4_dequantize_fp64(q, s)
    assert w.shape == (1, 128)
    assert w[0, :4].tolist() == [0.5, 3.5, -0.5, -4.0]
    assert w[0, 126:].tolist() == [-1.0, -3.5]
    assert np.count_nonzero(w) == 6


def test_groups_and_rows_take_their_own_scale():
    d_out, d_in = 3, 256
    q = np.full((d_out, d_in // 2), 0x11, dtype=np.uint8)     # every q = 1
    sc = np.array([[1.0, 2.0, 4.0], [0.25, 8.0, 0.5]], dtype=np.float32)   # [d_in/128, d_out]
    w = w4_dequantize_fp64(q, _bf16_bits_of(sc))
    for n in range(d_out):
        assert np.all(w[n, :128] == sc[0, n]) and np.all(w[n, 128:] == sc[1, n])


def test_every_nibble_value_round_trips():
    # quantise by hand (independent packing), decode with the oracle
    rng = np.random.default_rng(0)
    d_out, d_in = 5, 384
    qv = rng.integers(-8, 8, (d_out, d_in))
    sc = rng.uniform(0.01, 0.2, (d_in // W4_GROUP, d_out)).astype(np.float32)
    sc = (sc.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32)   # bf16-exact
    nib = (qv & 0xF).astype(np.uint8)
    packed = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    w = w4_dequantize_fp64(packed, _bf16_bits_of(sc))
    want = qv * np.repeat(sc.T.astype(np.float64), W4_GROUP, axis=1)
    assert np.array_equal(w, want)


def test_w4_projection_is_the_projection_of_the_decoded_weights():
    rng = np.random.default_rng(1)
    T, d_in, d_out, r = 20, 256, 48, 8
    x = rng.standard_normal((T, d_in))
    packed = rng.integers(0, 256, (d_out, d_in // 2)).astype(np.uint8)
    sc = _bf16_bits_of(np.full((d_in // 128, d_out), 0.0625))
    A = [rng.standard_normal((r, d_in))]
    B = [rng.standard_normal((d_out, r))]
    off, ids = [0, 7, 20], [1, 0]
    y = lora_linear_w4_fp64(x, off, ids, packed, sc, A, B, [1.5])
    w = w4_weights_bf16_fp64(packed, sc)
    # brute force for one row of each kind
    for t in (3, 15):
        base = np.array([sum(x[t, k] * w[n, k] for k in range(d_in)) for n in range(d_out)])
        if t < 7:
            u = A[0] @ x[t]
            base = base + 1.5 * (B[0] @ u)
        assert max_rel_err(y[t], base) < 1e-12
    assert max_rel_err(y, lora_linear_fp64(x, off, ids, w, A, B, [1.5])) == 0.0


def test_bf16_rounding_closed_forms():
    # 7 (1 + 2^-7) = 7.0546875 lies between the bf16 values 7.03125 and 7.0625: nearest 7.0625
    assert round_to_bf16_fp64([7 * (1 + 2.0 ** -7)]).tolist() == [7.0625]
    # ties go to the even significand: 3.0234375 is halfway between 3.015625 (odd) and 3.03125
    assert round_to_bf16_fp64([3 * (1 + 2.0 ** -7), -3 * (1 + 2.0 ** -7)]).tolist() == [3.03125, -3.03125]
    # 1 + 2^-8 is halfway between 1 (even) and 1 + 2^-7 (odd); 1 + 3 2^-8 between odd and even
    assert round_to_bf16_fp64([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8]).tolist() == [1.0, 1 + 2.0 ** -6]
    # bf16 values and zero are fixed points
    assert round_to_bf16_fp64([0.0, -0.0, 0.5, -4.0, 1 + 2.0 ** -7]).tolist() == [0.0, 0.0, 0.5, -4.0, 1 + 2.0 ** -7]
    with pytest.raises(ValueError):
        round_to_bf16_fp64([0.1])                    # not exact in binary32


def test_bf16_rounding_equals_the_library_conversion():
    # random binary32 values of every magnitude: the same as PyTorch's float32 -> bfloat16 cast
    rng = np.random.default_rng(2)
    f = (rng.standard_normal(20000) * np.exp2(rng.integers(-30, 30, 20000))).astype(np.float32)
    f[:64] = np.arange(64, dtype=np.float32) * np.float32(1 + 2.0 ** -9)     # many exact ties
    want = torch.from_numpy(f).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(round_to_bf16_fp64(f.astype(np.float64)), want)


def test_widened_weights_round_each_decoded_weight_once():
    rng = np.random.default_rng(3)
    d_out, d_in = 4, 256
    packed = rng.integers(0, 256, (d_out, d_in // 2)).astype(np.uint8)
    sc = _bf16_bits_of(np.array([[1 + 2.0 ** -7, 0.5, 0.1015625, 3.0], [0.25, 1.0078125, 2.0, 0.0625]]))
    exact = w4_dequantize_fp64(packed, sc)
    wide = w4_weights_bf16_fp64(packed, sc)
    assert np.array_equal(wide, round_to_bf16_fp64(exact))
    # power-of-two scales: q s is already a bf16 value
    assert np.array_equal(wide[1, :128], exact[1, :128]) and np.array_equal(wide[0, 128:], exact[0, 128:])
    # q = 7 or -3 with s = 1 + 2^-7 (row 0, first group): 7.0625 and -3.03125
    q = exact[0, :128] / (1 + 2.0 ** -7)
    assert np.all(wide[0, :128][q == 7] == 7.0625) and np.all(wide[0, :128][q == -3] == -3.03125)
    assert np.count_nonzero(wide != exact) > 0


def test_bad_scale_shape_is_rejected():
    with pytest.raises(ValueError):
        w4_dequantize_fp64(np.zeros((2, 64), dtype=np.uint8), np.zeros((2, 2), dtype=np.uint16))

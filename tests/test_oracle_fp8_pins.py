"""Pins of the 8-bit (e4m3, per-tensor scaled) oracle, independent of itself.

The e4m3 decode is pinned to hand-worked values of the format's definition
(OCP 8-bit floating point specification, E4M3: bias 7, no infinities, NaN at
S.1111.111, largest finite 448) and to torch's own float8_e4m3fn decode of
all 256 codes; plausible slips (bias 8, subnormals read as normals, 0x7E read
as NaN) are planted in copies here and must fail the hand values.  The
attention of dequantised inputs is pinned by closed forms: scores that are all
equal give O = mean of V, one key gives O = that key's V, and the descales
enter only as the products that define the dequantised tensors.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_82_gb300.inputs import E4M3_MAX, make_qkv_fp8, quantize_e4m3, u8_codes

# (code, value) worked by hand from the bit fields S.EEEE.MMM
HAND = [
    (0x00, 0.0),               # E=0 M=0
    (0x01, 2.0 ** -9),         # subnormal 1/8 * 2^-6, the smallest magnitude
    (0x07, 7 * 2.0 ** -9),     # largest subnormal
    (0x08, 2.0 ** -6),         # E=1: smallest normal
    (0x0F, 1.875 * 2.0 ** -6),
    (0x30, 0.5),               # E=6
    (0x38, 1.0),               # E=7 = bias
    (0x39, 1.125),
    (0x3C, 1.5),
    (0x40, 2.0),
    (0x4A, 5.0),               # E=9 M=2: 1.25 * 4
    (0x70, 128.0),             # E=14
    (0x77, 240.0),             # E=14 M=7: 1.875 * 128
    (0x78, 256.0),             # E=15 is an ordinary exponent
    (0x7D, 416.0),
    (0x7E, 448.0),             # largest finite
    (0x80, -0.0),
    (0x81, -(2.0 ** -9)),
    (0xB8, -1.0),
    (0xFE, -448.0),
]


def test_decode_hand_values():
    codes = np.array([c for c, _ in HAND], np.uint8)
    want = np.array([v for _, v in HAND])
    got = oracle.e4m3_to_f64(codes)
    np.testing.assert_array_equal(got, want)
    assert math.copysign(1.0, oracle.e4m3_to_f64(np.array([0x80], np.uint8))[0]) == -1.0


def test_decode_nan_codes_only():
    v = oracle.e4m3_to_f64(np.arange(256, dtype=np.uint8))
    assert set(np.flatnonzero(np.isnan(v))) == {0x7F, 0xFF}
    assert np.nanmax(np.abs(v)) == E4M3_MAX


def test_decode_matches_torch_for_every_code():
    c = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(c.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.e4m3_to_f64(c), ref)


def test_decode_positive_codes_increase():
    v = oracle.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(v) > 0)
    # negatives mirror positives bit for bit
    np.testing.assert_array_equal(oracle.e4m3_to_f64(np.arange(0x80, 0xFF, dtype=np.uint8)), -v)


def _mutant_bias8(c):
    c = np.asarray(c, np.int64)
    e, m = (c >> 3) & 15, (c & 7) / 8.0
    mag = np.where(e == 0, m * 2.0 ** -7, (1 + m) * 2.0 ** (e - 8.0))
    return np.where(c & 0x80, -mag, mag)


def _mutant_no_subnormal(c):
    c = np.asarray(c, np.int64)
    e, m = (c >> 3) & 15, (c & 7) / 8.0
    mag = (1 + m) * 2.0 ** (e - 7.0)
    return np.where(c & 0x80, -mag, mag)


def _mutant_ieee_like_top(c):
    v = oracle.e4m3_to_f64(c).copy()
    v[(np.asarray(c) & 0x78) == 0x78] = np.nan  # whole top exponent taken as inf/NaN
    return v


@pytest.mark.parametrize("mutant", [_mutant_bias8, _mutant_no_subnormal, _mutant_ieee_like_top])
def test_decode_pins_catch_mutants(mutant):
    codes = np.array([c for c, _ in HAND], np.uint8)
    want = np.array([v for _, v in HAND])
    got = mutant(codes)
    assert not np.array_equal(got, want, equal_nan=False)


def test_quantizer_uses_full_range_and_rounds_to_nearest():
    g = torch.Generator().manual_seed(5)
    x = torch.randn(4, 64, generator=g) * 3.0
    codes, d = quantize_e4m3(x)
    deq = oracle.e4m3_to_f64(u8_codes(codes)) * d
    assert abs(np.abs(deq).max() - float(x.abs().max())) <= 1e-6 * float(x.abs().max())
    # round to nearest: within half a step of the e4m3 grid at each magnitude
    xs = x.double().numpy() / d
    grid = np.sort(np.unique(np.abs(oracle.e4m3_to_f64(np.arange(0x7F, dtype=np.uint8)))))
    nearest = grid[np.abs(np.abs(xs)[..., None] - grid).argmin(-1)]
    np.testing.assert_allclose(np.abs(deq / d), nearest, rtol=0, atol=0)


def test_equal_scores_give_mean_of_v():
    """Q codes all zero: every score is 0, P is uniform, O = mean_j V_j, LSE = ln Sk."""
    (q, k, v), (dq, dk, dv) = make_qkv_fp8(1, 2, 5, 37, 128, seed=3)
    q = torch.zeros_like(q)
    o, lse = oracle.attn_fwd_fp8(u8_codes(q), u8_codes(k), u8_codes(v), dq, dk, dv, 0.1)
    vd = oracle.e4m3_to_f64(u8_codes(v)) * np.float32(dv)
    np.testing.assert_allclose(o, np.broadcast_to(vd.mean(axis=2, keepdims=True), o.shape),
                               rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse, math.log(37), rtol=1e-14)


def test_single_key_returns_its_value():
    (q, k, v), (dq, dk, dv) = make_qkv_fp8(2, 1, 3, 1, 128, seed=4)
    o, lse = oracle.attn_fwd_fp8(u8_codes(q), u8_codes(k), u8_codes(v), dq, dk, dv, 0.3)
    vd = oracle.e4m3_to_f64(u8_codes(v)) * np.float32(dv)
    np.testing.assert_allclose(o, np.broadcast_to(vd, o.shape), rtol=1e-14)
    qd = oracle.e4m3_to_f64(u8_codes(q)) * np.float32(dq)
    kd = oracle.e4m3_to_f64(u8_codes(k)) * np.float32(dk)
    np.testing.assert_allclose(lse, 0.3 * np.einsum("bhqd,bhkd->bhqk", qd, kd)[..., 0], rtol=1e-12)


def test_descales_enter_as_products():
    """Doubling descale_q is the same as doubling scale; doubling descale_v doubles O
    and leaves LSE; the result does not depend on how dq*dk is split."""
    (q, k, v), (dq, dk, dv) = make_qkv_fp8(1, 2, 40, 50, 128, seed=6)
    a = [u8_codes(t) for t in (q, k, v)]
    o1, l1 = oracle.attn_fwd_fp8(*a, dq * 2, dk, dv, 0.09, causal=False)
    o2, l2 = oracle.attn_fwd_fp8(*a, dq, dk, dv, 0.18, causal=False)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(l1, l2, rtol=1e-12)
    o3, l3 = oracle.attn_fwd_fp8(*a, dq, dk, dv * 2, 0.18, causal=False)
    np.testing.assert_allclose(o3, 2 * o2, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(l3, l2)
    o4, l4 = oracle.attn_fwd_fp8(*a, dk, dq, dv, 0.18, causal=False)
    np.testing.assert_allclose(o4, o2, rtol=1e-12, atol=1e-14)


def test_causal_first_row_sees_only_first_key():
    (q, k, v), (dq, dk, dv) = make_qkv_fp8(1, 1, 9, 9, 128, seed=8)
    o, _ = oracle.attn_fwd_fp8(*(u8_codes(t) for t in (q, k, v)), dq, dk, dv, 0.1, causal=True)
    vd = oracle.e4m3_to_f64(u8_codes(v)) * np.float32(dv)
    np.testing.assert_allclose(o[0, 0, 0], vd[0, 0, 0], rtol=1e-14)

"""Pins of the FP8 E4M3 / MX-scaling oracle (oracle/fp8.py), CPU only.

Each pin checks the oracle against something other than itself: the format's
defining values, a library conversion (torch's float8_e4m3fn, round to
nearest even), exact cases, and a rigorous error bound.
"""
import numpy as np
import pytest
import torch

import oracle.fp8 as fp8


def test_defining_values():
    dec = fp8.e4m3_decode
    assert dec(0x38) == 1.0 and dec(0x3C) == 1.5          # e = 7: 2^0
    assert dec(0x7E) == 448.0                             # largest finite
    assert dec(0x08) == 2.0 ** -6                         # smallest normal
    assert dec(0x01) == 2.0 ** -9 and dec(0x07) == 7 * 2.0 ** -9   # subnormals
    assert np.isnan(dec(0x7F)) and np.isnan(dec(0xFF))
    assert dec(0xB8) == -1.0 and np.signbit(dec(0x80))
    finite = dec(np.arange(256))
    assert np.isfinite(finite).sum() == 254
    assert len(np.unique(np.abs(finite[np.isfinite(finite)]))) == 127


def test_every_finite_code_round_trips():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(fp8.e4m3_encode(fp8.e4m3_decode(codes)), codes)


def test_ties_go_to_the_even_code():
    r = fp8.e4m3_round
    assert r(1 + 1 / 16) == 1.0          # between 1 (m = 0) and 1.125 (m = 1)
    assert r(1 + 3 / 16) == 1.25         # between 1.125 (m = 1) and 1.25 (m = 2)
    assert r(1.9375) == 2.0              # between 1.875 (m = 7) and 2.0 (next binade, m = 0)
    assert r(2.0 ** -10) == 0.0          # half the smallest subnormal
    assert r(7.5 * 2.0 ** -9) == 2.0 ** -6   # subnormal / normal boundary
    assert r(-(1 + 1 / 16)) == -1.0


def test_saturation_and_underflow():
    r = fp8.e4m3_round
    assert (r(np.array([448.0, 449.0, 464.0, 480.0, 1e9, np.inf])) == 448.0).all()
    assert r(-1e9) == -448.0
    assert r(0.75 * 2.0 ** -9) == 2.0 ** -9 and r(0.4 * 2.0 ** -9) == 0.0
    assert fp8.e4m3_encode(np.nan) == 0x7F


def test_rounding_matches_a_library_conversion():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(200000) * 2.0 ** rng.integers(-12, 9, 200000)).astype(np.float32)
    x = x[np.abs(x) < 464]               # torch turns larger magnitudes into NaN, not 448
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(fp8.e4m3_round(x.astype(np.float64)), ref)


def test_relative_error_in_the_normal_range():
    rng = np.random.default_rng(1)
    x = np.exp(rng.uniform(np.log(2.0 ** -6), np.log(448.0), 100000)) * rng.choice([-1, 1], 100000)
    assert (np.abs(fp8.e4m3_round(x) - x) <= 2.0 ** -4 * np.abs(x)).all()


@pytest.mark.parametrize("k", [-20, -3, 0, 1, 7, 30])
def test_mx_scale_is_the_block_exponent_minus_8(k):
    v = np.zeros((1, 32))
    v[0, 5] = 1.5 * 2.0 ** k             # amax in [2^k, 2^(k+1))
    v[0, 9] = -0.25 * 2.0 ** k
    P, X = fp8.mx_quantize(v)
    assert X[0, 0] == 2.0 ** (k - 8)
    assert P[0, 5] == 384.0 and P[0, 9] == -64.0
    np.testing.assert_array_equal(P * X[0, 0], v)     # both values representable


def test_mx_scaled_maximum_can_saturate():
    v = np.zeros((1, 32))
    v[0, 0] = 1.99                        # scaled by 2^-8: 509.4 > 448
    P, X = fp8.mx_quantize(v)
    assert X[0, 0] == 2.0 ** -8 and P[0, 0] == 448.0


def test_mx_blocks_are_independent_and_zero_blocks_stay_zero():
    rng = np.random.default_rng(2)
    v = rng.standard_normal((3, 96))
    v[1, 32:64] = 0.0
    P, X = fp8.mx_quantize(v)
    assert X.shape == (3, 3) and not P[1, 32:64].any()
    for b in range(3):
        Pb, Xb = fp8.mx_quantize(v[:, 32 * b:32 * (b + 1)])
        np.testing.assert_array_equal(Pb, P[:, 32 * b:32 * (b + 1)])
        np.testing.assert_array_equal(Xb[:, 0], X[:, b])


def _representable(rng, shape, k_scale):
    """Values X * P with P on the E4M3 grid, |P| <= 256, and one |P| = 256 per
    32-block, so that MX scaling reproduces them exactly."""
    codes = rng.integers(0, 0x77, shape)                   # magnitudes up to 224
    P = fp8.e4m3_decode(codes) * rng.choice([-1.0, 1.0], shape)
    R, K = shape
    for b in range(0, K, 32):
        P[:, b] = 256.0                                    # the block maximum
    X = 2.0 ** rng.integers(-k_scale, k_scale + 1, (R, (K + 31) // 32))
    return P * np.repeat(X, 32, axis=1)[:, :K]


def test_mx_gemm_exact_on_representable_inputs():
    rng = np.random.default_rng(3)
    A = _representable(rng, (24, 128), 4)
    B = _representable(rng, (40, 128), 4)
    np.testing.assert_allclose(fp8.mx_gemm(A, B), A @ B.T, rtol=1e-13, atol=0)


def test_mx_gemm_within_the_quantisation_bound():
    """|D_mx - A B^T| <= sum_k (|a| e_b + e_a |b| + e_a e_b) with e the
    per-element bound max(2^-4 |v|, |v| - 448 X, 2^-10 X)."""
    rng = np.random.default_rng(4)
    A, B = rng.standard_normal((32, 200)), rng.standard_normal((48, 200)) * 0.02
    D = fp8.mx_gemm(A, B)

    def bound(v):
        _, X = fp8.mx_quantize(v)
        Xe = np.repeat(X, 32, axis=1)[:, :v.shape[1]]
        return np.maximum.reduce([2.0 ** -4 * np.abs(v), np.abs(v) - 448 * Xe, 2.0 ** -10 * Xe])

    ea, eb = bound(A), bound(B)
    lim = np.abs(A) @ eb.T + ea @ np.abs(B).T + ea @ eb.T
    err = np.abs(D - A @ B.T)
    assert (err <= lim * (1 + 1e-12)).all()
    assert err.max() > 0                  # quantisation did change the result

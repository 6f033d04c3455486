"""FP8 E4M3 with MX block scaling, float64 numpy (oracle; test infrastructure only).

The Oases pages describe no low-precision variant; this is the reference for
an FP8 form of the block's GEMMs.  It restates two published definitions:

  * the E4M3 element format ("FP8 Formats for Deep Learning", Micikevicius et
    al., arXiv 2209.05433, Table 1; the same format is the FP8 E4M3 element
    type of the OCP Microscaling (MX) Formats Specification v1.0, §5.3):
    1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0
    holds the subnormals m * 2^-9; the all-ones exponent with mantissa 7 is
    NaN, so the largest finite value is 1.75 * 2^8 = 448 and there is no
    infinity.  A real number is encoded as the nearest finite value, ties to
    the even code (even mantissa), and magnitudes above 448 saturate to 448
    (the "satfinite" conversion a kernel would use);
  * MX block scaling (OCP MX v1.0, §5 and §6.2): a block of 32 consecutive
    values along the contraction shares one power-of-two scale
    X = 2^(floor(log2(max |v|)) - 8), 8 being the exponent of the largest
    power of two in E4M3; each element is stored as E4M3(v / X) and a dot
    product of two blocks is X_a X_b sum_i P_a[i] P_b[i].

The GEMM below is that definition written out: quantise A and B block by
block along K, then D[m, n] = sum over blocks of X_A[m, b] X_B[n, b] times the
block's dot product of the E4M3 values, in float64 (each block's sum is exact
in float64).  No blocking or reordering beyond that.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
EMAX_ELEM = 8      # exponent of the largest power of two representable in E4M3
MX_BLOCK = 32


def e4m3_decode(code) -> np.ndarray:
    """Value of each E4M3 code (uint8 array-like); NaN for the two NaN codes."""
    c = np.asarray(code, dtype=np.int64) & 0xFF
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * 2.0 ** (e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


# the 127 finite non-negative values, in code order 0x00 .. 0x7E (increasing)
_POS = e4m3_decode(np.arange(0x7F))


def e4m3_encode(x) -> np.ndarray:
    """Nearest finite E4M3 code of each value (ties to the even code), with
    magnitudes above 448 saturated to 448; NaN maps to the NaN code 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(_POS, a, side="left"), 0, len(_POS) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo, d_hi = a - _POS[lo], _POS[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo).astype(np.int64)
    code = np.where(np.signbit(x), code | 0x80, code)
    return np.where(np.isnan(x), 0x7F, code).astype(np.uint8)


def e4m3_round(x) -> np.ndarray:
    """x rounded to E4M3 (value of its code)."""
    return e4m3_decode(e4m3_encode(x))


def mx_quantize(v: np.ndarray, block: int = MX_BLOCK):
    """MX-scale the rows of v [R, K] in blocks of `block` along K (the last
    block may be shorter).  Returns (P [R, K] E4M3 values as float64,
    X [R, ceil(K / block)] power-of-two scales)."""
    v = np.asarray(v, dtype=np.float64)
    R, K = v.shape
    nb = (K + block - 1) // block
    P = np.zeros_like(v)
    X = np.ones((R, nb))
    for b in range(nb):
        blk = v[:, b * block:(b + 1) * block]
        amax = np.abs(blk).max(axis=1)
        # floor(log2(amax)) exactly: amax = f * 2^p with f in [0.5, 1)
        e = np.frexp(np.where(amax > 0, amax, 1.0))[1].astype(np.float64) - 1 - EMAX_ELEM
        e = np.clip(e, -127, 127)          # the E8M0 scale's range
        X[:, b] = np.where(amax > 0, 2.0 ** e, 1.0)
        P[:, b * block:(b + 1) * block] = e4m3_round(blk / X[:, b:b + 1])
    return P, X


def mx_gemm(A: np.ndarray, B: np.ndarray, block: int = MX_BLOCK) -> np.ndarray:
    """D[m, n] = sum_b X_A[m, b] X_B[n, b] sum_{k in block b} P_A[m, k] P_B[n, k]
    for A [M, K] and B [N, K] (both K-contiguous, as the block's GEMMs take
    them), MX-quantised along K."""
    PA, XA = mx_quantize(A, block)
    PB, XB = mx_quantize(B, block)
    K = A.shape[1]
    D = np.zeros((A.shape[0], B.shape[0]))
    for b in range((K + block - 1) // block):
        s = slice(b * block, (b + 1) * block)
        D += (XA[:, b:b + 1] * XB[:, b][None, :]) * (PA[:, s] @ PB[:, s].T)
    return D


def bf16_round(x) -> np.ndarray:
    """x rounded to the nearest bfloat16 value (8 significant bits, exponent
    range of float32), ties to the even significand: x = f 2^e with f in
    [0.5, 1) becomes round_half_even(f 2^8) 2^(e-8).  Values below the bf16
    normal range (2^-126) are rounded on the same grid as 2^-126."""
    x = np.asarray(x, dtype=np.float64)
    f, e = np.frexp(x)
    e = np.maximum(e, -125)
    return np.ldexp(np.round(np.ldexp(x, 8 - e)), e - 8)


def mx_product_bf16(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    """The MX-FP8 form of one of the block's products, A B^T: both operands as
    the block stores them (bf16), each MX-quantised along the contraction (the
    columns of both), multiplied as mx_gemm does."""
    return mx_gemm(bf16_round(A), bf16_round(B))

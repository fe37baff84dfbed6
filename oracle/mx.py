"""MXFP8: the recipe's validation format (oracle; test infrastructure only).

[4BL] §"Improving Gradient Stability", "Results Validation with MXFP8": the
dequantised-backward fix is first checked with the MXFP8 recipe.  Three runs are
compared: quantised forward and backward; quantised forward with a BF16 backward; and
quantised forward with a backward on the dequantised weights.  The pages name the format
but do not define it.  The reading here is the OCP Microscaling Formats (MX) v1.0
definition of MXFP8 with E4M3 elements:

* Values form blocks of 32 consecutive elements along the last (contraction) dimension.
* Each block shares one E8M0 scale: an unsigned power of two 2^(b - 127), with
  b = 0..254.  b = 255 is NaN and is never produced here.
* The shared exponent is floor(log2(amax_b)) - 8.  Here amax_b = max |x| over the block,
  and 8 is the exponent of E4M3's largest normal (448 = 1.75 * 2^8).  The exponent is
  clamped below at -127, which is b = 0; an all-zero block also takes b = 0.
* Each element is E4M3(x / 2^exponent): round to nearest, ties to even, saturating at
  +-448.  The top of the block's range, 448 < |x / 2^exponent| < 512, saturates.
* A zero magnitude encodes as +0.  This is the same reading as the NVFP4 codes, so that
  zero has one encoding.
* MX has no per-tensor scale: DQ(x) = value(code) * 2^(b - 127).

Arithmetic: x is BF16, with at most 8 significant bits, and the scale is a power of two.
So x / 2^exponent is exact in float64, and exact in float32 wherever it can round to a
non-zero E4M3 value (>= 2^-10).  No rounding happens before the single E4M3 rounding.
"""
from __future__ import annotations

import numpy as np

from . import formats as F

BLOCK = 32
E4M3_EMAX = 8             # floor(log2(448))
E8M0_BIAS = 127


def e8m0_decode(b) -> np.ndarray:
    """Value of each E8M0 scale byte: 2^(b - 127), float64; NaN for 0xFF."""
    b = np.asarray(b, dtype=np.int64)
    v = np.exp2((b - E8M0_BIAS).astype(np.float64))
    return np.where(b == 0xFF, np.nan, v)


def shared_exponent(amax) -> np.ndarray:
    """floor(log2(amax)) - 8, clamped to [-127, 127]; -127 for amax == 0 (int64)."""
    a = np.asarray(amax, dtype=np.float64)
    _, p = np.frexp(a)                 # a = m * 2^p, m in [0.5, 1): floor(log2 a) = p - 1
    e = (p.astype(np.int64) - 1) - E4M3_EMAX
    e = np.where(a == 0, -E8M0_BIAS, e)
    return np.clip(e, -E8M0_BIAS, E8M0_BIAS)


def e4m3_encode_signed(v) -> np.ndarray:
    """Signed E4M3 byte of float64 ``v``: RNE to the nearest finite value, saturating at
    +-448; a magnitude that rounds to zero encodes as +0."""
    v = np.asarray(v, dtype=np.float64)
    mag = F.e4m3_encode_rne_satfinite(np.abs(v).astype(np.float32))
    neg = np.signbit(v) & (mag != 0)
    return (mag | (neg.astype(np.uint8) << 7)).astype(np.uint8)


def quantize(x_bits: np.ndarray):
    """MXFP8 of a BF16 matrix (uint16 bit patterns [rows, cols], cols % 32 == 0).

    Returns (codes uint8 [rows, cols] E4M3 bytes, sf uint8 [rows, cols/32] E8M0 bytes,
    row-major)."""
    x = F.bf16_to_f32(x_bits).astype(np.float64)
    rows, cols = x.shape
    if cols % BLOCK != 0:
        raise ValueError("cols must be a multiple of 32")
    xb = x.reshape(rows, cols // BLOCK, BLOCK)
    amax = np.abs(xb).max(axis=2)
    e = shared_exponent(amax)                                  # [rows, cols/32]
    t = xb * np.exp2(-e.astype(np.float64))[:, :, None]        # exact (power of two)
    codes = e4m3_encode_signed(t).reshape(rows, cols)
    sf = (e + E8M0_BIAS).astype(np.uint8)
    return codes, sf


def dequantize_exact(codes: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """DQ = value(code) * 2^(b - 127) for codes [rows, cols] and row-major sf
    [rows, cols/32], exact in float64."""
    codes = np.asarray(codes, np.uint8)
    rows, cols = codes.shape
    v = F.e4m3_decode(codes)
    s = np.repeat(e8m0_decode(sf), BLOCK, axis=1)[:, :cols]
    return v * s


def dequantize(codes: np.ndarray, sf: np.ndarray, out: str = "bf16") -> np.ndarray:
    """DQ rounded once from the exact value: BF16 bit patterns (uint16) or float32."""
    d = dequantize_exact(codes, sf)
    if out == "bf16":
        return F.bf16_round(d)
    if out == "f32":
        with np.errstate(over="ignore"):
            return d.astype(np.float32)            # beyond float32's range: Inf
    raise ValueError(out)


def grouped_gemm(a_codes, a_sf, b_codes, b_sf, group_offsets, group_rows) -> np.ndarray:
    """MXFP8 x MXFP8 grouped GEMM, float64: for every expert e and row r of its group,
    D[r, n] = sum_k DQ(A)[r, k] * DQ(B_e)[n, k].

    a_codes [M, K], a_sf [M, K/32] (row-major); b_codes [E, N, K], b_sf [E, N, K/32];
    group_offsets [E+1] (row starts), group_rows [E].  Rows outside the groups are 0."""
    a = dequantize_exact(a_codes, a_sf)
    E, N, K = b_codes.shape
    out = np.zeros((a.shape[0], N), np.float64)
    for e in range(E):
        n = int(group_rows[e])
        if n == 0:
            continue
        r0 = int(group_offsets[e])
        b = dequantize_exact(b_codes[e], b_sf[e])
        out[r0:r0 + n] = a[r0:r0 + n] @ b.T
    return out

"""Element formats of NVFP4 and the BF16 boundary type (oracle; test infrastructure only).

[4BL] §Baseline: NVFP4 holds 4-bit floating-point values, one FP8 E4M3 scale per block
of 16 values and one FP32 scale for the whole tensor; together they recover a
higher-precision value.  The bit layouts of the two small formats are the OCP ones
(OCP Microscaling Formats v1.0 for E2M1, OCP 8-bit Floating Point for E4M3):

* E2M1: sign, 2 exponent bits (bias 1), 1 mantissa bit; magnitudes
  {0, 0.5, 1, 1.5, 2, 3, 4, 6}; no Inf or NaN.
* E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; subnormals below 2^-6 down to
  2^-9; largest finite 448 (0x7E); 0x7F / 0xFF are NaN; no Inf.
"""
from __future__ import annotations

import numpy as np

E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
E2M1_MAX = 6.0
E4M3_MAX = 448.0


# --------------------------------------------------------------------------- E2M1

def e2m1_decode(codes) -> np.ndarray:
    """Value of each 4-bit code (low nibble of each uint8), float64."""
    c = np.asarray(codes, dtype=np.uint8) & 0xF
    mag = E2M1_MAGNITUDES[c & 7]
    return np.where((c & 8) != 0, -mag, mag)


def e2m1_encode_rne(v) -> np.ndarray:
    """Round float32 ``v`` to the nearest E2M1 value, ties to the even code, saturating
    at +-6 (the clip/round staircase of [4BL] footnote 6 with qmax = 6).

    Reading: a value whose magnitude rounds to 0 is encoded as +0 (code 0x0), whatever
    its sign, so that zero has one encoding.
    """
    v = np.asarray(v, dtype=np.float32)
    a = np.abs(v).astype(np.float64)
    # lo = index of the largest grid magnitude <= a (a >= 0 so lo >= 0).
    lo = np.searchsorted(E2M1_MAGNITUDES, a, side="right") - 1
    lo = np.clip(lo, 0, 7)
    hi = np.minimum(lo + 1, 7)
    d_lo = a - E2M1_MAGNITUDES[lo]
    d_hi = E2M1_MAGNITUDES[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo)
    code = np.where(a >= E2M1_MAX, 7, code)
    sign = (np.signbit(v) & (code != 0)).astype(np.int64)
    return (code | (sign << 3)).astype(np.uint8)


def e2m1_encode_sr(v, r16) -> np.ndarray:
    """Stochastic rounding of float32 ``v`` to E2M1 ([4BL] §"Why is the NVFP4 pretraining
    recipe not sufficient for RL?": stochastic rounding makes the quantiser approximately
    unbiased).

    Reading (the pages give no bit rule): with lo <= |v| < hi the neighbouring grid
    magnitudes, p = (|v| - lo) / (hi - lo) is exact in float32; the value rounds up to hi
    iff the uniform 16-bit integer ``r16`` satisfies r16 < p * 65536, so P(up) =
    ceil(p * 2^16) / 2^16.  |v| >= 6 saturates to 6.  Zero magnitude encodes as +0.
    """
    v = np.asarray(v, dtype=np.float32)
    r16 = np.asarray(r16, dtype=np.uint32)
    a = np.abs(v)
    lo = np.searchsorted(E2M1_MAGNITUDES.astype(np.float32), a, side="right") - 1
    lo = np.clip(lo, 0, 7)
    hi = np.minimum(lo + 1, 7)
    lo_v = E2M1_MAGNITUDES.astype(np.float32)[lo]
    gap = (E2M1_MAGNITUDES.astype(np.float32)[hi] - lo_v)
    with np.errstate(divide="ignore", invalid="ignore"):
        p = np.where(gap > 0, (a - lo_v) / np.where(gap > 0, gap, np.float32(1)), np.float32(0))
    p = p.astype(np.float32)
    up = r16.astype(np.float32) < p * np.float32(65536.0)
    code = np.where(up, hi, lo)
    code = np.where(a >= np.float32(E2M1_MAX), 7, code)
    sign = (np.signbit(v) & (code != 0)).astype(np.int64)
    return (code | (sign << 3)).astype(np.uint8)


# Midpoints between neighbouring E2M1 magnitudes: m_i separates code i from code i + 1.
E2M1_MIDPOINTS = (E2M1_MAGNITUDES[:-1] + E2M1_MAGNITUDES[1:]) / 2      # 0.25, 0.75, ..., 5


def e2m1_round_quotient(x, s) -> np.ndarray:
    """E2M1 code of round(x / s): [4BL] footnote 6's clip(round(w / s), -6, 6) with the
    quotient taken exactly, ties to the even code, saturating at 6.

    ``x`` holds float32 values (here BF16 inputs), ``s`` float32 scales > 0, both given as
    float64 (broadcastable).  The quotient is never formed: |x| / s > m holds exactly when
    |x| > m * s, and every product m * s of a midpoint (at most 3 significant bits) with
    a float32 scale (24 bits) is exact in float64, so each comparison is exact.  The
    magnitude code is the number of midpoints strictly below |x| / s; at a midpoint
    itself (|x| == m_i * s) the tie goes to the even code of i and i + 1.  Zero
    magnitude encodes as +0 (the reading of ``e2m1_encode_rne``).
    """
    x = np.asarray(x, dtype=np.float64)
    s = np.asarray(s, dtype=np.float64)
    a = np.abs(x)
    code = np.zeros(np.broadcast(a, s).shape, dtype=np.int64)
    for i, m in enumerate(E2M1_MIDPOINTS):
        t = m * s                                  # exact
        code += a > t
        if i % 2 == 1:                             # tie between odd i and even i + 1: round up
            code += a == t
    sign = (np.signbit(x) & (code != 0)).astype(np.int64)
    return (code | (sign << 3)).astype(np.uint8)


def e2m1_sr_quotient(x, s, r16) -> np.ndarray:
    """Stochastic rounding of the exact quotient q = |x| / s to E2M1 (the rule of
    ``e2m1_encode_sr`` applied to q instead of a rounded float32 value).

    With lo <= q < hi the neighbouring magnitudes and p = (q - lo) / (hi - lo), q rounds
    up iff r16 < p * 2^16, i.e. iff |x| > (lo + r16 * (hi - lo) / 2^16) * s.  That
    threshold has at most 19 significant bits and s 24, so the product is exact in
    float64; lo itself is found exactly as the largest magnitude G with G * s <= |x|.
    q >= 6 saturates at 6.  Zero magnitude encodes as +0.
    """
    x = np.asarray(x, dtype=np.float64)
    s = np.asarray(s, dtype=np.float64)
    r16 = np.asarray(r16, dtype=np.float64)
    a = np.abs(x)
    lo = np.zeros(np.broadcast(a, s, r16).shape, dtype=np.int64)
    for j in range(1, 8):
        lo += a >= E2M1_MAGNITUDES[j] * s           # exact: G has at most 2 significant bits
    hi = np.minimum(lo + 1, 7)
    gap = E2M1_MAGNITUDES[hi] - E2M1_MAGNITUDES[lo]
    thresh = (E2M1_MAGNITUDES[lo] + r16 * gap / 65536.0) * s     # exact
    code = np.where(lo >= 7, 7, lo + (a > thresh))
    sign = (np.signbit(x) & (code != 0)).astype(np.int64)
    return (code | (sign << 3)).astype(np.uint8)


def pack_e2m1(codes: np.ndarray) -> np.ndarray:
    """Pack codes [..., 2n] into bytes [..., n]: element 2i in the low nibble, 2i+1 in the
    high nibble (reading: the pages do not give a packing)."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] & 0xF) | ((c[..., 1::2] & 0xF) << 4)


def unpack_e2m1(packed: np.ndarray) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = p & 0xF
    out[..., 1::2] = p >> 4
    return out


# --------------------------------------------------------------------------- E4M3

def e4m3_decode(b) -> np.ndarray:
    """Value of each E4M3 byte, float64 (NaN for 0x7F / 0xFF)."""
    b = np.asarray(b, dtype=np.int64)
    s = (b >> 7) & 1
    e = (b >> 3) & 0xF
    m = b & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


_E4M3_FINITE_POS = e4m3_decode(np.arange(0x7F))   # codes 0x00..0x7E, strictly increasing


def e4m3_encode_rne_satfinite(t) -> np.ndarray:
    """Round non-negative float32 ``t`` to the nearest finite E4M3 value, ties to the even
    code, saturating at 448 (RNE with satfinite).  Returns bytes (sign bit 0)."""
    a = np.asarray(t, dtype=np.float32).astype(np.float64)
    if np.any(a < 0) or np.any(np.isnan(a)):
        raise ValueError("block scales are non-negative and finite")
    lo = np.searchsorted(_E4M3_FINITE_POS, a, side="right") - 1
    lo = np.clip(lo, 0, 0x7E)
    hi = np.minimum(lo + 1, 0x7E)
    d_lo = a - _E4M3_FINITE_POS[lo]
    d_hi = _E4M3_FINITE_POS[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(take_hi, hi, lo)
    code = np.where(a >= E4M3_MAX, 0x7E, code)
    return code.astype(np.uint8)


# --------------------------------------------------------------------------- BF16

def bf16_to_f32(bits) -> np.ndarray:
    """BF16 bit patterns (uint16) -> float32 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def bf16_round(v) -> np.ndarray:
    """Round float64 (or float32) values to BF16, nearest with ties to even, in one
    rounding from the given value (no intermediate float32 rounding).  Returns uint16
    bit patterns.  Overflow beyond the largest finite BF16 by half an ulp or more gives
    Inf, as IEEE round-to-nearest does."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        _, e = np.frexp(a)                     # a = m * 2^e, m in [0.5, 1)
        unbiased = np.maximum(e - 1, -126)     # BF16 exponent (subnormals share -126)
        q = np.exp2(unbiased - 7.0)            # spacing of BF16 values at that exponent
        r = np.rint(a / q) * q                 # exact division; rint ties to even
        r = np.where(a == 0, 0.0, r)
        r = np.where(r >= 2.0 ** 128, np.inf, r)
        r = np.where(np.isnan(a), np.nan, r)
    out = np.where(np.signbit(v), -r, r).astype(np.float32)
    return (out.view(np.uint32) >> 16).astype(np.uint16)


# --------------------------------------------------------------- scale-factor layout

def sf_swizzled_size(rows: int, sf_cols: int) -> int:
    """Bytes of the tiled scale-factor layout for ``rows`` x ``sf_cols`` E4M3 scales."""
    return ((rows + 127) // 128) * ((sf_cols + 3) // 4) * 512


def sf_swizzle_offset(r, c, sf_cols: int):
    """Byte offset of scale (row r, block-column c) in the 128x4 tiled layout used by
    Blackwell block-scaled tensor-core MMAs (reading: the pages give no layout; this is
    the layout the hardware's block-scaled MMA consumes, 128 rows x 4 scales per 512-byte
    tile, tiles row-block-major):

        tile (r // 128, c // 4) at ((r // 128) * ceil(sf_cols / 4) + c // 4) * 512,
        inside the tile (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4).
    """
    r = np.asarray(r, dtype=np.int64)
    c = np.asarray(c, dtype=np.int64)
    ct = (sf_cols + 3) // 4
    return ((r // 128) * ct + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + (c % 4)


def sf_swizzle(sf: np.ndarray) -> np.ndarray:
    """Row-major scales [rows, sf_cols] -> tiled byte buffer (padding bytes are 0)."""
    rows, cols = sf.shape
    out = np.zeros(sf_swizzled_size(rows, cols), dtype=np.uint8)
    rr, cc = np.meshgrid(np.arange(rows), np.arange(cols), indexing="ij")
    out[sf_swizzle_offset(rr, cc, cols)] = sf
    return out


def sf_unswizzle(buf: np.ndarray, rows: int, sf_cols: int) -> np.ndarray:
    """Tiled byte buffer -> row-major scales [rows, sf_cols]."""
    rr, cc = np.meshgrid(np.arange(rows), np.arange(sf_cols), indexing="ij")
    return np.asarray(buf, dtype=np.uint8)[sf_swizzle_offset(rr, cc, sf_cols)]

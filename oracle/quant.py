"""NVFP4 quantiser (oracle; test infrastructure only).

What it computes ([4BL] §Baseline and §"Why is the NVFP4 pretraining recipe not
sufficient for RL?"): for a BF16 tensor, one FP32 global scale per *scope*, one E4M3
scale per block of 16 consecutive values along the last (contraction) dimension, and one
4-bit E2M1 code per value.  The scope is

* the whole tensor for a standalone tensor and for a weight matrix ("a single FP32
  global scale"); an expert's weight matrix is its own tensor;
* one token row for activations ("each token computes its own FP32 activation scale
  across the hidden dimension"), which keeps a token's codes independent of the rest
  of the batch.

Scale arithmetic (reading: the pages fix the formats, not the arithmetic).  The scale
steps are single IEEE float32 operations, round to nearest even, in this order, so that
a second implementation reproduces every scale bit for bit:

    amax   = max |x| over the scope                        (exact)
    g      = amax / 2688                                    2688 = 6 * 448; g is the
                                                            decode-direction global scale
    per block b of 16 values, amax_b = max |x| over b:
    sf_b   = E4M3_rne_satfinite( amax_b / (6 * g) )         the block scale byte
    s_b    = decode(sf_b) * g                               effective decode scale

and each element's code is [4BL] footnote 6's Q = clip(round(x / s_b), -6, 6) on the E2M1
grid with the quotient x / s_b taken exactly (round to nearest, ties to the even code,
or stochastic rounding), so that DQ(code) = value(code) * decode(sf_b) * g.  The exact
quotient is decided by comparisons in float64 (formats.e2m1_round_quotient /
e2m1_sr_quotient), never by a rounded float32 quotient or reciprocal.  Degenerate
cases: g == 0 (an all-zero scope) gives sf_b = 0 and zero codes; s_b == 0 (a block
scale that encodes or multiplies out to zero) gives zero codes, sf_b still the encoded
byte when g > 0.
"""
from __future__ import annotations

import numpy as np

from . import formats as F
from . import philox

GLOBAL_DIVISOR = np.float32(2688.0)     # 6 (E2M1 max) * 448 (E4M3 max)
SIX = np.float32(6.0)
BLOCK = 16


def _f32(x):
    return np.asarray(x, dtype=np.float32)


def global_scale(amax) -> np.ndarray:
    """g = amax / 2688 in float32."""
    return (_f32(amax) / GLOBAL_DIVISOR).astype(np.float32)


def quantize_rows(x32: np.ndarray, g_rows: np.ndarray, rounding: str = "rne",
                  seed: int = 0, rng_offset: int = 0, row_base: int = 0,
                  total_cols: int | None = None):
    """Quantise float32 rows ``x32`` [rows, cols] given the global scale of each row's
    scope ``g_rows`` [rows] (float32).  Returns (codes [rows, cols] uint8 nibbles,
    sf [rows, cols/16] uint8).  ``row_base`` / ``total_cols`` give the row-major element
    index used by stochastic rounding."""
    rows, cols = x32.shape
    assert cols % BLOCK == 0
    nb = cols // BLOCK
    xb = x32.reshape(rows, nb, BLOCK)
    amax_b = np.max(np.abs(xb), axis=2).astype(np.float32)            # [rows, nb]
    g = _f32(g_rows).reshape(rows, 1)
    six_g = (SIX * g).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        t = np.where(g > 0, amax_b / np.where(g > 0, six_g, np.float32(1)), np.float32(0))
    t = t.astype(np.float32)
    sf = F.e4m3_encode_rne_satfinite(t)
    s = (F.e4m3_decode(sf).astype(np.float32) * g).astype(np.float32)  # exact decode, fp32 mul
    live = s > 0                                                          # [rows, nb]
    x64 = xb.astype(np.float64)
    s64 = np.where(live, s, np.float32(1)).astype(np.float64)[:, :, None]
    if rounding == "rne":
        codes = F.e2m1_round_quotient(x64, s64)
    elif rounding == "sr":
        tc = cols if total_cols is None else total_cols
        idx = (np.arange(rows, dtype=np.uint64)[:, None] + np.uint64(row_base)) * np.uint64(tc) \
            + np.arange(cols, dtype=np.uint64)[None, :]
        r16 = philox.sr_bits16(idx, seed, rng_offset).reshape(rows, nb, BLOCK)
        codes = F.e2m1_sr_quotient(x64, s64, r16)
    else:
        raise ValueError(rounding)
    codes = np.where(live[:, :, None], codes, np.uint8(0)).astype(np.uint8)
    sf = np.where(g > 0, sf, np.uint8(0)).astype(np.uint8)
    return codes.reshape(rows, cols), sf


def quantize(x_bits: np.ndarray, scope: str = "tensor", rounding: str = "rne", seed: int = 0,
             rng_offset: int = 0, global_scale_in=None, group_rows: int | None = None,
             chunk_rows: int = 2048):
    """Quantise BF16 bits [rows, cols] to NVFP4.

    scope: "tensor" (one g), "row" (one g per row), "group" (one g per ``group_rows``
    consecutive rows, e.g. one expert's weight matrix in a stacked [E*N, K] tensor).
    ``global_scale_in`` overrides the computed g (float32 array of the scope's shape).
    Returns dict(codes=[rows, cols] nibbles, packed=[rows, cols/2] bytes,
    sf=[rows, cols/16] row-major bytes, g=[n_scopes] float32).
    """
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    rows, cols = x_bits.shape
    x32 = F.bf16_to_f32(x_bits)
    if scope == "tensor":
        amax = np.max(np.abs(x32)) if x32.size else np.float32(0)
        g = global_scale(np.array([amax])) if global_scale_in is None else _f32(global_scale_in).reshape(1)
        g_rows = np.broadcast_to(g, (rows,))
    elif scope == "row":
        amax = np.max(np.abs(x32), axis=1) if cols else np.zeros(rows, np.float32)
        g = global_scale(amax) if global_scale_in is None else _f32(global_scale_in).reshape(rows)
        g_rows = g
    elif scope == "group":
        assert group_rows and rows % group_rows == 0
        amax = np.max(np.abs(x32).reshape(rows // group_rows, -1), axis=1)
        g = global_scale(amax) if global_scale_in is None else _f32(global_scale_in).reshape(-1)
        g_rows = np.repeat(g, group_rows)
    else:
        raise ValueError(scope)
    codes = np.empty((rows, cols), dtype=np.uint8)
    sf = np.empty((rows, cols // BLOCK), dtype=np.uint8)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        codes[r0:r1], sf[r0:r1] = quantize_rows(x32[r0:r1], g_rows[r0:r1], rounding, seed,
                                                rng_offset, row_base=r0, total_cols=cols)
    return dict(codes=codes, packed=F.pack_e2m1(codes), sf=sf, g=np.asarray(g, dtype=np.float32))


def dequantize(codes: np.ndarray, sf: np.ndarray, g_rows) -> np.ndarray:
    """DQ: value(code) * decode(sf) * g per element, float64 (exact: the three factors
    have 2 + 4 + 24 significant bits).  ``codes`` are nibbles [rows, cols]."""
    codes = np.asarray(codes)
    rows, cols = codes.shape
    scale = np.repeat(F.e4m3_decode(sf), BLOCK, axis=1)
    return F.e2m1_decode(codes) * scale * np.asarray(g_rows, dtype=np.float64).reshape(rows, 1)


def dq_unscaled(codes: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """value(code) * decode(sf), float64 (the operand the block-scaled product sees)."""
    return F.e2m1_decode(codes) * np.repeat(F.e4m3_decode(sf), BLOCK, axis=1)

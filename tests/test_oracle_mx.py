"""Pins for the MXFP8 oracle (oracle/mx.py).  The expected values do not come from the
oracle itself.  They come from:

* the BF16 exponent field, read straight from the bits;
* hand-derived values at the top E4M3 binade (step 32 from 256 to 448);
* torch's float32 -> float8_e4m3fn cast, an independent RNE implementation;
* lossless round trips of every E4M3 value;
* float64 matmul of the unquantised values, where the quantisation is lossless;
* brute force.
"""
import numpy as np
import pytest
import torch

from oracle import formats as F
from oracle import mx as X
from nvfp4_w4a4_moe_quantize_gb300 import synthetic as S


def _bits(v):
    """float64 values that are exact in BF16 -> uint16 BF16 bit patterns."""
    b = F.bf16_round(np.asarray(v, np.float64))
    assert np.array_equal(F.bf16_to_f32(b).astype(np.float64), np.asarray(v, np.float64))
    return b


def test_e8m0_decode():
    got = X.e8m0_decode(np.array([0, 1, 126, 127, 128, 254, 255]))
    np.testing.assert_array_equal(got[:6], [2.0 ** -127, 2.0 ** -126, 0.5, 1.0, 2.0, 2.0 ** 127])
    assert np.isnan(got[6])


def test_scale_byte_is_the_exponent_field_minus_8_for_every_bf16_value():
    """Every positive finite BF16 value and zero, alone in a block of 32.  The E8M0
    byte is max(exponent field - 8, 0): floor(log2 amax) = field - 127 for normal
    values, minus 8, clamped at b = 0.  Subnormals and zero have field 0."""
    vals = np.arange(0x0000, 0x7F80, dtype=np.uint16)          # +0 .. largest finite
    x = np.zeros((vals.size, 32), np.uint16)
    x[:, 5] = vals
    codes, sf = X.quantize(x)
    field = (vals.astype(np.int64) >> 7) & 0xFF
    np.testing.assert_array_equal(sf[:, 0], np.maximum(field - 8, 0))
    # the other 31 elements are zero and encode as +0
    assert not np.any(np.delete(codes, 5, axis=1))


def test_top_binade_codes_from_the_mantissa():
    """For a normal amax with field >= 8, amax / 2^e = (128 + m7) * 2 is in [256, 510]
    (m7 is the 7-bit mantissa).  E4M3 there steps by 32 from 256 (0x78) to 448 (0x7E).
    The code is 0x78 + min(rne(m7 / 16), 6): rounding to the nearest step, ties to the
    even mantissa, saturating at 448."""
    m7 = np.arange(128)
    for field in (8, 9, 100, 127 + 5, 254):
        x = np.zeros((128, 32), np.uint16)
        x[:, 0] = (field << 7) | m7
        codes, sf = X.quantize(x)
        q = np.rint(m7 / 16.0)                  # numpy rint: ties to even
        np.testing.assert_array_equal(codes[:, 0], 0x78 + np.minimum(q, 6))
        np.testing.assert_array_equal(sf[:, 0], field - 8)


def test_hand_values_at_the_top_binade():
    """t = x / 2^e with e = 0 (block amax in [256, 512)).  Grid near the top:
    384 (0x7C), 416 (0x7D), 448 (0x7E)."""
    cases = {256.0: 0x78, 272.0: 0x78, 288.0: 0x79, 400.0: 0x7C, 404.0: 0x7D, 432.0: 0x7E,
             448.0: 0x7E, 464.0: 0x7E, 480.0: 0x7E, 510.0: 0x7E}
    for t, code in cases.items():
        x = np.zeros((1, 32))
        x[0, 3] = t
        x[0, 7] = -t
        codes, sf = X.quantize(_bits(x))
        assert sf[0, 0] == 127, t
        assert codes[0, 3] == code and codes[0, 7] == code | 0x80, (t, hex(codes[0, 3]))


@pytest.mark.parametrize("e", [-127, -60, -8, 0, 20, 119])
def test_element_codes_match_torch_float8_cast(e):
    """Blocks whose amax fixes the shared exponent at e.  Every element's code equals
    torch's float8_e4m3fn cast of x / 2^e wherever |x / 2^e| <= 448.  That cast is RNE,
    so it serves as an independent encoder.  A zero magnitude is +0."""
    rng = np.random.default_rng(1000 + e)
    t = rng.standard_normal((64, 32)) * np.exp2(rng.integers(-12, 9, (64, 32)))
    t = np.clip(t, -440, 440)
    t[:, 0] = 256.0 + 32.0 * rng.integers(0, 6, 64)           # amax in [256, 448]: exponent e
    x = F.bf16_to_f32(F.bf16_round(t * 2.0 ** e)).astype(np.float64)
    codes, sf = X.quantize(F.bf16_round(x))
    if e > -127:
        np.testing.assert_array_equal(sf, e + 127)
    else:
        # e = -127 is the clamp: the byte is 0 whatever the amax below 2^-119
        np.testing.assert_array_equal(sf, 0)
    tt = (x * 2.0 ** (-e)).reshape(-1)
    ref = torch.from_numpy(tt.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ref = np.where((ref & 0x7F) == 0, 0, ref)
    np.testing.assert_array_equal(codes.reshape(-1), ref)


@pytest.mark.parametrize("s", [-100, -20, -8, 0, 10, 100])
def test_lossless_round_trip_of_every_e4m3_value(s):
    """Every finite E4M3 value (both signs) times 2^s, in blocks that each also hold
    448 * 2^s (so the shared exponent is s), quantises back to its own code.  It
    dequantises to itself in BF16 and float32."""
    codes_in = np.concatenate([np.arange(0x00, 0x7F), np.arange(0x81, 0xFF)]).astype(np.uint8)
    vals = F.e4m3_decode(codes_in) * 2.0 ** s
    n = -(-vals.size // 31)
    x = np.zeros((n, 32))
    xc = np.zeros((n, 32), np.uint8)
    flat = np.zeros(n * 31)
    flat[:vals.size] = vals
    fc = np.zeros(n * 31, np.uint8)
    fc[:vals.size] = codes_in
    x[:, 1:] = flat.reshape(n, 31)
    xc[:, 1:] = fc.reshape(n, 31)
    x[:, 0] = 448.0 * 2.0 ** s
    xc[:, 0] = 0x7E
    codes, sf = X.quantize(_bits(x))
    np.testing.assert_array_equal(sf[:, 0], s + 127)
    np.testing.assert_array_equal(codes, xc)
    np.testing.assert_array_equal(F.bf16_to_f32(X.dequantize(codes, sf, "bf16")).astype(np.float64), x)
    np.testing.assert_array_equal(X.dequantize(codes, sf, "f32").astype(np.float64), x)


def test_quantisation_error_bound():
    """|DQ(Q(x)) - x| <= 2^e * bound(t), with t = x / 2^e.  In E4M3's normal range the
    bound is half a step, 2^(floor(log2|t|) - 4).  Below 2^-6 it is 2^-10.  In the
    saturated range (448, 512) it is |t| - 448."""
    x_bits = S.bf16_bits(S.randn_bf16((256, 512), 3.0, seed=5))
    codes, sf = X.quantize(x_bits)
    x = F.bf16_to_f32(x_bits).astype(np.float64)
    dq = X.dequantize_exact(codes, sf)
    scale = np.repeat(X.e8m0_decode(sf), 32, axis=1)
    t = np.abs(x) / scale
    with np.errstate(divide="ignore"):
        half_step = np.where(t >= 2.0 ** -6, np.exp2(np.floor(np.log2(np.maximum(t, 1e-300))) - 4), 2.0 ** -10)
    bound = np.where(t > 448, t - 448, half_step) * scale
    assert np.all(np.abs(dq - x) <= bound)
    assert np.all(t < 512)


def test_dequantize_matches_torch_bf16_cast():
    """Random codes and scale bytes: the exact product is representable in float32 (at
    most 4 significant bits, within [2^-136, 2^136)).  torch's float32 -> bfloat16
    cast (RNE) of it is the single rounding that DQ to BF16 must give."""
    rng = np.random.default_rng(9)
    codes = rng.integers(0, 256, (64, 256)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x12                       # no NaN codes
    sf = rng.integers(0, 255, (64, 8)).astype(np.uint8)        # 0..254
    exact = X.dequantize_exact(codes, sf)
    f32 = X.dequantize(codes, sf, "f32")
    finite = np.abs(exact) < 2.0 ** 128
    np.testing.assert_array_equal(f32.astype(np.float64)[finite], exact[finite])
    ref = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(X.dequantize(codes, sf, "bf16"), ref)


def test_grouped_gemm_lossless_equals_float64_matmul():
    """Operands made of E4M3 grid values times 2^s, each block holding a 448 * 2^s.
    The quantisation is lossless, so the oracle GEMM equals the float64 matmul of the
    unquantised values, group by group."""
    rng = np.random.default_rng(11)
    grid = F.e4m3_decode(np.arange(0, 0x7F))[::7]
    E, N, K = 3, 16, 128
    counts = np.array([5, 0, 9], np.int32)
    offsets = np.array([0, 128, 128, 256], np.int32)
    a = rng.choice(grid, (256, K)) * rng.choice([-1, 1], (256, K)) * 2.0 ** -6
    a[:, ::32] = 448 * 2.0 ** -6
    w = rng.choice(grid, (E, N, K)) * rng.choice([-1, 1], (E, N, K)) * 2.0 ** -12
    w[:, :, ::32] = 448 * 2.0 ** -12
    ac, asf = X.quantize(_bits(a))
    wc, wsf = X.quantize(_bits(w.reshape(E * N, K)))
    D = X.grouped_gemm(ac, asf, wc.reshape(E, N, K), wsf.reshape(E, N, K // 32), offsets, counts)
    for e in range(E):
        r0, n = offsets[e], counts[e]
        np.testing.assert_array_equal(D[r0:r0 + n], a[r0:r0 + n] @ w[e].T)
    rows = np.concatenate([np.arange(o, o + c) for o, c in zip(offsets[:-1], counts)])
    outside = np.setdiff1d(np.arange(256), rows)
    assert not np.any(D[outside])


def test_grouped_gemm_brute_force_tiny():
    """Triple loop over DQ values: one expert, 3 x 2 output, K = 64."""
    a_bits = S.bf16_bits(S.randn_bf16((3, 64), seed=12))
    w_bits = S.bf16_bits(S.randn_bf16((2, 64), 0.1, seed=13))
    ac, asf = X.quantize(a_bits)
    wc, wsf = X.quantize(w_bits)
    D = X.grouped_gemm(ac, asf, wc[None], wsf[None], np.array([0, 3]), np.array([3]))
    for r in range(3):
        for n in range(2):
            acc = 0.0
            for k in range(64):
                va = F.e4m3_decode(ac[r, k]) * 2.0 ** (int(asf[r, k // 32]) - 127)
                vw = F.e4m3_decode(wc[n, k]) * 2.0 ** (int(wsf[n, k // 32]) - 127)
                acc += va * vw
            assert D[r, n] == pytest.approx(acc, rel=1e-15, abs=1e-300)

"""Pins for the oracle's NVFP4 quantiser and Philox generator: a hand-worked example,
published known-answer vectors, the dequantisation error bound, scope invariants and
stochastic-rounding statistics."""
import numpy as np
import pytest

from conftest import golden_path, read_golden
from oracle import formats as F
from oracle import philox
from oracle import quant as Q
from nvfp4_w4a4_moe_quantize_gb300 import synthetic as S


def _hex_list(s):
    return [int(t, 16) for t in s.split()]


def test_philox_known_answers():
    for line in open(golden_path("philox4x32_10_kat.txt")):
        if line.startswith("#") or not line.strip():
            continue
        w = [int(t, 16) for t in line.split()]
        out = philox.philox4x32_10(np.array(w[0:4]), np.array(w[4:6]))
        assert list(out) == w[6:10]


def test_sr_bits_layout():
    """Element i takes 16 bits of block i//8: word (i%8)//2, low half for even i."""
    seed, off = 0x1234_5678_9ABC, 7
    idx = np.arange(40)
    bits = philox.sr_bits16(idx, seed, off)
    for i in idx:
        j = off + i // 8
        out = philox.philox4x32_10(np.array([j & 0xFFFFFFFF, j >> 32, 0, 0]),
                                   np.array([seed & 0xFFFFFFFF, seed >> 32]))
        word = int(out[(i % 8) // 2])
        assert bits[i] == ((word >> (16 * (i % 2))) & 0xFFFF)


def test_worked_example():
    gd = read_golden("quant_worked_example.txt")
    x = np.array(_hex_list(gd["x_bf16"]), np.uint16).reshape(1, 32)
    for scope in ("row", "tensor"):
        q = Q.quantize(x, scope=scope)
        assert q["g"][0] == np.float32(float(gd["g"]))
        assert list(q["sf"][0]) == _hex_list(gd["sf"])
        assert list(q["codes"][0]) == _hex_list(gd["codes"])
        assert list(q["packed"][0]) == _hex_list(gd["packed"])


def test_dequant_error_bound_and_max_block_scale():
    """|x - DQ(Q(x))| <= s_b (the largest half-gap of the E2M1 grid is 1, between 4 and 6,
    and the satfinite clip costs less than that), and the scope's largest block gets
    scale 448."""
    x = S.outlier_channels_bf16(64, 512, seed=3)
    bits = S.bf16_bits(x)
    x32 = F.bf16_to_f32(bits).astype(np.float64)
    for scope in ("tensor", "row"):
        q = Q.quantize(bits, scope=scope)
        g_rows = np.broadcast_to(q["g"], (64,)) if scope == "tensor" else q["g"]
        dq = Q.dequantize(q["codes"], q["sf"], g_rows)
        s = np.repeat(F.e4m3_decode(q["sf"]), 16, axis=1) * np.asarray(g_rows, np.float64)[:, None]
        assert np.all(np.abs(x32 - dq) <= s * (1 + 1e-6))
        if scope == "tensor":
            assert q["sf"].max() == 0x7E
        else:
            assert np.all(q["sf"].max(axis=1) == 0x7E)


def test_row_scope_is_batch_independent():
    """[4BL]: a token's codes must not depend on the other tokens in the batch."""
    bits = S.bf16_bits(S.randn_bf16((96, 256), seed=5))
    full = Q.quantize(bits, scope="row")
    part = Q.quantize(bits[17:40], scope="row")
    assert np.array_equal(full["codes"][17:40], part["codes"])
    assert np.array_equal(full["sf"][17:40], part["sf"])
    assert np.array_equal(full["g"][17:40], part["g"])
    # the tensor scope does depend on the batch (why activations use the row scope)
    t_full = Q.quantize(bits, scope="tensor")
    t_part = Q.quantize(bits[17:40], scope="tensor")
    assert not np.array_equal(t_full["codes"][17:40], t_part["codes"])


def test_group_scope_equals_per_tensor_on_each_group():
    bits = S.bf16_bits(S.randn_bf16((3 * 32, 128), 0.02, seed=6))
    grp = Q.quantize(bits, scope="group", group_rows=32)
    for e in range(3):
        one = Q.quantize(bits[32 * e:32 * (e + 1)], scope="tensor")
        assert np.array_equal(grp["codes"][32 * e:32 * (e + 1)], one["codes"])
        assert grp["g"][e] == one["g"][0]


def test_zero_and_tiny_scopes():
    z = np.zeros((2, 32), np.uint16)
    q = Q.quantize(z, scope="row")
    assert not q["codes"].any() and not q["sf"].any() and not q["g"].any()
    # a row of the smallest BF16 subnormals (2^-133): g = fl32(2^-133 / 2688) is the
    # float32 subnormal 24 * 2^-149, t = 2^-133 / (6 g) = 455.1 saturates to sf = 448, and
    # s = 448 g = 10752 * 2^-149 exactly; x / s = 65536 / 10752 = 6.095 rounds to 6
    tiny = np.full((1, 32), 0x0001, np.uint16)
    q = Q.quantize(tiny, scope="row")
    assert q["g"][0] == np.float32(24 * 2.0 ** -149)
    assert np.all(q["sf"] == 0x7E)
    assert np.all(q["codes"] == 7)
    dq = Q.dequantize(q["codes"], q["sf"], q["g"])
    assert np.all(dq == 6 * 448 * 24 * 2.0 ** -149)


def test_sr_outputs_are_neighbours_and_grid_values_stay():
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(20000) * 3).astype(np.float32)
    r16 = rng.integers(0, 1 << 16, v.size).astype(np.uint32)
    c = F.e2m1_encode_sr(v, r16)
    val = F.e2m1_decode(c)
    a = np.minimum(np.abs(v).astype(np.float64), 6.0)
    lo = F.E2M1_MAGNITUDES[np.clip(np.searchsorted(F.E2M1_MAGNITUDES, a, "right") - 1, 0, 7)]
    hi = F.E2M1_MAGNITUDES[np.minimum(np.searchsorted(F.E2M1_MAGNITUDES, a, "right"), 7)]
    ok = (np.abs(val) == lo) | (np.abs(val) == hi)
    assert ok.all()
    grid = np.array([0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -4], np.float32)
    for r in (0, 1, 0xFFFF):
        assert np.array_equal(F.e2m1_decode(F.e2m1_encode_sr(grid, np.full(grid.size, r))), grid)


def test_sr_is_unbiased():
    """Mean of DQ over many seeds is within 4 sigma of the value ([4BL]: SR makes the
    quantiser approximately unbiased; P(up) carries at most 2^-16 bias)."""
    x = np.array([[0.3, 1.1, 2.2, 3.7, -4.9, 0.05, 5.5, -1.3] * 2], np.float32)
    bits = F.bf16_round(x.astype(np.float64))
    x32 = F.bf16_to_f32(bits).astype(np.float64)
    n = 4096
    acc = np.zeros_like(x32)
    acc2 = np.zeros_like(x32)
    g = np.float32(6.0 / 2688)             # a fixed global scale, so every seed shares s_b
    for seed in range(n):
        q = Q.quantize(bits, scope="tensor", rounding="sr", seed=seed, global_scale_in=[g])
        dq = Q.dequantize(q["codes"], q["sf"], [g])
        acc += dq
        acc2 += dq * dq
    mean = acc / n
    var = acc2 / n - mean ** 2
    sigma = np.sqrt(np.maximum(var, 1e-30) / n)
    # E[DQ] = x up to the 2^-16 threshold granularity
    assert np.all(np.abs(mean - x32) <= 4 * sigma + 1e-4 * np.abs(x32))


def test_rne_sr_differ_only_in_rounding():
    bits = S.bf16_bits(S.randn_bf16((16, 64), seed=9))
    a = Q.quantize(bits, scope="row", rounding="rne")
    b = Q.quantize(bits, scope="row", rounding="sr", seed=3)
    assert np.array_equal(a["sf"], b["sf"]) and np.array_equal(a["g"], b["g"])
    assert not np.array_equal(a["codes"], b["codes"])


# --------------------------------------------------------------------------- exact quotient
# [4BL] footnote 6: Q = clip(round(w / s), qmin, qmax).  The pins below compute round(x / s)
# with exact rational arithmetic (fractions.Fraction), independently of the oracle's
# float64 comparisons, on the inputs where a rounded quotient would decide differently.

import math  # noqa: E402
from fractions import Fraction  # noqa: E402

_GRID = [Fraction(v) for v in (0, 0.5, 1, 1.5, 2, 3, 4, 6)]


def _round_rational(q: Fraction) -> int:
    """Magnitude code of round(q) on the E2M1 grid, ties to the even code, clip at 6."""
    if q >= 6:
        return 7
    lo = max(i for i in range(8) if _GRID[i] <= q)
    if _GRID[lo] == q:
        return lo
    hi = lo + 1
    d_lo, d_hi = q - _GRID[lo], _GRID[hi] - q
    if d_lo != d_hi:
        return lo if d_lo < d_hi else hi
    return lo if lo % 2 == 0 else hi


def _scales(q):
    """Effective decode scale s_b = decode(sf_b) * g of every element, float32 (the
    oracle's own scale steps are pinned separately by the worked example)."""
    rows = q["codes"].shape[0]
    g = np.broadcast_to(np.asarray(q["g"], np.float32), (rows,)) if q["g"].size == 1 else q["g"]
    return np.repeat((F.e4m3_decode(q["sf"]).astype(np.float32) * g[:, None]).astype(np.float32), 16, axis=1)


def test_round_of_exact_quotient_at_structured_near_ties():
    """N(0,1) rows, row scope: g = amax / 2688 is rounded, so x / s lands within an ulp of
    an E2M1 midpoint for many x that share digits with the row max.  Every element on
    which the float32 reciprocal product fl(x * fl(1/s)) or the float32 quotient fl(x / s)
    rounds differently from the exact quotient, plus a random sample, must get the code
    of the exact rational round(x / s)."""
    rng = np.random.default_rng(0)
    bits = F.bf16_round(rng.standard_normal((1500, 2048)))
    q = Q.quantize(bits, scope="row")
    x = F.bf16_to_f32(bits)
    s = _scales(q)
    with np.errstate(divide="ignore", over="ignore", invalid="ignore"):
        v_rcp = (x * (np.float32(1) / s).astype(np.float32)).astype(np.float32)
        v_div = (x / s).astype(np.float32)
    suspects = np.flatnonzero((F.e2m1_encode_rne(v_rcp) != q["codes"]).ravel() |
                              (F.e2m1_encode_rne(v_div) != q["codes"]).ravel())
    assert suspects.size > 100          # the structured near-ties are there
    sample = rng.choice(x.size, 3000, replace=False)
    for i in np.concatenate([suspects, sample]):
        xv, sv = Fraction(float(x.flat[i])), Fraction(float(s.flat[i]))
        mag = _round_rational(abs(xv) / sv)
        want = mag | (8 if (xv < 0 and mag) else 0)
        assert q["codes"].flat[i] == want, (i, float(x.flat[i]), float(s.flat[i]))


def test_round_of_exact_quotient_hand_case():
    """A row with max 3.34375 gives g = fl32(3.34375 / 2688), rounded up.  The block holding
    1.4296875 gets sf = 192 (0x74), so s = 192 g and x = 0.8359375 = 3.34375 / 4 has
    x / s = 3.5 / (1 + d) with d > 0, just below the midpoint 3.5: the code is 5 (3.0),
    not the 6 (4.0) that a tie-to-even at a rounded 3.5 would give."""
    row = np.zeros(32, np.float64)
    row[0] = 3.34375
    row[16] = 1.4296875
    row[17] = 0.8359375
    q = Q.quantize(F.bf16_round(row[None, :]), scope="row")
    g = np.float32(np.float32(3.34375) / np.float32(2688))
    assert q["g"][0] == g and Fraction(float(g)) > Fraction(3.34375) / 2688
    assert q["sf"][0, 1] == 0x74
    s = Fraction(float(np.float32(np.float32(192) * g)))
    assert Fraction(0.8359375) / s < Fraction(7, 2)
    assert q["codes"][0, 17] == 5


def test_rne_exact_ties_go_to_even():
    """Quotients that are exact midpoints (x = m * s with s a power of two times an odd
    number) round to the even code; one BF16 ulp either side rounds away from the tie."""
    s = np.float32(0.375)                       # 3 * 2^-3
    for m, tie_code in [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6)]:
        x = m * float(s)
        xb = F.bf16_round(np.array([x]))
        assert F.bf16_to_f32(xb)[0] == x        # representable
        assert F.e2m1_round_quotient(np.array([x]), float(s))[0] == tie_code
        assert F.e2m1_round_quotient(np.array([-x]), float(s))[0] == (tie_code | 8 if tie_code else 0)
        up = float(F.bf16_to_f32(xb + np.uint16(1))[0])
        dn = float(F.bf16_to_f32(xb - np.uint16(1))[0])
        assert F.e2m1_round_quotient(np.array([up]), float(s))[0] == _round_rational(Fraction(up) / Fraction(float(s)))
        assert F.e2m1_round_quotient(np.array([dn]), float(s))[0] == _round_rational(Fraction(dn) / Fraction(float(s)))


@pytest.mark.parametrize("x, s", [(0.8359375, 0.2388393), (1.3, 0.7), (0.11, 0.3), (5.9, 1.0), (2.0, 1.0),
                                  (0.7421875, 0.125 * 3), (4.5, 0.8)])
def test_sr_rounds_up_for_exactly_ceil_p_of_the_2_16_draws(x, s):
    """Stochastic rounding over all 65,536 values of the 16 random bits: the number that
    round up is ceil(p * 2^16) with p = (q - lo) / (hi - lo) of the exact quotient q = x / s
    (rational arithmetic), and every result is lo or hi."""
    xs = float(F.bf16_to_f32(F.bf16_round(np.array([x])))[0])
    ss = float(np.float32(s))
    r16 = np.arange(65536)
    codes = F.e2m1_sr_quotient(np.full(65536, xs), ss, r16)
    q = Fraction(xs) / Fraction(ss)
    lo = max(i for i in range(8) if _GRID[i] <= min(q, Fraction(6)))
    if lo == 7:
        assert np.all(codes == 7)
        return
    p = (q - _GRID[lo]) / (_GRID[lo + 1] - _GRID[lo])
    n_up = int(np.sum(codes == lo + 1))
    assert n_up == math.ceil(p * 65536)
    assert np.all((codes == lo) | (codes == lo + 1))
    # the draws that round up are exactly the smallest ones
    assert np.all(codes[:n_up] == lo + 1) and np.all(codes[n_up:] == lo)

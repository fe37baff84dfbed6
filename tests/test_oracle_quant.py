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
    # a row of the smallest BF16 subnormals: g and the scales underflow, codes decode to 0
    tiny = np.full((1, 32), 0x0001, np.uint16)
    q = Q.quantize(tiny, scope="row")
    dq = Q.dequantize(q["codes"], q["sf"], q["g"])
    assert np.all(np.isfinite(dq))


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
    # E[DQ] = s_b * (x * fl(1/s_b)) up to the 2^-16 threshold granularity
    assert np.all(np.abs(mean - x32) <= 4 * sigma + 1e-4 * np.abs(x32))


def test_rne_sr_differ_only_in_rounding():
    bits = S.bf16_bits(S.randn_bf16((16, 64), seed=9))
    a = Q.quantize(bits, scope="row", rounding="rne")
    b = Q.quantize(bits, scope="row", rounding="sr", seed=3)
    assert np.array_equal(a["sf"], b["sf"]) and np.array_equal(a["g"], b["g"])
    assert not np.array_equal(a["codes"], b["codes"])

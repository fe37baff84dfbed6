"""Pins for the oracle's MoE expert block: hand-worked routing and grouping examples,
brute force on tiny inputs, exact integer GEMMs, an independent float64 library GEMM,
mpmath references for SwiGLU and the combine, and an end-to-end case that is exact at
every stage."""
from fractions import Fraction

import numpy as np
import pytest
import torch

from conftest import read_golden
from oracle import formats as F
from oracle import moe as M
from oracle import quant as Q
from nvfp4_w4a4_moe_quantize_gb300 import synthetic as S


def _groups(s, conv=float):
    return [[conv(t) for t in g.split()] for g in s.split("|")]


# ------------------------------------------------------------------ routing

def test_routing_worked_example():
    gd = read_golden("routing_worked_example.txt")
    logits = np.array(_groups(gd["logits"]), np.float32)
    ids, w = M.route_topk(logits, 2)
    assert ids.tolist() == _groups(gd["ids"], int)
    np.testing.assert_allclose(w, np.array(_groups(gd["weights"])), rtol=1e-7)


def test_routing_brute_force():
    rng = np.random.default_rng(0)
    for renorm in (True, False):
        for T, E, k in [(7, 5, 2), (16, 8, 3), (9, 16, 8)]:
            logits = rng.integers(-3, 4, (T, E)).astype(np.float32)   # many ties
            ids, w = M.route_topk(logits, k, renormalize=renorm)
            for t in range(T):
                order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k]
                assert ids[t].tolist() == order
                ex = np.exp(logits[t].astype(np.float64) - logits[t].max())
                den = ex[order].sum() if renorm else ex.sum()
                np.testing.assert_allclose(w[t], ex[order] / den, rtol=1e-7)


# ------------------------------------------------------------------ permute

def test_permute_worked_example():
    gd = read_golden("permute_worked_example.txt")
    ids = np.array(_groups(gd["ids"], int))
    p = M.permute(ids, 3, align=int(gd["align"]))
    for key in ("counts", "offsets", "padded_offsets", "perm"):
        assert p[key].tolist() == [int(t) for t in gd[key].split()], key
    assert p["inv"].tolist() == _groups(gd["inv"], int)


def test_permute_brute_force():
    rng = np.random.default_rng(1)
    for T, E, k, align in [(50, 6, 2, 4), (200, 16, 4, 128), (3, 8, 3, 8), (0, 4, 2, 128)]:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]) if T else np.zeros((0, k), int)
        p = M.permute(ids, E, align=align)
        slot = 0
        inv = np.full((T, k), -1)
        perm = []
        for e in range(E):
            start = slot
            for t in range(T):
                for j in range(k):
                    if ids[t, j] == e:
                        inv[t, j] = slot
                        perm.append(t)
                        slot += 1
            while (slot - start) % align:
                perm.append(-1)
                slot += 1
        assert p["inv"].tolist() == inv.tolist()
        assert p["perm"].tolist() == perm


def test_permute_rejects_bad_ids():
    with pytest.raises(ValueError):
        M.permute(np.array([[0, 5]]), 4)


# ------------------------------------------------------------------ GEMM

def _e2m1_value(c):
    mag = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3),
           Fraction(4), Fraction(6)][c & 7]
    return -mag if c & 8 else mag


E4M3_SPEC = {0x38: Fraction(1), 0x30: Fraction(1, 2), 0x40: Fraction(2), 0x48: Fraction(4),
             0x3C: Fraction(3, 2), 0x08: Fraction(1, 64), 0x78: Fraction(256)}   # spec values


def test_grouped_gemm_exact_brute_force():
    """Small integer-valued case computed with exact rational arithmetic, using only code
    values from the E2M1 table and scale values from the E4M3 specification."""
    rng = np.random.default_rng(2)
    E, N, K = 3, 5, 64
    counts = np.array([2, 0, 3])
    padded = np.array([0, 4, 4, 8])
    Mtot = 8
    a_codes = rng.integers(0, 16, (Mtot, K)).astype(np.uint8)
    sf_keys = list(E4M3_SPEC)
    a_sf = rng.choice(sf_keys, (Mtot, K // 16)).astype(np.uint8)
    a_g = np.array([1.0, 0.5, 0, 0, 2.0, 0.25, 1.5, 0], np.float32)
    b_codes = rng.integers(0, 16, (E, N, K)).astype(np.uint8)
    b_sf = rng.choice(sf_keys, (E, N, K // 16)).astype(np.uint8)
    b_g = np.array([0.125, 3.0, 1.0], np.float32)
    D = M.grouped_gemm(a_codes, a_sf, a_g, b_codes, b_sf, b_g, padded, counts)
    for e in range(E):
        for r in range(int(padded[e]), int(padded[e]) + int(counts[e])):
            for n in range(N):
                acc = Fraction(0)
                for kk in range(K):
                    acc += (_e2m1_value(a_codes[r, kk]) * E4M3_SPEC[int(a_sf[r, kk // 16])]
                            * _e2m1_value(b_codes[e, n, kk]) * E4M3_SPEC[int(b_sf[e, n, kk // 16])])
                expect = acc * Fraction(float(a_g[r])) * Fraction(float(b_g[e]))
                assert D[r, n] == float(expect)
    assert np.isnan(D[2]).all() and np.isnan(D[7]).all()


def test_grouped_gemm_matches_torch_float64():
    x = S.bf16_bits(S.randn_bf16((64, 256), seed=11))
    w = S.bf16_bits(S.randn_bf16((2 * 32, 256), 0.02, seed=12))
    qa = Q.quantize(x, scope="row")
    qb = Q.quantize(w, scope="group", group_rows=32)
    D = M.grouped_gemm(qa["codes"], qa["sf"], qa["g"], qb["codes"].reshape(2, 32, 256),
                       qb["sf"].reshape(2, 32, 16), qb["g"], np.array([0, 32, 64]), np.array([30, 17]))
    ta = torch.from_numpy(Q.dequantize(qa["codes"], qa["sf"], qa["g"]))
    tb = torch.from_numpy(Q.dequantize(qb["codes"], qb["sf"], np.repeat(qb["g"], 32)))
    ref0 = (ta[:30] @ tb[:32].T).numpy()
    ref1 = (ta[32:49] @ tb[32:].T).numpy()
    np.testing.assert_allclose(D[:30], ref0, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(D[32:49], ref1, rtol=1e-12, atol=1e-15)


# ------------------------------------------------------------------ SwiGLU / combine

def _bf16_nearest_mp(mpmath, exact):
    """Nearest BF16 to an mpmath value, ties to even, by searching neighbours."""
    f32 = np.float32(float(exact))
    b = int((np.array([f32]).view(np.uint32)[0] >> 16))
    cands = []
    for c in range(b - 2, b + 3):
        c &= 0xFFFF
        v = F.bf16_to_f32(np.array([c], np.uint16))[0]
        if np.isfinite(v):
            cands.append((abs(mpmath.mpf(float(v)) - exact), c % 2, c, float(v)))
    best = min(x[0] for x in cands)
    win = sorted([x for x in cands if x[0] == best], key=lambda x: x[1])
    return win[0][2], win[0][3]


def test_swiglu_against_mpmath():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 60
    rng = np.random.default_rng(4)
    I = 64
    d = F.bf16_round(rng.standard_normal((8, 2 * I)) * 3)
    d[0, 0] = 0x0000                      # gate 0 -> h = 0
    d[0, 1] = 0xC2C8                      # gate -100 -> tiny
    h = M.swiglu(d, I)
    dv = F.bf16_to_f32(d)
    for r in range(8):
        for c in range(I):
            g, u = mpmath.mpf(float(dv[r, c])), mpmath.mpf(float(dv[r, I + c]))
            exact = g / (1 + mpmath.exp(-g)) * u
            if exact == 0:
                assert F.bf16_to_f32(h[r:r + 1, c:c + 1])[0, 0] == 0
                continue
            code, _ = _bf16_nearest_mp(mpmath, exact)
            if (code & 0x7FFF) == 0:
                assert (h[r, c] & 0x7FFF) == 0
            else:
                assert h[r, c] == code, (r, c)


def test_swiglu_backward_against_mpmath_derivative():
    """The SwiGLU backward against mpmath: dgate = dh * d/dg[silu(g) u], the derivative
    taken numerically by mpmath.diff of the forward expression (not the closed form the
    oracle uses), and dup = dh * silu(g).  Both are rounded once to BF16."""
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    rng = np.random.default_rng(6)
    I = 16
    d = F.bf16_round(rng.standard_normal((6, 2 * I)) * 3)
    d[0, 0] = 0x0000                      # g = 0: dgate = dh * u / 2, dup = 0
    d[0, 1] = 0x41F0                      # g = 30: silu' ~ 1
    d[0, 2] = 0xC1F0                      # g = -30: silu' ~ -29 e^-30
    dh = F.bf16_round(rng.standard_normal((6, I)))
    out = M.swiglu_backward(d, dh, I)
    dv, dhv = F.bf16_to_f32(d), F.bf16_to_f32(dh)
    for r in range(6):
        for c in range(I):
            g, u, gh = (mpmath.mpf(float(dv[r, c])), mpmath.mpf(float(dv[r, I + c])),
                        mpmath.mpf(float(dhv[r, c])))
            dg = gh * mpmath.diff(lambda z: z / (1 + mpmath.exp(-z)) * u, g)
            du = gh * g / (1 + mpmath.exp(-g))
            for col, exact in ((c, dg), (I + c, du)):
                if exact == 0:
                    assert (out[r, col] & 0x7FFF) == 0, (r, col)
                    continue
                code, _ = _bf16_nearest_mp(mpmath, exact)
                assert out[r, col] == code, (r, col)
    # g = 0: silu'(0) = 1/2, silu(0) = 0
    g0 = F.bf16_to_f32(out[0:1, 0:1])[0, 0]
    assert g0 == F.bf16_to_f32(F.bf16_round(np.array([[0.5 * dhv[0, 0] * dv[0, I]]])))[0, 0]
    assert (out[0, I] & 0x7FFF) == 0


def test_expert_wgrad_brute_force_and_exact_case():
    """Expert wgrad against a brute-force triple loop over the dequantised operands (tiny
    sizes).  Also an exact case: E2M1 grid values times 448 * 2^-k, with every 16-token
    block reaching 6 * 448 * 2^-k, quantise losslessly (g = 2^-k, block scales 448), so dW
    equals the float64 product of the unquantised values."""
    rng = np.random.default_rng(13)
    counts = [3, 0, 17]
    N, H = 16, 16
    dy = F.bf16_round(rng.standard_normal((sum(counts), N)) * 1e-2)
    x = F.bf16_round(rng.standard_normal((sum(counts), H)))
    dw, ops = M.expert_wgrad(dy, x, counts, rounding_dy="sr", seed=4)
    assert dw.shape == (3, N, H)
    assert not np.any(dw[1])                            # an expert with no tokens
    qa, qb = ops[2]
    a = Q.dq_unscaled(qa["codes"], qa["sf"]) * qa["g"][0]
    b = Q.dq_unscaled(qb["codes"], qb["sf"]) * qb["g"][0]
    for n_ in range(N):
        for h_ in range(H):
            acc = sum(a[n_, t] * b[h_, t] for t in range(a.shape[1]))
            assert dw[2, n_, h_] == pytest.approx(acc, rel=1e-12, abs=1e-300)
    # exact case: one expert, 32 tokens, RNE on both operands; amax = 2688 * 2^-k makes
    # g = 2^-k and every block scale 448, so the quantisation is lossless
    grid = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0])
    s_dy, s_x = 448 * 2.0 ** -14, 448 * 2.0 ** -8
    dyv = rng.choice(grid, (32, N)) * rng.choice([-1, 1], (32, N)) * s_dy
    xv = rng.choice(grid, (32, H)) * rng.choice([-1, 1], (32, H)) * s_x
    dyv[0::16, :] = 6 * s_dy                            # each 16-token block reaches 6 * scale
    xv[0::16, :] = 6 * s_x
    dw2, _ = M.expert_wgrad(F.bf16_round(dyv), F.bf16_round(xv), [32], rounding_dy="rne")
    np.testing.assert_array_equal(dw2[0], dyv.T @ xv)


def test_combine_against_mpmath():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 60
    rng = np.random.default_rng(5)
    T, k, H, Mr = 6, 3, 16, 24
    y = F.bf16_round(rng.standard_normal((Mr, H)))
    inv = np.stack([rng.permutation(Mr)[:k] for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    out = M.combine(y, inv, w)
    yv = F.bf16_to_f32(y)
    for t in range(T):
        for c in range(H):
            exact = sum(mpmath.mpf(float(w[t, j])) * mpmath.mpf(float(yv[inv[t, j], c])) for j in range(k))
            code, _ = _bf16_nearest_mp(mpmath, exact)
            assert out[t, c] == code


# ------------------------------------------------------------------ end to end

def _exact_case():
    """Inputs whose quantisation is lossless and whose GEMM sums are small dyadic
    rationals, so every stage up to the gate/up output is exact.

    Each x value is an E2M1 grid value times s = 448 * 2^-11 and every 16-block holds
    6 * s = 1.3125, so the row scale is g = 1.3125 / 2688 = 2^-11 exactly, every block
    scale is 448 and DQ(Q(x)) = x.  The weights do the same with g = 2^-13."""
    T, H, I, E, k = 16, 64, 64, 2, 2
    rng = np.random.default_rng(6)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -2, -3, -4, -6])
    s_x, s_w = 448 * 2.0 ** -11, 448 * 2.0 ** -13
    xv = rng.choice(grid, (T, H)) * s_x
    xv[:, ::16] = 6 * s_x
    w13 = rng.choice(grid, (E, 2 * I, H)) * s_w
    w13[:, :, ::16] = 6 * s_w
    w2 = rng.choice(grid, (E, H, I)) * s_w
    w2[:, :, ::16] = 6 * s_w
    ids = np.array([[t % E, (t + 1) % E] for t in range(T)], np.int32)
    topk_w = np.full((T, k), 0.5, np.float32)
    return (F.bf16_round(xv), ids, topk_w, F.bf16_round(w13), F.bf16_round(w2), xv, w13)


def test_forward_exact_case_lossless_quantisation_and_exact_gemm():
    x, ids, tw, w13, w2, xv, w13v = _exact_case()
    r = M.moe_forward(x, ids, tw, w13, w2)
    # lossless: DQ(Q(x)) == x exactly for every token
    q = r["aq"]["token_q"]
    assert np.array_equal(Q.dequantize(q["codes"], q["sf"], q["g"]), xv)
    pw = r["prepared"]
    for e in range(2):
        g_e = np.repeat(pw["w13_g"][e], 128)
        assert np.array_equal(Q.dequantize(pw["w13_codes"][e], pw["w13_sf"][e], g_e), w13v[e])
    # gate/up: exact rational products equal the float64 GEMM bit for bit
    pi = r["perm"]
    for slot in np.nonzero(pi["perm"] >= 0)[0][:6]:
        t = pi["perm"][slot]
        e = int(np.searchsorted(pi["padded_offsets"], slot, side="right") - 1)
        for n in (0, 5, 77):
            exact = sum(Fraction(float(xv[t, kk])) * Fraction(float(w13v[e, n, kk])) for kk in range(64))
            assert r["d"][slot, n] == float(exact)


def test_forward_batched_equals_token_by_token():
    shape = S.WORKLOADS["tiny"]
    x, logits, w13, w2 = S.moe_inputs(shape, seed=0)
    xb, w13b, w2b = S.bf16_bits(x[:40]), S.bf16_bits(w13), S.bf16_bits(w2)
    ids, tw = M.route_topk(logits[:40].numpy(), shape.k)
    r = M.moe_forward(xb, ids, tw, w13b, w2b)
    toks = [0, 7, 39]
    per = M.moe_forward_tokens(xb, ids, tw, r["prepared"], toks)
    assert np.array_equal(per, r["out"][toks])


def test_forward_row_invariance():
    """A token's output bits do not depend on the rest of the batch ([LBP] §The
    Cross-Engine Alignment Problem; [4BL] per-token scales)."""
    shape = S.WORKLOADS["tiny"]
    x, logits, w13, w2 = S.moe_inputs(shape, seed=1)
    xb, w13b, w2b = S.bf16_bits(x[:64]), S.bf16_bits(w13), S.bf16_bits(w2)
    ids, tw = M.route_topk(logits[:64].numpy(), shape.k)
    full = M.moe_forward(xb, ids, tw, w13b, w2b)
    part = M.moe_forward(xb[10:30], ids[10:30], tw[10:30], w13b, w2b, prepared=full["prepared"])
    assert np.array_equal(full["out"][10:30], part["out"])

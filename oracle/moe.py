"""MoE expert block over NVFP4 operands (oracle; test infrastructure only).

The block the pages build their speed-up on ([LBP] §"What W4A4 GEMM Actually Changes":
native W4A4 GEMM on the expert layers; [4BL] §"Why is the NVFP4 pretraining recipe not
sufficient for RL?", baseline recipe: only the MoE layers are quantised; [miniTE]
§Development: NVFP4 kernels, scaling and grouped GEMMs):

    route      top-k experts per token from router logits
    permute    group the (token, slot) pairs by expert
    quantise   x per token row (per-token FP32 scale) -> NVFP4
    gate/up    grouped W4A4 GEMM   D = DQ(x_q) DQ(W13_e)^T       -> BF16
    SwiGLU     h = silu(gate) * up                              -> BF16
    requant    h per routed row -> NVFP4
    down       grouped W4A4 GEMM   y = DQ(h_q) DQ(W2_e)^T        -> BF16
    combine    out[t] = sum_j w[t, j] * y[slot(t, j)]           -> BF16

Readings taken where the pages are silent (each repeated at its function):
routing weights are the softmax renormalised over the chosen k; slots are grouped by
expert ascending and, inside an expert, by token ascending, each expert's group starting
at a multiple of 128 rows; W13 holds the gate rows first and the up rows second; the
pipeline rounds to BF16 exactly where an unfused pipeline crosses a kernel boundary
(D, h, y, out), each from the exact (float64) value.
"""
from __future__ import annotations

import numpy as np

from . import formats as F
from . import quant as Q

ROW_ALIGN = 128


# --------------------------------------------------------------------------- routing

def route_topk(logits: np.ndarray, k: int, renormalize: bool = True):
    """Top-k experts per token, in descending logit order, ties to the lower expert id;
    weights = softmax over the chosen k (renormalize=True) or the full softmax
    probabilities of the chosen experts (renormalize=False), computed in float64 and
    returned as float32.  Softmax is monotone, so the ids come from the logits directly.
    """
    logits = np.asarray(logits, dtype=np.float32)
    order = np.argsort(-logits, axis=1, kind="stable")[:, :k]
    top = np.take_along_axis(logits, order, axis=1).astype(np.float64)
    m = top[:, :1]
    e = np.exp(top - m)
    if renormalize:
        w = e / e.sum(axis=1, keepdims=True)
    else:
        mall = logits.astype(np.float64).max(axis=1, keepdims=True)
        w = np.exp(top - mall) / np.exp(logits.astype(np.float64) - mall).sum(axis=1, keepdims=True)
    return order.astype(np.int32), w.astype(np.float32)


# --------------------------------------------------------------------------- permute

def permute(topk_ids: np.ndarray, num_experts: int, align: int = ROW_ALIGN):
    """Group the T*k (token, j) entries by expert.

    Returns dict(counts [E], offsets [E+1] (unpadded exclusive scan), padded_offsets
    [E+1] (each expert's rows start at a multiple of ``align``), inv [T, k] = slot of
    (t, j), perm [padded_offsets[E]] = token of each slot or -1 for padding).
    Slot order (reading): experts ascending; inside an expert, tokens ascending -- a
    stable counting sort of the row-major flattened ids, since a token names an expert
    at most once.
    """
    ids = np.asarray(topk_ids, dtype=np.int64)
    T, k = ids.shape
    flat = ids.reshape(-1)
    if flat.size and (flat.min() < 0 or flat.max() >= num_experts):
        raise ValueError("expert id out of range")
    counts = np.bincount(flat, minlength=num_experts).astype(np.int64)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    padded = np.concatenate([[0], np.cumsum((counts + align - 1) // align * align)])
    order = np.argsort(flat, kind="stable")                  # entries grouped by expert
    rank = np.empty_like(order)
    rank[order] = np.arange(flat.size) - offsets[flat[order]]  # rank inside the expert
    slot = padded[flat] + rank
    perm = np.full(int(padded[-1]), -1, dtype=np.int64)
    perm[slot] = np.arange(flat.size) // k
    return dict(counts=counts.astype(np.int32), offsets=offsets.astype(np.int32),
                padded_offsets=padded.astype(np.int32), inv=slot.reshape(T, k).astype(np.int32),
                perm=perm.astype(np.int32))


# --------------------------------------------------------------------------- GEMM

def grouped_gemm(a_codes, a_sf, a_g, b_codes, b_sf, b_g, padded_offsets, counts):
    """D[r, n] = gA[r] * gB[e] * sum_kk value(a)[r,kk] sf_a[r,kk/16] value(b_e)[n,kk] sf_b[n,kk/16]
    for every row r of expert e's group (rows padded_offsets[e] .. + counts[e]); float64.

    a_codes [M, K] nibbles, a_sf [M, K/16], a_g [M]; b_codes [E, N, K], b_sf [E, N, K/16],
    b_g [E].  Rows outside every group are NaN.  The products of the exact float64
    dequantised operands are summed by numpy's float64 matmul (a library primitive; the
    rounding error is ~1e-16 relative, far below the kernel's float32 accumulation).
    """
    M, K = a_codes.shape
    E, N, _ = b_codes.shape
    out = np.full((M, N), np.nan)
    for e in range(E):
        r0 = int(padded_offsets[e])
        n = int(counts[e])
        if n == 0:
            continue
        A = Q.dq_unscaled(a_codes[r0:r0 + n], a_sf[r0:r0 + n])
        B = Q.dq_unscaled(b_codes[e], b_sf[e])
        acc = A @ B.T
        scale = np.asarray(a_g[r0:r0 + n], dtype=np.float64)[:, None] * np.float64(b_g[e])
        out[r0:r0 + n] = acc * scale
    return out


def expert_wgrad(dy_bits: np.ndarray, x_bits: np.ndarray, counts, rounding_dy: str = "sr", seed: int = 0):
    """Weight gradient of every expert in W4A4: dW_e[n, h] = sum over expert e's tokens t of
    dY[t, n] * X[t, h], with both operands quantised along the tokens (the contraction) --
    dY_e^T and X_e^T each as one tensor (one FP32 global scale per expert matrix, blocks of
    16 consecutive tokens), the gradient with stochastic rounding and seed ``seed + e``, the
    activations with RNE -- and each expert's token count zero-padded to a multiple of 256
    ([4BL] §"Why is the NVFP4 pretraining recipe not sufficient for RL?": stochastic
    rounding for gradients; the transposed quantisation of the backward's operands).

    dy_bits [T, N] and x_bits [T, H] hold the tokens grouped by expert (counts[e] rows
    each, in order).  Returns dW [E, N, H] in float64 (the exact GEMM of the dequantised
    operands) and the per-expert operands (codes, sf, g of dY_e^T and X_e^T)."""
    counts = [int(c) for c in counts]
    N, H = dy_bits.shape[1], x_bits.shape[1]
    out = np.zeros((len(counts), N, H))
    ops = []
    r = 0
    for e, n in enumerate(counts):
        tp = max(256, (n + 255) // 256 * 256)
        dyt = np.zeros((N, tp), np.uint16)
        xt = np.zeros((H, tp), np.uint16)
        dyt[:, :n] = dy_bits[r:r + n].T
        xt[:, :n] = x_bits[r:r + n].T
        qa = Q.quantize(dyt, scope="tensor", rounding=rounding_dy, seed=seed + e)
        qb = Q.quantize(xt, scope="tensor")
        a = Q.dq_unscaled(qa["codes"], qa["sf"]) * np.float64(qa["g"][0])
        b = Q.dq_unscaled(qb["codes"], qb["sf"]) * np.float64(qb["g"][0])
        out[e] = a @ b.T
        ops.append((qa, qb))
        r += n
    return out, ops


def gemm_rows(a_codes_rows, a_sf_rows, a_g_rows, b_codes_e, b_sf_e, b_g_e):
    """The same product for a few rows against one expert's matrix (sampled checks)."""
    A = Q.dq_unscaled(a_codes_rows, a_sf_rows)
    B = Q.dq_unscaled(b_codes_e, b_sf_e)
    return (A @ B.T) * (np.asarray(a_g_rows, np.float64)[:, None] * np.float64(b_g_e))


# --------------------------------------------------------------------------- SwiGLU

def silu(z: np.ndarray) -> np.ndarray:
    """silu(z) = z / (1 + exp(-z)) in float64 (exp overflow for z < -709 gives -0)."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu(d_bits: np.ndarray, inter: int) -> np.ndarray:
    """h = BF16(silu(gate) * up) with gate = columns [0, I) and up = columns [I, 2I) of the
    BF16 gate/up output (reading: the pages do not give the column order).  The product
    is formed in float64 and rounded once to BF16."""
    d = F.bf16_to_f32(d_bits).astype(np.float64)
    gate, up = d[:, :inter], d[:, inter:2 * inter]
    return F.bf16_round(silu(gate) * up)


def swiglu_backward(d_bits: np.ndarray, dh_bits: np.ndarray, inter: int) -> np.ndarray:
    """Gradient of h = silu(gate) * up for the backward pass, with gate and up read from the
    BF16 gate/up output as in ``swiglu`` and dh the BF16 gradient of h:

        dgate = dh * up * silu'(gate),  silu'(g) = s(g) * (1 + g * (1 - s(g))),  s = sigmoid
        dup   = dh * silu(gate)

    formed in float64 and each rounded once to BF16.  Returns the BF16 bits of
    [dgate | dup], shaped like d_bits (columns [0, I) and [I, 2I)).  Reading: the pages
    do not give the backward's precision; the forward's rule (float64, one rounding) is
    kept."""
    d = F.bf16_to_f32(d_bits).astype(np.float64)
    dh = F.bf16_to_f32(dh_bits).astype(np.float64)
    g, u = d[:, :inter], d[:, inter:2 * inter]
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-g))
    dsilu = s * (1.0 + g * (1.0 - s))
    out = np.empty_like(d)
    out[:, :inter] = dh * u * dsilu
    out[:, inter:2 * inter] = dh * (g * s)
    return F.bf16_round(out)


# --------------------------------------------------------------------------- combine

def combine(y_bits: np.ndarray, inv: np.ndarray, topk_w: np.ndarray) -> np.ndarray:
    """out[t] = BF16( sum_j w[t, j] * y[inv[t, j]] ), float64 sum, one rounding."""
    y = F.bf16_to_f32(y_bits).astype(np.float64)
    w = np.asarray(topk_w, dtype=np.float32).astype(np.float64)
    acc = np.zeros((inv.shape[0], y.shape[1]))
    for j in range(inv.shape[1]):
        acc += w[:, j:j + 1] * y[inv[:, j]]
    return F.bf16_round(acc)


# --------------------------------------------------------------------------- forward

def prepare_weights(w13_bits: np.ndarray, w2_bits: np.ndarray):
    """Quantise each expert's W13 [2I, H] and W2 [H, I] as its own tensor (one FP32 global
    scale per expert matrix: [4BL]'s weight recipe applied to each expert's weight)."""
    E, N13, H = w13_bits.shape
    _, N2, I = w2_bits.shape
    q13 = Q.quantize(w13_bits.reshape(E * N13, H), scope="group", group_rows=N13)
    q2 = Q.quantize(w2_bits.reshape(E * N2, I), scope="group", group_rows=N2)
    return dict(
        w13_codes=q13["codes"].reshape(E, N13, H), w13_sf=q13["sf"].reshape(E, N13, H // 16),
        w13_g=q13["g"],
        w2_codes=q2["codes"].reshape(E, N2, I), w2_sf=q2["sf"].reshape(E, N2, I // 16),
        w2_g=q2["g"])


def quantize_tokens_scatter(x_bits: np.ndarray, perm_info: dict):
    """Per-token NVFP4 of x, each token row written to each of its k slots
    ([4BL] §"Why is the NVFP4 pretraining recipe not sufficient for RL?": per-token FP32
    scale).  Padding slots hold zero codes, zero scales and g = 0."""
    q = Q.quantize(x_bits, scope="row")
    M = int(perm_info["padded_offsets"][-1])
    T, H = x_bits.shape
    perm = perm_info["perm"]
    live = perm >= 0
    codes = np.zeros((M, H), np.uint8)
    sf = np.zeros((M, H // 16), np.uint8)
    g = np.zeros(M, np.float32)
    codes[live] = q["codes"][perm[live]]
    sf[live] = q["sf"][perm[live]]
    g[live] = q["g"][perm[live]]
    return dict(codes=codes, sf=sf, g=g, token_q=q)


def moe_forward(x_bits, topk_ids, topk_w, w13_bits, w2_bits, prepared=None, num_experts=None):
    """The expert block, returning out (BF16 bits [T, H]) and every intermediate."""
    T, H = x_bits.shape
    E = w13_bits.shape[0] if num_experts is None else num_experts
    I = w2_bits.shape[2]
    pw = prepare_weights(w13_bits, w2_bits) if prepared is None else prepared
    pi = permute(topk_ids, E)
    aq = quantize_tokens_scatter(x_bits, pi)
    d = grouped_gemm(aq["codes"], aq["sf"], aq["g"], pw["w13_codes"], pw["w13_sf"], pw["w13_g"],
                     pi["padded_offsets"], pi["counts"])
    live = pi["perm"] >= 0
    d_bits = np.zeros(d.shape, np.uint16)
    d_bits[live] = F.bf16_round(d[live])
    h_bits = np.zeros((d.shape[0], I), np.uint16)
    h_bits[live] = swiglu(d_bits[live], I)
    hq = Q.quantize(h_bits[live], scope="row")
    M = d.shape[0]
    h_codes = np.zeros((M, I), np.uint8)
    h_sf = np.zeros((M, I // 16), np.uint8)
    h_g = np.zeros(M, np.float32)
    h_codes[live], h_sf[live], h_g[live] = hq["codes"], hq["sf"], hq["g"]
    y = grouped_gemm(h_codes, h_sf, h_g, pw["w2_codes"], pw["w2_sf"], pw["w2_g"],
                     pi["padded_offsets"], pi["counts"])
    y_bits = np.zeros(y.shape, np.uint16)
    y_bits[live] = F.bf16_round(y[live])
    out = combine(y_bits, pi["inv"], topk_w)
    return dict(out=out, perm=pi, aq=aq, d=d, d_bits=d_bits, h_bits=h_bits, h_codes=h_codes,
                h_sf=h_sf, h_g=h_g, y=y, y_bits=y_bits, prepared=pw)


def moe_forward_tokens(x_bits, topk_ids, topk_w, prepared, tokens):
    """out rows for a subset of tokens only, computed token by token (bounded CPU sample
    of a large workload; each token's result does not depend on the others).
    ``prepared`` maps each weight field to something indexable by expert id (the arrays
    of prepare_weights, or dicts holding only the experts the tokens use)."""
    H = x_bits.shape[1]
    out = np.zeros((len(tokens), H), np.uint16)
    for n, t in enumerate(tokens):
        q = Q.quantize(x_bits[t:t + 1], scope="row")
        acc = np.zeros(H)
        for j in range(topk_ids.shape[1]):
            e = int(topk_ids[t, j])
            d = gemm_rows(q["codes"], q["sf"], q["g"], prepared["w13_codes"][e],
                          prepared["w13_sf"][e], prepared["w13_g"][e])
            d_bits = F.bf16_round(d)
            h_bits = swiglu(d_bits, d.shape[1] // 2)
            hq = Q.quantize(h_bits, scope="row")
            y = gemm_rows(hq["codes"], hq["sf"], hq["g"], prepared["w2_codes"][e],
                          prepared["w2_sf"][e], prepared["w2_g"][e])
            y_bits = F.bf16_round(y)
            acc += np.float64(np.float32(topk_w[t, j])) * F.bf16_to_f32(y_bits)[0].astype(np.float64)
        out[n] = F.bf16_round(acc[None, :])[0]
    return out

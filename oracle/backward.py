"""Backward pass of the NVFP4 W4A4 expert block (oracle; test infrastructure only).

The quantised backward of [4BL] §"Why is the NVFP4 pretraining recipe not sufficient for
RL?" -- the pretraining recipe runs the backward GEMMs in NVFP4 too, with stochastic
rounding so that the gradient quantisation is approximately unbiased -- which is recipe
(a), "quantized forward and backward", of [4BL] §"Improving Gradient Stability" (Results
Validation).  It differentiates the forward of ``moe.moe_forward``:

    combine      dy[slot(t,j)] = w[t,j] dout[t]          dw[t,j] = <dout[t], y[slot(t,j)]>
    down         dh  = dy W2_e        (dgrad)            dW2_e  = dy_e^T h_e   (wgrad)
    SwiGLU       [dgate | dup] = swiglu_backward(D, dh)
    gate/up      dxs = dD W13_e       (dgrad)            dW13_e = dD_e^T x_e   (wgrad)
    un-permute   dx[t] = sum_j dxs[slot(t,j)]

Readings (the pages give no bit-level rule for the backward; each is stated where used):

* Every backward GEMM is W4A4: both operands NVFP4, quantised along that GEMM's own
  contraction (the forward's row-wise quantisation does not serve: a dgrad contracts over
  the output features, a wgrad over the tokens).  Gradients (dy, dD) use stochastic
  rounding, weights and activations round to nearest.
* dgrad: the gradient per routed row (one FP32 scale per row, blocks of 16 along the
  features, the forward's per-token rule); each expert's weight matrix transposed, one
  FP32 scale per expert matrix, blocks of 16 along the contraction.
* wgrad: both operands transposed per expert -- blocks of 16 consecutive tokens of the
  expert's group, one FP32 scale per expert matrix -- the group zero-padded to a multiple
  of 256 tokens (at least 256).
* Philox key of each stochastic quantisation: seed + (((stream << 10) + expert) << 40)
  (mod 2^64) with stream 0 = dgrad of the down projection (dy by rows), 1 = its wgrad
  (dy^T per expert), 2 = dgrad of gate/up (dD by rows), 3 = its wgrad (dD^T per expert);
  rng_offset 0; element index = row-major index in the quantised matrix (the slot layout
  [M, N] for rows, the expert's zero-padded [N, tokens] for transposes).
* BF16 wherever an unfused pipeline crosses a kernel boundary (dy, dh, dD, the per-slot
  dxs, dx), each rounded once from the exact value; the weight gradients and dw are
  returned exact (float64).
* Columns of D, dD and W13 in the canonical order [gate | up].
"""
from __future__ import annotations

import numpy as np

from . import formats as F
from . import moe as M
from . import quant as Q

STREAM_DGRAD_DOWN, STREAM_WGRAD_DOWN, STREAM_DGRAD_GATEUP, STREAM_WGRAD_GATEUP = 0, 1, 2, 3
WGRAD_TOKEN_ALIGN = 256


def sr_key(seed: int, stream: int, expert: int = 0) -> int:
    """The Philox key (64 bits) of one stochastic quantisation of the backward."""
    return (int(seed) + ((((stream << 10) + expert)) << 40)) & 0xFFFFFFFFFFFFFFFF


def combine_backward(dout_bits: np.ndarray, inv: np.ndarray, topk_w: np.ndarray, y_bits: np.ndarray,
                     n_slots: int):
    """Backward of out[t] = sum_j w[t,j] y[slot(t,j)]: dy[slot(t,j)] = BF16(w[t,j] dout[t]) (the
    product exact in float64, rounded once), slots of no token zero; dw[t,j] =
    sum_h dout[t,h] y[slot(t,j),h] in float64."""
    dout = F.bf16_to_f32(dout_bits).astype(np.float64)
    y = F.bf16_to_f32(y_bits).astype(np.float64)
    w = np.asarray(topk_w, np.float32).astype(np.float64)
    T, k = inv.shape
    dy = np.zeros((n_slots, dout.shape[1]), np.uint16)
    dw = np.zeros((T, k))
    for j in range(k):
        dy[inv[:, j]] = F.bf16_round(w[:, j:j + 1] * dout)
        dw[:, j] = np.sum(dout * y[inv[:, j]], axis=1)
    return dy, dw


def quantize_weights_transposed(w_bits: np.ndarray):
    """Each expert matrix W_e [N, K] as W_e^T [K, N], quantised along N (round to nearest, one
    FP32 scale per expert matrix): the B operand of the dgrad GEMM dX = dY W_e."""
    E, N, K = w_bits.shape
    wt = np.ascontiguousarray(w_bits.transpose(0, 2, 1)).reshape(E * K, N)
    q = Q.quantize(wt, scope="group", group_rows=K)
    return dict(codes=q["codes"].reshape(E, K, N), sf=q["sf"].reshape(E, K, N // 16), g=q["g"])


def dgrad(grad_bits: np.ndarray, wq_t: dict, padded_offsets, counts, seed: int, stream: int):
    """dX[r] = dY[r] W_e for the rows r of each expert's group: dY [M, N] (slot layout, BF16)
    quantised per row along N with stochastic rounding, times the transposed weights.
    Returns (dX float64 [M, K] -- NaN outside the groups -- and dY's quantisation)."""
    q = Q.quantize(grad_bits, scope="row", rounding="sr", seed=sr_key(seed, stream))
    d = M.grouped_gemm(q["codes"], q["sf"], q["g"], wq_t["codes"], wq_t["sf"], wq_t["g"], padded_offsets,
                       counts)
    return d, q


def wgrad(grad_bits: np.ndarray, act_bits: np.ndarray, padded_offsets, counts, seed: int, stream: int):
    """dW_e = dY_e^T X_e over each expert's tokens (rows padded_offsets[e] .. + counts[e] of the
    slot layout): both operands transposed and quantised along the tokens, dY with
    stochastic rounding, X to nearest.  Returns dW float64 [E, N, K] and the operands'
    quantisations per expert."""
    E = len(counts)
    N, K = grad_bits.shape[1], act_bits.shape[1]
    out = np.zeros((E, N, K))
    ops = []
    for e in range(E):
        r0, n = int(padded_offsets[e]), int(counts[e])
        tp = max(WGRAD_TOKEN_ALIGN, -(-n // WGRAD_TOKEN_ALIGN) * WGRAD_TOKEN_ALIGN)
        gt = np.zeros((N, tp), np.uint16)
        at = np.zeros((K, tp), np.uint16)
        gt[:, :n] = grad_bits[r0:r0 + n].T
        at[:, :n] = act_bits[r0:r0 + n].T
        qa = Q.quantize(gt, scope="tensor", rounding="sr", seed=sr_key(seed, stream, e))
        qb = Q.quantize(at, scope="tensor")
        a = Q.dq_unscaled(qa["codes"], qa["sf"]) * np.float64(qa["g"][0])
        b = Q.dq_unscaled(qb["codes"], qb["sf"]) * np.float64(qb["g"][0])
        out[e] = a @ b.T
        ops.append((qa, qb))
    return out, ops


def unpermute_sum(dxs_bits: np.ndarray, inv: np.ndarray) -> np.ndarray:
    """dx[t] = BF16(sum_j dxs[slot(t,j)]) (float64 sum, one rounding)."""
    return M.combine(dxs_bits, inv, np.ones(inv.shape, np.float32))


def moe_backward(dout_bits, fwd: dict, x_bits, topk_w, w13_bits, w2_bits, seed: int = 0):
    """The whole backward of the expert block from the forward's intermediates (``fwd`` as
    ``moe.moe_forward`` returns them).  Returns every stage: dy, dw (router weights), dh,
    dW2 [E, H, I], dD (canonical [dgate | dup]), dxs (per slot), dW13 [E, 2I, H], dx."""
    pi = fwd["perm"]
    padded, counts, inv = pi["padded_offsets"], pi["counts"], pi["inv"]
    n = int(padded[-1])
    live = pi["perm"] >= 0
    I = w2_bits.shape[2]
    dy, dw = combine_backward(dout_bits, inv, topk_w, fwd["y_bits"], n)
    w2q_t = quantize_weights_transposed(w2_bits)                      # [E, I, H], blocks along H
    dh64, _ = dgrad(dy, w2q_t, padded, counts, seed, STREAM_DGRAD_DOWN)
    dh = np.zeros((n, I), np.uint16)
    dh[live] = F.bf16_round(dh64[live])
    dw2, _ = wgrad(dy, fwd["h_bits"], padded, counts, seed, STREAM_WGRAD_DOWN)
    dD = np.zeros((n, 2 * I), np.uint16)
    dD[live] = M.swiglu_backward(fwd["d_bits"][live], dh[live], I)
    w13q_t = quantize_weights_transposed(w13_bits)                    # [E, H, 2I], blocks along 2I
    dxs64, _ = dgrad(dD, w13q_t, padded, counts, seed, STREAM_DGRAD_GATEUP)
    dxs = np.zeros(dxs64.shape, np.uint16)
    dxs[live] = F.bf16_round(dxs64[live])
    x_slots = np.zeros((n, x_bits.shape[1]), np.uint16)
    x_slots[live] = x_bits[pi["perm"][live]]
    dw13, _ = wgrad(dD, x_slots, padded, counts, seed, STREAM_WGRAD_GATEUP)
    dx = unpermute_sum(dxs, inv)
    return dict(dy=dy, dw=dw, dh=dh, dw2=dw2, dD=dD, dxs=dxs, dw13=dw13, dx=dx)

"""GPU parity of the expert block's W4A4 backward (moe_expert_backward) against the
oracle's backward, stage by stage over the GPU's own inputs to each stage:

  transposed weights, dy and the router-weight gradient, the quantised gradient rows,
  dh (dgrad of the down projection), D recomputed, the SwiGLU backward, the quantised dD
  rows, dxs (dgrad of gate/up) and dx, the per-expert transposed wgrad operands and both
  weight gradients.

Quantised codes, scales and global scales are bit-exact (stochastic rounding included:
both sides draw the same Philox bits); GEMM outputs are within the GEMM tolerance of
the float64 GEMM over the same quantised operands; sums within their float32 bounds."""
import numpy as np
import pytest
import torch

from gpu_util import (bf16_tensor, check_bf16_against, combine_violations, dev, npy, rel_err_floor, u16,
                      untile_host)
from oracle import backward as B
from oracle import formats as F
from oracle import moe as M
from oracle import quant as Q
from nvfp4_w4a4_moe_quantize_gb300 import synthetic as S

pytestmark = pytest.mark.gpu


def _src_interleave(I):
    j = np.arange(2 * I)
    chunk, within = j // 128, j % 128
    return np.where(within < 64, chunk * 64 + within, I + chunk * 64 + within - 64)


def _views(buf, lay, i, n, dtype):
    nbytes = n * torch.empty((), dtype=dtype).element_size()
    return buf[lay[i]:lay[i] + nbytes].view(dtype)


def _run(lib, shape, seed=0, bwd_seed=123, x_scale=1.0):
    x, logits, w13, w2 = S.moe_inputs(shape, seed=seed)
    if x_scale != 1.0:
        x = (x.float() * x_scale).bfloat16()
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    ids, w = M.route_topk(logits.numpy(), k)
    pw = lib.moe_prepare_weights(w13.cuda(), w2.cuda())
    pt = lib.moe_prepare_weights_backward(w13.cuda(), w2.cuda())
    fws = lib.moe_forward_workspace(T, k, pw, "cuda")
    xc = x.cuda()
    lib.moe_expert_forward(xc, dev(ids), dev(w), pw, workspace=fws)
    dout = S.randn_bf16((T, H), 1e-3, seed=seed + 77)
    bws = lib.moe_backward_workspace(T, k, pw, "cuda")
    dx, dw, dw13, dw2 = lib.moe_expert_backward(dout.cuda(), xc, dev(w), pw, pt, fws, seed=bwd_seed, workspace=bws)
    assert lib.nvfp4_status_check() == 0
    return dict(x=x, w13=w13, w2=w2, ids=ids, w=w, dout=dout, pw=pw, pt=pt, fws=fws, bws=bws, dx=dx, dw=dw,
                dw13=dw13, dw2=dw2, seed=bwd_seed)


def _check_backward(lib, shape, r, wgrad_values=True):
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    Ip = (I + 255) // 256 * 256
    flay = lib.moe_forward_workspace_layout(T, k, E, H, I)
    blay = lib.moe_backward_workspace_layout(T, k, E, H, I)
    mcap = flay[13]
    fws, bws = r["fws"], r["bws"]
    counts = npy(_views(fws, flay, 0, E, torch.int32))
    padded = npy(_views(fws, flay, 2, E + 1, torch.int32))
    inv = npy(_views(fws, flay, 3, T * k, torch.int32)).reshape(T, k)
    perm = npy(_views(fws, flay, 4, mcap, torch.int32))
    n = int(padded[-1])
    live = np.nonzero(perm[:n] >= 0)[0]
    pi = M.permute(r["ids"], E)
    np.testing.assert_array_equal(padded, pi["padded_offsets"])
    h_gpu = u16(_views(fws, flay, 8, mcap * I, torch.bfloat16).view(mcap, I))[:n]
    y_gpu = u16(_views(fws, flay, 12, mcap * H, torch.bfloat16).view(mcap, H))[:n]
    w13b, w2b, xb = S.bf16_bits(r["w13"]), S.bf16_bits(r["w2"]), S.bf16_bits(r["x"])
    seed = r["seed"]

    # transposed weights (prepared once): bit exact, padding rows of W2^T zero
    w13q_t = B.quantize_weights_transposed(w13b)
    w2q_t = B.quantize_weights_transposed(w2b)
    c13, sf13 = untile_host(npy(r["pt"].w13t), E * H, 2 * I, 256)
    np.testing.assert_array_equal(c13.reshape(E, H, 2 * I), w13q_t["codes"])
    np.testing.assert_array_equal(sf13.reshape(E, H, 2 * I // 16), w13q_t["sf"])
    np.testing.assert_array_equal(npy(r["pt"].w13t_g), w13q_t["g"])
    c2, sf2 = untile_host(npy(r["pt"].w2t), E * Ip, H, 256)
    c2, sf2 = c2.reshape(E, Ip, H), sf2.reshape(E, Ip, H // 16)
    np.testing.assert_array_equal(c2[:, :I], w2q_t["codes"])
    np.testing.assert_array_equal(sf2[:, :I], w2q_t["sf"])
    assert not c2[:, I:].any() and not sf2[:, I:].any()
    np.testing.assert_array_equal(npy(r["pt"].w2t_g), w2q_t["g"])

    # 1. un-permute backward: dy bit exact; dw within the float32 summation bound
    dy_gpu = u16(_views(bws, blay, 0, mcap * H, torch.bfloat16).view(mcap, H))[:n]
    dy_ref, dw_ref = B.combine_backward(S.bf16_bits(r["dout"]), inv, r["w"], y_gpu, n)
    np.testing.assert_array_equal(dy_gpu[live], dy_ref[live])
    dv = F.bf16_to_f32(S.bf16_bits(r["dout"])).astype(np.float64)
    yv = F.bf16_to_f32(y_gpu).astype(np.float64)
    mag = np.stack([np.sum(np.abs(dv * yv[inv[:, j]]), axis=1) for j in range(k)], axis=1)
    assert np.all(np.abs(npy(r["dw"]) - dw_ref) <= (H + 2) * 2.0 ** -24 * mag + 1e-30)

    # 2. dy rows quantised (stochastic rounding, stream 0), then dh = Q(dy) Q(W2^T); the
    #    padding slots hold whatever the workspace held (never read by the kernels): zero
    #    them for the oracle, which quantises the whole slot layout (row index = slot)
    pad = np.ones(n, bool)
    pad[live] = False
    dy_gpu = dy_gpu.copy()
    dy_gpu[pad] = 0
    dyq_c, dyq_sf = untile_host(npy(bws[blay[1]:blay[2]]), mcap, H, 128)
    q_dy = Q.quantize(dy_gpu, scope="row", rounding="sr", seed=B.sr_key(seed, B.STREAM_DGRAD_DOWN))
    np.testing.assert_array_equal(dyq_c[live], q_dy["codes"][live])
    np.testing.assert_array_equal(dyq_sf[live], q_dy["sf"][live])
    np.testing.assert_array_equal(npy(_views(bws, blay, 2, mcap, torch.float32))[live], q_dy["g"][live])
    dh_gpu = u16(_views(bws, blay, 3, mcap * Ip, torch.bfloat16).view(mcap, Ip))[:n]
    dh_ref = M.grouped_gemm(q_dy["codes"], q_dy["sf"], q_dy["g"], w2q_t["codes"], w2q_t["sf"], w2q_t["g"], padded,
                            counts)
    nbad, worst = check_bf16_against(dh_gpu[live][:, :I], dh_ref[live])
    assert nbad == 0, worst

    # 3. D recomputed: the forward's own h is the SwiGLU of it, bit for bit; SwiGLU backward
    d_gpu = u16(_views(bws, blay, 4, mcap * 2 * I, torch.bfloat16).view(mcap, 2 * I))[:n]
    d_can = np.empty_like(d_gpu)
    d_can[:, _src_interleave(I)] = d_gpu
    np.testing.assert_array_equal(M.swiglu(d_can[live], I), h_gpu[live])
    dD_gpu = u16(_views(bws, blay, 5, mcap * 2 * I, torch.bfloat16).view(mcap, 2 * I))[:n].copy()
    dD_gpu[pad] = 0
    dD_ref = M.swiglu_backward(d_can[live], dh_gpu[live][:, :I], I)
    for part in (slice(0, I), slice(I, 2 * I)):
        nbad, worst = check_bf16_against(dD_gpu[live][:, part], F.bf16_to_f32(dD_ref[:, part]).astype(np.float64))
        assert nbad == 0, (part, worst)

    # 4. dD rows quantised (stream 2), dxs = Q(dD) Q(W13^T), dx = sum over the slots
    dDq_c, dDq_sf = untile_host(npy(bws[blay[6]:blay[7]]), mcap, 2 * I, 128)
    q_dD = Q.quantize(dD_gpu, scope="row", rounding="sr", seed=B.sr_key(seed, B.STREAM_DGRAD_GATEUP))
    np.testing.assert_array_equal(dDq_c[live], q_dD["codes"][live])
    np.testing.assert_array_equal(dDq_sf[live], q_dD["sf"][live])
    np.testing.assert_array_equal(npy(_views(bws, blay, 7, mcap, torch.float32))[live], q_dD["g"][live])
    dxs_gpu = u16(_views(bws, blay, 8, mcap * H, torch.bfloat16).view(mcap, H))[:n]
    dxs_ref = M.grouped_gemm(q_dD["codes"], q_dD["sf"], q_dD["g"], w13q_t["codes"], w13q_t["sf"], w13q_t["g"],
                             padded, counts)
    nbad, worst = check_bf16_against(dxs_gpu[live], dxs_ref[live])
    assert nbad == 0, worst
    assert combine_violations(u16(r["dx"]), dxs_gpu, inv, np.ones((T, k), np.float32)) == 0

    # 5. weight gradients: per-expert transposed operands bit exact, GEMMs within tolerance
    kofs = npy(_views(bws, blay, 9, E + 1, torch.int32))
    kb = np.maximum(1, (counts + 255) // 256)
    np.testing.assert_array_equal(kofs, np.concatenate([[0], np.cumsum(kb)]))
    gexp = npy(_views(bws, blay, 11, 4 * E, torch.float32))
    x_slots = np.zeros((n, H), np.uint16)
    x_slots[live] = xb[perm[live]]
    for (gsrc, asrc, Fa, Fb, Fbp, stream, slot, ia, ib, got) in (
            (dy_gpu, h_gpu, H, I, Ip, B.STREAM_WGRAD_DOWN, 0, 12, 13, r["dw2"]),
            (dD_gpu, x_slots, 2 * I, H, H, B.STREAM_WGRAD_GATEUP, 1, 14, 15, r["dw13"])):
        ref, ops = B.wgrad(gsrc, asrc, padded, counts, seed, stream)
        kb_cap = blay[16]
        abuf = npy(bws[blay[ia]:blay[ia] + (Fa // 128) * kb_cap * 128 * 144])
        bbuf = npy(bws[blay[ib]:blay[ib] + (Fbp // 256) * kb_cap * 256 * 144])
        for e in range(E):
            tp = 256 * int(kb[e])
            qa, qb = ops[e]
            a0 = (Fa // 128) * int(kofs[e]) * 128 * 144
            ac, asf = untile_host(abuf[a0:a0 + (Fa // 128) * int(kb[e]) * 128 * 144], Fa, tp, 128)
            np.testing.assert_array_equal(ac, qa["codes"], err_msg=f"A codes, expert {e}")
            np.testing.assert_array_equal(asf, qa["sf"], err_msg=f"A scales, expert {e}")
            b0 = (Fbp // 256) * int(kofs[e]) * 256 * 144
            bc, bsf = untile_host(bbuf[b0:b0 + (Fbp // 256) * int(kb[e]) * 256 * 144], Fbp, tp, 256)
            np.testing.assert_array_equal(bc[:Fb], qb["codes"], err_msg=f"B codes, expert {e}")
            np.testing.assert_array_equal(bsf[:Fb], qb["sf"], err_msg=f"B scales, expert {e}")
            assert not bc[Fb:].any()
            assert gexp[2 * slot * E + e] == qa["g"][0] and gexp[2 * slot * E + E + e] == qb["g"][0]
        if not wgrad_values:
            continue
        mx, nw = rel_err_floor(npy(got).reshape(-1), ref.reshape(-1))
        assert mx <= 1e-3, (stream, mx, nw)


@pytest.mark.parametrize("shape", [
    S.MoEShape("tiny-bwd", T=512, H=256, I=128, E=8, k=2, routing="normal"),
    S.MoEShape("edge-bwd", T=300, H=512, I=384, E=16, k=4, routing="zipf"),   # empty experts, I % 256 != 0
])
def test_backward_stagewise(cuda_lib, shape):
    r = _run(cuda_lib, shape)
    _check_backward(cuda_lib, shape, r)


def test_backward_tiny_activations(cuda_lib):
    """Activations scaled by 2^-120: the per-row global scales of x and dD are float32
    subnormals, so the per-expert maxima of the wgrad operands come from reading the rows
    rather than from the scales.  Every stage matches the oracle, the per-expert wgrad
    operands and their global scales bit for bit; the weight-gradient values themselves
    are not compared (the product of the two per-expert scales, about 2^-265, is below the
    float32 range of the GEMM epilogue's scale, while the float64 reference keeps it)."""
    shape = S.MoEShape("tiny-bwd", T=256, H=256, I=128, E=4, k=2, routing="normal")
    r = _run(cuda_lib, shape, x_scale=2.0 ** -120)
    _check_backward(cuda_lib, shape, r, wgrad_values=False)


def test_backward_is_deterministic_and_seeded(cuda_lib):
    shape = S.MoEShape("tiny-bwd", T=256, H=256, I=128, E=4, k=2, routing="normal")
    a = _run(cuda_lib, shape, bwd_seed=5)
    b = _run(cuda_lib, shape, bwd_seed=5)
    c = _run(cuda_lib, shape, bwd_seed=6)
    for key in ("dx", "dw", "dw13", "dw2"):
        assert torch.equal(a[key], b[key]), key
    assert not torch.equal(a["dw13"], c["dw13"])      # another Philox key draws other roundings

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


def _run(lib, shape, seed=0, bwd_seed=123, x_scale=1.0, d_scale=1.0):
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
    if d_scale != 1.0:
        dout = (dout.float() * d_scale).bfloat16()
    bws = lib.moe_backward_workspace(T, k, pw, "cuda")
    dx, dw, dw13, dw2 = lib.moe_expert_backward(dout.cuda(), xc, dev(w), pw, pt, fws, seed=bwd_seed, workspace=bws)
    assert lib.nvfp4_status_check() == 0
    return dict(x=x, w13=w13, w2=w2, ids=ids, w=w, dout=dout, pw=pw, pt=pt, fws=fws, bws=bws, dx=dx, dw=dw,
                dw13=dw13, dw2=dw2, seed=bwd_seed)


def _check_backward(lib, shape, r, wgrad_values=True, upto_dy_quant=False):
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
    if upto_dy_quant:
        return
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


def test_backward_subnormal_gradients(cuda_lib):
    """Output gradients scaled by 2^-118 (about 2^-128, float32 subnormals): every
    product w dout and so every dy = BF16(w dout) is a subnormal, rounded once from the
    exact product (where the float32 product sits on a BF16 midpoint, an FMA residual
    would itself underflow); dy and dw, and dy's per-row quantisation (codes, scales and
    the subnormal global scales), match the oracle bit for bit.  The GEMMs that follow are
    not compared: the product of dy's global scale (about 2^-139) and the weights' is
    below the float32 range of the GEMM epilogue's scale, while the float64 reference
    keeps it (as in test_backward_tiny_activations)."""
    shape = S.MoEShape("tiny-bwd", T=256, H=256, I=128, E=4, k=2, routing="normal")
    r = _run(cuda_lib, shape, d_scale=2.0 ** -118)
    d = S.bf16_bits(r["dout"])
    assert np.any((d & 0x7F80) == 0) and np.any(d & 0x7FFF), "subnormal gradients"
    _check_backward(cuda_lib, shape, r, upto_dy_quant=True)


def test_backward_is_deterministic_and_seeded(cuda_lib):
    shape = S.MoEShape("tiny-bwd", T=256, H=256, I=128, E=4, k=2, routing="normal")
    a = _run(cuda_lib, shape, bwd_seed=5)
    b = _run(cuda_lib, shape, bwd_seed=5)
    c = _run(cuda_lib, shape, bwd_seed=6)
    for key in ("dx", "dw", "dw13", "dw2"):
        assert torch.equal(a[key], b[key]), key
    assert not torch.equal(a["dw13"], c["dw13"])      # another Philox key draws other roundings


def _tiled_block(buf, block, K, R=128):
    """Codes and row-major scales of one R-row block of a GEMM-tiled buffer (device)."""
    nbytes = (K // 256) * R * 144
    return untile_host(npy(buf[block * nbytes:(block + 1) * nbytes]), R, K, R)


def test_backward_learner_size_sampled(cuda_lib):
    """The learner-step workload at full size (T=32768, H=2048, I=768, 128 experts, top-8,
    uniform routing, dout N(0, 1e-3)), through the calls and sizes the bench times.  Two
    experts are checked stage by stage on a 128-row block of their groups (dy, the
    SR-quantised dy and dD rows and their scales bit exact; dh, dD and dxs within the GEMM
    and SwiGLU tolerances; the recomputed D gives the forward's h bit for bit), dx on the
    tokens of those rows, and each of the two experts' weight gradients whole: the
    transposed operands bit exact and dW within the GEMM tolerance."""
    lib = cuda_lib
    shape = S.WORKLOADS["learner"]
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    Ip = (I + 255) // 256 * 256
    x, logits, w13, w2 = S.moe_inputs(shape, seed=0)
    dout = S.randn_bf16((T, H), 1e-3, 9)
    seed = 7
    xc = x.cuda()
    ids, w = lib.moe_route_topk(logits.cuda(), k)
    pw = lib.moe_prepare_weights(w13.cuda(), w2.cuda())
    pt = lib.moe_prepare_weights_backward(w13.cuda(), w2.cuda())
    fws = lib.moe_forward_workspace(T, k, pw, "cuda")
    lib.moe_expert_forward(xc, ids, w, pw, workspace=fws)
    bws = lib.moe_backward_workspace(T, k, pw, "cuda")
    dx, _, dw13, dw2 = lib.moe_expert_backward(dout.cuda(), xc, w, pw, pt, fws, seed=seed, workspace=bws)
    assert lib.nvfp4_status_check() == 0

    flay = lib.moe_forward_workspace_layout(T, k, E, H, I)
    blay = lib.moe_backward_workspace_layout(T, k, E, H, I)
    mcap = flay[13]
    counts = npy(_views(fws, flay, 0, E, torch.int32))
    padded = npy(_views(fws, flay, 2, E + 1, torch.int32))
    inv = npy(_views(fws, flay, 3, T * k, torch.int32)).reshape(T, k)
    perm_d = _views(fws, flay, 4, mcap, torch.int32)
    h_d = _views(fws, flay, 8, mcap * I, torch.bfloat16).view(mcap, I)
    dy_d = _views(bws, blay, 0, mcap * H, torch.bfloat16).view(mcap, H)
    dh_d = _views(bws, blay, 3, mcap * Ip, torch.bfloat16).view(mcap, Ip)
    d_d = _views(bws, blay, 4, mcap * 2 * I, torch.bfloat16).view(mcap, 2 * I)
    dD_d = _views(bws, blay, 5, mcap * 2 * I, torch.bfloat16).view(mcap, 2 * I)
    dxs_d = _views(bws, blay, 8, mcap * H, torch.bfloat16).view(mcap, H)
    g_dy = _views(bws, blay, 2, mcap, torch.float32)
    g_dD = _views(bws, blay, 7, mcap, torch.float32)
    kofs = npy(_views(bws, blay, 9, E + 1, torch.int32))
    gexp = npy(_views(bws, blay, 11, 4 * E, torch.float32))
    w_np, dout_b, xb = npy(w), S.bf16_bits(dout), S.bf16_bits(x)
    w13b, w2b = S.bf16_bits(w13), S.bf16_bits(w2)
    kb_cap = blay[16]

    for e in (0, 77):
        assert counts[e] >= 128
        r0 = int(padded[e])
        rows = slice(r0, r0 + 128)
        tok = npy(perm_d[rows]).astype(np.int64)
        jj = np.array([int(np.nonzero(inv[t] == r0 + i)[0][0]) for i, t in enumerate(tok)])
        # dy = BF16(w dout), bit exact
        dy_b = u16(dy_d[rows])
        dyv = F.bf16_to_f32(dout_b[tok]).astype(np.float64) * w_np[tok, jj].astype(np.float64)[:, None]
        np.testing.assert_array_equal(dy_b, F.bf16_round(dyv))
        # the SR-quantised dy rows (row-major element index over the slot layout)
        q_dy = Q.quantize(dy_b, scope="row", rounding="sr", seed=B.sr_key(seed, B.STREAM_DGRAD_DOWN),
                          rng_offset=r0 * H // 8)
        c, sf = _tiled_block(bws[blay[1]:blay[2]], r0 // 128, H)
        np.testing.assert_array_equal(c, q_dy["codes"])
        np.testing.assert_array_equal(sf, q_dy["sf"])
        np.testing.assert_array_equal(npy(g_dy[rows]), q_dy["g"])
        # dh = Q(dy) Q(W2_e^T)
        w2q_t = B.quantize_weights_transposed(w2b[e:e + 1])
        one = (np.array([0, 128]), np.array([128]))
        dh_ref = M.grouped_gemm(q_dy["codes"], q_dy["sf"], q_dy["g"], w2q_t["codes"], w2q_t["sf"], w2q_t["g"], *one)
        dh_b = u16(dh_d[rows])
        nbad, worst = check_bf16_against(dh_b[:, :I], dh_ref)
        assert nbad == 0, (e, "dh", worst)
        # D recomputed gives the forward's h; the SwiGLU backward
        d_b = u16(d_d[rows])
        d_can = np.empty_like(d_b)
        d_can[:, _src_interleave(I)] = d_b
        np.testing.assert_array_equal(M.swiglu(d_can, I), u16(h_d[rows]))
        dD_b = u16(dD_d[rows])
        dD_ref = M.swiglu_backward(d_can, dh_b[:, :I], I)
        for part in (slice(0, I), slice(I, 2 * I)):
            nbad, worst = check_bf16_against(dD_b[:, part], F.bf16_to_f32(dD_ref[:, part]).astype(np.float64))
            assert nbad == 0, (e, "dD", worst)
        # the SR-quantised dD rows, then dxs = Q(dD) Q(W13_e^T)
        q_dD = Q.quantize(dD_b, scope="row", rounding="sr", seed=B.sr_key(seed, B.STREAM_DGRAD_GATEUP),
                          rng_offset=r0 * 2 * I // 8)
        c, sf = _tiled_block(bws[blay[6]:blay[7]], r0 // 128, 2 * I)
        np.testing.assert_array_equal(c, q_dD["codes"])
        np.testing.assert_array_equal(sf, q_dD["sf"])
        np.testing.assert_array_equal(npy(g_dD[rows]), q_dD["g"])
        w13q_t = B.quantize_weights_transposed(w13b[e:e + 1])
        dxs_ref = M.grouped_gemm(q_dD["codes"], q_dD["sf"], q_dD["g"], w13q_t["codes"], w13q_t["sf"], w13q_t["g"],
                                 *one)
        nbad, worst = check_bf16_against(u16(dxs_d[rows]), dxs_ref)
        assert nbad == 0, (e, "dxs", worst)
        # dx of these rows' tokens: the sum of their k slots' dxs
        ts = tok[:32]
        slots = inv[ts]
        dxs_rows = u16(dxs_d[torch.from_numpy(slots.reshape(-1)).long().cuda()]).reshape(len(ts) * k, H)
        assert combine_violations(u16(dx[torch.from_numpy(ts).cuda()]), dxs_rows,
                                  np.arange(len(ts) * k).reshape(len(ts), k), np.ones((len(ts), k), np.float32)) == 0

        # weight gradients of expert e, whole: transposed operands and dW
        n = int(counts[e])
        gr = slice(r0, r0 + n)
        tp = 256 * int(kofs[e + 1] - kofs[e])
        for (gsrc, asrc, Fa, Fb, Fbp, stream, slot, ia, ib, got) in (
                (u16(dy_d[gr]), u16(h_d[gr]), H, I, Ip, B.STREAM_WGRAD_DOWN, 0, 12, 13, dw2),
                (u16(dD_d[gr]), xb[npy(perm_d[gr]).astype(np.int64)], 2 * I, H, H, B.STREAM_WGRAD_GATEUP, 1, 14, 15,
                 dw13)):
            gt = np.zeros((Fa, tp), np.uint16)
            at = np.zeros((Fb, tp), np.uint16)
            gt[:, :n] = gsrc.T
            at[:, :n] = asrc.T
            qa = Q.quantize(gt, scope="tensor", rounding="sr", seed=B.sr_key(seed, stream, e))
            qb = Q.quantize(at, scope="tensor")
            abuf = bws[blay[ia]:blay[ia] + (Fa // 128) * kb_cap * 128 * 144]
            bbuf = bws[blay[ib]:blay[ib] + (Fbp // 256) * kb_cap * 256 * 144]
            a0 = (Fa // 128) * int(kofs[e]) * 128 * 144
            ac, asf = untile_host(npy(abuf[a0:a0 + (Fa // 128) * (tp // 256) * 128 * 144]), Fa, tp, 128)
            np.testing.assert_array_equal(ac, qa["codes"], err_msg=f"A codes, expert {e}")
            np.testing.assert_array_equal(asf, qa["sf"], err_msg=f"A scales, expert {e}")
            b0 = (Fbp // 256) * int(kofs[e]) * 256 * 144
            bc, bsf = untile_host(npy(bbuf[b0:b0 + (Fbp // 256) * (tp // 256) * 256 * 144]), Fbp, tp, 256)
            np.testing.assert_array_equal(bc[:Fb], qb["codes"], err_msg=f"B codes, expert {e}")
            np.testing.assert_array_equal(bsf[:Fb], qb["sf"], err_msg=f"B scales, expert {e}")
            assert gexp[2 * slot * E + e] == qa["g"][0] and gexp[2 * slot * E + E + e] == qb["g"][0]
            ref = (Q.dq_unscaled(qa["codes"], qa["sf"]) * np.float64(qa["g"][0])) @ \
                  (Q.dq_unscaled(qb["codes"], qb["sf"]) * np.float64(qb["g"][0])).T
            mx, nw = rel_err_floor(npy(got[e]).reshape(-1), ref.reshape(-1))
            assert mx <= 1e-3, (e, stream, mx, nw)

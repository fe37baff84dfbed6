"""GPU parity of the MoE expert block against the oracle: routing, grouping, combine,
SwiGLU + requantisation, weight preparation and the whole forward, stage by stage, plus
the execution-alignment properties (row invariance, determinism)."""
import numpy as np
import pytest
import torch

from gpu_util import (bf16_tensor, bf16_ulp, check_bf16_against, combine_violations, dev, npy, rel_err_floor, u16,
                      untile_host)
from oracle import formats as F
from oracle import moe as M
from oracle import quant as Q
from nvfp4_w4a4_moe_quantize_gb300 import synthetic as S

pytestmark = pytest.mark.gpu


def interleave_src(I: int) -> np.ndarray:
    """Column (or row) j of the 64-chunk gate/up interleave holds canonical index src[j]."""
    j = np.arange(2 * I)
    chunk, within = j // 128, j % 128
    return np.where(within < 64, chunk * 64 + within, I + chunk * 64 + within - 64)


def _ws_views(ws, lay, T, k, E, H, I):
    mcap = lay[13]
    Ip = (I + 255) // 256 * 256

    def view(i, n, dtype):
        nbytes = n * torch.empty((), dtype=dtype).element_size()
        return ws[lay[i]:lay[i] + nbytes].view(dtype)
    return dict(
        counts=view(0, E, torch.int32), offsets=view(1, E + 1, torch.int32), padded=view(2, E + 1, torch.int32),
        inv=view(3, T * k, torch.int32).view(T, k), perm=view(4, mcap, torch.int32),
        aq=ws[lay[5]:lay[7]], ga=view(7, mcap, torch.float32),
        h=view(8, mcap * I, torch.bfloat16).view(mcap, I), hq=ws[lay[9]:lay[11]],
        gh=view(11, mcap, torch.float32), y=view(12, mcap * H, torch.bfloat16).view(mcap, H), mcap=mcap, Ip=Ip)


# ------------------------------------------------------------------ routing / grouping

@pytest.mark.parametrize("T,E,k,kind", [(512, 8, 2, "normal"), (8192, 128, 8, "zipf"), (333, 1000, 32, "normal")])
def test_route_topk(cuda_lib, T, E, k, kind):
    logits = S.router_logits_zipf(T, E, seed=3) if kind == "zipf" else S.router_logits_normal(T, E, seed=3)
    for renorm in (True, False):
        ids, w = cuda_lib.moe_route_topk(logits.cuda(), k, renorm)
        rid, rw = M.route_topk(logits.numpy(), k, renorm)
        np.testing.assert_array_equal(npy(ids), rid)
        np.testing.assert_allclose(npy(w), rw, rtol=1e-6, atol=1e-12)


def test_route_topk_ties(cuda_lib):
    logits = torch.randint(-2, 3, (256, 16), generator=torch.Generator().manual_seed(1)).float()
    ids, w = cuda_lib.moe_route_topk(logits.cuda(), 4)
    rid, rw = M.route_topk(logits.numpy(), 4)
    np.testing.assert_array_equal(npy(ids), rid)
    np.testing.assert_allclose(npy(w), rw, rtol=1e-6)


@pytest.mark.parametrize("T,E,k", [(512, 8, 2), (8192, 128, 8), (1, 4, 4), (3000, 1024, 3)])
def test_permute(cuda_lib, T, E, k):
    logits = S.router_logits_zipf(T, E, seed=T)
    rid, _ = M.route_topk(logits.numpy(), k)
    p = cuda_lib.moe_permute(dev(rid), E)
    r = M.permute(rid, E)
    for key in ("counts", "offsets", "padded_offsets", "inv"):
        np.testing.assert_array_equal(npy(p[key]), r[key], err_msg=key)
    n = int(r["padded_offsets"][-1])
    np.testing.assert_array_equal(npy(p["perm"])[:n], r["perm"])
    assert cuda_lib.nvfp4_status_check() == 0


def test_permute_bad_ids_set_status(cuda_lib):
    ids = torch.tensor([[0, 1], [2, 9], [-1, 3]], dtype=torch.int32, device="cuda")
    p = cuda_lib.moe_permute(ids, 4)
    assert cuda_lib.nvfp4_status_check() == cuda_lib.Status.DEVICE_STATUS
    assert cuda_lib.nvfp4_status_check() == 0                       # cleared
    inv = npy(p["inv"])
    assert inv[1, 1] == -1 and inv[2, 0] == -1
    assert npy(p["counts"]).tolist() == [1, 1, 1, 1]


def test_combine(cuda_lib):
    T, k, H, Mr = 300, 8, 2048, 4000
    rng = np.random.default_rng(3)
    y = F.bf16_round(rng.standard_normal((Mr, H)))
    inv = np.stack([rng.permutation(Mr)[:k] for _ in range(T)]).astype(np.int32)
    w = rng.random((T, k)).astype(np.float32)
    out = u16(cuda_lib.moe_combine(bf16_tensor(y), dev(inv), dev(w)))
    ref = M.combine(y, inv, w)
    # float32 products and sums in order j: |err| <= (k+1) 2^-24 sum|w y| before rounding
    assert combine_violations(out, y, inv, w) == 0
    assert np.mean(out == ref) > 0.999


# ------------------------------------------------------------------ SwiGLU + requant

def test_swiglu_quantize_bit_exact(cuda_lib):
    rows, I = 300, 768
    rng = np.random.default_rng(5)
    d_can = F.bf16_round(rng.standard_normal((rows, 2 * I)) * rng.choice([0.1, 1, 4, 30], (rows, 1)))
    d_can[0, :I] = F.bf16_round(np.linspace(-120, 120, I))          # saturated gates
    d_can[1, :5] = 0
    d_can[2, I:I + 7] = 0x8000
    perm = np.arange(rows, dtype=np.int32)
    perm[7] = -1
    d_il = d_can[:, interleave_src(I)]
    h, hq, hsf, gh = cuda_lib.moe_swiglu_quantize(bf16_tensor(d_il), dev(perm), I)
    live = perm >= 0
    ref_h = M.swiglu(d_can, I)
    np.testing.assert_array_equal(u16(h)[live], ref_h[live])
    q = Q.quantize(ref_h[live], scope="row")
    np.testing.assert_array_equal(npy(hq)[live], q["packed"])
    np.testing.assert_array_equal(npy(gh)[live], q["g"])
    sf = F.sf_unswizzle(npy(hsf), rows, I // 16)
    np.testing.assert_array_equal(sf[live], q["sf"])


def _swiglu_hard_pairs(n_random=8_000_000, seed=11):
    """(gate, up) BF16 pairs whose SwiGLU value lies near a BF16 rounding midpoint: the
    cases the float32 fast path hands to its slower exact path.  Three families:
    (a) random pairs whose float64 value is within 2^-14 BF16 ulp of a midpoint;
    (b) gate in [8, 48] with gate*up exactly a midpoint, where silu(gate)*up sits just
        below it by exp(-gate) (the float64 reference ties to even once 1 + exp(-gate)
        rounds to 1, above gate = 36.74);
    (c) range edges: |gate| near and beyond 80, tiny and huge products;
    (d) family (b) with up scaled by 2^-118 .. 2^-132: products at the bottom of the
        float32 normal range and below it (BF16 subnormals), where the residual of a
        float32 product can itself underflow."""
    rng = np.random.default_rng(seed)
    bf = lambda v: F.bf16_to_f32(F.bf16_round(v)).astype(np.float64)  # noqa: E731
    g = bf(rng.standard_normal(n_random) * rng.choice([0.05, 0.3, 1, 4, 20], n_random))
    u = bf(rng.standard_normal(n_random) * rng.choice([0.01, 1, 100], n_random))
    ref = M.silu(g) * u
    _, ex = np.frexp(np.abs(ref))
    pos = np.abs(ref) / np.exp2(ex - 8.0)                  # in BF16 ulps; midpoints at .5
    near = (np.abs(pos - np.floor(pos) - 0.5) < 2.0 ** -14) & (ref != 0)
    ga, ua = g[near], u[near]
    gs = bf(np.linspace(8, 48, 321))
    us = bf(rng.standard_normal(3000) * 2)
    G2, U2 = (a.ravel() for a in np.meshgrid(gs, us))
    prod = (G2.astype(np.float32) * U2.astype(np.float32)).view(np.uint32)
    mid = (prod & 0xFFFF) == 0x8000
    gb, ub = G2[mid], U2[mid]
    # large |gate|, and gates at or below the float32 normal range with large up (silu(gate)
    # itself subnormal)
    gc = bf(np.array([79.5, 80, 80.5, 81, -79.5, -80, -80.5, -81, -87, -88.5, -100, -200, 1e-20, -1e-20, 1e-3, 3e4,
                      16.5, -17, 24, -30, 1e-39, -3e-40, 2e-41, 1.2e-38, -5e-39, 3e-30]))
    uc = bf(np.array([1.5, -3, 1e30, 2e-30, 1e38, -1e37, 1e35, 7e38, 1e-30, 1e25, 5e-39, 1.0, 1e20, 1e-10, 3e33,
                      -2e-35, 3.0, -1e10, 7.0, 2e20, 1e30, -3e35, 1e38, 2e25, 7e33, 1e30]))
    gd, ud = [], []
    for sc in (-118, -124, -128, -132):
        U4 = bf(us * 2.0 ** sc)
        G4, U4 = (a.ravel() for a in np.meshgrid(gs, U4))
        p4 = (G4.astype(np.float32) * U4.astype(np.float32)).view(np.uint32)
        idx = np.flatnonzero((p4 & 0xFFFF) == 0x8000)
        idx = idx[rng.permutation(idx.size)[:5000]]
        gd.append(G4[idx])
        ud.append(U4[idx])
    return (np.concatenate([ga, gb, gc] + gd), np.concatenate([ua, ub, uc] + ud), (ga.size, gb.size))


def test_swiglu_hard_cases_bit_exact(cuda_lib):
    """Near-midpoint SwiGLU values: every h bit equals the oracle's float64 rounding."""
    g, u, (na, nb) = _swiglu_hard_pairs()
    assert na > 2000 and nb > 2000
    I = 1024
    rows = (g.size + I - 1) // I
    pad = rows * I - g.size
    g = np.concatenate([g, np.ones(pad)])
    u = np.concatenate([u, np.ones(pad)])
    d_can = np.concatenate([F.bf16_round(g).reshape(rows, I), F.bf16_round(u).reshape(rows, I)], axis=1)
    perm = np.arange(rows, dtype=np.int32)
    h, _, _, _ = cuda_lib.moe_swiglu_quantize(bf16_tensor(d_can[:, interleave_src(I)]), dev(perm), I)
    got, ref = u16(h), M.swiglu(d_can, I)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, [(float(g.reshape(rows, I)[r, c]), float(u.reshape(rows, I)[r, c]), hex(got[r, c]),
                            hex(ref[r, c])) for r, c in bad[:8]]


def test_swiglu_quantize_pads_k(cuda_lib):
    """I = 128: h is quantised into a 256-wide (zero-padded) row for the down GEMM."""
    rows, I = 130, 128
    d_can = S.bf16_bits(S.randn_bf16((rows, 2 * I), seed=8))
    perm = np.arange(rows, dtype=np.int32)
    _, hq, hsf, gh = cuda_lib.moe_swiglu_quantize(bf16_tensor(d_can[:, interleave_src(I)]), dev(perm), I)
    q = Q.quantize(M.swiglu(d_can, I), scope="row")
    hq = npy(hq)
    np.testing.assert_array_equal(hq[:, :64], q["packed"])
    assert not hq[:, 64:].any()
    sf = F.sf_unswizzle(npy(hsf), rows, 16)
    np.testing.assert_array_equal(sf[:, :8], q["sf"])
    assert not sf[:, 8:].any()


# ------------------------------------------------------------------ weights

@pytest.mark.parametrize("name", ["tiny"])
def test_prepare_weights(cuda_lib, name):
    shape = S.WORKLOADS[name]
    _, _, w13, w2 = S.moe_inputs(shape, seed=0)
    pw = cuda_lib.moe_prepare_weights(w13.cuda(), w2.cuda())
    ref = M.prepare_weights(S.bf16_bits(w13), S.bf16_bits(w2))
    E, H, I = shape.E, shape.H, shape.I
    src = interleave_src(I)
    c13, sf13 = untile_host(npy(pw.w13), E * 2 * I, H, 256)
    np.testing.assert_array_equal(c13.reshape(E, 2 * I, H), ref["w13_codes"][:, src, :])
    np.testing.assert_array_equal(sf13.reshape(E, 2 * I, H // 16), ref["w13_sf"][:, src, :])
    np.testing.assert_array_equal(npy(pw.w13_g), ref["w13_g"])
    Ip = pw.Ip
    c2, sf2 = untile_host(npy(pw.w2), E * H, Ip, 256)
    c2, sf2 = c2.reshape(E, H, Ip), sf2.reshape(E, H, Ip // 16)
    np.testing.assert_array_equal(c2[:, :, :I], ref["w2_codes"])
    assert not c2[:, :, I:].any()
    np.testing.assert_array_equal(sf2[:, :, :I // 16], ref["w2_sf"])
    assert not sf2[:, :, I // 16:].any()
    np.testing.assert_array_equal(npy(pw.w2_g), ref["w2_g"])


# ------------------------------------------------------------------ forward

def _forward(lib, x, ids, w, pw, T, k):
    ws = lib.moe_forward_workspace(T, k, pw, "cuda")
    out = lib.moe_expert_forward(x, ids, w, pw, workspace=ws)
    assert lib.nvfp4_status_check() == 0
    lay = lib.moe_forward_workspace_layout(T, k, pw.E, pw.H, pw.I)
    return out, _ws_views(ws, lay, T, k, pw.E, pw.H, pw.I)


def _stage_checks(lib, r, v, out, w_np, pw, I):
    """Compare the forward's intermediates with the oracle stage by stage, on every routed
    row and every token (the contract of the fused pipeline):
      grouping arrays and the per-token quantisation scattered into the slots: bit exact;
      h from the fused gate/up GEMM + SwiGLU epilogue: within the GEMM tolerance of the
        oracle's h (a float32-accumulated D can round to the neighbouring BF16 value);
      the requantisation of h: the GPU's own h through the oracle quantiser, bit exact;
      the down GEMM: the float64 GEMM over the GPU's own quantised h, within one BF16 ulp
        plus the float32-accumulation allowance;
      the weighted un-permute: the GPU's own y through the combine bound, element-wise."""
    pi = r["perm"]
    n = int(pi["padded_offsets"][-1])
    for key, ref in (("counts", pi["counts"]), ("padded", pi["padded_offsets"]), ("inv", pi["inv"])):
        np.testing.assert_array_equal(npy(v[key]), ref, err_msg=key)
    perm = npy(v["perm"])[:n]
    np.testing.assert_array_equal(perm, pi["perm"])
    live = np.nonzero(pi["perm"] >= 0)[0]
    H, Ip = pw.H, v["Ip"]
    aq_codes, aq_sf = untile_host(npy(v["aq"]), v["mcap"], H, 128)
    np.testing.assert_array_equal(aq_codes[live], r["aq"]["codes"][live])
    np.testing.assert_array_equal(aq_sf[live], r["aq"]["sf"][live])
    np.testing.assert_array_equal(npy(v["ga"])[live], r["aq"]["g"][live])
    # h against the oracle's h (its own D)
    h_gpu = u16(v["h"])[live]
    h_ref = r["h_bits"][live]
    hv, hr = F.bf16_to_f32(h_gpu).astype(np.float64), F.bf16_to_f32(h_ref).astype(np.float64)
    tau = 1e-2 * np.sqrt(np.mean(hr * hr))
    assert np.all(np.abs(hv - hr) <= 4 * bf16_ulp(hr) + 1e-2 * np.maximum(np.abs(hr), tau))
    # requantisation of the GPU's own h: every routed row, bit exact (columns I..Ip-1 zero)
    hq_codes, hq_sf = untile_host(npy(v["hq"]), v["mcap"], Ip, 128)
    qh = Q.quantize(h_gpu, scope="row")
    np.testing.assert_array_equal(hq_codes[live][:, :I], qh["codes"])
    np.testing.assert_array_equal(hq_sf[live][:, :I // 16], qh["sf"])
    np.testing.assert_array_equal(npy(v["gh"])[live], qh["g"])
    assert not hq_codes[live][:, I:].any() and not hq_sf[live][:, I // 16:].any()
    # down GEMM over the GPU's own hq / gH: every routed row
    pr = r["prepared"]
    gh = npy(v["gh"])[:n]
    yref = M.grouped_gemm(hq_codes[:n, :I], hq_sf[:n, :I // 16], gh, pr["w2_codes"], pr["w2_sf"], pr["w2_g"],
                          pi["padded_offsets"], pi["counts"])
    y_all = u16(v["y"])
    nbad, worst = check_bf16_against(y_all[live], yref[live])
    assert nbad == 0, worst
    # weighted un-permute of the GPU's own y: every token, element-wise
    assert combine_violations(u16(out), y_all, pi["inv"], w_np) == 0


def test_forward_tiny_stagewise(cuda_lib):
    shape = S.WORKLOADS["tiny"]
    x, logits, w13, w2 = S.moe_inputs(shape, seed=0)
    ids, w = M.route_topk(logits.numpy(), shape.k)
    pw = cuda_lib.moe_prepare_weights(w13.cuda(), w2.cuda())
    out, v = _forward(cuda_lib, x.cuda(), dev(ids), dev(w), pw, shape.T, shape.k)
    r = M.moe_forward(S.bf16_bits(x), ids, w, S.bf16_bits(w13), S.bf16_bits(w2))
    _stage_checks(cuda_lib, r, v, out, w, pw, shape.I)
    got = F.bf16_to_f32(u16(out)).astype(np.float64)
    ref = F.bf16_to_f32(r["out"]).astype(np.float64)
    mx, nw = rel_err_floor(got, ref)
    assert nw < 1e-2, nw


@pytest.mark.parametrize("T,H,I,E,k,routing", [
    (1, 256, 128, 4, 1, "normal"),        # one token, one slot; I padded to 256 for the down GEMM
    (1, 256, 128, 4, 4, "normal"),        # one token routed to every expert
    (300, 256, 128, 1, 1, "normal"),      # a single expert: one group with a ragged last tile
    (130, 512, 384, 16, 4, "zipf"),       # I not a multiple of 256, many empty experts
    (64, 2048, 2048, 2, 2, "normal"),     # the largest H and I the forward takes
])
def test_forward_edge_shapes_stagewise(cuda_lib, T, H, I, E, k, routing):
    """The forward at the edges of its shape range, stage by stage against the oracle."""
    shape = S.MoEShape("edge", T=T, H=H, I=I, E=E, k=k, routing=routing)
    x, logits, w13, w2 = S.moe_inputs(shape, seed=7)
    ids, w = M.route_topk(logits.numpy(), k)
    pw = cuda_lib.moe_prepare_weights(w13.cuda(), w2.cuda())
    out, v = _forward(cuda_lib, x.cuda(), dev(ids), dev(w), pw, T, k)
    r = M.moe_forward(S.bf16_bits(x), ids, w, S.bf16_bits(w13), S.bf16_bits(w2))
    _stage_checks(cuda_lib, r, v, out, w, pw, I)
    got = F.bf16_to_f32(u16(out)).astype(np.float64)
    ref = F.bf16_to_f32(r["out"]).astype(np.float64)
    _, nw = rel_err_floor(got, ref)
    assert nw < 1e-2, nw


def test_forward_exact_operands_bit_exact_through_requant(cuda_lib):
    """Lossless inputs (grid values times powers of two): the gate/up output is exact, so
    the whole chain up to the requantised h must match the oracle bit for bit."""
    T, H, I, E, k = 256, 256, 128, 4, 2
    rng = np.random.default_rng(9)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -2, -3, -4, -6])
    s_x, s_w = 448 * 2.0 ** -11, 448 * 2.0 ** -13
    xv = rng.choice(grid, (T, H)) * s_x
    xv[:, ::16] = 6 * s_x
    w13 = rng.choice(grid, (E, 2 * I, H)) * s_w
    w13[:, :, ::16] = 6 * s_w
    w2v = rng.choice(grid, (E, H, I)) * s_w
    w2v[:, :, ::16] = 6 * s_w
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    wts = rng.random((T, k)).astype(np.float32)
    xb, w13b, w2b = F.bf16_round(xv), F.bf16_round(w13), F.bf16_round(w2v)
    pw = cuda_lib.moe_prepare_weights(bf16_tensor(w13b), bf16_tensor(w2b))
    out, v = _forward(cuda_lib, bf16_tensor(xb), dev(ids), dev(wts), pw, T, k)
    r = M.moe_forward(xb, ids, wts, w13b, w2b)
    live = np.nonzero(r["perm"]["perm"] >= 0)[0]
    # exact gate/up output -> identical BF16 D -> correctly rounded h -> identical codes
    np.testing.assert_array_equal(u16(v["h"])[live], r["h_bits"][live])
    hq, hsf = untile_host(npy(v["hq"]), v["mcap"], v["Ip"], 128)
    np.testing.assert_array_equal(hq[live][:, :I], r["h_codes"][live])
    np.testing.assert_array_equal(hsf[live][:, :I // 16], r["h_sf"][live])
    np.testing.assert_array_equal(npy(v["gh"])[live], r["h_g"][live])
    nbad, worst = check_bf16_against(u16(v["y"])[live], r["y"][live])
    assert nbad == 0, worst
    assert combine_violations(u16(out), u16(v["y"]), r["perm"]["inv"], wts) == 0


def test_forward_matches_chain_of_standalone_kernels(cuda_lib):
    """The fused forward equals the unfused chain of library calls over the same operands,
    bit for bit: row-major grouped GEMM (BF16 D) -> moe_swiglu_quantize -> row-major
    grouped GEMM -> moe_combine.  Operands are taken from the forward's own tiled buffers
    (untiled on the host), so this checks the fused SwiGLU epilogue, the tiled GEMM and the
    tiled requantisation against the standalone kernels."""
    shape = S.WORKLOADS["tiny"]
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    x, logits, w13, w2 = S.moe_inputs(shape, seed=2)
    ids, w = cuda_lib.moe_route_topk(logits.cuda(), k)
    pw = cuda_lib.moe_prepare_weights(w13.cuda(), w2.cuda())
    out, v = _forward(cuda_lib, x.cuda(), ids, w, pw, T, k)
    mcap, Ip = v["mcap"], pw.Ip
    n = int(npy(v["padded"])[-1])
    live = npy(v["perm"])[:n] >= 0
    rm = lambda buf, rows, K, R: untile_host(npy(buf), rows, K, R)   # noqa: E731
    a_c, a_sf = rm(v["aq"], mcap, H, 128)
    w13_c, w13_sf = rm(pw.w13, E * 2 * I, H, 256)
    D = cuda_lib.nvfp4_grouped_gemm(dev(F.pack_e2m1(a_c)), dev(F.sf_swizzle(a_sf)), v["ga"],
                                    dev(F.pack_e2m1(w13_c)), dev(F.sf_swizzle(w13_sf)), pw.w13_g,
                                    v["padded"], v["counts"], 2 * I, H, E)
    h, hq, hsf, gh = cuda_lib.moe_swiglu_quantize(D[:n], v["perm"][:n], I)
    np.testing.assert_array_equal(u16(h)[:n][live], u16(v["h"])[:n][live])
    f_hq, f_hsf = rm(v["hq"], mcap, Ip, 128)
    np.testing.assert_array_equal(F.unpack_e2m1(npy(hq))[live], f_hq[:n][live])
    np.testing.assert_array_equal(F.sf_unswizzle(npy(hsf), n, Ip // 16)[live], f_hsf[:n][live])
    np.testing.assert_array_equal(npy(gh)[live], npy(v["gh"])[:n][live])
    w2_c, w2_sf = rm(pw.w2, E * H, Ip, 256)
    hq_full = torch.zeros(mcap, Ip // 2, dtype=torch.uint8, device="cuda")
    hq_full[:n] = hq
    hsf_full = dev(F.sf_swizzle(np.concatenate([F.sf_unswizzle(npy(hsf), n, Ip // 16),
                                                np.zeros((mcap - n, Ip // 16), np.uint8)])))
    gh_full = torch.zeros(mcap, dtype=torch.float32, device="cuda")
    gh_full[:n] = gh
    y = cuda_lib.nvfp4_grouped_gemm(hq_full, hsf_full, gh_full, dev(F.pack_e2m1(w2_c)), dev(F.sf_swizzle(w2_sf)),
                                    pw.w2_g, v["padded"], v["counts"], H, Ip, E)
    np.testing.assert_array_equal(u16(y)[:n][live], u16(v["y"])[:n][live])
    o2 = cuda_lib.moe_combine(y, v["inv"], w)
    np.testing.assert_array_equal(u16(o2), u16(out))


def test_forward_row_invariance_and_determinism_tiny(cuda_lib):
    shape = S.WORKLOADS["tiny"]
    x, logits, w13, w2 = S.moe_inputs(shape, seed=4)
    ids, w = cuda_lib.moe_route_topk(logits.cuda(), shape.k)
    pw = cuda_lib.moe_prepare_weights(w13.cuda(), w2.cuda())
    xc = x.cuda()
    full = u16(cuda_lib.moe_expert_forward(xc, ids, w, pw))
    again = u16(cuda_lib.moe_expert_forward(xc, ids, w, pw))
    np.testing.assert_array_equal(full, again)
    for lo, hi in [(0, 1), (100, 333), (511, 512)]:
        part = u16(cuda_lib.moe_expert_forward(xc[lo:hi].contiguous(), ids[lo:hi].contiguous(),
                                               w[lo:hi].contiguous(), pw))
        np.testing.assert_array_equal(part, full[lo:hi])
    # a permuted token order gives the permuted output
    pidx = torch.randperm(shape.T, generator=torch.Generator().manual_seed(0)).cuda()
    permuted = u16(cuda_lib.moe_expert_forward(xc[pidx].contiguous(), ids[pidx].contiguous(),
                                               w[pidx].contiguous(), pw))
    np.testing.assert_array_equal(permuted, full[npy(pidx)])


@pytest.mark.slow
@pytest.mark.parametrize("name", ["forward", "learner"])
def test_forward_full_size_sampled_and_row_invariant(cuda_lib, name):
    """The Qwen3-30B-A3B-shaped forward in the launch configuration the benchmark times
    (forward: T=16384, Zipf routing; learner: T=32768, uniform routing; H=2048, I=768,
    E=128, top-8).  Grouping, per-token quantisation, the requantisation of h and the
    weighted un-permute are checked on every row and token; the two GEMMs (with SwiGLU)
    on sampled rows, and out end to end on sampled tokens.  Then the first 1024 tokens
    re-run alone must give identical rows."""
    shape = S.WORKLOADS[name]
    x, logits, w13, w2 = S.moe_inputs(shape, seed=0)
    ids, w = cuda_lib.moe_route_topk(logits.cuda(), shape.k)
    rid, rw = M.route_topk(logits.numpy(), shape.k)
    np.testing.assert_array_equal(npy(ids), rid)
    pw = cuda_lib.moe_prepare_weights(w13.cuda(), w2.cuda())
    xc = x.cuda()
    out, v = _forward(cuda_lib, xc, ids, w, pw, shape.T, shape.k)
    # grouping and per-token quantisation: everything
    pi = M.permute(rid, shape.E)
    n = int(pi["padded_offsets"][-1])
    np.testing.assert_array_equal(npy(v["inv"]), pi["inv"])
    np.testing.assert_array_equal(npy(v["perm"])[:n], pi["perm"])
    xb = S.bf16_bits(x)
    qx = Q.quantize(xb, scope="row")
    live = np.nonzero(pi["perm"] >= 0)[0]
    tok = pi["perm"][live]
    aq_c, aq_sf = untile_host(npy(v["aq"]), v["mcap"], shape.H, 128)
    np.testing.assert_array_equal(aq_c[live], qx["codes"][tok])
    np.testing.assert_array_equal(aq_sf[live], qx["sf"][tok])
    np.testing.assert_array_equal(npy(v["ga"])[live], qx["g"][tok])
    # sampled routed rows through the gate/up GEMM + SwiGLU against the oracle, and the
    # down GEMM of the same rows over the GPU's own quantised h
    rng = np.random.default_rng(0)
    sample = np.sort(rng.choice(live, 96, replace=False))
    experts = np.searchsorted(pi["padded_offsets"], sample, side="right") - 1
    w13b, w2b = S.bf16_bits(w13), S.bf16_bits(w2)
    h_all = u16(v["h"])
    y_all = u16(v["y"])
    gh_all = npy(v["gh"])
    hq_c, hq_sf = untile_host(npy(v["hq"]), v["mcap"], v["Ip"], 128)
    I = shape.I
    cache = {}
    for s_row, e in zip(sample, experts):
        if e not in cache:
            cache[e] = (Q.quantize(w13b[e], scope="tensor"), Q.quantize(w2b[e], scope="tensor"))
        q13, q2 = cache[e]
        t = pi["perm"][s_row]
        dref = M.gemm_rows(qx["codes"][t:t + 1], qx["sf"][t:t + 1], qx["g"][t:t + 1], q13["codes"], q13["sf"],
                           q13["g"][0])
        href = M.swiglu(F.bf16_round(dref), I)
        hv = F.bf16_to_f32(h_all[s_row:s_row + 1]).astype(np.float64)
        hr = F.bf16_to_f32(href).astype(np.float64)
        assert np.all(np.abs(hv - hr) <= 4 * bf16_ulp(hr) + 1e-2 * np.abs(hr).max()), s_row
        yref = M.gemm_rows(hq_c[s_row:s_row + 1, :I], hq_sf[s_row:s_row + 1, :I // 16], gh_all[s_row:s_row + 1],
                           q2["codes"], q2["sf"], q2["g"][0])
        nbad, worst = check_bf16_against(y_all[s_row:s_row + 1], yref)
        assert nbad == 0, (s_row, worst)
    # requantisation of the GPU's own h: every routed row, bit exact
    qh = Q.quantize(h_all[live], scope="row")
    np.testing.assert_array_equal(hq_c[live][:, :I], qh["codes"])
    np.testing.assert_array_equal(hq_sf[live][:, :I // 16], qh["sf"])
    np.testing.assert_array_equal(gh_all[live], qh["g"])
    # weighted un-permute of the GPU's own y: every token, element-wise
    assert combine_violations(u16(out), y_all, pi["inv"], npy(w)) == 0
    # sampled tokens end to end
    toks = [0, 1, 4095, 8191, shape.T - 1]
    sub_e = sorted(set(rid[toks].reshape(-1).tolist()))
    pref = {"w13_codes": {}, "w13_sf": {}, "w13_g": {}, "w2_codes": {}, "w2_sf": {}, "w2_g": {}}
    for e in sub_e:
        q13, q2 = cache.get(e) or (Q.quantize(w13b[e], scope="tensor"), Q.quantize(w2b[e], scope="tensor"))
        pref["w13_codes"][e], pref["w13_sf"][e], pref["w13_g"][e] = q13["codes"], q13["sf"], q13["g"][0]
        pref["w2_codes"][e], pref["w2_sf"][e], pref["w2_g"][e] = q2["codes"], q2["sf"], q2["g"][0]
    oref = M.moe_forward_tokens(xb, rid, rw, pref, toks)
    got = F.bf16_to_f32(u16(out)[toks]).astype(np.float64)
    ref = F.bf16_to_f32(oref).astype(np.float64)
    _, nw = rel_err_floor(got, ref)
    assert nw < 1e-2, nw
    # row invariance: the first 1024 tokens alone
    part = u16(cuda_lib.moe_expert_forward(xc[:1024].contiguous(), ids[:1024].contiguous(),
                                           w[:1024].contiguous(), pw))
    np.testing.assert_array_equal(part, u16(out)[:1024])


@pytest.mark.slow
def test_gateup_workload_full_size_sampled(cuda_lib):
    """The gate/up grouped-GEMM workload (T=8192 top-8 of 128 experts, Zipf(1.1) routing:
    65,536 routed rows, K=2048, N=1536, BF16 out), in the launch the benchmark times:
    nvfp4_grouped_gemm_tiled with the plain store over the forward's own grouped operand.
    Sampled rows are checked against the oracle GEMM; output columns follow the prepared
    W13 row order (gate and up interleaved in chunks of 64)."""
    shape = S.WORKLOADS["gateup"]
    T, H, I, E, k = shape.T, shape.H, shape.I, shape.E, shape.k
    x, logits, w13, w2 = S.moe_inputs(shape, seed=1)
    ids, w = cuda_lib.moe_route_topk(logits.cuda(), k)
    rid, _ = M.route_topk(logits.numpy(), k)
    pw = cuda_lib.moe_prepare_weights(w13.cuda(), w2.cuda())
    _, v = _forward(cuda_lib, x.cuda(), ids, w, pw, T, k)
    pi = M.permute(rid, E)
    d = cuda_lib.nvfp4_grouped_gemm_tiled(v["aq"], v["ga"], pw.w13, pw.w13_g, v["padded"], v["counts"], v["mcap"],
                                          2 * I, H, E, out_dtype=torch.bfloat16)
    assert cuda_lib.nvfp4_status_check() == 0
    d_all = u16(d)
    orig = interleave_src(I)   # column j of the prepared order holds W13 row orig[j]
    live = np.nonzero(pi["perm"] >= 0)[0]
    rng = np.random.default_rng(1)
    sample = np.sort(rng.choice(live, 64, replace=False))
    experts = np.searchsorted(pi["padded_offsets"], sample, side="right") - 1
    xb, w13b = S.bf16_bits(x), S.bf16_bits(w13)
    qx = Q.quantize(xb, scope="row")
    cache = {}
    for s_row, e in zip(sample, experts):
        if e not in cache:
            cache[e] = Q.quantize(w13b[e], scope="tensor")
        q13 = cache[e]
        t = pi["perm"][s_row]
        dref = M.gemm_rows(qx["codes"][t:t + 1], qx["sf"][t:t + 1], qx["g"][t:t + 1], q13["codes"], q13["sf"],
                           q13["g"][0])
        nbad, worst = check_bf16_against(d_all[s_row:s_row + 1], dref[:, orig])
        assert nbad == 0, (s_row, worst)


@pytest.mark.parametrize("sizes", [(1, 7, 64), (3, 16, 33)])
def test_decode_shaped_launches_match_the_learner_shaped_launch(cuda_lib, sizes):
    """Execution alignment between a sampler-shaped and a learner-shaped launch ("Low-Bit
    Precision Training Is Ready for Production...", §"The Cross-Engine Alignment Problem"):
    tokens run through decode-size batches (1 to 64 tokens, one or a few row tiles per
    expert, most experts empty) give exactly the bits the same tokens get inside the full
    16,384-token batch of the forward workload, whose groups span many row tiles."""
    shape = S.WORKLOADS["forward"]
    x, logits, w13, w2 = S.moe_inputs(shape, seed=3)
    ids, w = cuda_lib.moe_route_topk(logits.cuda(), shape.k)
    pw = cuda_lib.moe_prepare_weights(w13.cuda(), w2.cuda())
    xc = x.cuda()
    learner = u16(cuda_lib.moe_expert_forward(xc, ids, w, pw))
    start = 5000
    for n in sizes:
        sl = slice(start, start + n)
        dec = u16(cuda_lib.moe_expert_forward(xc[sl].contiguous(), ids[sl].contiguous(), w[sl].contiguous(), pw))
        np.testing.assert_array_equal(dec, learner[sl])
        # the router too: top-k of a decode batch equals the rows of the full launch
        dids, dw = cuda_lib.moe_route_topk(logits[sl].contiguous().cuda(), shape.k)
        np.testing.assert_array_equal(npy(dids), npy(ids)[sl])
        np.testing.assert_array_equal(npy(dw), npy(w)[sl])
        start += n

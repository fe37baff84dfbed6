"""GPU parity of the W4A4 grouped GEMM against the oracle over the same quantised
operands: exact cases bit for bit, random cases within 1e-3 relative (float32 output)
or one BF16 ulp plus that allowance (BF16 output), ragged groups of 0, 1, 127, 128 and
129+ rows, several row / column / K tiles."""
import numpy as np
import pytest
import torch

from gpu_util import check_bf16_against, dev, npy, rel_err_floor, u16
from oracle import formats as F
from oracle import moe as M
from oracle import quant as Q
from nvfp4_w4a4_moe_quantize_gb300 import synthetic as S

pytestmark = pytest.mark.gpu


def _groups(counts):
    counts = np.asarray(counts, np.int64)
    padded = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)])
    return counts.astype(np.int32), padded.astype(np.int32)


def _operands_from_oracle(a_bits, counts, w_bits, a_scope="row"):
    """Quantise with the oracle and lay the operands out the way the kernel reads them."""
    E, N, K = w_bits.shape
    counts, padded = _groups(counts)
    M = int(padded[-1]) if padded[-1] > 0 else 128
    qa = Q.quantize(a_bits, scope=a_scope)
    a_codes = np.zeros((M, K), np.uint8)
    a_sf = np.zeros((M, K // 16), np.uint8)
    a_g = np.zeros(M, np.float32)
    r = 0
    for e in range(E):
        n = int(counts[e])
        a_codes[padded[e]:padded[e] + n] = qa["codes"][r:r + n]
        a_sf[padded[e]:padded[e] + n] = qa["sf"][r:r + n]
        a_g[padded[e]:padded[e] + n] = qa["g"][r:r + n] if a_scope == "row" else qa["g"][0]
        r += n
    qb = Q.quantize(w_bits.reshape(E * N, K), scope="group", group_rows=N)
    ops = dict(a_codes=a_codes, a_sf=a_sf, a_g=a_g, b_codes=qb["codes"].reshape(E, N, K),
               b_sf=qb["sf"].reshape(E, N, K // 16), b_g=qb["g"], counts=counts, padded=padded, M=M)
    return ops


def _run_gpu(lib, ops, N, K, out_dtype):
    E = ops["b_codes"].shape[0]
    A = dev(F.pack_e2m1(ops["a_codes"]))
    SFA = dev(F.sf_swizzle(ops["a_sf"]))
    B = dev(F.pack_e2m1(ops["b_codes"].reshape(E * N, K)))
    SFB = dev(F.sf_swizzle(ops["b_sf"].reshape(E * N, K // 16)))
    D = lib.nvfp4_grouped_gemm(A, SFA, dev(ops["a_g"]), B, SFB, dev(ops["b_g"]), dev(ops["padded"]),
                               dev(ops["counts"]), N, K, E, out_dtype=out_dtype)
    assert lib.nvfp4_status_check() == 0
    return D


def _oracle(ops):
    return M.grouped_gemm(ops["a_codes"], ops["a_sf"], ops["a_g"], ops["b_codes"], ops["b_sf"], ops["b_g"],
                          ops["padded"], ops["counts"])


def _valid_rows(ops):
    return np.concatenate([np.arange(p, p + c) for p, c in zip(ops["padded"][:-1], ops["counts"])]).astype(int)


@pytest.mark.parametrize("N", [128, 256])
def test_gemm_single_tile_exact(cuda_lib, N):
    """One expert, one 128xN tile (both tile widths of the kernel), K = 256; E2M1 grid
    values times powers of two so every partial sum is exact in float32: the result
    must be bit-exact."""
    rng = np.random.default_rng(0)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -2, -3, -4, -6])
    s_a, s_w = 448 * 2.0 ** -11, 448 * 2.0 ** -13
    xa = rng.choice(grid, (128, 256)) * s_a
    xa[:, ::16] = 6 * s_a
    w = rng.choice(grid, (1, N, 256)) * s_w
    w[:, :, ::16] = 6 * s_w
    ops = _operands_from_oracle(F.bf16_round(xa), [128], F.bf16_round(w))
    ref = _oracle(ops)
    D = npy(_run_gpu(cuda_lib, ops, N, 256, torch.float32))
    np.testing.assert_array_equal(D, ref.astype(np.float32))
    np.testing.assert_array_equal(ref, (xa @ w[0].T))          # lossless quantisation


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("N", [384, 512])
def test_gemm_ragged_groups(cuda_lib, out_dtype, N):
    E, K = 6, 512
    counts = [0, 1, 127, 128, 129, 300]
    a_bits = S.bf16_bits(S.randn_bf16((sum(counts), K), seed=31))
    w_bits = S.bf16_bits(S.randn_bf16((E, N, K), 0.02, seed=32))
    ops = _operands_from_oracle(a_bits, counts, w_bits)
    ref = _oracle(ops)
    D = _run_gpu(cuda_lib, ops, N, K, out_dtype)
    rows = _valid_rows(ops)
    if out_dtype == torch.float32:
        mx, nw = rel_err_floor(npy(D)[rows], ref[rows])
        assert mx <= 1e-3, (mx, nw)
        assert nw <= 1e-5
    else:
        nbad, worst = check_bf16_against(u16(D)[rows], ref[rows])
        assert nbad == 0, worst


def test_gemm_qwen_shaped_k_and_many_experts(cuda_lib):
    """K = 2048 (8 K-stages), N = 1536, 16 experts with Zipf-like group sizes."""
    E, N, K = 16, 1536, 2048
    rng = np.random.default_rng(7)
    counts = list(rng.integers(0, 400, E))
    counts[3] = 0
    a_bits = S.bf16_bits(S.randn_bf16((sum(counts), K), seed=41))
    w_bits = S.bf16_bits(S.randn_bf16((E, N, K), 0.02, seed=42))
    ops = _operands_from_oracle(a_bits, counts, w_bits)
    ref = _oracle(ops)
    D = npy(_run_gpu(cuda_lib, ops, N, K, torch.float32))
    rows = _valid_rows(ops)
    mx, nw = rel_err_floor(D[rows], ref[rows])
    assert mx <= 1e-3, (mx, nw)


@pytest.mark.parametrize("N", [128, 256])
def test_gemm_leaves_rows_outside_groups_untouched(cuda_lib, N):
    E, K = 2, 256
    counts = [5, 130]
    a_bits = S.bf16_bits(S.randn_bf16((sum(counts), K), seed=51))
    w_bits = S.bf16_bits(S.randn_bf16((E, N, K), 0.02, seed=52))
    ops = _operands_from_oracle(a_bits, counts, w_bits)
    A = dev(F.pack_e2m1(ops["a_codes"]))
    out = torch.full((ops["M"], N), 7.0, dtype=torch.float32, device="cuda")
    cuda_lib.nvfp4_grouped_gemm(A, dev(F.sf_swizzle(ops["a_sf"])), dev(ops["a_g"]),
                                dev(F.pack_e2m1(ops["b_codes"].reshape(E * N, K))),
                                dev(F.sf_swizzle(ops["b_sf"].reshape(E * N, K // 16))), dev(ops["b_g"]),
                                dev(ops["padded"]), dev(ops["counts"]), N, K, E, out=out)
    o = npy(out)
    valid = np.zeros(ops["M"], bool)
    valid[_valid_rows(ops)] = True
    assert np.all(o[~valid] == 7.0)
    assert not np.any(o[valid] == 7.0)


def test_gemm_is_deterministic(cuda_lib):
    E, N, K = 4, 256, 1024
    counts = [300, 17, 0, 200]
    a_bits = S.bf16_bits(S.randn_bf16((sum(counts), K), seed=61))
    w_bits = S.bf16_bits(S.randn_bf16((E, N, K), 0.02, seed=62))
    ops = _operands_from_oracle(a_bits, counts, w_bits)
    d1 = npy(_run_gpu(cuda_lib, ops, N, K, torch.float32))
    d2 = npy(_run_gpu(cuda_lib, ops, N, K, torch.float32))
    rows = _valid_rows(ops)
    np.testing.assert_array_equal(d1[rows], d2[rows])


# ------------------------------------------------------------------ GEMM-tiled operands

@pytest.fixture(params=["pair", "single"])
def cta_mode(request, monkeypatch):
    """The GEMM-tiled kernel in both forms: one CTA per M=128 tile (the default) and a
    CTA pair per M=256 tile (NVFP4_GEMM_CTA_PAIR=1)."""
    monkeypatch.setenv("NVFP4_GEMM_CTA_PAIR", "1" if request.param == "pair" else "0")
    return request.param


def _run_tiled(lib, ops, N, K, out_dtype=torch.float32, epilogue=0):
    from gpu_util import pack_tiled_host
    E = ops["b_codes"].shape[0]
    A = dev(pack_tiled_host(ops["a_codes"], ops["a_sf"], 128))
    B = dev(pack_tiled_host(ops["b_codes"].reshape(E * N, K), ops["b_sf"].reshape(E * N, K // 16), 256))
    D = lib.nvfp4_grouped_gemm_tiled(A, dev(ops["a_g"]), B, dev(ops["b_g"]), dev(ops["padded"]), dev(ops["counts"]),
                                     ops["M"], N, K, E, out_dtype=out_dtype, epilogue=epilogue)
    assert lib.nvfp4_status_check() == 0
    return D


def test_tiled_gemm_exact_single_tile(cuda_lib, cta_mode):
    rng = np.random.default_rng(0)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -2, -3, -4, -6])
    s_a, s_w = 448 * 2.0 ** -11, 448 * 2.0 ** -13
    xa = rng.choice(grid, (128, 512)) * s_a
    xa[:, ::16] = 6 * s_a
    w = rng.choice(grid, (1, 256, 512)) * s_w
    w[:, :, ::16] = 6 * s_w
    ops = _operands_from_oracle(F.bf16_round(xa), [128], F.bf16_round(w))
    D = npy(_run_tiled(cuda_lib, ops, 256, 512))
    np.testing.assert_array_equal(D, (xa @ w[0].T).astype(np.float32))


def _lossless_blocks(rng, rows, K, s, kmin=2):
    """Values on the E2M1 grid times s * 2^(k-4), one k in [kmin, 4] per 16-value block,
    each block holding a +-6 (so its scale is exactly s * 2^(k-4)) and each row one block
    with k = 4 (so the row's global scale is exact): quantisation is lossless and every
    partial sum of a K <= 512 product is a float32 number."""
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6, -0.5, -1, -2, -3, -4, -6])
    k = rng.integers(kmin, 5, (rows, K // 16))
    k[:, 0] = 4
    x = rng.choice(grid, (rows, K)) * s * np.repeat(2.0 ** (k - 4), 16, axis=1)
    x[:, ::16] = rng.choice([-6.0, 6.0], (rows, K // 16)) * s * 2.0 ** (k - 4)
    return x


def test_tiled_gemm_exact_block_scales_and_odd_row_blocks(cuda_lib, cta_mode):
    """Bit-exact products with a different scale in every 16-value block of A and of W,
    on groups of 3, 1 and 2 row blocks (the CTA pair's last pair of a group with an odd
    block count has an empty second half): any scale read from the wrong row, column or
    K block shows."""
    rng = np.random.default_rng(7)
    E, N, K = 3, 512, 512
    counts = [269, 128, 256]
    xa = _lossless_blocks(rng, sum(counts), K, 448 * 2.0 ** -11)
    w = np.stack([_lossless_blocks(rng, N, K, 448 * 2.0 ** -13) for _ in range(E)])
    ops = _operands_from_oracle(F.bf16_round(xa), counts, F.bf16_round(w))
    D = npy(_run_tiled(cuda_lib, ops, N, K))
    r = 0
    for e, c in enumerate(counts):
        p = int(ops["padded"][e])
        want = (xa[r:r + c] @ w[e].T).astype(np.float32)
        np.testing.assert_array_equal(D[p:p + c], want)
        r += c


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_tiled_gemm_ragged_groups_matches_oracle_and_row_major_kernel(cuda_lib, out_dtype, cta_mode):
    E, N, K = 6, 512, 768
    counts = [0, 1, 127, 128, 129, 300]
    a_bits = S.bf16_bits(S.randn_bf16((sum(counts), K), seed=71))
    w_bits = S.bf16_bits(S.randn_bf16((E, N, K), 0.02, seed=72))
    ops = _operands_from_oracle(a_bits, counts, w_bits)
    ref = _oracle(ops)
    Dt = _run_tiled(cuda_lib, ops, N, K, out_dtype)
    Dr = _run_gpu(cuda_lib, ops, N, K, out_dtype)
    rows = _valid_rows(ops)
    if out_dtype == torch.float32:
        mx, nw = rel_err_floor(npy(Dt)[rows], ref[rows])
        assert mx <= 1e-3, (mx, nw)
    else:
        nbad, worst = check_bf16_against(u16(Dt)[rows], ref[rows])
        assert nbad == 0, worst
    # same MMA sequence as the row-major kernel: identical bits
    np.testing.assert_array_equal(npy(Dt.view(torch.int32) if out_dtype == torch.float32 else Dt.view(torch.int16))[rows],
                                  npy(Dr.view(torch.int32) if out_dtype == torch.float32 else Dr.view(torch.int16))[rows])


def test_pack_tiled_matches_host_layout(cuda_lib):
    from gpu_util import pack_tiled_host
    rows, K = 300, 512
    bits = S.bf16_bits(S.randn_bf16((rows, K), seed=81))
    x = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).cuda()
    codes, sf, _ = cuda_lib.nvfp4_quantize(x, cuda_lib.SCALE_PER_ROW)
    q = Q.quantize(bits, scope="row")
    for R in (128, 256):
        got = npy(cuda_lib.nvfp4_pack_tiled(codes, sf, rows, K, R))
        np.testing.assert_array_equal(got, pack_tiled_host(q["codes"], q["sf"], R))


def test_tiled_swiglu_epilogue_equals_standalone_swiglu(cuda_lib, cta_mode):
    """gate/up GEMM with the SwiGLU epilogue == BF16 GEMM output followed by the
    standalone SwiGLU kernel (64-row interleaved gate/up weights), bit for bit."""
    E, I, K = 3, 256, 512
    counts = [200, 0, 77]
    a_bits = S.bf16_bits(S.randn_bf16((sum(counts), K), seed=91))
    w_bits = S.bf16_bits(S.randn_bf16((E, 2 * I, K), 0.05, seed=92))
    ops = _operands_from_oracle(a_bits, counts, w_bits)
    # rows whose global scale is blown up or shrunk: gate values below -80 and products
    # outside [2^-100, 2^100] leave the float32 path for many values of one row, so the
    # epilogue's deferred exact path runs with more than two values per row and tile,
    # in full 32-row slabs and in the partial slab of the last group
    ops["a_g"][0:64] *= 3000.0
    ops["a_g"][64:96] *= 1e-30
    ops["a_g"][256 + 40:256 + 77] *= 3000.0
    h_fused = u16(_run_tiled(cuda_lib, ops, 2 * I, K, epilogue=1))
    D = _run_gpu(cuda_lib, ops, 2 * I, K, torch.bfloat16)
    perm = np.full(ops["M"], -1, np.int32)
    perm[_valid_rows(ops)] = 0
    h, _, _, _ = cuda_lib.moe_swiglu_quantize(D, dev(perm), I)
    rows = _valid_rows(ops)
    np.testing.assert_array_equal(h_fused[rows], u16(h)[rows])
    # and against the oracle's SwiGLU of the same BF16 gate/up values
    j = np.arange(2 * I)
    src = np.where(j % 128 < 64, (j // 128) * 64 + j % 128, I + (j // 128) * 64 + j % 128 - 64)
    d_il = u16(D)[rows]
    d_can = np.empty_like(d_il)
    d_can[:, src] = d_il
    np.testing.assert_array_equal(h_fused[rows], M.swiglu(d_can, I))
    gate = F.bf16_to_f32(d_can[:, :I])
    assert (gate < -80).sum() > 2000            # the exact path did run, many per row


@pytest.mark.parametrize("N", [128, 256])
@pytest.mark.parametrize("fault", ["rows_over_span", "offsets_past_m_total", "unaligned_offset"])
def test_gemm_rejects_inconsistent_group_arrays(cuda_lib, N, fault, cta_mode):
    """Group arrays that break the documented contract (rows[e] larger than its padded
    span, offsets past M_total, a start that is not a multiple of 128) set the device
    status and leave D untouched, on both tile widths and on the GEMM-tiled kernel."""
    E, K = 2, 256
    counts = [100, 60]
    a_bits = S.bf16_bits(S.randn_bf16((sum(counts), K), seed=51))
    w_bits = S.bf16_bits(S.randn_bf16((E, N, K), 0.02, seed=52))
    ops = _operands_from_oracle(a_bits, counts, w_bits)
    rows, padded = ops["counts"].copy(), ops["padded"].copy()
    if fault == "rows_over_span":
        rows[0] = 129
    elif fault == "offsets_past_m_total":
        padded[-1] = ops["M"] + 128
    else:
        padded[1] = 64
    A = dev(F.pack_e2m1(ops["a_codes"]))
    SFA = dev(F.sf_swizzle(ops["a_sf"]))
    B = dev(F.pack_e2m1(ops["b_codes"].reshape(E * N, K)))
    SFB = dev(F.sf_swizzle(ops["b_sf"].reshape(E * N, K // 16)))
    sentinel = torch.full((ops["M"], N), 7.0, dtype=torch.float32, device="cuda")
    D = sentinel.clone()
    cuda_lib.nvfp4_grouped_gemm(A, SFA, dev(ops["a_g"]), B, SFB, dev(ops["b_g"]), dev(padded), dev(rows), N, K, E,
                                out=D)
    assert cuda_lib.nvfp4_status_check() == cuda_lib.Status.DEVICE_STATUS
    assert torch.equal(D, sentinel)
    if N == 256:
        At = cuda_lib.nvfp4_pack_tiled(A, SFA, ops["M"], K, 128)
        Bt = cuda_lib.nvfp4_pack_tiled(B, SFB, E * N, K, 256)
        D2 = sentinel.clone()
        cuda_lib.nvfp4_grouped_gemm_tiled(At, dev(ops["a_g"]), Bt, dev(ops["b_g"]), dev(padded), dev(rows),
                                          ops["M"], N, K, E, out=D2)
        assert cuda_lib.nvfp4_status_check() == cuda_lib.Status.DEVICE_STATUS
        assert torch.equal(D2, sentinel)

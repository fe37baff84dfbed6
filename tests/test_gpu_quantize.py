"""GPU parity of the NVFP4 quantiser against the oracle: codes, scales and global scales
bit for bit, in every scope and rounding mode, including ragged shapes and degenerate
inputs."""
import numpy as np
import pytest
import torch

from conftest import read_golden
from gpu_util import bf16_tensor, dev, npy, u16
from oracle import formats as F
from oracle import quant as Q
from nvfp4_w4a4_moe_quantize_gb300 import synthetic as S

pytestmark = pytest.mark.gpu

MODES = {"tensor": 0, "row": 1, "group": 2}


def _gpu_quant(lib, bits, scope, rounding="rne", seed=0, off=0, group_rows=0, g_in=None):
    x = bf16_tensor(bits)
    codes, sf, g = lib.nvfp4_quantize(x, MODES[scope], 1 if rounding == "sr" else 0, seed, off, group_rows,
                                      None if g_in is None else dev(np.asarray(g_in, np.float32)))
    assert lib.nvfp4_status_check() == 0
    return npy(codes), npy(sf), npy(g)


def _compare(lib, bits, scope, rounding="rne", seed=0, off=0, group_rows=0, g_in=None):
    rows, cols = bits.shape
    codes, sf, g = _gpu_quant(lib, bits, scope, rounding, seed, off, group_rows, g_in)
    ref = Q.quantize(bits, scope=scope, rounding=rounding, seed=seed, rng_offset=off,
                     group_rows=group_rows or None, global_scale_in=g_in)
    np.testing.assert_array_equal(g[:ref["g"].size], ref["g"])
    np.testing.assert_array_equal(codes, ref["packed"])
    np.testing.assert_array_equal(sf, F.sf_swizzle(ref["sf"]))
    return ref


@pytest.mark.parametrize("scope", ["tensor", "row"])
@pytest.mark.parametrize("shape", [(1, 16), (3, 48), (130, 272), (257, 2048), (64, 4096)])
def test_quantize_rne_matches_oracle(cuda_lib, scope, shape):
    bits = S.bf16_bits(S.outlier_channels_bf16(*shape, seed=shape[0] * 7 + shape[1]))
    _compare(cuda_lib, bits, scope)


@pytest.mark.parametrize("shape", [(130, 272), (256, 2048)])
def test_quantize_sr_matches_oracle(cuda_lib, shape):
    bits = S.bf16_bits(S.randn_bf16(shape, seed=11))
    for seed, off in [(0, 0), (0xDEADBEEF12345, 77)]:
        _compare(cuda_lib, bits, "tensor", "sr", seed, off)
        _compare(cuda_lib, bits, "row", "sr", seed, off)


@pytest.mark.parametrize("scope", ["tensor", "row"])
@pytest.mark.parametrize("shape", [(5, 64), (130, 2048), (33, 4096)])
def test_quantize_rowmajor_scales(cuda_lib, scope, shape):
    """The row-major scale layout: the same codes and g as the tiled call, and scales that
    equal the oracle's [rows, cols/16] bytes (the tiled layout's padding does not exist)."""
    bits = S.bf16_bits(S.outlier_channels_bf16(*shape, seed=shape[0] + 3))
    x = bf16_tensor(bits)
    codes, sf, g = cuda_lib.nvfp4_quantize(x, MODES[scope], sf_layout=cuda_lib.SF_ROWMAJOR)
    assert cuda_lib.nvfp4_status_check() == 0
    ref = Q.quantize(bits, scope=scope)
    assert tuple(sf.shape) == (shape[0], shape[1] // 16)
    np.testing.assert_array_equal(npy(sf), ref["sf"])
    np.testing.assert_array_equal(npy(codes), ref["packed"])
    np.testing.assert_array_equal(npy(g)[:ref["g"].size], ref["g"])
    for rounding in (1,):
        c2, sf2, _ = cuda_lib.nvfp4_quantize(x, MODES[scope], rounding, 5, 9, sf_layout=cuda_lib.SF_ROWMAJOR)
        ref2 = Q.quantize(bits, scope=scope, rounding="sr", seed=5, rng_offset=9)
        np.testing.assert_array_equal(npy(c2), ref2["packed"])
        np.testing.assert_array_equal(npy(sf2), ref2["sf"])


def test_quantize_group_scope(cuda_lib):
    bits = S.bf16_bits(S.randn_bf16((4 * 96, 512), 0.02, seed=5))
    _compare(cuda_lib, bits, "group", group_rows=96)


def test_worked_example_on_gpu(cuda_lib):
    gd = read_golden("quant_worked_example.txt")
    x = np.array([int(t, 16) for t in gd["x_bf16"].split()], np.uint16).reshape(1, 32)
    codes, sf, g = _gpu_quant(cuda_lib, x, "row")
    assert list(codes[0]) == [int(t, 16) for t in gd["packed"].split()]
    assert list(F.sf_unswizzle(sf, 1, 2)[0]) == [int(t, 16) for t in gd["sf"].split()]
    assert g[0] == np.float32(float(gd["g"]))


def test_every_bf16_value_and_every_tie(cuda_lib):
    """All finite BF16 patterns, quantised with forced global scales so that every E2M1
    tie, the saturation region and E4M3 subnormal block scales all occur."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    fin = np.isfinite(F.bf16_to_f32(bits))
    bits = bits[fin]
    bits = bits[: bits.size // 256 * 256].reshape(-1, 256)
    for g in (np.float32(2.0 ** -10), np.float32(1.0), np.float32(1e-20), np.float32(6.0 / 2688)):
        _compare(cuda_lib, bits, "tensor", g_in=[g])
        _compare(cuda_lib, bits, "tensor", "sr", 3, 0, g_in=[g])
    _compare(cuda_lib, bits, "row")


def test_degenerate_rows(cuda_lib):
    bits = np.zeros((5, 64), np.uint16)
    bits[1] = 0x0001                         # smallest subnormal
    bits[2, ::3] = 0x8000                    # negative zeros
    bits[3] = F.bf16_round(np.linspace(-1e-38, 1e-38, 64))
    bits[4, 7] = 0x7F7F                      # largest finite BF16
    for scope in ("row", "tensor"):
        _compare(cuda_lib, bits, scope)


def test_quantize_is_deterministic(cuda_lib):
    bits = S.bf16_bits(S.randn_bf16((512, 2048), seed=21))
    a = _gpu_quant(cuda_lib, bits, "tensor", "sr", 5)
    b = _gpu_quant(cuda_lib, bits, "tensor", "sr", 5)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)


def test_quantiser_workload_full_size(cuda_lib):
    """The standalone-quantiser workload at full size (16384 x 2048, 1% outlier channels),
    per-tensor scale, RNE and SR, against the oracle over the whole tensor."""
    bits = S.bf16_bits(S.outlier_channels_bf16(*S.QUANTISER_SHAPE, seed=0))
    _compare(cuda_lib, bits, "tensor")
    _compare(cuda_lib, bits, "tensor", "sr", 0, 0)


def test_bad_arguments_raise(cuda_lib):
    x = torch.zeros(4, 24, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cuda_lib.NVFP4Error):
        cuda_lib.nvfp4_quantize(x)


@pytest.mark.parametrize("scope", ["tensor", "row", "group"])
@pytest.mark.parametrize("shape", [(1, 16), (130, 272), (256, 2048)])
def test_dequantize_matches_oracle(cuda_lib, scope, shape):
    """DQ(Q(x)) on the GPU equals the oracle's exact float64 dequantisation rounded once:
    BF16 and float32 outputs, bit for bit -- including rows whose tiny global scale puts
    values in the BF16 subnormal range and rows of zeros."""
    rows, cols = shape
    rng = np.random.default_rng(rows + cols)
    x = rng.standard_normal((rows, cols)) * rng.choice([1e-36, 1e-3, 1.0, 300.0], (rows, 1))
    x[0, :16] = 0.0
    xb = F.bf16_round(x)
    group_rows = 2 if scope == "group" and rows % 2 == 0 else 0
    if scope == "group" and group_rows == 0:
        pytest.skip("group scope needs rows divisible by the group")
    q = Q.quantize(xb, scope=scope, group_rows=group_rows if group_rows else None)
    codes = dev(F.pack_e2m1(q["codes"]))
    sf = dev(F.sf_swizzle(q["sf"]))
    g = dev(np.asarray(q["g"], np.float32))
    mode = {"tensor": cuda_lib.SCALE_PER_TENSOR, "row": cuda_lib.SCALE_PER_ROW, "group": cuda_lib.SCALE_PER_GROUP}[scope]
    g_rows = np.asarray(q["g"], np.float64)
    if scope == "tensor":
        g_rows = np.full(rows, g_rows[0])
    elif scope == "group":
        g_rows = np.repeat(g_rows, group_rows)
    exact = Q.dequantize(q["codes"], q["sf"], g_rows)
    got_bf16 = u16(cuda_lib.nvfp4_dequantize(codes, sf, g, cols, mode, group_rows))
    np.testing.assert_array_equal(got_bf16, F.bf16_round(exact))
    got_f32 = npy(cuda_lib.nvfp4_dequantize(codes, sf, g, cols, mode, group_rows, out_dtype=torch.float32))
    np.testing.assert_array_equal(got_f32.view(np.uint32), exact.astype(np.float32).view(np.uint32))


def test_dequantize_every_scale_and_code(cuda_lib):
    """DQ of every (E4M3 scale byte, E2M1 code) pair under per-row global scales from the
    subnormal BF16 range to near the top of the float32 range: BF16 and float32 outputs
    equal the oracle's exact dequantisation rounded once, bit for bit."""
    sfb = np.arange(127, dtype=np.uint8)                     # every finite E4M3 scale byte
    gs = np.array([1.0, 1.0 / 2688, 3.7e-5, 2.0 ** -126, 1e-38, 7.1e-42, 1e-30, 3e30, 2.0 ** 120, 0.0], np.float32)
    rows = sfb.size * gs.size
    codes = np.tile(np.arange(16, dtype=np.uint8), (rows, 1))
    sf = np.tile(sfb, gs.size).reshape(rows, 1)
    g_rows = np.repeat(gs, sfb.size)
    exact = Q.dequantize(codes, sf, g_rows.astype(np.float64))
    c = dev(F.pack_e2m1(codes))
    s_ = dev(F.sf_swizzle(sf))
    g = dev(g_rows)
    got_bf16 = u16(cuda_lib.nvfp4_dequantize(c, s_, g, 16, cuda_lib.SCALE_PER_ROW, 0))
    np.testing.assert_array_equal(got_bf16, F.bf16_round(exact))
    got_f32 = npy(cuda_lib.nvfp4_dequantize(c, s_, g, 16, cuda_lib.SCALE_PER_ROW, 0, out_dtype=torch.float32))
    np.testing.assert_array_equal(got_f32.view(np.uint32), exact.astype(np.float32).view(np.uint32))


@pytest.mark.parametrize("scope", ["tensor", "row", "group"])
@pytest.mark.parametrize("rounding", ["rne", "sr"])
@pytest.mark.parametrize("shape", [(3, 48, 40), (1, 256, 2048), (2, 2048, 72)])
def test_quantize_transposed_matches_oracle(cuda_lib, scope, rounding, shape):
    """Transposed quantisation (blocks of 16 along the original rows) equals the oracle's
    quantisation of the stacked transposes, codes / scales / global scales bit for bit,
    for every scope and both roundings (group = one scale per stacked matrix)."""
    B, R, C = shape
    rng = np.random.default_rng(B * R + C)
    x = rng.standard_normal((B, R, C)) * rng.choice([1e-3, 1.0, 40.0], (B, 1, C))
    xb = F.bf16_round(x)
    xt = np.ascontiguousarray(xb.transpose(0, 2, 1)).reshape(B * C, R)
    group_rows = C if scope == "group" else 0
    q = Q.quantize(xt, scope=scope, rounding=rounding, seed=11, group_rows=group_rows if group_rows else None)
    mode = {"tensor": cuda_lib.SCALE_PER_TENSOR, "row": cuda_lib.SCALE_PER_ROW, "group": cuda_lib.SCALE_PER_GROUP}[scope]
    rnd = cuda_lib.ROUND_RNE if rounding == "rne" else cuda_lib.ROUND_STOCHASTIC
    codes, sf, g = cuda_lib.nvfp4_quantize_transposed(bf16_tensor(xb.reshape(B, R, C)), mode, rnd, seed=11,
                                                      group_rows=group_rows)
    np.testing.assert_array_equal(npy(codes), q["packed"])
    np.testing.assert_array_equal(F.sf_unswizzle(npy(sf), B * C, R // 16), q["sf"])
    np.testing.assert_array_equal(npy(g), np.asarray(q["g"], np.float32))


def test_down_projection_dgrad_w4a4(cuda_lib):
    """The dgrad GEMM of the down projection in W4A4: dh[r, i] = sum_h dY[r, h] W2_e[h, i]
    with dY quantised per row along H and each expert's W2 quantised transposed (blocks
    along H, one global scale per expert) -- the grouped GEMM over those operands against
    the oracle's float64 GEMM over the same dequantised operands."""
    from oracle import moe as M
    from gpu_util import check_bf16_against
    E, H, I = 3, 256, 256
    counts = np.array([200, 0, 77])
    padded = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)]).astype(np.int32)
    Mt = int(padded[-1])
    rng = np.random.default_rng(21)
    w2 = F.bf16_round(rng.standard_normal((E, H, I)) * 0.02)
    dy = np.zeros((Mt, H), np.uint16)
    for e in range(E):
        dy[padded[e]:padded[e] + counts[e]] = F.bf16_round(rng.standard_normal((counts[e], H)) * 1e-3)
    # GPU operands
    qa_c, qa_sf, qa_g = cuda_lib.nvfp4_quantize(bf16_tensor(dy), cuda_lib.SCALE_PER_ROW)
    qb_c, qb_sf, qb_g = cuda_lib.nvfp4_quantize_transposed(bf16_tensor(w2), cuda_lib.SCALE_PER_GROUP, group_rows=I)
    dh = cuda_lib.nvfp4_grouped_gemm(qa_c, qa_sf, qa_g, qb_c, qb_sf, qb_g, dev(padded),
                                     dev(counts.astype(np.int32)), I, H, E)
    # oracle: the same quantisation, then the float64 grouped GEMM
    qa = Q.quantize(dy, scope="row")
    w2t = np.ascontiguousarray(w2.transpose(0, 2, 1)).reshape(E * I, H)
    qb = Q.quantize(w2t, scope="group", group_rows=I)
    np.testing.assert_array_equal(npy(qb_c), qb["packed"])
    ref = M.grouped_gemm(qa["codes"], qa["sf"], qa["g"], qb["codes"].reshape(E, I, H), qb["sf"].reshape(E, I, H // 16),
                         qb["g"], padded, counts)
    rows = np.concatenate([np.arange(p, p + c) for p, c in zip(padded[:-1], counts)]).astype(int)
    nbad, worst = check_bf16_against(u16(dh)[rows], ref[rows])
    assert nbad == 0, worst


def test_expert_wgrad_w4a4_with_stochastic_rounding(cuda_lib):
    """The wgrad GEMM of an expert layer in W4A4: dW_e[n, h] = sum over the expert's
    tokens t of dY[t, n] X[t, h].  The contraction runs over each expert's own (ragged)
    token count, zero-padded to 256; dY is quantised transposed (blocks of 16 along tokens)
    with Philox stochastic rounding, X transposed with RNE, one global scale per expert
    matrix.  One GEMM per expert against the oracle's float64 GEMM over the same operands."""
    from oracle import moe as M
    from gpu_util import check_bf16_against
    N, H = 256, 256
    counts = [300, 77, 512]
    rng = np.random.default_rng(33)
    for e, n_tok in enumerate(counts):
        Tp = (n_tok + 255) // 256 * 256
        x = np.zeros((Tp, H), np.uint16)
        dy = np.zeros((Tp, N), np.uint16)
        x[:n_tok] = F.bf16_round(rng.standard_normal((n_tok, H)))
        dy[:n_tok] = F.bf16_round(rng.standard_normal((n_tok, N)) * 1e-3)
        seed = 100 + e
        a_c, a_sf, a_g = cuda_lib.nvfp4_quantize_transposed(bf16_tensor(dy), cuda_lib.SCALE_PER_TENSOR,
                                                            cuda_lib.ROUND_STOCHASTIC, seed=seed)
        b_c, b_sf, b_g = cuda_lib.nvfp4_quantize_transposed(bf16_tensor(x), cuda_lib.SCALE_PER_TENSOR)
        offs = dev(np.array([0, N], np.int32))
        dw = cuda_lib.nvfp4_grouped_gemm(a_c, a_sf, a_g.expand(N).contiguous(), b_c, b_sf, b_g, offs,
                                         dev(np.array([N], np.int32)), H, Tp, 1)
        qa = Q.quantize(np.ascontiguousarray(dy.T), scope="tensor", rounding="sr", seed=seed)
        qb = Q.quantize(np.ascontiguousarray(x.T), scope="tensor")
        np.testing.assert_array_equal(npy(a_c), qa["packed"])
        np.testing.assert_array_equal(npy(b_c), qb["packed"])
        ref = M.grouped_gemm(qa["codes"], qa["sf"], np.full(N, qa["g"][0]), qb["codes"][None], qb["sf"][None],
                             np.asarray(qb["g"], np.float64)[:1], np.array([0, N]), np.array([N]))
        nbad, worst = check_bf16_against(u16(dw), ref)
        assert nbad == 0, (e, worst)

"""GPU parity of the MXFP8 calls (mxfp8_quantize, mxfp8_dequantize, mxfp8_grouped_gemm)
against the MXFP8 oracle.  Codes, scales and DQ must match bit for bit.  The GEMM must be
bit-exact where every partial sum is exact in float32, and otherwise within 1e-3
relative (float32 out), or one BF16 ulp plus that (BF16 out).  Cases: ragged groups of
0, 1, 127, 128, 129 and 300 rows, several row / column / K tiles, and the edge values of
the format."""
import numpy as np
import pytest
import torch

from gpu_util import bf16_tensor, check_bf16_against, dev, npy, rel_err_floor, u16
from oracle import formats as F
from oracle import mx as X
from nvfp4_w4a4_moe_quantize_gb300 import synthetic as S

pytestmark = pytest.mark.gpu


def _quant_gpu(lib, bits, ld=None):
    rows, cols = bits.shape
    if ld is None:
        x = bf16_tensor(bits)
    else:
        full = np.zeros((rows, ld), np.uint16)
        full[:, :cols] = bits
        x = bf16_tensor(full)[:, :cols]
    codes, sf = lib.mxfp8_quantize(x)
    assert lib.nvfp4_status_check() == 0
    return npy(codes), npy(sf)


@pytest.mark.parametrize("shape,ld", [((1, 128), None), ((37, 256), None), ((129, 384), 392),
                                      ((300, 2048), None), ((1024, 1024), None)])
def test_quantize_matches_oracle(cuda_lib, shape, ld):
    bits = S.bf16_bits(S.randn_bf16(shape, 1.0, seed=shape[0] * 7 + shape[1]))
    # a spread of magnitudes so blocks take very different scales
    x = F.bf16_to_f32(bits).astype(np.float64)
    rng = np.random.default_rng(shape[0])
    x *= np.exp2(rng.integers(-40, 40, (shape[0], shape[1] // 32))).repeat(32, axis=1)
    bits = F.bf16_round(x)
    codes, sf = _quant_gpu(cuda_lib, bits, ld)
    rc, rsf = X.quantize(bits)
    np.testing.assert_array_equal(codes, rc)
    np.testing.assert_array_equal(sf, F.sf_swizzle(rsf))


def test_quantize_edge_values(cuda_lib):
    """Zero blocks, negative zero, BF16 subnormals, the largest finite BF16, values at
    and above the E4M3 saturation point, single-element blocks and ties, both signs."""
    rows = []
    rows.append(np.zeros(32))
    rows.append(np.full(32, -0.0))
    sub = F.bf16_to_f32(np.arange(1, 33, dtype=np.uint16)).astype(np.float64)      # subnormals
    rows.append(sub)
    rows.append(-sub)
    big = np.full(32, F.bf16_to_f32(np.array([0x7F7F], np.uint16))[0], np.float64)
    big[1::2] *= -1
    rows.append(big)
    top = np.array([256, 272, 288, 400, 404, 432, 448, 464, 480, 510] + [0] * 22, np.float64)
    rows.append(top)
    rows.append(-top * 2.0 ** -100)
    one = np.zeros(32)
    one[17] = 2.0 ** -126
    rows.append(one)
    mixed = np.array([2.0 ** k for k in range(-12, 20)], np.float64)
    rows.append(mixed)
    rows.append(-mixed[::-1] * 2.0 ** 90)
    tiny = np.zeros(32)
    tiny[0] = 1.0                              # shared exponent -8: t = x * 2^8
    tiny[1:] = 2.0 ** -18                      # t = 2^-10, the tie between 0 and 2^-9: +0
    tiny[2] = -2.0 ** -17                      # t = -2^-9, the smallest subnormal
    tiny[3] = -3 * 2.0 ** -19                  # t = -1.5 * 2^-10: rounds to -2^-9
    tiny[4] = -2.0 ** -19                      # t = -2^-11: rounds to zero, encoded +0
    rows.append(tiny)
    blocks = np.array(rows)
    # 4 blocks per row of 128 columns; repeat the pattern over 3 rows x 128 columns
    n = -(-blocks.shape[0] // 4) * 4
    pad = np.zeros((n - blocks.shape[0], 32))
    x = np.concatenate([blocks, pad]).reshape(-1, 128)
    x = np.concatenate([x, x[::-1], -x])
    bits = F.bf16_round(x)
    codes, sf = _quant_gpu(cuda_lib, bits)
    rc, rsf = X.quantize(bits)
    np.testing.assert_array_equal(codes, rc)
    np.testing.assert_array_equal(sf, F.sf_swizzle(rsf))


@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("rows,cols,ldo", [(1, 128, 128), (200, 256, 264), (333, 1024, 1024)])
def test_dequantize_matches_oracle(cuda_lib, out_dtype, rows, cols, ldo):
    rng = np.random.default_rng(rows + cols)
    codes = rng.integers(0, 256, (rows, cols)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x33                       # no NaN codes
    sf = rng.integers(0, 255, (rows, cols // 32)).astype(np.uint8)
    sf[:, ::5] = rng.integers(100, 140, sf[:, ::5].shape)      # many in the common range
    out = torch.zeros(rows, ldo, dtype=out_dtype, device="cuda")
    cuda_lib.mxfp8_dequantize(dev(codes), dev(F.sf_swizzle(sf)), out=out[:, :cols])
    assert cuda_lib.nvfp4_status_check() == 0
    if out_dtype == torch.bfloat16:
        got = u16(out[:, :cols])
        ref = X.dequantize(codes, sf, "bf16")
        np.testing.assert_array_equal(got, ref)
    else:
        got = npy(out[:, :cols])
        ref = X.dequantize(codes, sf, "f32")
        np.testing.assert_array_equal(got.view(np.uint32), ref.view(np.uint32))
    assert not np.any(npy(out[:, cols:].float()))             # the pitch padding is untouched


def test_dequantize_of_quantize_round_trip(cuda_lib):
    bits = S.bf16_bits(S.randn_bf16((256, 512), 2.0, seed=77))
    codes, sf = cuda_lib.mxfp8_quantize(bf16_tensor(bits))
    dq = cuda_lib.mxfp8_dequantize(codes, sf)
    rc, rsf = X.quantize(bits)
    np.testing.assert_array_equal(u16(dq), X.dequantize(rc, rsf, "bf16"))


# --------------------------------------------------------------------------- grouped GEMM

def _groups(counts):
    counts = np.asarray(counts, np.int64)
    padded = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)])
    return counts.astype(np.int32), padded.astype(np.int32)


def _operands(a_bits, counts, w_bits):
    E, N, K = w_bits.shape
    counts, padded = _groups(counts)
    M = int(padded[-1]) if padded[-1] > 0 else 128
    ac, asf = X.quantize(a_bits)
    a_codes = np.zeros((M, K), np.uint8)
    a_sf = np.zeros((M, K // 32), np.uint8)
    r = 0
    for e in range(E):
        n = int(counts[e])
        a_codes[padded[e]:padded[e] + n] = ac[r:r + n]
        a_sf[padded[e]:padded[e] + n] = asf[r:r + n]
        r += n
    wc, wsf = X.quantize(w_bits.reshape(E * N, K))
    return dict(a_codes=a_codes, a_sf=a_sf, b_codes=wc.reshape(E, N, K), b_sf=wsf.reshape(E, N, K // 32),
                counts=counts, padded=padded, M=M)


def _run(lib, ops, N, K, out_dtype):
    E = ops["b_codes"].shape[0]
    D = lib.mxfp8_grouped_gemm(dev(ops["a_codes"]), dev(F.sf_swizzle(ops["a_sf"])),
                               dev(ops["b_codes"].reshape(E * N, K)),
                               dev(F.sf_swizzle(ops["b_sf"].reshape(E * N, K // 32))),
                               dev(ops["padded"]), dev(ops["counts"]), N, K, E, out_dtype=out_dtype)
    assert lib.nvfp4_status_check() == 0
    return D


def _oracle(ops):
    return X.grouped_gemm(ops["a_codes"], ops["a_sf"], ops["b_codes"], ops["b_sf"], ops["padded"], ops["counts"])


def _rows(ops):
    return np.concatenate([np.arange(p, p + c) for p, c in zip(ops["padded"][:-1], ops["counts"])]).astype(int)


@pytest.mark.parametrize("N", [128, 256])
@pytest.mark.parametrize("K", [128, 256, 512])
def test_mx_gemm_single_tile_exact(cuda_lib, K, N):
    """One expert, one 128 x N tile (both tile kernels: 128 columns, and 256 columns on a
    CTA pair whose second tile is a discarded duplicate).  Operands are E4M3 grid values times powers of
    two, with every block holding its 448 so the quantisation is lossless; every partial
    sum is exact in float32.  The result must be bit-exact and equal the float64 matmul
    of the unquantised values."""
    rng = np.random.default_rng(K)
    grid = F.e4m3_decode(np.array([0x00, 0x38, 0x40, 0x48]))   # 0, 1, 2, 4: partial sums stay on 2^-14 below 2^8
    xa = rng.choice(grid, (128, K)) * rng.choice([-1, 1], (128, K)) * 2.0 ** -6
    xa[:, ::32] = 448 * 2.0 ** -6
    w = rng.choice(grid, (1, N, K)) * rng.choice([-1, 1], (1, N, K)) * 2.0 ** -8
    w[:, :, ::32] = 448 * 2.0 ** -8
    ops = _operands(F.bf16_round(xa), [128], F.bf16_round(w))
    ref = _oracle(ops)
    np.testing.assert_array_equal(ref, xa @ w[0].T)
    D = npy(_run(cuda_lib, ops, N, K, torch.float32))
    np.testing.assert_array_equal(D, ref.astype(np.float32))


@pytest.mark.parametrize("N", [128, 256])
@pytest.mark.parametrize("span,tol", [(4, 0.0), (20, 1e-4)])
def test_mx_gemm_scale_bytes_reach_every_k_block(cuda_lib, span, tol, N):
    """Each 32-value block gets its own power-of-two scale on both sides (exponents in
    [-span, 0)).  A wrong byte within a scale word (the op's scale-factor id) or a wrong
    scale tile changes the result by powers of two.  span = 4: every partial sum is
    exact in float32 (block sums 2989 * 2^(3..9) over 16 blocks), so the result must be
    bit-exact.  span = 20: the tensor cores' float32 accumulation over widely spread
    terms is allowed 1e-4."""
    rng = np.random.default_rng(5 + span)
    K = 512
    xa = np.ones((128, K)) * 448
    w = np.ones((1, N, K)) * 448
    sa = rng.integers(-span, 0, (128, K // 32))
    sw = rng.integers(-span, 0, (N, K // 32))
    xa *= np.exp2(sa).repeat(32, axis=1)
    w[0] *= np.exp2(sw).repeat(32, axis=1)
    xa[:, 3::32] *= -0.5
    ops = _operands(F.bf16_round(xa), [128], F.bf16_round(w))
    ref = _oracle(ops)
    np.testing.assert_array_equal(ref, xa @ w[0].T)
    D = npy(_run(cuda_lib, ops, N, K, torch.float32))
    if tol == 0.0:
        np.testing.assert_array_equal(D, ref.astype(np.float32))
    else:
        mx, _ = rel_err_floor(D, ref)
        assert mx <= tol, mx


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("N,K", [(128, 256), (384, 640), (512, 384)])
def test_mx_gemm_ragged_groups(cuda_lib, out_dtype, N, K):
    E = 6
    counts = [0, 1, 127, 128, 129, 300]
    a_bits = S.bf16_bits(S.randn_bf16((sum(counts), K), seed=51))
    w_bits = S.bf16_bits(S.randn_bf16((E, N, K), 0.02, seed=52))
    ops = _operands(a_bits, counts, w_bits)
    ref = _oracle(ops)
    D = _run(cuda_lib, ops, N, K, out_dtype)
    rows = _rows(ops)
    if out_dtype == torch.float32:
        mx, nw = rel_err_floor(npy(D)[rows], ref[rows])
        assert mx <= 1e-3, (mx, nw)
        assert nw <= 1e-5
    else:
        nbad, worst = check_bf16_against(u16(D)[rows], ref[rows])
        assert nbad == 0, worst


def test_mx_gemm_qwen_shaped(cuda_lib):
    """K = 2048 (16 K-stages), N = 1536, 16 experts with uneven group sizes, activations
    quantised on the GPU by mxfp8_quantize (the composed path of an MXFP8 expert GEMM)."""
    E, N, K = 16, 1536, 2048
    rng = np.random.default_rng(8)
    counts = list(rng.integers(0, 400, E))
    counts[5] = 0
    a_bits = S.bf16_bits(S.randn_bf16((sum(counts), K), seed=61))
    w_bits = S.bf16_bits(S.randn_bf16((E, N, K), 0.02, seed=62))
    ops = _operands(a_bits, counts, w_bits)
    ref = _oracle(ops)
    # the activation operand quantised on the GPU, rows placed into the padded groups
    counts_a, padded = _groups(counts)
    xa = np.zeros((ops["M"], K), np.uint16)
    r = 0
    for e in range(E):
        xa[padded[e]:padded[e] + counts_a[e]] = a_bits[r:r + counts_a[e]]
        r += counts_a[e]
    A, SFA = cuda_lib.mxfp8_quantize(bf16_tensor(xa))
    B, SFB = cuda_lib.mxfp8_quantize(bf16_tensor(w_bits.reshape(E * N, K)))
    D = cuda_lib.mxfp8_grouped_gemm(A, SFA, B, SFB, dev(padded), dev(counts_a), N, K, E, out_dtype=torch.float32)
    assert cuda_lib.nvfp4_status_check() == 0
    rows = _rows(ops)
    np.testing.assert_array_equal(npy(A)[rows], ops["a_codes"][rows])
    mx, nw = rel_err_floor(npy(D)[rows], ref[rows])
    assert mx <= 1e-3, (mx, nw)


def test_mx_argument_checks(cuda_lib):
    x = torch.zeros(4, 96, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(Exception) as ei:
        cuda_lib.mxfp8_quantize(x)
    assert "UNSUPPORTED" in str(ei.value).upper() or "status 2" in str(ei.value)
    codes = torch.zeros(128, 128, dtype=torch.uint8, device="cuda")
    sf = torch.zeros(512, dtype=torch.uint8, device="cuda")
    offs = torch.tensor([0, 128], dtype=torch.int32, device="cuda")
    rows = torch.tensor([128], dtype=torch.int32, device="cuda")
    with pytest.raises(Exception):
        cuda_lib.mxfp8_grouped_gemm(codes, sf, codes, sf, offs, rows, 128, 192, 1)   # K % 128 != 0

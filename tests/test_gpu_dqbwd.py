"""GPU parity of the dequantised backward ("The 4-bitter Lesson...", §"Improving Gradient
Stability": the backward GEMMs use the dequantised weights DQ(Q(W)), so that the
gradient is that of the forward actually run).  The pieces are the BF16 grouped GEMM
(bf16_grouped_gemm) and the transpose that puts DQ(W) in the K-major form of a dgrad
operand (bf16_transpose).  Then the recipe's dgrad through the down projection:
NVFP4 Q, DQ to BF16, transpose, BF16 grouped GEMM, against the oracle."""
import numpy as np
import pytest
import torch

from gpu_util import bf16_tensor, check_bf16_against, dev, npy, rel_err_floor, u16
from oracle import formats as F
from oracle import quant as Q
from nvfp4_w4a4_moe_quantize_gb300 import synthetic as S

pytestmark = pytest.mark.gpu


def _groups(counts):
    counts = np.asarray(counts, np.int64)
    padded = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)])
    return counts.astype(np.int32), padded.astype(np.int32)


def _rows(counts, padded):
    return np.concatenate([np.arange(p, p + c) for p, c in zip(padded[:-1], counts)]).astype(int)


def _ref(a, b, counts, padded):
    """float64 grouped GEMM: D[r, n] = sum_k a[r, k] b[e, n, k] for the rows of group e."""
    out = np.zeros((a.shape[0], b.shape[1]))
    for e in range(b.shape[0]):
        r0, n = int(padded[e]), int(counts[e])
        out[r0:r0 + n] = a[r0:r0 + n] @ b[e].T
    return out


@pytest.mark.parametrize("N", [128, 256])
def test_bf16_grouped_gemm_exact(cuda_lib, N):
    """Small integers times powers of two: every product and partial sum is exact in
    float32, so the float32 output must equal the float64 GEMM bit for bit.  Ragged groups
    of 0, 1, 127, 128, 129 and 300 rows; K = 512 (8 stages)."""
    rng = np.random.default_rng(N)
    counts, padded = _groups([0, 1, 127, 128, 129, 300])
    E, K, Mt = len(counts), 512, int(padded[-1])
    a = rng.integers(-4, 5, (Mt, K)) * 2.0 ** -3
    b = rng.integers(-4, 5, (E, N, K)) * 2.0 ** -5
    D = cuda_lib.bf16_grouped_gemm(bf16_tensor(F.bf16_round(a)), bf16_tensor(F.bf16_round(b.reshape(E * N, K))),
                                   dev(padded), dev(counts), N, K, E, out_dtype=torch.float32)
    assert cuda_lib.nvfp4_status_check() == 0
    rows = _rows(counts, padded)
    np.testing.assert_array_equal(npy(D)[rows], _ref(a, b, counts, padded)[rows].astype(np.float32))


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_bf16_grouped_gemm_random(cuda_lib, out_dtype):
    """Gaussian BF16 operands, N = 384 (three 128-column tiles), K = 640: float32 output
    within 1e-3 relative (floored), BF16 output within one ulp plus that allowance."""
    rng = np.random.default_rng(3)
    counts, padded = _groups([5, 260, 0, 131])
    E, N, K, Mt = len(counts), 384, 640, int(padded[-1])
    a = F.bf16_round(rng.standard_normal((Mt, K)))
    b = F.bf16_round(rng.standard_normal((E * N, K)) * 0.02)
    D = cuda_lib.bf16_grouped_gemm(bf16_tensor(a), bf16_tensor(b), dev(padded), dev(counts), N, K, E,
                                   out_dtype=out_dtype)
    assert cuda_lib.nvfp4_status_check() == 0
    ref = _ref(F.bf16_to_f32(a).astype(np.float64), F.bf16_to_f32(b).astype(np.float64).reshape(E, N, K),
               counts, padded)
    rows = _rows(counts, padded)
    if out_dtype == torch.float32:
        mx, nw = rel_err_floor(npy(D)[rows], ref[rows])
        assert mx <= 1e-3, (mx, nw)
    else:
        nbad, worst = check_bf16_against(u16(D)[rows], ref[rows])
        assert nbad == 0, worst


def test_bf16_transpose(cuda_lib):
    rng = np.random.default_rng(4)
    x = rng.integers(0, 1 << 16, (3 * 40, 72)).astype(np.uint16)
    out = cuda_lib.bf16_transpose(bf16_tensor(x), batches=3)
    ref = x.reshape(3, 40, 72).transpose(0, 2, 1).reshape(3 * 72, 40)
    np.testing.assert_array_equal(u16(out), ref)


def test_dequantised_backward_dgrad_of_the_down_projection(cuda_lib):
    """The recipe's dgrad through the down projection, dh[r, i] = sum_h dY[r, h] W2_e[h, i],
    computed with the dequantised weights.  Quantise W2 as the forward does (one global
    scale per expert, blocks along I).  DQ to BF16 (rounded once), transpose each
    expert's matrix to [I, H], then the BF16 grouped GEMM over the routed dY.  The oracle
    takes the same steps in float64: its DQ rounded to BF16 once, then the exact GEMM."""
    E, H, I = 4, 512, 256
    rng = np.random.default_rng(8)
    counts, padded = _groups([200, 0, 77, 300])
    Mt = int(padded[-1])
    w2 = F.bf16_round(rng.standard_normal((E * H, I)) * 0.02)
    dy = np.zeros((Mt, H), np.uint16)
    for e in range(E):
        dy[padded[e]:padded[e] + counts[e]] = F.bf16_round(rng.standard_normal((counts[e], H)) * 1e-3)
    # GPU: Q (per-expert scope), DQ to BF16, transpose, BF16 grouped GEMM
    c, sf, g = cuda_lib.nvfp4_quantize(bf16_tensor(w2), cuda_lib.SCALE_PER_GROUP, group_rows=H)
    dq = cuda_lib.nvfp4_dequantize(c, sf, g, I, cuda_lib.SCALE_PER_GROUP, group_rows=H)
    dqt = cuda_lib.bf16_transpose(dq, batches=E)
    for out_dtype in (torch.float32, torch.bfloat16):
        dh = cuda_lib.bf16_grouped_gemm(bf16_tensor(dy), dqt, dev(padded), dev(counts), I, H, E,
                                        out_dtype=out_dtype)
        assert cuda_lib.nvfp4_status_check() == 0
        # oracle
        q = Q.quantize(w2, scope="group", group_rows=H)
        dq_ref = F.bf16_round(Q.dequantize(q["codes"], q["sf"], np.repeat(q["g"], H)))
        if out_dtype == torch.float32:
            np.testing.assert_array_equal(u16(dq), dq_ref)
        wq = F.bf16_to_f32(dq_ref).astype(np.float64).reshape(E, H, I).transpose(0, 2, 1)
        ref = _ref(F.bf16_to_f32(dy).astype(np.float64), wq, counts, padded)
        rows = _rows(counts, padded)
        if out_dtype == torch.float32:
            mx, nw = rel_err_floor(npy(dh)[rows], ref[rows])
            assert mx <= 1e-3, (mx, nw)
        else:
            nbad, worst = check_bf16_against(u16(dh)[rows], ref[rows])
            assert nbad == 0, worst


def test_bf16_gemm_argument_checks(cuda_lib):
    a = torch.zeros(128, 96, dtype=torch.bfloat16, device="cuda")   # K % 64 != 0
    offs = torch.tensor([0, 128], dtype=torch.int32, device="cuda")
    rows = torch.tensor([128], dtype=torch.int32, device="cuda")
    with pytest.raises(Exception):
        cuda_lib.bf16_grouped_gemm(a, a, offs, rows, 128, 96, 1)


@pytest.mark.parametrize("rows,I", [(1, 8), (333, 768), (64, 128)])
def test_swiglu_backward_matches_oracle(cuda_lib, rows, I):
    """The SwiGLU backward between the down-projection dgrad and the gate/up dgrad: float32
    on the device against the oracle's float64, each result within one BF16 ulp plus the
    float32 round-off allowance where silu' cancels."""
    from oracle import moe as M
    rng = np.random.default_rng(rows + I)
    gu = F.bf16_round(rng.standard_normal((rows, 2 * I)) * 3)
    gu[0, 0] = 0x0000                                  # gate 0
    if I > 1:
        gu[0, 1] = 0xC2C8                              # gate -100: e^-g overflows, s = 0
    dh = F.bf16_round(rng.standard_normal((rows, I)))
    got = u16(cuda_lib.moe_swiglu_backward(bf16_tensor(gu), bf16_tensor(dh)))
    assert cuda_lib.nvfp4_status_check() == 0
    ref = M.swiglu_backward(gu, dh, I)
    for part in (slice(0, I), slice(I, 2 * I)):
        nbad, worst = check_bf16_against(got[:, part], F.bf16_to_f32(ref[:, part]).astype(np.float64))
        assert nbad == 0, (part, worst)

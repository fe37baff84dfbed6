"""The C-ABI library: it builds for sm_103a, loads without a GPU, exports every function
the header declares, and its host-side logic (sizes, layouts, argument checks that
return before any CUDA call) behaves as documented.  No compute call is made here."""
import ctypes

import pytest

import nvfp4_w4a4_moe_quantize_gb300 as L
from nvfp4_w4a4_moe_quantize_gb300 import build as B


@pytest.fixture(scope="module")
def lib():
    B.build()
    return L.load()


def test_every_declared_function_is_exported(lib):
    names = L.header_functions()
    expected = {"nvfp4_quantize", "nvfp4_grouped_gemm", "moe_expert_forward", "moe_route_topk", "moe_permute",
                "moe_combine", "moe_swiglu_quantize", "moe_prepare_weights", "nvfp4_status_check",
                "nvfp4_status_string", "nvfp4_sf_bytes", "moe_weights_sizes", "nvfp4_workspace_size",
                "moe_forward_workspace_layout", "nvfp4_grouped_gemm_tiled", "nvfp4_pack_tiled",
                "nvfp4_tiled_bytes", "nvfp4_quantize_noalloc", "nvfp4_dequantize", "nvfp4_quantize_transposed",
                "mxfp8_quantize", "mxfp8_dequantize", "mxfp8_grouped_gemm", "mxfp8_sf_bytes",
                "bf16_grouped_gemm", "bf16_transpose", "moe_swiglu_backward", "moe_weights_t_sizes",
                "moe_prepare_weights_backward", "moe_expert_backward", "moe_backward_workspace_layout"}
    assert expected <= set(names)
    for n in names:
        assert hasattr(lib, n), n
        assert n in L._SIGS, n


def test_sf_bytes_and_weight_sizes(lib):
    assert L.nvfp4_sf_bytes(16384, 2048) == 128 * 32 * 512
    assert L.nvfp4_sf_bytes(1, 16) == 512
    assert L.nvfp4_sf_bytes(129, 80) == 2 * 2 * 512
    sizes = (ctypes.c_size_t * 4)()
    assert lib.moe_weights_sizes(128, 2048, 768, sizes) == 0
    # GEMM-tiled: 256-row blocks of 256 K-values, 144 bytes per row per block (128 codes + 16 scales)
    assert list(sizes) == [128 * 1536 // 256 * 8 * 256 * 144, 512, 128 * 2048 // 256 * 3 * 256 * 144, 512]
    # I not a multiple of 256: the down projection's K is zero-padded to 256
    assert lib.moe_weights_sizes(8, 256, 128, sizes) == 0
    assert sizes[2] == 8 * 256 // 256 * 1 * 256 * 144
    assert L.nvfp4_tiled_bytes(129, 512, 128) == 2 * 2 * 128 * 144
    assert L.nvfp4_tiled_bytes(100, 300, 128) == 0          # K not a multiple of 256


def test_forward_workspace_layout(lib):
    T, k, E, H, I = 16384, 8, 128, 2048, 768
    lay = L.moe_forward_workspace_layout(T, k, E, H, I)
    mcap = lay[13]
    assert mcap == (T * k + E * 127 + 127) // 128 * 128
    offs = [lay[i] for i in range(13)]
    assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert lay[12] + mcap * H * 2 <= lay[14]
    assert lib.nvfp4_workspace_size(L.OP_MOE_FORWARD, T, k, E, H, I) == lay[14]
    assert lay[6] == lay[5] and lay[10] == lay[9]              # scales live inside the tiles
    assert lay[7] - lay[5] >= mcap // 128 * 8 * 128 * 144      # Aq tiled, K = H
    assert lay[11] - lay[9] >= mcap // 128 * 3 * 128 * 144     # hq tiled, K = Ip


def test_host_argument_checks_return_before_any_cuda_call(lib):
    null = ctypes.c_void_p(0)
    # cols not a multiple of 16
    assert lib.nvfp4_quantize(null, 4, 24, 24, 0, 0, 0, 0, 0, null, null, null, null, 0, null, 0, null) == L.Status.INVALID_ARG
    # an unknown scale layout; row-major scales need whole 64-value groups
    assert lib.nvfp4_quantize(null, 4, 64, 64, 0, 0, 0, 0, 0, null, null, null, null, 7, null, 0, null) == L.Status.INVALID_ARG
    assert lib.nvfp4_quantize(null, 4, 48, 48, 0, 0, 0, 0, 0, null, null, null, null, L.SF_ROWMAJOR, null, 0,
                              null) == L.Status.UNSUPPORTED
    # K not a multiple of 256
    assert lib.nvfp4_grouped_gemm(null, null, null, null, null, null, null, null, 128, 128, 192, 1, null, 0, 128,
                                  null) == L.Status.UNSUPPORTED
    # k > 32
    assert lib.moe_route_topk(null, 4, 64, 33, 1, null, null, null) == L.Status.INVALID_ARG
    # H not a multiple of 8 in the combine
    assert lib.moe_combine(null, null, null, 4, 2, 12, null, null) == L.Status.INVALID_ARG
    # empty inputs are a no-op
    assert lib.nvfp4_quantize(null, 0, 32, 32, 0, 0, 0, 0, 0, null, null, null, null, 0, null, 0, null) == L.Status.OK
    assert lib.nvfp4_status_string(L.Status.WORKSPACE) == b"workspace too small"


def test_python_binding_rejects_cpu_tensors(lib):
    torch = pytest.importorskip("torch")
    with pytest.raises(ValueError):
        L.moe_route_topk(torch.zeros(4, 8), 2)

"""Host-side argument checks of the C ABI's MXFP8, BF16-GEMM and SwiGLU-backward entry
points, run on the CPU.  Every case here is rejected (or finishes as an empty call)
before the library touches a device: sizes, alignment and null pointers are checked
first.  So placeholder addresses stand in for device buffers and are never dereferenced."""
import ctypes

import pytest

import nvfp4_w4a4_moe_quantize_gb300 as L

OK, INVALID, UNSUPPORTED = L.Status.OK, L.Status.INVALID_ARG, L.Status.UNSUPPORTED
P = ctypes.c_void_p(0x10000)        # 16-byte aligned placeholder, never dereferenced
P4 = ctypes.c_void_p(0x10004)       # 4-byte aligned only
NULL = ctypes.c_void_p(0)


@pytest.fixture(scope="module")
def lib():
    return L.load()


def test_mxfp8_sf_bytes(lib):
    assert lib.mxfp8_sf_bytes(130, 256) == 2 * 2 * 512
    assert lib.mxfp8_sf_bytes(1, 128) == 512
    assert lib.mxfp8_sf_bytes(0, 128) == 0


def test_mxfp8_quantize_checks(lib):
    assert lib.mxfp8_quantize(P, 4, 96, 96, P, P, NULL) == UNSUPPORTED        # cols % 128
    assert lib.mxfp8_quantize(P, 4, 128, 120, P, P, NULL) == INVALID          # ld < cols
    assert lib.mxfp8_quantize(P, 4, 128, 132, P, P, NULL) == INVALID          # ld % 8
    assert lib.mxfp8_quantize(P, -1, 128, 128, P, P, NULL) == INVALID
    assert lib.mxfp8_quantize(NULL, 4, 128, 128, P, P, NULL) == INVALID
    assert lib.mxfp8_quantize(P4, 4, 128, 128, P, P, NULL) == INVALID         # x not 16-byte aligned
    assert lib.mxfp8_quantize(P, 0, 128, 128, P, P, NULL) == OK               # empty: nothing enqueued


def test_mxfp8_dequantize_checks(lib):
    assert lib.mxfp8_dequantize(P, P, 4, 96, P, 0, 96, NULL) == UNSUPPORTED
    assert lib.mxfp8_dequantize(P, P, 4, 128, P, 7, 128, NULL) == INVALID     # out dtype
    assert lib.mxfp8_dequantize(P, P, 4, 128, P, 0, 64, NULL) == INVALID      # ldo < cols
    assert lib.mxfp8_dequantize(P, NULL, 4, 128, P, 0, 128, NULL) == INVALID
    assert lib.mxfp8_dequantize(P, P, 0, 128, P, 0, 128, NULL) == OK


def test_mxfp8_grouped_gemm_checks(lib):
    g = (P, P, P, P, P4, P4)
    assert lib.mxfp8_grouped_gemm(*g, 128, 128, 192, 1, P, 0, 128, NULL) == UNSUPPORTED   # K % 128
    assert lib.mxfp8_grouped_gemm(*g, 128, 96, 128, 1, P, 0, 128, NULL) == UNSUPPORTED    # N % 128
    assert lib.mxfp8_grouped_gemm(*g, 100, 128, 128, 1, P, 0, 128, NULL) == INVALID       # M_total % 128
    assert lib.mxfp8_grouped_gemm(*g, 128, 128, 128, 0, P, 0, 128, NULL) == INVALID       # E = 0
    assert lib.mxfp8_grouped_gemm(*g, 128, 128, 128, 1025, P, 0, 128, NULL) == INVALID    # E > 1024
    assert lib.mxfp8_grouped_gemm(*g, 128, 256, 128, 1, P, 0, 128, NULL) == INVALID       # ldd < N
    assert lib.mxfp8_grouped_gemm(*g, 128, 128, 128, 1, P, 5, 128, NULL) == INVALID       # out dtype
    assert lib.mxfp8_grouped_gemm(P4, P, P, P, P4, P4, 128, 128, 128, 1, P, 0, 128, NULL) == INVALID
    assert lib.mxfp8_grouped_gemm(*g, 0, 128, 128, 1, P, 0, 128, NULL) == OK


def test_bf16_grouped_gemm_checks(lib):
    g = (P, P, P4, P4)
    assert lib.bf16_grouped_gemm(*g, 128, 128, 96, 1, P, 0, 128, NULL) == UNSUPPORTED     # K % 64
    assert lib.bf16_grouped_gemm(*g, 128, 192, 128, 1, P, 0, 192, NULL) == UNSUPPORTED    # N % 128
    assert lib.bf16_grouped_gemm(*g, 128, 128, 128, 1, P, 0, 120, NULL) == INVALID        # ldd
    assert lib.bf16_grouped_gemm(P, NULL, P4, P4, 128, 128, 128, 1, P, 0, 128, NULL) == INVALID
    assert lib.bf16_grouped_gemm(*g, 0, 128, 128, 1, P, 0, 128, NULL) == OK


def test_bf16_transpose_checks(lib):
    assert lib.bf16_transpose(P, 1, 4, 8, 6, P, NULL) == INVALID              # ld < C
    assert lib.bf16_transpose(NULL, 1, 4, 8, 8, P, NULL) == INVALID
    assert lib.bf16_transpose(P, 0, 4, 8, 8, P, NULL) == OK                   # nothing to do


def test_swiglu_backward_checks(lib):
    assert lib.moe_swiglu_backward(P, P, 4, 12, P, NULL) == INVALID           # I % 8
    assert lib.moe_swiglu_backward(P, P4, 4, 16, P, NULL) == INVALID          # dh not 16-byte aligned
    assert lib.moe_swiglu_backward(P, P, 4, 16, NULL, NULL) == INVALID
    assert lib.moe_swiglu_backward(P, P, 0, 16, P, NULL) == OK

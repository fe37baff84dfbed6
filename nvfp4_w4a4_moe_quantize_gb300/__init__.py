"""NVFP4 W4A4 mixture-of-experts expert block for GB300 (sm_103a).

Python binding of the C ABI in ``include/nvfp4moe.h``: every function here marshals
torch tensors into raw device pointers, sizes and the current CUDA stream, and calls the
CUDA library ``_build/libnvfp4moe.so`` (built in-tree by ``build.py``).  PyTorch supplies
device memory and streams only; every step of the path runs in the library's kernels.
There is no fallback: if the library cannot be loaded, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

from . import build as _build

__all__ = [
    "load", "library_path", "Status", "NVFP4Error",
    "nvfp4_quantize", "nvfp4_quantize_noalloc", "nvfp4_quantize_transposed", "nvfp4_dequantize",
    "nvfp4_grouped_gemm", "moe_route_topk", "moe_permute", "moe_combine",
    "moe_swiglu_quantize", "moe_prepare_weights", "moe_expert_forward", "moe_forward_workspace",
    "moe_forward_workspace_layout", "nvfp4_status_check", "nvfp4_sf_bytes", "NVFP4MoEWeights",
    "nvfp4_grouped_gemm_tiled", "nvfp4_pack_tiled", "nvfp4_tiled_bytes",
    "mxfp8_quantize", "mxfp8_dequantize", "mxfp8_grouped_gemm", "mxfp8_sf_bytes",
    "bf16_grouped_gemm", "bf16_transpose", "moe_swiglu_backward",
    "SCALE_PER_TENSOR", "SCALE_PER_ROW", "SCALE_PER_GROUP", "ROUND_RNE", "ROUND_STOCHASTIC",
    "SF_SWIZZLED_128x4", "SF_ROWMAJOR",
    "NVFP4MoEWeightsT", "moe_prepare_weights_backward", "moe_expert_backward", "moe_backward_workspace",
    "moe_backward_workspace_layout",
]

SCALE_PER_TENSOR, SCALE_PER_ROW, SCALE_PER_GROUP = 0, 1, 2
ROUND_RNE, ROUND_STOCHASTIC = 0, 1
SF_SWIZZLED_128x4, SF_ROWMAJOR = 0, 1
OUT_BF16, OUT_F32 = 0, 1
OP_QUANTIZE, OP_PREPARE_WEIGHTS, OP_MOE_FORWARD, OP_MOE_PERMUTE, OP_QUANTIZE_T = 0, 1, 2, 3, 4
OP_MOE_BACKWARD, OP_PREPARE_WEIGHTS_T = 5, 6

_lib = None
_vp, _i64, _i32, _u64, _sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint64, ctypes.c_size_t


class Status:
    OK, INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA, DEVICE_STATUS, TIMEOUT = range(7)


class NVFP4Error(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} (status {code})")


class _Weights(ctypes.Structure):
    _fields_ = [("E", _i32), ("H", _i64), ("I", _i64), ("w13", _vp), ("w13_g", _vp), ("w2", _vp),
                ("w2_g", _vp)]


class _WeightsT(ctypes.Structure):
    _fields_ = [("E", _i32), ("H", _i64), ("I", _i64), ("w13t", _vp), ("w13t_g", _vp), ("w2t", _vp),
                ("w2t_g", _vp)]


_SIGS = {
    "nvfp4_sf_bytes": (_sz, [_i64, _i64]),
    "nvfp4_tiled_bytes": (_sz, [_i64, _i64, _i32]),
    "nvfp4_grouped_gemm_tiled": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp,
                                                ctypes.c_int, _i64, _i32, _vp]),
    "nvfp4_pack_tiled": (ctypes.c_int, [_vp, _vp, _i64, _i64, _i32, _vp, _vp]),
    "moe_weights_sizes": (ctypes.c_int, [_i32, _i64, _i64, ctypes.POINTER(_sz)]),
    "nvfp4_workspace_size": (_sz, [ctypes.c_int, _i64, _i64, _i64, _i64, _i64]),
    "nvfp4_status_check": (ctypes.c_int, [_vp]),
    "nvfp4_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "nvfp4_quantize": (ctypes.c_int, [_vp, _i64, _i64, _i64, ctypes.c_int, _i64, ctypes.c_int, _u64, _u64,
                                      _vp, _vp, _vp, _vp, ctypes.c_int, _vp, _sz, _vp]),
    "nvfp4_quantize_noalloc": (ctypes.c_int, [_vp, _i64, _i64, _i64, ctypes.c_int, _i64, ctypes.c_int, _u64, _u64,
                                              _vp, _vp, _vp, _vp, _vp]),
    "nvfp4_quantize_transposed": (ctypes.c_int, [_vp, _i64, _i64, _i64, _i64, ctypes.c_int, _i64, ctypes.c_int,
                                                 _u64, _u64, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "nvfp4_dequantize": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i64, ctypes.c_int, _i64, _vp, ctypes.c_int, _i64,
                                        _vp]),
    "nvfp4_grouped_gemm": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32,
                                          _vp, ctypes.c_int, _i64, _vp]),
    "bf16_grouped_gemm": (ctypes.c_int, [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, ctypes.c_int, _i64, _vp]),
    "bf16_transpose": (ctypes.c_int, [_vp, _i64, _i64, _i64, _i64, _vp, _vp]),
    "moe_swiglu_backward": (ctypes.c_int, [_vp, _vp, _i64, _i64, _vp, _vp]),
    "mxfp8_sf_bytes": (_sz, [_i64, _i64]),
    "mxfp8_quantize": (ctypes.c_int, [_vp, _i64, _i64, _i64, _vp, _vp, _vp]),
    "mxfp8_dequantize": (ctypes.c_int, [_vp, _vp, _i64, _i64, _vp, ctypes.c_int, _i64, _vp]),
    "mxfp8_grouped_gemm": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i32, _vp, ctypes.c_int,
                                          _i64, _vp]),
    "moe_route_topk": (ctypes.c_int, [_vp, _i64, _i32, _i32, ctypes.c_int, _vp, _vp, _vp]),
    "moe_permute": (ctypes.c_int, [_vp, _i64, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "moe_combine": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i32, _i64, _vp, _vp]),
    "moe_swiglu_quantize": (ctypes.c_int, [_vp, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp]),
    "moe_prepare_weights": (ctypes.c_int, [_vp, _vp, _i32, _i64, _i64, ctypes.POINTER(_Weights), _vp, _sz,
                                           _vp]),
    "moe_expert_forward": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i32, ctypes.POINTER(_Weights), _vp, _vp,
                                          _sz, _vp]),
    "moe_forward_workspace_layout": (ctypes.c_int, [_i64, _i32, _i32, _i64, _i64, ctypes.POINTER(_i64)]),
    "moe_weights_t_sizes": (ctypes.c_int, [_i32, _i64, _i64, ctypes.POINTER(_sz)]),
    "moe_prepare_weights_backward": (ctypes.c_int, [_vp, _vp, _i32, _i64, _i64, ctypes.POINTER(_WeightsT), _vp,
                                                    _sz, _vp]),
    "moe_expert_backward": (ctypes.c_int, [_vp, _vp, _vp, _i64, _i32, ctypes.POINTER(_Weights),
                                           ctypes.POINTER(_WeightsT), _vp, _sz, _u64, _vp, _vp, _vp, _vp, _vp, _sz,
                                           _vp]),
    "moe_backward_workspace_layout": (ctypes.c_int, [_i64, _i32, _i32, _i64, _i64, ctypes.POINTER(_i64)]),
}


def library_path() -> str:
    return _build.LIB


def header_functions() -> list:
    """Names of the functions declared in include/nvfp4moe.h."""
    src = open(os.path.join(_build.INCLUDE, "nvfp4moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b([a-z][a-z0-9_]*)\s*\(", src)) - {"if", "sizeof"})


def load(path: str | None = None):
    """Load the CUDA library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"CUDA library not built ({path}); run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(code: int) -> str:
    try:
        return load().nvfp4_status_string(code).decode()
    except Exception:  # noqa: BLE001 - only used for messages
        return "unknown"


def _check(code: int, what: str):
    if code != Status.OK:
        raise NVFP4Error(code, what)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t):
    if not t.is_cuda:
        raise ValueError("tensors must be on a CUDA device")
    return t.device


def nvfp4_sf_bytes(rows: int, cols: int) -> int:
    return int(load().nvfp4_sf_bytes(rows, cols))


def nvfp4_tiled_bytes(rows: int, K: int, block_rows: int) -> int:
    return int(load().nvfp4_tiled_bytes(rows, K, block_rows))


def nvfp4_status_check(stream=None) -> int:
    """Synchronise the stream; return (and clear) the device status word."""
    return int(load().nvfp4_status_check(_stream(stream)))


# --------------------------------------------------------------------------- quantiser

def nvfp4_quantize(x: torch.Tensor, mode: int = SCALE_PER_TENSOR, rounding: int = ROUND_RNE, seed: int = 0,
                   rng_offset: int = 0, group_rows: int = 0, global_scale: torch.Tensor | None = None,
                   out=None, workspace: torch.Tensor | None = None, sf_layout: int = SF_SWIZZLED_128x4,
                   stream=None):
    """NVFP4 of a BF16 matrix [rows, cols].  Returns (codes [rows, cols/2] uint8,
    scales uint8 (tiled [nvfp4_sf_bytes], or [rows, cols/16] with SF_ROWMAJOR),
    g float32 [1 | rows | rows/group_rows])."""
    lib = load()
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    dev = _dev(x)
    n_g = 1 if mode == SCALE_PER_TENSOR else (rows if mode == SCALE_PER_ROW else rows // max(group_rows, 1))
    if out is None:
        codes = torch.empty(rows, cols // 2, dtype=torch.uint8, device=dev)
        if sf_layout == SF_ROWMAJOR:
            sf = torch.empty(rows, cols // 16, dtype=torch.uint8, device=dev)
        else:
            sf = torch.empty(max(nvfp4_sf_bytes(rows, cols), 16), dtype=torch.uint8, device=dev)
        g = torch.empty(max(n_g, 1), dtype=torch.float32, device=dev)
    else:
        codes, sf, g = out
    ws_bytes = int(lib.nvfp4_workspace_size(OP_QUANTIZE, rows, cols, 0, 0, 0))
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    _check(lib.nvfp4_quantize(_p(x), rows, cols, x.stride(0), mode, group_rows, rounding, seed, rng_offset,
                              _p(global_scale), _p(g), _p(codes), _p(sf), sf_layout, _p(workspace),
                              workspace.numel(), _stream(stream)), "nvfp4_quantize")
    return codes, sf, g


def nvfp4_quantize_noalloc(x: torch.Tensor, mode: int = SCALE_PER_TENSOR, rounding: int = ROUND_RNE,
                           seed: int = 0, rng_offset: int = 0, group_rows: int = 0,
                           global_scale: torch.Tensor | None = None, out=None, stream=None):
    """nvfp4_quantize without a workspace: the library keeps the amax scratch in its own
    fixed device array (for callers that cannot allocate).  Outputs as nvfp4_quantize."""
    lib = load()
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.stride(1) == 1
    rows, cols = x.shape
    dev = _dev(x)
    n_g = 1 if mode == SCALE_PER_TENSOR else (rows if mode == SCALE_PER_ROW else rows // max(group_rows, 1))
    if out is None:
        codes = torch.empty(rows, cols // 2, dtype=torch.uint8, device=dev)
        sf = torch.empty(max(nvfp4_sf_bytes(rows, cols), 16), dtype=torch.uint8, device=dev)
        g = torch.empty(max(n_g, 1), dtype=torch.float32, device=dev)
    else:
        codes, sf, g = out
    _check(lib.nvfp4_quantize_noalloc(_p(x), rows, cols, x.stride(0), mode, group_rows, rounding, seed, rng_offset,
                                      _p(global_scale), _p(g), _p(codes), _p(sf), _stream(stream)),
           "nvfp4_quantize_noalloc")
    return codes, sf, g


def nvfp4_quantize_transposed(x: torch.Tensor, mode: int = SCALE_PER_TENSOR, rounding: int = ROUND_RNE,
                              seed: int = 0, rng_offset: int = 0, group_rows: int = 0,
                              global_scale: torch.Tensor | None = None, stream=None):
    """NVFP4 of the transposes of BF16 matrices: x [R, C] or [batches, R, C] -> codes of
    the stacked transposes [batches*C, R/2], tiled scales and g, exactly as nvfp4_quantize
    of that transposed matrix (blocks of 16 along R)."""
    lib = load()
    assert x.dtype == torch.bfloat16 and x.stride(-1) == 1
    x3 = x if x.dim() == 3 else x.unsqueeze(0)
    assert x3.is_contiguous() or x.dim() == 2
    batches, R, C = x3.shape
    ld = x.stride(-2)
    rows_t = batches * C
    dev = _dev(x)
    n_g = 1 if mode == SCALE_PER_TENSOR else (rows_t if mode == SCALE_PER_ROW else rows_t // max(group_rows, 1))
    codes = torch.empty(rows_t, R // 2, dtype=torch.uint8, device=dev)
    sf = torch.empty(max(nvfp4_sf_bytes(rows_t, R), 16), dtype=torch.uint8, device=dev)
    g = torch.empty(max(n_g, 1), dtype=torch.float32, device=dev)
    ws = torch.empty(int(lib.nvfp4_workspace_size(OP_QUANTIZE_T, rows_t, R, 0, 0, 0)), dtype=torch.uint8, device=dev)
    _check(lib.nvfp4_quantize_transposed(_p(x), batches, R, C, ld, mode, group_rows, rounding, seed, rng_offset,
                                         _p(global_scale), _p(g), _p(codes), _p(sf), _p(ws), ws.numel(),
                                         _stream(stream)), "nvfp4_quantize_transposed")
    return codes, sf, g


def nvfp4_dequantize(codes: torch.Tensor, sf: torch.Tensor, g: torch.Tensor, cols: int,
                     mode: int = SCALE_PER_TENSOR, group_rows: int = 0, out_dtype=torch.bfloat16,
                     out: torch.Tensor | None = None, stream=None):
    """DQ: out[rows, cols] = value(code) * block scale * global scale, rounded once to
    out_dtype (BF16 or float32), from nvfp4_quantize's codes, tiled scales and g."""
    lib = load()
    rows = codes.shape[0]
    if out is None:
        out = torch.empty(rows, cols, dtype=out_dtype, device=_dev(codes))
    _check(lib.nvfp4_dequantize(_p(codes), _p(sf), _p(g), rows, cols, mode, group_rows, _p(out),
                                1 if out.dtype == torch.float32 else 0, out.stride(0), _stream(stream)),
           "nvfp4_dequantize")
    return out


# --------------------------------------------------------------------------- GEMM

def nvfp4_grouped_gemm(A, SFA, gA, B, SFB, gB, group_offsets, group_rows, N: int, K: int, E: int,
                       out_dtype=torch.bfloat16, out: torch.Tensor | None = None, stream=None):
    """D[M_total, N] = grouped W4A4 GEMM (rows outside the groups are left unwritten)."""
    lib = load()
    M_total = A.shape[0]
    if out is None:
        out = torch.empty(M_total, N, dtype=out_dtype, device=_dev(A))
    code = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check(lib.nvfp4_grouped_gemm(_p(A), _p(SFA), _p(gA), _p(B), _p(SFB), _p(gB), _p(group_offsets),
                                  _p(group_rows), M_total, N, K, E, _p(out), code, out.stride(0),
                                  _stream(stream)), "nvfp4_grouped_gemm")
    return out


# --------------------------------------------------------------------------- dequantised backward

def bf16_grouped_gemm(A, B, group_offsets, group_rows, N: int, K: int, E: int, out_dtype=torch.bfloat16,
                      out: torch.Tensor | None = None, stream=None):
    """D[M_total, N] = grouped BF16 GEMM: A [M_total, K] BF16, B [E*N, K] BF16 (rows outside
    the groups are left unwritten)."""
    lib = load()
    M_total = A.shape[0]
    if out is None:
        out = torch.empty(M_total, N, dtype=out_dtype, device=_dev(A))
    code = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check(lib.bf16_grouped_gemm(_p(A), _p(B), _p(group_offsets), _p(group_rows), M_total, N, K, E, _p(out), code,
                                 out.stride(0), _stream(stream)), "bf16_grouped_gemm")
    return out


def bf16_transpose(x: torch.Tensor, batches: int = 1, stream=None):
    """out[b*C + c, r] = x[b*R + r, c] for x = `batches` stacked [R, C] BF16 matrices."""
    lib = load()
    rows, C = x.shape
    R = rows // batches
    out = torch.empty(batches * C, R, dtype=torch.bfloat16, device=_dev(x))
    _check(lib.bf16_transpose(_p(x), batches, R, C, x.stride(0), _p(out), _stream(stream)), "bf16_transpose")
    return out


def moe_swiglu_backward(gu: torch.Tensor, dh: torch.Tensor, out: torch.Tensor | None = None, stream=None):
    """[dgate | dup] (BF16 [rows, 2I]) of h = silu(gate) * up, from gu = [gate | up] and dh."""
    lib = load()
    rows, I = dh.shape
    if out is None:
        out = torch.empty(rows, 2 * I, dtype=torch.bfloat16, device=_dev(dh))
    _check(lib.moe_swiglu_backward(_p(gu.contiguous()), _p(dh.contiguous()), rows, I, _p(out), _stream(stream)),
           "moe_swiglu_backward")
    return out


# --------------------------------------------------------------------------- MXFP8

def mxfp8_sf_bytes(rows: int, cols: int) -> int:
    return int(load().mxfp8_sf_bytes(rows, cols))


def mxfp8_quantize(x: torch.Tensor, codes: torch.Tensor | None = None, sf: torch.Tensor | None = None,
                   stream=None):
    """MXFP8 of a BF16 matrix [rows, cols] (cols % 128 == 0): E4M3 codes [rows, cols]
    and E8M0 scales (one per 32 values, 128x4 tiled).  Returns (codes, sf)."""
    lib = load()
    if x.dtype != torch.bfloat16 or x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be a 2-D BF16 tensor with unit column stride")
    rows, cols = x.shape
    if codes is None:
        codes = torch.empty(rows, cols, dtype=torch.uint8, device=_dev(x))
    if sf is None:
        sf = torch.empty(max(mxfp8_sf_bytes(rows, cols), 1), dtype=torch.uint8, device=_dev(x))
    _check(lib.mxfp8_quantize(_p(x), rows, cols, x.stride(0), _p(codes), _p(sf), _stream(stream)),
           "mxfp8_quantize")
    return codes, sf


def mxfp8_dequantize(codes: torch.Tensor, sf: torch.Tensor, out_dtype=torch.bfloat16,
                     out: torch.Tensor | None = None, stream=None):
    """MXFP8 DQ: out[rows, cols] = value(code) * 2^(b - 127), rounded once to out_dtype."""
    lib = load()
    rows, cols = codes.shape
    if out is None:
        out = torch.empty(rows, cols, dtype=out_dtype, device=_dev(codes))
    _check(lib.mxfp8_dequantize(_p(codes), _p(sf), rows, cols, _p(out), 1 if out.dtype == torch.float32 else 0,
                                out.stride(0), _stream(stream)), "mxfp8_dequantize")
    return out


def mxfp8_grouped_gemm(A, SFA, B, SFB, group_offsets, group_rows, N: int, K: int, E: int,
                       out_dtype=torch.bfloat16, out: torch.Tensor | None = None, stream=None):
    """D[M_total, N] = grouped MXFP8 x MXFP8 GEMM (rows outside the groups are left unwritten)."""
    lib = load()
    M_total = A.shape[0]
    if out is None:
        out = torch.empty(M_total, N, dtype=out_dtype, device=_dev(A))
    code = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check(lib.mxfp8_grouped_gemm(_p(A), _p(SFA), _p(B), _p(SFB), _p(group_offsets), _p(group_rows), M_total, N, K,
                                  E, _p(out), code, out.stride(0), _stream(stream)), "mxfp8_grouped_gemm")
    return out


EPILOGUE_STORE, EPILOGUE_SWIGLU = 0, 1


def nvfp4_grouped_gemm_tiled(A_tiled, gA, B_tiled, gB, group_offsets, group_rows, M_total: int, N: int, K: int,
                             E: int, out_dtype=torch.bfloat16, epilogue: int = EPILOGUE_STORE,
                             out: torch.Tensor | None = None, stream=None):
    """Grouped GEMM over GEMM-tiled operands.  EPILOGUE_SWIGLU returns h [M_total, N/2]."""
    lib = load()
    dev = _dev(A_tiled)
    if out is None:
        if epilogue == EPILOGUE_SWIGLU:
            out = torch.empty(M_total, N // 2, dtype=torch.bfloat16, device=dev)
        else:
            out = torch.empty(M_total, N, dtype=out_dtype, device=dev)
    code = OUT_F32 if out.dtype == torch.float32 else OUT_BF16
    _check(lib.nvfp4_grouped_gemm_tiled(_p(A_tiled), _p(gA), _p(B_tiled), _p(gB), _p(group_offsets), _p(group_rows),
                                        M_total, N, K, E, _p(out), code, out.stride(0), epilogue, _stream(stream)),
           "nvfp4_grouped_gemm_tiled")
    return out


def nvfp4_pack_tiled(codes: torch.Tensor, sf: torch.Tensor, rows: int, K: int, block_rows: int, stream=None):
    """Row-major codes + 128x4 tiled scales -> the GEMM-tiled layout (block_rows 128 / 256)."""
    lib = load()
    out = torch.empty(nvfp4_tiled_bytes(rows, K, block_rows), dtype=torch.uint8, device=_dev(codes))
    _check(lib.nvfp4_pack_tiled(_p(codes), _p(sf), rows, K, block_rows, _p(out), _stream(stream)),
           "nvfp4_pack_tiled")
    return out


# --------------------------------------------------------------------------- MoE helpers

def moe_route_topk(logits: torch.Tensor, k: int, renormalize: bool = True, out=None, stream=None):
    lib = load()
    T, E = logits.shape
    if out is None:
        ids = torch.empty(T, k, dtype=torch.int32, device=_dev(logits))
        w = torch.empty(T, k, dtype=torch.float32, device=logits.device)
    else:
        ids, w = out
    _check(lib.moe_route_topk(_p(logits.contiguous()), T, E, k, int(renormalize), _p(ids), _p(w),
                              _stream(stream)), "moe_route_topk")
    return ids, w


def moe_mcap(T: int, k: int, E: int) -> int:
    return (T * k + E * 127 + 127) // 128 * 128


def moe_permute(ids: torch.Tensor, E: int, stream=None):
    lib = load()
    T, k = ids.shape
    dev = _dev(ids)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    padded = torch.empty(E + 1, dtype=torch.int32, device=dev)
    inv = torch.empty(T, k, dtype=torch.int32, device=dev)
    perm = torch.full((moe_mcap(T, k, E),), -2, dtype=torch.int32, device=dev)
    ws = torch.empty(int(lib.nvfp4_workspace_size(OP_MOE_PERMUTE, T, k, E, 0, 0)), dtype=torch.uint8, device=dev)
    _check(lib.moe_permute(_p(ids.contiguous()), T, k, E, _p(counts), _p(offsets), _p(padded), _p(inv), _p(perm),
                           _p(ws), ws.numel(), _stream(stream)), "moe_permute")
    return dict(counts=counts, offsets=offsets, padded_offsets=padded, inv=inv, perm=perm)


def moe_combine(y: torch.Tensor, inv: torch.Tensor, w: torch.Tensor, stream=None):
    lib = load()
    T, k = inv.shape
    H = y.shape[1]
    out = torch.empty(T, H, dtype=torch.bfloat16, device=_dev(y))
    _check(lib.moe_combine(_p(y), _p(inv.contiguous()), _p(w.contiguous()), T, k, H, _p(out), _stream(stream)),
           "moe_combine")
    return out


def moe_swiglu_quantize(d: torch.Tensor, perm: torch.Tensor, I: int, want_h: bool = True, stream=None):
    """h = BF16(silu(gate) * up) over the interleaved gate/up output, then per-row NVFP4."""
    lib = load()
    rows = d.shape[0]
    dev = _dev(d)
    Ip = (I + 255) // 256 * 256
    h = torch.empty(rows, I, dtype=torch.bfloat16, device=dev) if want_h else None
    hq = torch.empty(rows, Ip // 2, dtype=torch.uint8, device=dev)
    hsf = torch.empty(nvfp4_sf_bytes(rows, Ip), dtype=torch.uint8, device=dev)
    gh = torch.empty(rows, dtype=torch.float32, device=dev)
    _check(lib.moe_swiglu_quantize(_p(d), _p(perm), rows, I, _p(h), _p(hq), _p(hsf), _p(gh), _stream(stream)),
           "moe_swiglu_quantize")
    return h, hq, hsf, gh


class NVFP4MoEWeights:
    """Quantised expert weights (GEMM-tiled device buffers) plus the C struct that points
    at them."""

    def __init__(self, E: int, H: int, I: int, device):
        lib = load()
        sizes = (_sz * 4)()
        _check(lib.moe_weights_sizes(E, H, I, sizes), "moe_weights_sizes")
        Ip = (I + 255) // 256 * 256
        self.E, self.H, self.I, self.Ip = E, H, I, Ip
        self.w13 = torch.empty(sizes[0], dtype=torch.uint8, device=device)
        self.w13_g = torch.empty(E, dtype=torch.float32, device=device)
        self.w2 = torch.empty(sizes[2], dtype=torch.uint8, device=device)
        self.w2_g = torch.empty(E, dtype=torch.float32, device=device)
        self.struct = _Weights(E, H, I, self.w13.data_ptr(), self.w13_g.data_ptr(), self.w2.data_ptr(),
                               self.w2_g.data_ptr())


def moe_prepare_weights(w13: torch.Tensor, w2: torch.Tensor, stream=None) -> NVFP4MoEWeights:
    """Quantise W13 [E, 2I, H] (gate rows then up rows) and W2 [E, H, I], BF16."""
    lib = load()
    E, N13, H = w13.shape
    I = N13 // 2
    assert w2.shape == (E, H, I)
    pw = NVFP4MoEWeights(E, H, I, _dev(w13))
    ws = torch.empty(int(lib.nvfp4_workspace_size(OP_PREPARE_WEIGHTS, E, 0, 0, 0, 0)), dtype=torch.uint8,
                     device=w13.device)
    _check(lib.moe_prepare_weights(_p(w13.contiguous()), _p(w2.contiguous()), E, H, I, ctypes.byref(pw.struct),
                                   _p(ws), ws.numel(), _stream(stream)), "moe_prepare_weights")
    pw._ws = ws
    return pw


def moe_forward_workspace_layout(T: int, k: int, E: int, H: int, I: int) -> list:
    lib = load()
    out = (_i64 * 15)()
    _check(lib.moe_forward_workspace_layout(T, k, E, H, I, out), "moe_forward_workspace_layout")
    return list(out)


def moe_forward_workspace(T: int, k: int, weights: NVFP4MoEWeights, device) -> torch.Tensor:
    lib = load()
    n = int(lib.nvfp4_workspace_size(OP_MOE_FORWARD, T, k, weights.E, weights.H, weights.I))
    return torch.empty(n, dtype=torch.uint8, device=device)


def moe_expert_forward(x: torch.Tensor, ids: torch.Tensor, w: torch.Tensor, weights: NVFP4MoEWeights,
                       out: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None):
    """out[T, H] BF16 = the NVFP4 W4A4 expert block over routed tokens."""
    lib = load()
    T, H = x.shape
    k = ids.shape[1]
    if out is None:
        out = torch.empty(T, H, dtype=torch.bfloat16, device=_dev(x))
    if workspace is None:
        workspace = moe_forward_workspace(T, k, weights, x.device)
    _check(lib.moe_expert_forward(_p(x), _p(ids), _p(w), T, k, ctypes.byref(weights.struct), _p(out),
                                  _p(workspace), workspace.numel(), _stream(stream)), "moe_expert_forward")
    return out


# --------------------------------------------------------------------------- backward (W4A4)

class NVFP4MoEWeightsT:
    """Transposed quantised expert weights for the backward's dgrad GEMMs (GEMM-tiled
    device buffers) plus the C struct that points at them."""

    def __init__(self, E: int, H: int, I: int, device):
        lib = load()
        sizes = (_sz * 4)()
        _check(lib.moe_weights_t_sizes(E, H, I, sizes), "moe_weights_t_sizes")
        self.E, self.H, self.I, self.Ip = E, H, I, (I + 255) // 256 * 256
        self.w13t = torch.empty(sizes[0], dtype=torch.uint8, device=device)
        self.w13t_g = torch.empty(E, dtype=torch.float32, device=device)
        self.w2t = torch.empty(sizes[2], dtype=torch.uint8, device=device)
        self.w2t_g = torch.empty(E, dtype=torch.float32, device=device)
        self.struct = _WeightsT(E, H, I, self.w13t.data_ptr(), self.w13t_g.data_ptr(), self.w2t.data_ptr(),
                                self.w2t_g.data_ptr())


def moe_prepare_weights_backward(w13: torch.Tensor, w2: torch.Tensor, stream=None) -> NVFP4MoEWeightsT:
    """Quantise W13^T and W2^T per expert (along the dgrad contractions) from the BF16
    W13 [E, 2I, H] and W2 [E, H, I]."""
    lib = load()
    E, N13, H = w13.shape
    I = N13 // 2
    pt = NVFP4MoEWeightsT(E, H, I, _dev(w13))
    ws = torch.empty(int(lib.nvfp4_workspace_size(OP_PREPARE_WEIGHTS_T, E, 0, 0, 0, 0)), dtype=torch.uint8,
                     device=w13.device)
    _check(lib.moe_prepare_weights_backward(_p(w13.contiguous()), _p(w2.contiguous()), E, H, I,
                                            ctypes.byref(pt.struct), _p(ws), ws.numel(), _stream(stream)),
           "moe_prepare_weights_backward")
    pt._ws = ws
    return pt


def moe_backward_workspace_layout(T: int, k: int, E: int, H: int, I: int) -> list:
    lib = load()
    out = (_i64 * 18)()
    _check(lib.moe_backward_workspace_layout(T, k, E, H, I, out), "moe_backward_workspace_layout")
    return list(out)


def moe_backward_workspace(T: int, k: int, weights: NVFP4MoEWeights, device) -> torch.Tensor:
    lib = load()
    n = int(lib.nvfp4_workspace_size(OP_MOE_BACKWARD, T, k, weights.E, weights.H, weights.I))
    return torch.empty(n, dtype=torch.uint8, device=device)


def moe_expert_backward(dout: torch.Tensor, x: torch.Tensor, w: torch.Tensor, weights: NVFP4MoEWeights,
                        weights_t: NVFP4MoEWeightsT, fwd_workspace: torch.Tensor, seed: int = 0, out=None,
                        workspace: torch.Tensor | None = None, stream=None):
    """The expert block's W4A4 backward for the forward whose workspace is fwd_workspace.
    Returns (dx [T, H] BF16, dw [T, k] f32, dw13 [E, 2I, H] f32, dw2 [E, H, I] f32)."""
    lib = load()
    T, H = x.shape
    k = w.shape[1]
    E, I = weights.E, weights.I
    dev = _dev(x)
    if out is None:
        out = (torch.empty(T, H, dtype=torch.bfloat16, device=dev), torch.empty(T, k, dtype=torch.float32, device=dev),
               torch.empty(E, 2 * I, H, dtype=torch.float32, device=dev),
               torch.empty(E, H, I, dtype=torch.float32, device=dev))
    dx, dw, dw13, dw2 = out
    if workspace is None:
        workspace = moe_backward_workspace(T, k, weights, dev)
    _check(lib.moe_expert_backward(_p(dout.contiguous()), _p(x), _p(w.contiguous()), T, k, ctypes.byref(weights.struct),
                                   ctypes.byref(weights_t.struct), _p(fwd_workspace), fwd_workspace.numel(), seed,
                                   _p(dx), _p(dw), _p(dw13), _p(dw2), _p(workspace), workspace.numel(),
                                   _stream(stream)), "moe_expert_backward")
    return dx, dw, dw13, dw2

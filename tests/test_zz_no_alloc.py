"""The quantiser entry point for callers that cannot allocate device memory.

Some callers of this library have no allocator they may use (a host plug-in handed only
its input and output tensors, for example), so they cannot provide the workspace that
nvfp4_quantize takes for its amax scratch.  nvfp4_quantize_noalloc keeps that scratch in
a fixed device array inside the library.  This test calls it through the C ABI and checks
its outputs against nvfp4_quantize's, bit for bit (the quantiser's parity tolerance), on
two calls in a row -- the second with a smaller amax, so stale scratch from the first
call would show.  The file is named to be collected last."""
import ctypes

import numpy as np
import pytest
import torch

from nvfp4_w4a4_moe_quantize_gb300 import synthetic as S

pytestmark = pytest.mark.gpu


def _noalloc_via_cabi(lib, x, mode, group_rows=0, rounding=0, seed=0):
    rows, cols = x.shape
    n_g = 1 if mode == lib.SCALE_PER_TENSOR else (rows if mode == lib.SCALE_PER_ROW else rows // group_rows)
    codes = torch.empty(rows, cols // 2, dtype=torch.uint8, device=x.device)
    sf = torch.empty(lib.nvfp4_sf_bytes(rows, cols), dtype=torch.uint8, device=x.device)
    g = torch.empty(n_g, dtype=torch.float32, device=x.device)
    c = lib.load()
    st = c.nvfp4_quantize_noalloc(ctypes.c_void_p(x.data_ptr()), rows, cols, x.stride(0), mode, group_rows,
                                  rounding, seed, 0, None, ctypes.c_void_p(g.data_ptr()),
                                  ctypes.c_void_p(codes.data_ptr()), ctypes.c_void_p(sf.data_ptr()),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.status_string(st)
    return codes, sf, g


@pytest.mark.parametrize("mode,group_rows", [(0, 0), (2, 64)])
def test_noalloc_matches_workspace_entry_point_twice(cuda_lib, mode, group_rows):
    big = S.outlier_channels_bf16(512, 2048, seed=1).cuda()
    small = (S.randn_bf16((512, 2048), 0.01, seed=2)).cuda()      # smaller amax on the second call
    for x in (big, small):
        got = _noalloc_via_cabi(cuda_lib, x, mode, group_rows, rounding=0)
        ref = cuda_lib.nvfp4_quantize(x, mode, 0, 0, 0, group_rows)
        for a, b in zip(got, ref):
            np.testing.assert_array_equal(a.cpu().numpy(), b[:a.numel()].cpu().numpy().reshape(a.shape))
    assert cuda_lib.nvfp4_status_check() == 0


def test_noalloc_rejects_too_many_scopes(cuda_lib):
    x = torch.zeros(8192, 16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cuda_lib.NVFP4Error):
        cuda_lib.nvfp4_quantize_noalloc(x, cuda_lib.SCALE_PER_GROUP, group_rows=1)

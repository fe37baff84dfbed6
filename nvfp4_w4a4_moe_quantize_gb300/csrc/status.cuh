// Device status word: kernels record bad input or an expired wait here instead of
// trapping; the host reads and clears it with nvfp4_status_check().
#pragma once

namespace nvfp4 {

enum : int { kStatusOk = 0, kStatusBadInput = 5, kStatusTimeout = 6 };

__device__ __forceinline__ void set_status(int* status, int code) {
  if (status != nullptr) atomicCAS(status, 0, code);   // first error wins
}

}  // namespace nvfp4

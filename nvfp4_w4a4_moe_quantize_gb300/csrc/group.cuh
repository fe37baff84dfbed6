// Expert group of a 128-row tile: the largest e with offsets[e] <= row0 (groups with no
// rows have offsets[e] == offsets[e+1] and are skipped by the search).
#pragma once
#include <cstdint>

namespace nvfp4 {

__device__ __forceinline__ int find_group(const int32_t* off, int E, int32_t row0) {
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= row0) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

}  // namespace nvfp4

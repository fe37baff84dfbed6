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

// Checks the group arrays of a grouped GEMM (already in shared memory) before any tile
// is touched: offsets[0..E] non-decreasing multiples of 128 starting at >= 0 with
// offsets[E] <= m_total, and 0 <= rows[e] <= offsets[e+1] - offsets[e].  Every thread of
// the block must call it (it ends with a block-wide vote); the result is the same in all
// of them.
__device__ __forceinline__ bool groups_valid(const int32_t* off, const int32_t* rows, int E, int64_t m_total) {
  int bad = 0;
  for (int i = threadIdx.x; i < E; i += blockDim.x) {
    const int32_t a = off[i], b = off[i + 1], r = rows[i];
    if (a < 0 || (a & 127) != 0 || b < a || (b & 127) != 0 || r < 0 || r > b - a) bad = 1;
  }
  if (threadIdx.x == 0 && (E < 1 || (int64_t)off[E] > m_total)) bad = 1;
  return __syncthreads_or(bad) == 0;
}

// The K-block prefix sums of a ragged-K grouped GEMM (already in shared memory):
// kofs[0] == 0, every expert at least one block, kofs[E] <= cap.  Block-wide, like
// groups_valid.
__device__ __forceinline__ bool kblocks_valid(const int32_t* kofs, int E, int64_t cap) {
  int bad = 0;
  for (int i = threadIdx.x; i < E; i += blockDim.x)
    if (kofs[i + 1] - kofs[i] < 1) bad = 1;
  if (threadIdx.x == 0 && (E < 1 || kofs[0] != 0 || (int64_t)kofs[E] > cap)) bad = 1;
  return __syncthreads_or(bad) == 0;
}

}  // namespace nvfp4

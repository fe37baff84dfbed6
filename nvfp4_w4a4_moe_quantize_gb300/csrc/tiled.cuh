// GEMM-tiled operand layout.
//
// An NVFP4 operand with K columns is stored as blocks of R rows (R = 128 for activations,
// 256 for weights) by 256 K-values.  Block (b, kb) starts at byte (b * (K/256) + kb) * R*144
// and holds
//   R * 128 bytes of codes in the order the tensor cores read a 128-byte-swizzled K-major
//     tile: row rr at rr*128, its 16-byte chunk j at ((j ^ (rr % 8)) * 16);
//   (R/128) * 2048 bytes of E4M3 scales: for row group g = rr/128 and k-group q of 64
//     values, a 512-byte 32x4 atom at g*2048 + q*512, scale (rr, c) at
//     (rr%32)*16 + ((rr%128)/32)*4 + c%4.
// A block is the exact shared-memory image of one pipeline stage, so the GEMM fetches it
// with a single bulk copy.
#pragma once
#include <cstdint>

namespace nvfp4 {

__host__ __device__ inline int64_t tiled_block_bytes(int R) { return (int64_t)R * 144; }
__host__ __device__ inline int64_t tiled_bytes(int64_t rows, int64_t K, int R) {
  return ((rows + R - 1) / R) * (K / 256) * tiled_block_bytes(R);
}

// R is 128 or 256, so the row block is a shift, not a division.
__host__ __device__ inline int tiled_log2_rows(int R) { return R == 256 ? 8 : 7; }

// byte b (< K/2) of the codes of row r
__host__ __device__ inline int64_t tiled_code_offset(int64_t r, int64_t b, int64_t kblocks, int R) {
  const int64_t blk = r >> tiled_log2_rows(R), rr = r & (R - 1), kb = b >> 7, bb = b & 127;
  return (blk * kblocks + kb) * tiled_block_bytes(R) + rr * 128 + ((((bb >> 4) ^ (rr & 7))) << 4) + (bb & 15);
}

// scale column c (< K/16) of row r
__host__ __device__ inline int64_t tiled_sf_offset(int64_t r, int64_t c, int64_t kblocks, int R) {
  const int64_t blk = r >> tiled_log2_rows(R), rr = r & (R - 1), kb = c >> 4, cc = c & 15;
  const int64_t rg = rr >> 7, r128 = rr & 127;
  return (blk * kblocks + kb) * tiled_block_bytes(R) + (int64_t)R * 128 + rg * 2048 + (cc >> 2) * 512 +
         (r128 & 31) * 16 + (r128 >> 5) * 4 + (cc & 3);
}

}  // namespace nvfp4

// Data movement into the GEMM-tiled operand layout (tiled.cuh): packing of row-major
// codes and scales, and the gather of token rows into the expert-grouped routed slots
// ("Low-Bit Precision Training Is Ready for Production...", §"What W4A4 GEMM Actually
// Changes": the expert GEMMs read these operands).
#include <cuda_runtime.h>

#include "launch.h"
#include "pdl.cuh"
#include "ptx.cuh"
#include "tiled.cuh"

namespace nvfp4 {

// Row-major codes [rows, K/2] + 128x4 tiled scales -> GEMM-tiled layout with R-row blocks;
// rows rows .. round_up(rows, R) - 1 are written as zeros.  One thread per 16-byte code
// chunk or 32-bit scale word of the output.
__global__ void __launch_bounds__(256) pack_tiled_kernel(const uint8_t* __restrict__ codes,
                                                         const uint8_t* __restrict__ sf, int64_t rows, int64_t K,
                                                         int R, uint8_t* __restrict__ out) {
  const int64_t kb = K / 256, rows_pad = (rows + R - 1) / R * R;
  const int64_t chunks = K / 32, words = K / 64, per_row = chunks + words;
  const int64_t total = rows_pad * per_row;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / per_row, u = i - r * per_row;
    if (u < chunks) {
      const uint4 v = r < rows ? *reinterpret_cast<const uint4*>(codes + r * (K / 2) + 16 * u) : make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(out + tiled_code_offset(r, 16 * u, kb, R)) = v;
    } else {
      const int64_t w = u - chunks;
      const uint32_t v = r < rows ? *reinterpret_cast<const uint32_t*>(
                                        sf + ((r >> 7) * words + w) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4)
                                  : 0u;
      *reinterpret_cast<uint32_t*>(out + tiled_sf_offset(r, 4 * w, kb, R)) = v;
    }
  }
}

// Gather of routed rows into the GEMM-tiled layout (128-row blocks): slot r of the
// expert-grouped order receives token perm[r]'s row of the per-token operand -- row-major
// codes `src` [T, K/2] and row-major scales `src_sf` [T, K/16] -- for every 256-K block,
// and its global scale.  Slots with perm[r] < 0 (group padding) get zero codes and
// scales.  One warp per (128-row block, K block) chunk of the output, assembled in shared
// memory: each lane first loads the 16 scale bytes of its four rows (lane + 32 i) into
// registers, then asynchronous 16-byte copies move each row's 128 code bytes (8 lanes per
// row, swizzled for the destination row), the scales go to the 128x4 image with four
// 16-byte shared stores per lane, and one bulk store writes the 18 KB image as whole
// lines.  The per-token operand is small next to L2, so the k-fold reads hit there; a
// row's scales of a K block are one 16-byte read.
__global__ void __launch_bounds__(32) gather_tiled_kernel(const uint8_t* __restrict__ src,
                                                          const uint8_t* __restrict__ src_sf,
                                                          const float* __restrict__ src_g,
                                                          const int32_t* __restrict__ perm,
                                                          const int32_t* __restrict__ n_rows_dev, int64_t max_rows,
                                                          int64_t kblocks, uint8_t* __restrict__ dst,
                                                          float* __restrict__ dst_g,
                                                          uint32_t* __restrict__ amax_zero) {
  grid_dep_sync();
  constexpr int R = 128;
  constexpr int64_t kChunk = R * 144;
  extern __shared__ __align__(128) uint8_t gsm[];
  const int lane = threadIdx.x;
  const uint32_t sb = smem_u32(gsm);
  int64_t rows = *n_rows_dev;
  if (rows > max_rows) rows = max_rows;
  const int64_t chunks = rows / R * kblocks;
  const int64_t code_row = kblocks * 128, sf_row = kblocks * 16;
  for (int64_t c = blockIdx.x; c < chunks; c += gridDim.x) {
    const int64_t b = c / kblocks, kb = c - (c / kblocks) * kblocks;
    int32_t pr[4];   // tokens of rows lane + 32 i of this block
#pragma unroll
    for (int i = 0; i < 4; ++i) pr[i] = perm[b * R + lane + 32 * i];
    uint4 sv[4];     // scale words 0..3 of this K block for rows lane + 32 i
#pragma unroll
    for (int i = 0; i < 4; ++i)
      sv[i] = pr[i] >= 0 ? *reinterpret_cast<const uint4*>(src_sf + (int64_t)pr[i] * sf_row + kb * 16)
                         : make_uint4(0u, 0u, 0u, 0u);
    if (lane == 0) bulk_wait_read<0>();   // the previous chunk's store has read the buffer
    __syncwarp();
    // codes: row rr's 16-byte chunk j, swizzled for the destination row
#pragma unroll
    for (int p = 0; p < 32; ++p) {
      const int rr = 4 * p + (lane >> 3), j = lane & 7;
      const int32_t t = __shfl_sync(0xFFFFFFFFu, pr[p >> 3], rr & 31);
      const uint32_t d = sb + rr * 128 + ((j ^ (rr & 7)) << 4);
      if (t >= 0) {
        cp_async_16(d, src + (int64_t)t * code_row + kb * 128 + j * 16);
      } else {
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(d), "r"(0u) : "memory");
      }
    }
    // scales: word q of row rr sits at q * 512 + (rr & 31) * 16 + (rr >> 5) * 4, so the
    // four rows of a lane fill one 16-byte slot per word
    {
      const uint32_t d = sb + R * 128 + lane * 16;
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(d), "r"(sv[0].x), "r"(sv[1].x), "r"(sv[2].x),
                   "r"(sv[3].x)
                   : "memory");
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(d + 512), "r"(sv[0].y), "r"(sv[1].y),
                   "r"(sv[2].y), "r"(sv[3].y)
                   : "memory");
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(d + 1024), "r"(sv[0].z), "r"(sv[1].z),
                   "r"(sv[2].z), "r"(sv[3].z)
                   : "memory");
      asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(d + 1536), "r"(sv[0].w), "r"(sv[1].w),
                   "r"(sv[2].w), "r"(sv[3].w)
                   : "memory");
    }
    cp_async_wait_all();
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      bulk_store(dst + (b * kblocks + kb) * kChunk, gsm, (uint32_t)kChunk);
      bulk_commit();
    }
    if (kb == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (pr[i] >= 0) dst_g[b * R + lane + 32 * i] = src_g[pr[i]];
        if (amax_zero != nullptr) amax_zero[b * R + lane + 32 * i] = 0u;
      }
    }
  }
  if (lane == 0) bulk_wait_all<0>();   // the last store is complete before the CTA exits
  __syncwarp();
}

cudaError_t launch_gather_tiled(const uint8_t* src, const uint8_t* src_sf, const float* src_g, const int32_t* perm,
                                const int32_t* n_rows_dev, int64_t max_rows, int64_t K, uint8_t* dst, float* dst_g,
                                uint32_t* amax_zero, cudaStream_t s) {
  constexpr int kSmem = 128 * 144;
  const int64_t chunks = max_rows / 128 * (K / 256);
  if (chunks == 0) return cudaSuccess;
  static std::atomic<bool> attr_set[64];   // the attribute is set once per device
  {
    const cudaError_t err = set_smem_attr_once(attr_set, (const void*)gather_tiled_kernel, kSmem);
    if (err != cudaSuccess) return err;
  }
  // one warp per block and one 18 KB chunk image per warp: 12 per SM fit in shared memory
  int64_t blocks = chunks;
  if (blocks > 12 * (int64_t)num_sms()) blocks = 12 * (int64_t)num_sms();
  return launch_pdl(false, gather_tiled_kernel, dim3((unsigned)blocks), dim3(32), kSmem, s, src, src_sf, src_g, perm,
                    n_rows_dev, max_rows, K / 256, dst, dst_g, amax_zero);
}

// out[b*C + c, r] = x[b*R + r, c] for `batches` stacked [R, C] BF16 matrices (pitch ld):
// 32 x 32 tiles through shared memory (one padding column: no bank conflicts), loads and
// stores both along rows.
__global__ void __launch_bounds__(256) transpose_bf16_kernel(const uint16_t* __restrict__ x, int64_t R, int64_t C,
                                                             int64_t ld, uint16_t* __restrict__ out) {
  __shared__ uint16_t tile[32][33];
  const int64_t b = blockIdx.z, c0 = (int64_t)blockIdx.x * 32, r0 = (int64_t)blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  for (int j = ty; j < 32; j += 8) {
    const int64_t r = r0 + j, c = c0 + tx;
    if (r < R && c < C) tile[j][tx] = x[(b * R + r) * ld + c];
  }
  __syncthreads();
  for (int j = ty; j < 32; j += 8) {
    const int64_t c = c0 + j, r = r0 + tx;
    if (r < R && c < C) out[(b * C + c) * R + r] = tile[tx][j];
  }
}

cudaError_t launch_transpose_bf16(const void* x, int64_t batches, int64_t R, int64_t C, int64_t ld, void* out,
                                  cudaStream_t s) {
  if (batches == 0 || R == 0 || C == 0) return cudaSuccess;
  const dim3 grid((unsigned)((C + 31) / 32), (unsigned)((R + 31) / 32), (unsigned)batches);
  transpose_bf16_kernel<<<grid, 256, 0, s>>>(static_cast<const uint16_t*>(x), R, C, ld, static_cast<uint16_t*>(out));
  return cudaGetLastError();
}

cudaError_t launch_pack_tiled(const uint8_t* codes, const uint8_t* sf, int64_t rows, int64_t K, int R, uint8_t* out,
                              cudaStream_t s) {
  const int64_t rows_pad = (rows + R - 1) / R * R;
  const int64_t total = rows_pad * (K / 32 + K / 64);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 16 * num_sms()) blocks = 16 * num_sms();
  pack_tiled_kernel<<<(int)blocks, 256, 0, s>>>(codes, sf, rows, K, R, out);
  return cudaGetLastError();
}

}  // namespace nvfp4

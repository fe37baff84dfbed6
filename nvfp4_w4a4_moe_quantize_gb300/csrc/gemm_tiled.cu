// W4A4 grouped GEMM over GEMM-tiled operands (see tiled.cuh), the kernel of the expert
// block's two projections ("Low-Bit Precision Training Is Ready for Production...",
// §"What W4A4 GEMM Actually Changes"; "miniTE identifies and closes the execution gap
// ...", §Development: grouped GEMMs):
//     D[r, n] = (gA[r] * gB[e]) * sum_k value(A)[r,k] sf_A[r,k/16] value(B_e)[n,k] sf_B[n,k/16]
//
// On this GPU an asynchronous copy costs a fixed ~0.2 us of issue time per operation
// and per issuing thread, so a stage built from separate code and scale-factor copies is
// paced by the copy count, not by bytes.  In the tiled layout every 128-row x 256-K block
// of A (18 KB) and every 256-row x 256-K block of B (36 KB) is the exact shared-memory
// image of a stage -- swizzled codes followed by their scales -- so a stage is two bulk
// copies, issued by two producer warps in parallel.
//
// One CTA per SM, 11 warps:
//   warp 0 / 1  producers of the A / B block of each stage (cp.async.bulk + mbarrier);
//   warp 2      MMA issuer: tcgen05.cp of the stage's scales into TMEM, four
//               tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X (M=128, N=256,
//               K=64) into a 256-column TMEM accumulator, tcgen05.commit;
//   warps 3-10  epilogue, two per TMEM lane quadrant (128 columns each): drain the
//               accumulator into registers, release it, scale by gA[r]*gB[e] in float32
//               and store BF16 / float32 rows of the group -- or, in the SwiGLU mode of
//               the gate/up projection, form h = BF16(silu(gate) * up) from the BF16-
//               rounded gate and up columns and store h only.
// Tiles are (128-row block) x (256 columns), row-block-major; no split-K, fixed K order.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "group.cuh"
#include "launch.h"
#include "ptx.cuh"
#include "swiglu.cuh"
#include "tiled.cuh"

namespace nvfp4 {

namespace gt {
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kStages = 4;
constexpr int kABlock = 128 * 144;          // 16 KB codes + 2 KB scales
constexpr int kBBlock = 256 * 144;          // 32 KB codes + 4 KB scales
constexpr int kACodes = 128 * 128;
constexpr int kBCodes = 256 * 128;
constexpr int kTmemCols = 512;
constexpr int kAccCols = kBN;
constexpr int kSFCol0 = kAccCols;
constexpr int kSFStageCols = 16 + 32;       // A: 4 x 4 columns, B: 4 x 8 columns
constexpr int kEpiWarps = 8;
constexpr int kFirstEpiWarp = 3;
constexpr int kThreads = 32 * (kFirstEpiWarp + kEpiWarps);
constexpr int kMaxE = 512;

struct Smem {
  uint8_t a[kStages][kABlock];
  uint8_t b[kStages][kBBlock];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t accf;
  uint64_t acce;
  uint32_t tmem_base;
  int abort;
  int32_t offsets[kMaxE + 1];
  int32_t rows[kMaxE];
  float gb[kMaxE];
};
static_assert(kABlock % 1024 == 0 && kBBlock % 1024 == 0, "1024-byte aligned stage images");
static_assert(kSFCol0 + kStages * kSFStageCols <= kTmemCols, "TMEM budget");
static_assert(sizeof(Smem) + 1024 <= 232448, "shared memory budget");
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
}  // namespace gt

template <bool kSwiGLU>
__global__ void __launch_bounds__(gt::kThreads, 1)
    grouped_gemm_tiled_kernel(const uint8_t* __restrict__ A, const uint8_t* __restrict__ B, const GemmArgs g) {
  using namespace gt;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  for (int i = threadIdx.x; i <= g.E; i += blockDim.x) sm.offsets[i] = g.offsets[i];
  for (int i = threadIdx.x; i < g.E; i += blockDim.x) {
    sm.rows[i] = g.rows[i];
    sm.gb[i] = g.gb[i];
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 2);            // the A and the B producer arrive
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(&sm.accf, 1);
    mbar_init(&sm.acce, kEpiWarps * 32);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;

  const int n_tiles = g.N / kBN;
  const int m_tiles = sm.offsets[g.E] / kBM;
  const int total = m_tiles * n_tiles;
  const int kblocks = g.K / 256;

  if (warp < 2) {
    if (lane == 0) {
      const bool is_a = warp == 0;
      uint32_t stage = 0, phase = 0;
      for (int t = blockIdx.x; t < total; t += gridDim.x) {
        const int m_tile = t / n_tiles, n_tile = t - (t / n_tiles) * n_tiles;
        int64_t blk;
        if (is_a) {
          blk = m_tile;
        } else {
          const int e = find_group(sm.offsets, g.E, m_tile * kBM);
          blk = (int64_t)e * n_tiles + n_tile;
        }
        const uint8_t* src = (is_a ? A : B) + blk * kblocks * (int64_t)(is_a ? kABlock : kBBlock);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&sm.empty[stage], phase ^ 1u, g.status, abort)) goto producer_done;
          const uint32_t bytes = is_a ? kABlock : kBBlock;
          mbar_arrive_expect_tx(&sm.full[stage], bytes);
          bulk_load(is_a ? sm.a[stage] : sm.b[stage], src + (int64_t)kb * bytes, bytes, &sm.full[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    producer_done:;
    }
  } else if (warp == 2) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_nvf4(kBM, kBN);
      uint32_t stage = 0, phase = 0;
      int it = 0;
      for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
        if (!mbar_wait(&sm.acce, (it & 1) ^ 1u, g.status, abort)) break;   // accumulator drained
        tc_fence_after();
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&sm.full[stage], phase, g.status, abort)) goto mma_done;
          tc_fence_after();
          const uint32_t sfa_t = tmem + kSFCol0 + stage * kSFStageCols;
          const uint32_t sfb_t = sfa_t + 16;
          const uint32_t sa = smem_u32(sm.a[stage]), sb = smem_u32(sm.b[stage]);
          const uint32_t ssfa = sa + kACodes, ssfb = sb + kBCodes;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            tc_cp_32x128b_warpx4(sfa_t + 4 * j, smem_desc(ssfa + 512 * j, 0, 128, 0));
            tc_cp_32x128b_warpx4(sfb_t + 8 * j, smem_desc(ssfb + 512 * j, 0, 128, 0));
            tc_cp_32x128b_warpx4(sfb_t + 8 * j + 4, smem_desc(ssfb + 2048 + 512 * j, 0, 128, 0));
          }
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint64_t adesc = smem_desc(sa + 32 * j, 16, 1024, 2);
            const uint64_t bdesc = smem_desc(sb + 32 * j, 16, 1024, 2);
            tc_mma_nvf4(tmem, adesc, bdesc, idesc, sfa_t + 4 * j, sfb_t + 8 * j, (kb | j) != 0 ? 1u : 0u);
          }
          tc_commit(&sm.empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        tc_commit(&sm.accf);
      }
    mma_done:;
    }
  } else {
    // epilogue: lane quadrant q = warp % 4, column half of the tile = (warp - 3) / 4
    const int q = warp & 3;
    const int half = (warp - kFirstEpiWarp) >> 2;
    const int elt = g.out_f32 ? 4 : 2;
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      const int m_tile = t / n_tiles, n_tile = t - (t / n_tiles) * n_tiles;
      const int32_t row0 = m_tile * kBM;
      const int e = find_group(sm.offsets, g.E, row0);
      const int32_t in_group = sm.rows[e] - (row0 - sm.offsets[e]);
      const bool valid = q * 32 + lane < in_group;
      const int64_t row = (int64_t)row0 + q * 32 + lane;
      const float ga = valid ? g.ga[row] : 0.0f;
      if (!mbar_wait(&sm.accf, it & 1, g.status, abort)) break;
      tc_fence_after();
      const float scale = __fmul_rn(ga, sm.gb[e]);
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + half * 128;
      uint32_t v[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) NVFP4_TMEM_LD_X32(taddr + 32 * c, v[c]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&sm.acce);
      if (!valid) continue;
      if (kSwiGLU) {
        // columns [0, 64) of this half are gate, [64, 128) up, for h columns
        // n_tile*128 + half*64 + [0, 64) (64-row gate/up interleave of W13)
        __nv_bfloat16* hp = g.h + row * g.I + (int64_t)n_tile * 128 + half * 64;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
#pragma unroll
          for (int u8 = 0; u8 < 4; ++u8) {
            uint32_t w[4];
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              uint32_t hb[2];
#pragma unroll
              for (int s2 = 0; s2 < 2; ++s2) {
                const int i = 8 * u8 + 2 * p + s2;
                const float gate = __bfloat162float(__float2bfloat16_rn(__fmul_rn(__uint_as_float(v[c][i]), scale)));
                const float up = __bfloat162float(__float2bfloat16_rn(__fmul_rn(__uint_as_float(v[c + 2][i]), scale)));
                hb[s2] = swiglu_bf16(gate, up);
              }
              w[p] = hb[0] | (hb[1] << 16);
            }
            *reinterpret_cast<uint4*>(hp + 32 * c + 8 * u8) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      } else {
        uint8_t* dp = static_cast<uint8_t*>(g.d) + (row * g.ldd + (int64_t)n_tile * kBN + half * 128) * elt;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (g.out_f32) {
#pragma unroll
            for (int u4 = 0; u4 < 8; ++u4)
              *reinterpret_cast<float4*>(dp + (32 * c + 4 * u4) * 4) =
                  make_float4(__fmul_rn(__uint_as_float(v[c][4 * u4]), scale),
                              __fmul_rn(__uint_as_float(v[c][4 * u4 + 1]), scale),
                              __fmul_rn(__uint_as_float(v[c][4 * u4 + 2]), scale),
                              __fmul_rn(__uint_as_float(v[c][4 * u4 + 3]), scale));
          } else {
#pragma unroll
            for (int u4 = 0; u4 < 4; ++u4) {
              uint32_t w[4];
#pragma unroll
              for (int p = 0; p < 4; ++p) {
                const __nv_bfloat162 b2 =
                    __floats2bfloat162_rn(__fmul_rn(__uint_as_float(v[c][8 * u4 + 2 * p]), scale),
                                          __fmul_rn(__uint_as_float(v[c][8 * u4 + 2 * p + 1]), scale));
                w[p] = *reinterpret_cast<const uint32_t*>(&b2);
              }
              *reinterpret_cast<uint4*>(dp + (32 * c + 8 * u4) * 2) = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, kTmemCols);
}

template <bool kSwiGLU>
static cudaError_t launch_tiled(const uint8_t* A, const uint8_t* B, const GemmArgs& g, int64_t max_m_tiles,
                                cudaStream_t s) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !attr_set[dev]) {
    cudaError_t err = cudaFuncSetAttribute(grouped_gemm_tiled_kernel<kSwiGLU>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gt::kSmemBytes);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64) attr_set[dev] = true;
  }
  const int64_t tiles = max_m_tiles * (g.N / gt::kBN);
  if (tiles == 0) return cudaSuccess;
  int grid = num_sms();
  if (tiles < grid) grid = (int)tiles;
  grouped_gemm_tiled_kernel<kSwiGLU><<<grid, gt::kThreads, gt::kSmemBytes, s>>>(A, B, g);
  return cudaGetLastError();
}

cudaError_t launch_grouped_gemm_tiled(const uint8_t* A, const uint8_t* B, const GemmArgs& g, int64_t max_m_tiles,
                                      bool swiglu, cudaStream_t s) {
  return swiglu ? launch_tiled<true>(A, B, g, max_m_tiles, s) : launch_tiled<false>(A, B, g, max_m_tiles, s);
}

int tiled_max_experts() { return gt::kMaxE; }

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

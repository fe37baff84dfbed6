// W4A4 grouped GEMM with 128 x 256 output tiles over row-major operands: the same
// computation as grouped_gemm.cu ("Low-Bit Precision Training Is Ready for
// Production...", §"What W4A4 GEMM Actually Changes"), issued as M=128, N=256, K=64
// block-scaled MMAs.  An N=256 instruction costs the tensor pipe about the same time as
// an N=128 one, so this shape doubles the work per instruction; it is used whenever N is
// a multiple of 256.
//
// One persistent CTA per SM; every CTA loads its own operands (TMA boxes of 128 rows:
// one for A, two for the 256 weight rows, plus the matching scale blocks by bulk copy),
// so no CTA ever waits on another.  Tiles are (128-row block of the padded group layout)
// x (256 output columns), row-block-major, so CTAs running at the same time share A
// tiles and one expert's weights in L2.
//
// One 256-column TMEM accumulator per CTA (the scale factors of the stages take the rest
// of TMEM), 4 stages of 54 KB, and 8 epilogue warps (two per TMEM lane quadrant, 128
// columns each) that drain the accumulator into registers at once and release it before
// converting and storing.  Rows outside the groups are never written.
//
// Instantiated with kMX, the same kernel runs the MXFP8 grouped GEMM (E4M3 operands,
// E8M0 scales per 32 values, no global scales; see grouped_gemm.cu): a stage holds 128
// K-values, one 512-byte scale tile per 128 rows, and four
// kind::mxf8f6f4.block_scale.scale_vec::1X MMAs (K = 32) that pick byte j of the scale
// words through their scale-factor ids.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "group.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace nvfp4 {

namespace g256 {
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBKBytes = 128;                // 256 FP4 values of K per stage
#ifndef NVFP4_N256_STAGES
#define NVFP4_N256_STAGES 4
#endif
constexpr int kStages = NVFP4_N256_STAGES;   // build-time tunable
constexpr int kABytes = kBM * kBKBytes;      // 16 KB
constexpr int kBBytes = kBN * kBKBytes;      // 32 KB
constexpr int kSFABytes = 4 * 512;           // 4 k-groups x (128 rows x 4 scales)
constexpr int kSFBBytes = 2 * 4 * 512;       // 2 row groups of 128
constexpr int kTmemCols = 512;
constexpr int kAccCols = kBN;                // one accumulator: 128 lanes x 256 float32
constexpr int kSFCol0 = kAccCols;
constexpr int kSFStageCols = 16 + 32;        // A: 4 x 4 columns, B: 4 x 8 columns
constexpr int kEpiWarps = 8;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kMaxE = 512;

struct Smem {
  uint8_t a[kStages][kABytes];
  uint8_t b[kStages][kBBytes];
  uint8_t sfa[kStages][kSFABytes];
  uint8_t sfb[kStages][kSFBBytes];
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
static_assert(kSFCol0 + kStages * kSFStageCols <= kTmemCols, "TMEM budget");
static_assert(sizeof(Smem) + 1024 <= 232448, "shared memory budget");
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
}  // namespace g256

template <bool kMX>
__global__ void __launch_bounds__(g256::kThreads, 1)
    grouped_gemm_n256_kernel(const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmb,
                             const GemmArgs g) {
  using namespace g256;
  constexpr int kStageK = kMX ? 128 : 256;            // K values per stage
  constexpr int kSFA = kMX ? 512 : kSFABytes;         // A's scales per stage
  constexpr int kSFB128 = kMX ? 512 : 2048;           // scales per stage of one 128-row half of B
  constexpr uint32_t kTx = kABytes + kBBytes + kSFA + 2 * kSFB128;
  constexpr int kSFTiles = kMX ? 1 : 4;               // 512-byte scale tiles per stage and 128 rows
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  for (int i = threadIdx.x; i <= g.E; i += blockDim.x) sm.offsets[i] = g.offsets[i];
  for (int i = threadIdx.x; i < g.E; i += blockDim.x) {
    sm.rows[i] = g.rows[i];
    sm.gb[i] = kMX ? 1.0f : g.gb[i];
  }
  __syncthreads();
  if (!groups_valid(sm.offsets, sm.rows, g.E, g.m_total)) {   // nothing is read or written
    if (threadIdx.x == 0) set_status(g.status, kStatusBadInput);
    return;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    mbar_init(&sm.accf, 1);
    mbar_init(&sm.acce, kEpiWarps * 32);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tma);
    prefetch_tensormap(&tmb);
  }
  if (warp == 1) {
    tmem_alloc(&sm.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;

  const int n_tiles = g.N / kBN;
  const int total = sm.offsets[g.E] / kBM * n_tiles;
  const int kblocks = g.K / kStageK;
  const int64_t sf_kgroups = g.K / (kMX ? 128 : 64);

  if (warp == 0) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      for (int t = blockIdx.x; t < total; t += gridDim.x) {
        const int m_tile = t / n_tiles, n_tile = t - (t / n_tiles) * n_tiles;
        const int32_t row0 = m_tile * kBM;
        const int e = find_group(sm.offsets, g.E, row0);
        const int32_t brow = e * g.N + n_tile * kBN;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&sm.empty[stage], phase ^ 1u, g.status, abort)) goto producer_done;
          mbar_arrive_expect_tx(&sm.full[stage], kTx);
          tma_load_2d(sm.a[stage], &tma, kb * kBKBytes, row0, &sm.full[stage]);
#pragma unroll
          for (int h = 0; h < 2; ++h)
            tma_load_2d(sm.b[stage] + h * (kBBytes / 2), &tmb, kb * kBKBytes, brow + h * 128, &sm.full[stage]);
          bulk_load(sm.sfa[stage], g.sfa + ((int64_t)m_tile * sf_kgroups + kb * kSFTiles) * 512, kSFA,
                    &sm.full[stage]);
#pragma unroll
          for (int h = 0; h < 2; ++h)
            bulk_load(sm.sfb[stage] + h * kSFB128,
                      g.sfb + ((int64_t)(brow / 128 + h) * sf_kgroups + kb * kSFTiles) * 512, kSFB128,
                      &sm.full[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    producer_done:;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = kMX ? idesc_mxf8(kBM, kBN, 0) : idesc_nvf4(kBM, kBN);
      uint32_t stage = 0, phase = 0;
      int it = 0;
      for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&sm.full[stage], phase, g.status, abort)) goto mma_done;
          tc_fence_after();
          const uint32_t sfa_t = tmem + kSFCol0 + stage * kSFStageCols;
          const uint32_t sfb_t = sfa_t + 16;
          const uint32_t sa = smem_u32(sm.a[stage]), sb = smem_u32(sm.b[stage]);
          const uint32_t ssfa = smem_u32(sm.sfa[stage]), ssfb = smem_u32(sm.sfb[stage]);
          // The first stage's scale copies go out before the accumulator wait: they do not
          // touch the accumulator, and tcgen05 ops of one thread execute in issue order.
          const bool first = kb == 0;
          if constexpr (kMX) {
            tc_cp_32x128b_warpx4(sfa_t, smem_desc(ssfa, 0, 128, 0));
            tc_cp_32x128b_warpx4(sfb_t, smem_desc(ssfb, 0, 128, 0));
            tc_cp_32x128b_warpx4(sfb_t + 4, smem_desc(ssfb + 512, 0, 128, 0));
            if (first) {
              if (!mbar_wait(&sm.acce, (it & 1) ^ 1u, g.status, abort)) goto mma_done;   // accumulator drained
              tc_fence_after();
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint64_t adesc = smem_desc(sa + 32 * j, 16, 1024, 2);
              const uint64_t bdesc = smem_desc(sb + 32 * j, 16, 1024, 2);
              tc_mma_mxf8(tmem, adesc, bdesc, idesc_mxf8(kBM, kBN, (uint32_t)j), sfa_t, sfb_t,
                          (kb | j) != 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              tc_cp_32x128b_warpx4(sfa_t + 4 * j, smem_desc(ssfa + 512 * j, 0, 128, 0));
              tc_cp_32x128b_warpx4(sfb_t + 8 * j, smem_desc(ssfb + 512 * j, 0, 128, 0));
              tc_cp_32x128b_warpx4(sfb_t + 8 * j + 4, smem_desc(ssfb + 2048 + 512 * j, 0, 128, 0));
            }
            if (first) {
              if (!mbar_wait(&sm.acce, (it & 1) ^ 1u, g.status, abort)) goto mma_done;   // accumulator drained
              tc_fence_after();
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint64_t adesc = smem_desc(sa + 32 * j, 16, 1024, 2);
              const uint64_t bdesc = smem_desc(sb + 32 * j, 16, 1024, 2);
              tc_mma_nvf4(tmem, adesc, bdesc, idesc, sfa_t + 4 * j, sfb_t + 8 * j, (kb | j) != 0 ? 1u : 0u);
            }
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
    // epilogue: warps 2..9.  Lane quadrant q = warp % 4, column half = (warp - 2) / 4.
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int elt = g.out_f32 ? 4 : 2;
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      const int m_tile = t / n_tiles, n_tile = t - (t / n_tiles) * n_tiles;
      const int32_t row0 = m_tile * kBM;
      const int e = find_group(sm.offsets, g.E, row0);
      const int32_t in_group = sm.rows[e] - (row0 - sm.offsets[e]);   // valid rows of this tile
      const bool valid = q * 32 + lane < in_group;
      const int64_t row = (int64_t)row0 + q * 32 + lane;
      const float ga = kMX ? 1.0f : (valid ? g.ga[row] : 0.0f);
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
      if (valid) {
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
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

bool n256_supported(const GemmArgs& g) { return g.N % g256::kBN == 0 && g.E <= g256::kMaxE; }

template <bool kMX>
static cudaError_t launch_n256(const CUtensorMap& tma, const CUtensorMap& tmb, const GemmArgs& g,
                               int64_t max_m_tiles, cudaStream_t s) {
  static std::atomic<bool> attr_set[64];
  cudaError_t err = set_smem_attr_once(attr_set, (const void*)grouped_gemm_n256_kernel<kMX>, (int)g256::kSmemBytes);
  if (err != cudaSuccess) return err;
  const int64_t tiles = max_m_tiles * (g.N / g256::kBN);
  if (tiles == 0) return cudaSuccess;
  int grid = num_sms();
  if (tiles < grid) grid = (int)tiles;
  grouped_gemm_n256_kernel<kMX><<<grid, g256::kThreads, g256::kSmemBytes, s>>>(tma, tmb, g);
  return cudaGetLastError();
}

cudaError_t launch_grouped_gemm_n256(const CUtensorMap& tma, const CUtensorMap& tmb, const GemmArgs& g,
                                     int64_t max_m_tiles, cudaStream_t s) {
  return launch_n256<false>(tma, tmb, g, max_m_tiles, s);
}

cudaError_t launch_grouped_gemm_n256_mx(const CUtensorMap& tma, const CUtensorMap& tmb, const GemmArgs& g,
                                        int64_t max_m_tiles, cudaStream_t s) {
  return launch_n256<true>(tma, tmb, g, max_m_tiles, s);
}

}  // namespace nvfp4

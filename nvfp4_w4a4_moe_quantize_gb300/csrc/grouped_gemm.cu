// W4A4 grouped GEMM over ragged expert groups on the 5th-generation tensor cores.
//
// "Low-Bit Precision Training Is Ready for Production...", §"What W4A4 GEMM Actually
// Changes": with both operands in 4 bits the GEMM itself runs at FP4 tensor-core rate;
// "miniTE identifies and closes the execution gap...", §Development: grouped GEMMs
// over the experts.  For every row r of expert e's group:
//     D[r, n] = (gA[r] * gB[e]) * sum_k value(A)[r,k] sf_A[r,k/16] value(B_e)[n,k] sf_B[n,k/16]
//
// Design (one CTA per SM, persistent, 6 warps):
//   warp 0  TMA producer: A tile 128 x 256 codes and B tile 128 x 256 codes per stage
//           (128-byte swizzled boxes), plus the matching 2 KB scale-factor blocks of A and
//           B by bulk copy -- the tiled scale layout keeps them contiguous.
//   warp 1  MMA issuer: copies the stage's scales into TMEM (tcgen05.cp 32x128b.warpx4),
//           then four tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X (M=128, N=128,
//           K=64) into a TMEM accumulator; tcgen05.commit frees the stage.  Two
//           accumulators let the epilogue of one tile overlap the main loop of the next.
//   warps 2-5  epilogue: tcgen05.ld 32 lanes x 32 columns, scale by gA[r] * gB[e] in
//           float32, round to BF16 (or keep float32); whole 32-row blocks of a group go
//           through a swizzled shared-memory box and a TMA store, the last partial block
//           of a group is stored row by row, so rows outside the groups are never written.
// Tiles are (128-row block of the padded group layout) x (128 output columns); tile t
// is row block t / (N/128), column block t % (N/128), so CTAs running at the same time
// share A tiles and one expert's weights in L2.  The K loop has a fixed order and no
// split, so every output element has one accumulation order whatever the batch.
//
// The same kernel is also the BF16 grouped GEMM of the dequantised backward ("The
// 4-bitter Lesson...", §"Improving Gradient Stability": the backward GEMMs take the
// dequantised weights DQ(Q(W)), in BF16): kind::f16 MMAs (M=128, N=128, K=16) on BF16
// operands, 64 K-values per stage, no scale factors, no global scales.
//
// Instantiated with the MX format it is the MXFP8 grouped GEMM of the recipe's
// validation format ("The 4-bitter Lesson...", §"Improving Gradient Stability", Results
// Validation with MXFP8): E4M3 operands with one E8M0 scale per 32 values of K, no global
// scales.  A stage is then 128 K-values (one 128-byte swizzle row of 8-bit codes).  The
// stage's scales are one 512-byte tile of the 128x4 layout per 128 rows, copied into TMEM
// with one tcgen05.cp.  Four tcgen05.mma.kind::mxf8f6f4.block_scale.scale_vec::1X
// (K = 32 each) follow; MMA j reads byte j of each 32-bit scale word through the
// scale-factor ids of its instruction descriptor.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "group.cuh"
#include "launch.h"
#include "ptx.cuh"

namespace nvfp4 {

enum : int { kGemmNVF4 = 0, kGemmMXF8 = 1, kGemmBF16 = 2 };

namespace gg {
constexpr int kBM = 128;          // rows per tile (one per TMEM lane)
constexpr int kBN = 128;          // output columns per tile
constexpr int kBKBytes = 128;     // K bytes per stage = 256 FP4 values (one 128-byte swizzle row)
constexpr int kStages = 5;
constexpr int kABytes = kBM * kBKBytes;
constexpr int kBBytes = kBN * kBKBytes;
constexpr int kSFABytes = 4 * 512;           // 4 k-groups of 64 x 128 rows
constexpr int kSFBBytes = (kBN / 128) * 4 * 512;
constexpr int kTmemCols = 512;
constexpr int kAccCols = kBN;                // one accumulator: 128 lanes x kBN float32
constexpr int kSFCol0 = 2 * kAccCols;        // scale factors after the two accumulators
constexpr int kSFStageCols = 16 + 4 * 4 * (kBN / 128);
constexpr int kEpiWarps = 4;
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kMaxE = 1024;
constexpr int kOutBox = 32 * 128;            // one 32-row x 128-byte swizzled store box

struct Smem {
  uint8_t a[kStages][kABytes];
  uint8_t b[kStages][kBBytes];
  uint8_t sfa[kStages][kSFABytes];
  uint8_t sfb[kStages][kSFBBytes];
  uint8_t out[kEpiWarps][2][kOutBox];        // double-buffered store staging per epilogue warp
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t accf[2];
  uint64_t acce[2];
  uint32_t tmem_base;
  int abort;
  int32_t offsets[kMaxE + 1];
  int32_t rows[kMaxE];
  float gb[kMaxE];
};
static_assert(kSFCol0 + kStages * kSFStageCols <= kTmemCols, "TMEM budget");
static_assert(sizeof(Smem) + 1024 <= 232448, "shared memory budget");
constexpr size_t kSmemBytes = sizeof(Smem) + 1024;
}  // namespace gg

template <int kFmt>
__global__ void __launch_bounds__(gg::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tma, const __grid_constant__ CUtensorMap tmb,
                        const __grid_constant__ CUtensorMap tmd, const GemmArgs g) {
  using namespace gg;
  // per stage: K values, bytes of A's scales, bytes of one 128-row block of B's scales
  constexpr bool kMX = kFmt == kGemmMXF8, kBF = kFmt == kGemmBF16;
  constexpr int kStageK = kBF ? 64 : (kMX ? 128 : 256);
  constexpr int kSFA = kBF ? 0 : (kMX ? 512 : kSFABytes);
  constexpr int kSFB128 = kBF ? 0 : (kMX ? 512 : 2048);
  constexpr uint32_t kTx = kABytes + kBBytes + kSFA + (kBN / 128) * kSFB128;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  for (int i = threadIdx.x; i <= g.E; i += blockDim.x) sm.offsets[i] = g.offsets[i];
  for (int i = threadIdx.x; i < g.E; i += blockDim.x) {
    sm.rows[i] = g.rows[i];
    sm.gb[i] = kFmt != kGemmNVF4 ? 1.0f : g.gb[i];
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
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sm.accf[a], 1);
      mbar_init(&sm.acce[a], kEpiWarps * 32);
    }
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tma);
    prefetch_tensormap(&tmb);
    prefetch_tensormap(&tmd);
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
  const int m_tiles = sm.offsets[g.E] / kBM;
  const int total = m_tiles * n_tiles;
  const int kblocks = g.K / kStageK;
  const int64_t sf_kgroups = g.K / (kMX ? 128 : 64);   // 512-byte scale tiles per 128-row block
  constexpr int kSFTiles = kMX ? 1 : 4;                 // scale tiles per stage and 128 rows

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
          tma_load_2d(sm.b[stage], &tmb, kb * kBKBytes, brow, &sm.full[stage]);
          if constexpr (!kBF) {
            bulk_load(sm.sfa[stage], g.sfa + ((int64_t)m_tile * sf_kgroups + kb * kSFTiles) * 512, kSFA,
                      &sm.full[stage]);
#pragma unroll
            for (int h = 0; h < kBN / 128; ++h)
              bulk_load(sm.sfb[stage] + h * kSFB128,
                        g.sfb + ((int64_t)(brow / 128 + h) * sf_kgroups + kb * kSFTiles) * 512, kSFB128,
                        &sm.full[stage]);
          }
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
      constexpr uint32_t idesc = kBF ? idesc_bf16(kBM, kBN) : (kMX ? idesc_mxf8(kBM, kBN, 0) : idesc_nvf4(kBM, kBN));
      uint32_t stage = 0, phase = 0;
      int it = 0;
      for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
        const uint32_t acc = it & 1, acc_phase = (it >> 1) & 1;
        if (!mbar_wait(&sm.acce[acc], acc_phase ^ 1u, g.status, abort)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem + acc * kAccCols;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&sm.full[stage], phase, g.status, abort)) goto mma_done;
          tc_fence_after();
          const uint32_t sfa_t = tmem + kSFCol0 + stage * kSFStageCols;
          const uint32_t sfb_t = sfa_t + 16;
          const uint32_t sa = smem_u32(sm.a[stage]), sb = smem_u32(sm.b[stage]);
          const uint32_t ssfa = smem_u32(sm.sfa[stage]), ssfb = smem_u32(sm.sfb[stage]);
          if constexpr (kBF) {
            // 64 BF16 values of K per 128-byte row: four K=16 steps of 32 bytes
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint64_t adesc = smem_desc(sa + 32 * j, 16, 1024, 2);
              const uint64_t bdesc = smem_desc(sb + 32 * j, 16, 1024, 2);
              tc_mma_f16(d_tmem, adesc, bdesc, idesc, (kb | j) != 0 ? 1u : 0u);
            }
          } else if constexpr (kMX) {
            tc_cp_32x128b_warpx4(sfa_t, smem_desc(ssfa, 0, 128, 0));
#pragma unroll
            for (int h = 0; h < kBN / 128; ++h) tc_cp_32x128b_warpx4(sfb_t + 4 * h, smem_desc(ssfb + 512 * h, 0, 128, 0));
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint64_t adesc = smem_desc(sa + 32 * j, 16, 1024, 2);
              const uint64_t bdesc = smem_desc(sb + 32 * j, 16, 1024, 2);
              tc_mma_mxf8(d_tmem, adesc, bdesc, idesc_mxf8(kBM, kBN, (uint32_t)j), sfa_t, sfb_t,
                          (kb | j) != 0 ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              tc_cp_32x128b_warpx4(sfa_t + 4 * j, smem_desc(ssfa + 512 * j, 0, 128, 0));
#pragma unroll
              for (int h = 0; h < kBN / 128; ++h)
                tc_cp_32x128b_warpx4(sfb_t + 4 * (kBN / 128) * j + 4 * h,
                                     smem_desc(ssfb + 2048 * h + 512 * j, 0, 128, 0));
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint64_t adesc = smem_desc(sa + 32 * j, 16, 1024, 2);
              const uint64_t bdesc = smem_desc(sb + 32 * j, 16, 1024, 2);
              tc_mma_nvf4(d_tmem, adesc, bdesc, idesc, sfa_t + 4 * j, sfb_t + 4 * (kBN / 128) * j,
                          (kb | j) != 0 ? 1u : 0u);
            }
          }
          tc_commit(&sm.empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        tc_commit(&sm.accf[acc]);
      }
    mma_done:;
    }
  } else {
    // epilogue: warps 2..5; TMEM lane quadrant = warp % 4.  Each warp owns 32 rows of the
    // tile.  When all 32 rows belong to the group, the rows are staged in a 128-byte
    // swizzled shared-memory box and written by a TMA store (full lines); otherwise the
    // valid rows are stored thread by thread, so rows outside the groups stay untouched.
    const int q = warp & 3;
    const int ew = warp - 2;
    const int elt = g.out_f32 ? 4 : 2;
    const int box_cols = 128 / elt;
    uint32_t cur = 0;
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      const uint32_t acc = it & 1, acc_phase = (it >> 1) & 1;
      const int m_tile = t / n_tiles, n_tile = t - (t / n_tiles) * n_tiles;
      const int32_t row0 = m_tile * kBM;
      const int e = find_group(sm.offsets, g.E, row0);
      const int32_t in_group = sm.rows[e] - (row0 - sm.offsets[e]);   // valid rows of this tile
      const bool valid = q * 32 + lane < in_group;
      const bool full_warp = q * 32 + 32 <= in_group;
      const int64_t row = (int64_t)row0 + q * 32 + lane;
      const float ga = kFmt != kGemmNVF4 ? 1.0f : (valid ? g.ga[row] : 0.0f);   // load before the wait
      if (!mbar_wait(&sm.accf[acc], acc_phase, g.status, abort)) break;
      tc_fence_after();
      const float scale = __fmul_rn(ga, sm.gb[e]);
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + acc * kAccCols;
      // the whole 128-column accumulator row in four loads, one wait, then hand the
      // accumulator back to the MMA warp before converting and storing
      uint32_t vall[kBN / 32][32];
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c) NVFP4_TMEM_LD_X32(taddr + 32 * c, vall[c]);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&sm.acce[acc]);
#pragma unroll
      for (int c0 = 0; c0 < kBN; c0 += 32) {
        const uint32_t (&v)[32] = vall[c0 / 32];
        const int64_t n0 = (int64_t)n_tile * kBN + c0;
        uint32_t w[32];
        int nw;
        if (g.out_f32) {
#pragma unroll
          for (int u = 0; u < 32; ++u) w[u] = __float_as_uint(__fmul_rn(__uint_as_float(v[u]), scale));
          nw = 32;
        } else {
#pragma unroll
          for (int u = 0; u < 16; ++u) {
            const __nv_bfloat162 b2 = __floats2bfloat162_rn(__fmul_rn(__uint_as_float(v[2 * u]), scale),
                                                            __fmul_rn(__uint_as_float(v[2 * u + 1]), scale));
            w[u] = *reinterpret_cast<const uint32_t*>(&b2);
          }
          nw = 16;
        }
        if (full_warp) {
          const int boff = (c0 * elt) & 127;        // byte offset of this chunk inside its box row
          if (boff == 0) {
            if (lane == 0) bulk_wait_read<1>();   // the group that last read this buffer is done
            __syncwarp();
          }
          uint8_t* buf = sm.out[ew][cur];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            if (u * 4 < nw) {
              const int j = (boff >> 4) + u;
              *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) =
                  make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
            }
          }
          if (boff + 32 * elt == 128) {   // box complete: hand it to the TMA engine
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmd, buf, (int32_t)(n0 + 32 - box_cols), row0 + q * 32);
              bulk_commit();
            }
            cur ^= 1u;
          }
        } else if (valid) {
          uint8_t* dp = static_cast<uint8_t*>(g.d) + (row * g.ldd + n0) * elt;
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (u * 4 < nw)
              *reinterpret_cast<uint4*>(dp + 16 * u) = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        }
      }
    }
    if (lane == 0) bulk_wait_all<0>();
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int kFmt>
static cudaError_t launch_gg(const CUtensorMap& tma, const CUtensorMap& tmb, const CUtensorMap& tmd,
                             const GemmArgs& g, int64_t max_m_tiles, cudaStream_t s) {
  static std::atomic<bool> attr_set[64];   // the attribute is set once per device
  cudaError_t err = set_smem_attr_once(attr_set, (const void*)grouped_gemm_kernel<kFmt>, (int)gg::kSmemBytes);
  if (err != cudaSuccess) return err;
  const int64_t tiles = max_m_tiles * (g.N / gg::kBN);
  if (tiles == 0) return cudaSuccess;
  int grid = num_sms();
  if (tiles < grid) grid = (int)tiles;
  grouped_gemm_kernel<kFmt><<<grid, gg::kThreads, gg::kSmemBytes, s>>>(tma, tmb, tmd, g);
  return cudaGetLastError();
}

cudaError_t launch_grouped_gemm(const CUtensorMap& tma, const CUtensorMap& tmb, const CUtensorMap& tmd,
                                const GemmArgs& g, int64_t max_m_tiles, cudaStream_t s) {
  return launch_gg<kGemmNVF4>(tma, tmb, tmd, g, max_m_tiles, s);
}

cudaError_t launch_grouped_gemm_mx(const CUtensorMap& tma, const CUtensorMap& tmb, const CUtensorMap& tmd,
                                   const GemmArgs& g, int64_t max_m_tiles, cudaStream_t s) {
  return launch_gg<kGemmMXF8>(tma, tmb, tmd, g, max_m_tiles, s);
}

cudaError_t launch_grouped_gemm_bf16(const CUtensorMap& tma, const CUtensorMap& tmb, const CUtensorMap& tmd,
                                     const GemmArgs& g, int64_t max_m_tiles, cudaStream_t s) {
  return launch_gg<kGemmBF16>(tma, tmb, tmd, g, max_m_tiles, s);
}

}  // namespace nvfp4

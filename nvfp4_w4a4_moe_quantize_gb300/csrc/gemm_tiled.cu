// W4A4 grouped GEMM over GEMM-tiled operands (see tiled.cuh), the kernel of the expert
// block's two projections ("Low-Bit Precision Training Is Ready for Production...",
// §"What W4A4 GEMM Actually Changes"; "miniTE identifies and closes the execution gap
// ...", §Development: grouped GEMMs):
//     D[r, n] = (gA[r] * gB[e]) * sum_k value(A)[r,k] sf_A[r,k/16] value(B_e)[n,k] sf_B[n,k/16]
//
// Measured on this GPU, a stage filled by many small asynchronous copies (2 KB scale
// blocks next to tensor-map boxes) ran far below one filled by a few large ones, and the
// main loop is bound by the bytes each SM keeps in flight.  In the tiled layout every
// 128-row x 256-K block of A (18 KB) and every 256-row x 256-K block of B (36 KB) is the
// exact shared-memory image of a stage -- swizzled codes followed by their scales -- so a
// stage is two bulk copies, issued by two producer warps in parallel, and three stages
// (162 KB) stay in flight.
//
// One CTA per SM:
//   warp 0 / 1  producers of the A / B block of each stage (cp.async.bulk + mbarrier);
//   warp 2      MMA issuer: four tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X
//               (M=128, N=256, K=64) per stage into a 256-column TMEM accumulator,
//               tcgen05.commit;
//   last 4      scale warps, one per TMEM lane quadrant: each reads the stage's twelve
//               512-byte scale blocks from shared memory and writes them into its 32 TMEM
//               lanes with tcgen05.st, in the image a tcgen05.cp.32x128b.warpx4 of the
//               block would leave (every quadrant holds the block's 32 x 16 bytes).  Done
//               by tcgen05.cp, the twelve copies share the tensor pipe with the four MMAs
//               and, measured on this GPU, stretch a stage from 512 to about 800 cycles;
//               tcgen05.st leaves the pipe to the MMAs;
//   warps 3..   epilogue (8 warps, two per TMEM lane quadrant, for the plain store; 16,
//               four per quadrant, for SwiGLU): drain the accumulator into registers,
//               release it, scale by gA[r]*gB[e] in float32 and write BF16 / float32 rows
//               of the group -- or, in the SwiGLU mode of the gate/up projection, form
//               h = BF16(silu(gate) * up) from the BF16-rounded gate and up columns and
//               write h only.  Each warp stages its 32-row box in a swizzled shared-memory
//               buffer and hands it to one TMA store: a thread-per-row register layout
//               stored directly would cost one 16-byte L2 request per row and chunk, and
//               paced the kernel when K is small.  The 32-row slab of a group's last,
//               partial tile is stored row by row, so rows outside the groups are never
//               written.
// Tiles are (128-row block) x (256 columns), row-block-major; no split-K, fixed K order.
#include <cstddef>
#include <cstdlib>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "group.cuh"
#include "launch.h"
#include "pdl.cuh"
#include "ptx.cuh"
#include "swiglu.cuh"
#include "tiled.cuh"

namespace nvfp4 {

namespace gt {
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kOutBytes = 32 * 1024;        // staged output boxes of all epilogue warps
constexpr int kABlock = 128 * 144;          // 16 KB codes + 2 KB scales
constexpr int kBBlock = 256 * 144;          // 32 KB codes + 4 KB scales
constexpr int kACodes = 128 * 128;
constexpr int kBCodes = 256 * 128;
constexpr int kBHalfCodes = 128 * 128;      // one CTA's half of a B block's codes (pair mode)
constexpr int kBScales = 256 * 16;
constexpr int kTmemCols = 512;
constexpr int kAccCols = kBN;
constexpr int kSFCol0 = kAccCols;
constexpr int kSFStageCols = 16 + 32;       // A: 4 x 4 columns, B: 4 x 8 columns
constexpr int kFirstEpiWarp = 3;
constexpr int kScaleWarps = 4;              // one per TMEM lane quadrant
// Epilogue warps: 8 for the plain store (two per TMEM lane quadrant, 128 columns each);
// 16 for the SwiGLU epilogue, whose per-value arithmetic needs the latency hiding of four
// warps per quadrant (each one 32-column gate slice and its up slice).
__host__ __device__ constexpr int epi_warps(bool swiglu) { return swiglu ? 16 : 8; }
__host__ __device__ constexpr int threads(bool swiglu, bool pair) {
  return 32 * (kFirstEpiWarp + epi_warps(swiglu) + kScaleWarps) + 0 * pair;
}
constexpr int kMaxE = 512;

// One pipeline stage in shared memory.  One SM per tile (kPair false): the A block
// (codes, then scales) at 0 and the whole B block (codes, then scales) after it.  CTA
// pair: this CTA's half of B's codes at 0, the A block at 16 KB (its scales at 32 KB) and
// all of B's scales (both halves' rows, which each SM's MMA reads) at 34 KB.
template <bool kPair>
struct Layout {
  static constexpr int kStages = kPair ? 4 : 3;
  static constexpr int kStageBytes = kPair ? kBHalfCodes + kABlock + kBScales : kABlock + kBBlock;
  static constexpr int kA = kPair ? kBHalfCodes : 0;
  static constexpr int kB = kPair ? 0 : kABlock;
  static constexpr int kSFA = kA + kACodes;
  static constexpr int kSFB = kPair ? kBHalfCodes + kABlock : kABlock + kBCodes;
};

template <bool kPair>
struct Smem {
  uint8_t stage[Layout<kPair>::kStages][Layout<kPair>::kStageBytes];
  uint8_t out[kOutBytes];     // TMA store boxes: 1024-byte aligned (128-byte swizzle), as the stages
  uint64_t full[Layout<kPair>::kStages];
  uint64_t empty[Layout<kPair>::kStages];
  uint64_t sfull[Layout<kPair>::kStages];     // the stage's scale bytes have landed
  uint64_t sfready[Layout<kPair>::kStages];   // the stage's scales are in TMEM (pair: in both CTAs')
  uint64_t accf;
  uint64_t acce;
  uint64_t fin;               // the MMA issuer's last operations have completed
  uint32_t tmem_base;
  int abort;
  int32_t offsets[kMaxE + 1];
  int32_t rows[kMaxE];
  float gb[kMaxE];
  int32_t pairs[kMaxE + 1];   // CTA pair: row-block pairs before group e
};
static_assert(kABlock % 1024 == 0 && kBBlock % 1024 == 0 && kBHalfCodes % 1024 == 0, "1024-byte aligned images");
static_assert(Layout<false>::kStageBytes % 1024 == 0 && Layout<true>::kStageBytes % 1024 == 0, "stage alignment");
static_assert(kSFCol0 + Layout<false>::kStages * kSFStageCols <= kTmemCols, "TMEM budget");
static_assert(kSFCol0 + Layout<true>::kStages * kSFStageCols <= kTmemCols, "TMEM budget");
static_assert(sizeof(Smem<false>) + 1024 <= 232448 && sizeof(Smem<true>) + 1024 <= 232448, "shared memory budget");
static_assert(offsetof(Smem<false>, out) % 1024 == 0 && offsetof(Smem<true>, out) % 1024 == 0,
              "TMA store boxes 1024-byte aligned");
template <bool kPair>
constexpr size_t smem_bytes() { return sizeof(Smem<kPair>) + 1024; }
}  // namespace gt

// BF16 pair (a s in the low half, b s in the high half) of two accumulator values scaled
// by s: both IEEE products by one paired multiply, both roundings by one paired
// conversion (round to nearest even) -- the same bits as two multiplies and a
// __floats2bfloat162_rn.
__device__ __forceinline__ uint32_t bf16x2_scaled(uint32_t a, uint32_t b, float s) {
  float pa, pb;
  asm("{\n .reg .b64 x, y, d;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %4};\n"
      " mul.rn.f32x2 d, x, y;\n mov.b64 {%0, %1}, d;\n}"
      : "=f"(pa), "=f"(pb)
      : "r"(a), "r"(b), "f"(s));
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(pb), "f"(pa));
  return r;
}

// One lane's 128-byte row of a warp's 32-row output box, written 128-byte swizzled (16-byte
// chunk j at (j ^ (row % 8)) * 16, the TMA SWIZZLE_128B image), then one TMA store of the
// box at column x, row y.  The buffer is reused only after the previous store read it.
__device__ __forceinline__ void store_box(uint8_t* buf, const uint32_t (&w)[32], int lane,
                                          const CUtensorMap* map, int32_t x, int32_t y) {
  if (lane == 0) bulk_wait_read<0>();
  __syncwarp();
#pragma unroll
  for (int j = 0; j < 8; ++j)
    *reinterpret_cast<uint4*>(buf + lane * 128 + ((j ^ (lane & 7)) << 4)) =
        make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, buf, x, y);
    bulk_commit();
  }
}

// What one tile reads and writes.  Grouped rows (kRagged false): tile t is row block
// t / n_tiles of the padded group layout and column block t % n_tiles; its expert is the
// group holding the row block; K = g.K.  Ragged K (kRagged true, the weight gradients):
// expert e = t / (m_tiles * n_tiles) owns g.m_rows rows of A and of D and its own
// contraction of 256 * kb_e values (kb_e = kofs[e+1] - kofs[e]); A's blocks of expert e
// start at block (m_rows / 128) * kofs[e], B's at (N / 256) * kofs[e], each row block's
// kb_e K-blocks consecutive.
struct TileJob {
  const uint8_t* a;    // first K-block of A
  const uint8_t* b;    // first K-block of B
  int kblocks;
  int e, n_tile;
  int32_t row0;        // first output row
  int32_t in_group;    // valid rows of the tile (>= 128: all; <= 0: none)
  bool has_a;          // false: the pair's second row block lies past its group (no A load)
};

template <bool kRagged>
__device__ __forceinline__ TileJob tile_job(const GemmArgs& g, const int32_t* offsets, const int32_t* rows,
                                            const uint8_t* A, const uint8_t* B, int t, int n_tiles, int m_tiles,
                                            int kblocks) {
  TileJob j;
  if (kRagged) {
    const int per_e = m_tiles * n_tiles;
    j.e = t / per_e;
    const int rem = t - j.e * per_e;
    const int m_tile = rem / n_tiles;
    j.n_tile = rem - m_tile * n_tiles;
    const int32_t k0 = offsets[j.e];
    j.kblocks = offsets[j.e + 1] - k0;
    j.a = A + ((int64_t)m_tiles * k0 + (int64_t)m_tile * j.kblocks) * gt::kABlock;
    j.b = B + ((int64_t)n_tiles * k0 + (int64_t)j.n_tile * j.kblocks) * gt::kBBlock;
    j.row0 = j.e * g.m_rows + m_tile * gt::kBM;
    j.in_group = gt::kBM;
  } else {
    const int m_tile = t / n_tiles;
    j.n_tile = t - m_tile * n_tiles;
    j.row0 = m_tile * gt::kBM;
    j.e = find_group(offsets, g.E, j.row0);
    j.kblocks = kblocks;
    j.a = A + (int64_t)m_tile * kblocks * gt::kABlock;
    j.b = B + ((int64_t)j.e * n_tiles + j.n_tile) * kblocks * gt::kBBlock;
    j.in_group = rows[j.e] - (j.row0 - offsets[j.e]);
  }
  j.has_a = true;
  return j;
}

// CTA pair: unit p of a group is the pair of row blocks (2 jj, 2 jj + 1) of the group
// (jj = p - pairs[e]), CTA `rank` of the pair taking block 2 jj + rank; a group with an odd
// number of row blocks leaves its last pair's second block empty (that CTA loads no A and
// stores nothing; its half of the MMA is discarded).  Both row blocks are one expert's, so
// the pair shares B's column tile.
__device__ __forceinline__ TileJob tile_job_pair(const GemmArgs& g, const int32_t* offsets, const int32_t* rows,
                                                 const int32_t* pairs, const uint8_t* A, const uint8_t* B, int t,
                                                 int n_tiles, int kblocks, uint32_t rank) {
  TileJob j;
  const int p = t / n_tiles;
  j.n_tile = t - p * n_tiles;
  j.e = find_group(pairs, g.E, p);
  const int32_t blocks_e = (offsets[j.e + 1] - offsets[j.e]) / gt::kBM;
  const int32_t jb = 2 * (p - pairs[j.e]) + (int32_t)rank;   // row block within the group
  j.has_a = jb < blocks_e;
  j.row0 = offsets[j.e] + jb * gt::kBM;
  j.kblocks = kblocks;
  j.a = A + (int64_t)(j.row0 / gt::kBM) * kblocks * gt::kABlock;
  j.b = B + ((int64_t)j.e * n_tiles + j.n_tile) * kblocks * gt::kBBlock;
  j.in_group = j.has_a ? rows[j.e] - (j.row0 - offsets[j.e]) : 0;
  return j;
}

// kMode: 0 plain store, 1 SwiGLU epilogue, 2 plain store with ragged K per expert.
// kPair: a cluster of two CTAs on two SMs shares each M=256 x N=256 tile (cta_group::2):
// CTA 0 issues the MMAs; each CTA loads its own A block, its half of B's codes and all of
// B's scales into its own shared memory (no shared loads), and its scale warps write its
// own TMEM; CTA 1's warp 2 tells CTA 0 when a stage of CTA 1 is full and its scales are in
// CTA 1's TMEM; CTA 0's commits free the stages and fill the accumulators of both; both
// CTAs' epilogues release the accumulator to CTA 0.
template <int kMode, bool kPair>
__global__ void __launch_bounds__(gt::threads(kMode == 1, kPair), 1)
    grouped_gemm_tiled_kernel(const uint8_t* __restrict__ A, const uint8_t* __restrict__ B,
                              const __grid_constant__ CUtensorMap tmd, const GemmArgs g) {
  grid_dep_sync();
  using namespace gt;
  using L = Layout<kPair>;
  constexpr int kStages = L::kStages;
  constexpr bool kSwiGLU = kMode == 1, kRagged = kMode == 2;
  static_assert(!(kPair && kRagged), "the CTA pair runs the grouped-row modes");
  constexpr int kEpiWarps = epi_warps(kSwiGLU);
  extern __shared__ uint8_t smem_raw[];
  Smem<kPair>& sm = *reinterpret_cast<Smem<kPair>*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;

  for (int i = threadIdx.x; i <= g.E; i += blockDim.x) sm.offsets[i] = g.offsets[i];
  for (int i = threadIdx.x; i < g.E; i += blockDim.x) {
    sm.rows[i] = kRagged ? 0 : g.rows[i];
    sm.gb[i] = g.gb[i];
  }
  __syncthreads();
  // nothing is read or written unless the group arrays are consistent (ragged K: g.offsets
  // are the K-block prefix sums, every expert at least one block, at most g.m_total blocks);
  // both CTAs of a pair read the same arrays and leave together, before any cluster step
  if (kRagged ? !kblocks_valid(sm.offsets, g.E, g.m_total) : !groups_valid(sm.offsets, sm.rows, g.E, g.m_total)) {
    if (threadIdx.x == 0) set_status(g.status, kStatusBadInput);
    return;
  }
  if (threadIdx.x == 0) {
    if (kPair) {
      sm.pairs[0] = 0;
      for (int e = 0; e < g.E; ++e)
        sm.pairs[e + 1] = sm.pairs[e] + ((sm.offsets[e + 1] - sm.offsets[e]) / kBM + 1) / 2;
    }
    for (int s = 0; s < kStages; ++s) {
      // the A and the B producer arrive; in a pair CTA 0 also hears from CTA 1's warp 2
      mbar_init(&sm.full[s], kPair && rank == 0 ? 3 : 2);
      mbar_init(&sm.empty[s], 1);
      mbar_init(&sm.sfull[s], 2);
      mbar_init(&sm.sfready[s], kScaleWarps);
    }
    mbar_init(&sm.accf, 1);
    mbar_init(&sm.fin, 1);
    // one arrival per epilogue warp (pair: of either CTA, on CTA 0's barrier)
    mbar_init(&sm.acce, kPair ? 2 * kEpiWarps : kEpiWarps);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 2) {
    if (kPair) {
      tmem_alloc_pair(&sm.tmem_base, kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&sm.tmem_base, kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync();   // both CTAs' barriers exist before any remote arrival
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  volatile int* abort = &sm.abort;
  auto wait = [&](uint64_t* bar, uint32_t parity) {
    return kPair ? mbar_wait_cluster(bar, parity, g.status, abort) : mbar_wait(bar, parity, g.status, abort);
  };

  const int n_tiles = g.N / kBN;
  const int m_tiles = kRagged ? g.m_rows / kBM : sm.offsets[g.E] / kBM;   // ragged: per expert
  const int total = kRagged ? g.E * m_tiles * n_tiles : (kPair ? sm.pairs[g.E] : m_tiles) * n_tiles;
  const int kblocks = g.K / 256;
  const int first = kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int stride = kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  auto job_of = [&](int t) {
    return kPair ? tile_job_pair(g, sm.offsets, sm.rows, sm.pairs, A, B, t, n_tiles, kblocks, rank)
                 : tile_job<kRagged>(g, sm.offsets, sm.rows, A, B, t, n_tiles, m_tiles, kblocks);
  };

  if (warp < 2) {
    if (lane == 0) {
      const bool is_a = warp == 0;
      uint32_t stage = 0, phase = 0;
      for (int t = first; t < total; t += stride) {
        const TileJob job = job_of(t);
        for (int kb = 0; kb < job.kblocks; ++kb) {
          if (!wait(&sm.empty[stage], phase ^ 1u)) goto producer_done;
          uint8_t* st = sm.stage[stage];
          if (!kPair) {
            // the scale bytes first, on their own barrier: the scale warps move them into
            // TMEM while the codes are still arriving
            const uint8_t* src = is_a ? job.a + (int64_t)kb * kABlock : job.b + (int64_t)kb * kBBlock;
            const uint32_t codes = is_a ? kACodes : kBCodes, scales = is_a ? kABlock - kACodes : kBScales;
            uint8_t* dst = st + (is_a ? L::kA : L::kB);
            mbar_arrive_expect_tx(&sm.sfull[stage], scales);
            bulk_load(dst + codes, src + codes, scales, &sm.sfull[stage]);
            mbar_arrive_expect_tx(&sm.full[stage], codes);
            bulk_load(dst, src, codes, &sm.full[stage]);
          } else if (is_a) {
            // pair: this CTA's A block (scales first, on the scale barrier), or nothing
            // for the empty half of a group's last pair
            if (job.has_a) {
              const uint8_t* src = job.a + (int64_t)kb * kABlock;
              mbar_arrive_expect_tx(&sm.sfull[stage], kABlock - kACodes);
              bulk_load(st + L::kSFA, src + kACodes, kABlock - kACodes, &sm.sfull[stage]);
              mbar_arrive_expect_tx(&sm.full[stage], kACodes);
              bulk_load(st + L::kA, src, kACodes, &sm.full[stage]);
            } else {
              mbar_arrive(&sm.sfull[stage]);
              mbar_arrive(&sm.full[stage]);
            }
          } else {
            // pair: all of B's scales (each SM's MMA reads them all), then this CTA's half
            // of B's codes
            const uint8_t* src = job.b + (int64_t)kb * kBBlock;
            mbar_arrive_expect_tx(&sm.sfull[stage], kBScales);
            bulk_load(st + L::kSFB, src + kBCodes, kBScales, &sm.sfull[stage]);
            mbar_arrive_expect_tx(&sm.full[stage], kBHalfCodes);
            bulk_load(st + L::kB, src + rank * kBHalfCodes, kBHalfCodes, &sm.full[stage]);
          }
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    producer_done:;
    }
  } else if (warp == 2) {
    if (rank == 0) {
      // The whole warp runs the loop (its waits, descriptors and TMEM addresses are
      // warp-uniform values); lane 0 issues the tcgen05 operations.  Measured: one lane
      // alone running it spent about 300 cycles a stage on its scalar work, sharing the
      // issue slots of its SM sub-partition with five busy warps.
      constexpr uint32_t idesc = idesc_nvf4(kPair ? 2 * kBM : kBM, kBN);
      // operand descriptors of stage 0; stage s and K-step j add (s * stage bytes + 32 j) / 16
      // to the start-address field (every address stays below 2^18, so no carry leaves it)
      const uint32_t st0 = smem_u32(sm.stage[0]);
      const uint64_t adesc0 = smem_desc(st0 + L::kA, 16, 1024, 2), bdesc0 = smem_desc(st0 + L::kB, 16, 1024, 2);
      constexpr uint32_t kStageDesc = L::kStageBytes >> 4;
      const bool leader = lane == 0;
      uint32_t stage = 0, phase = 0;
      int it = 0;
      for (int t = first; t < total; t += stride, ++it) {
        const int kbt = kRagged ? tile_job<true>(g, sm.offsets, sm.rows, A, B, t, n_tiles, m_tiles, kblocks).kblocks
                                : kblocks;
        for (int kb = 0; kb < kbt; ++kb) {
          bool ok = wait(&sm.full[stage], phase);
          ok = ok && wait(&sm.sfready[stage], phase);
          if (!__all_sync(0xFFFFFFFFu, ok)) goto mma_done;
          tc_fence_after();
          const uint32_t sfa_t = tmem + kSFCol0 + stage * kSFStageCols;
          const uint32_t sfb_t = sfa_t + 16;
          const uint64_t adesc = adesc0 + stage * kStageDesc, bdesc = bdesc0 + stage * kStageDesc;
          if (kb == 0) {
            if (!__all_sync(0xFFFFFFFFu, wait(&sm.acce, (it & 1) ^ 1u))) goto mma_done;
            tc_fence_after();
          }
          if (leader) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (kPair)
                tc_mma_nvf4_pair(tmem, adesc + 2 * j, bdesc + 2 * j, idesc, sfa_t + 4 * j, sfb_t + 8 * j,
                                 (kb | j) != 0 ? 1u : 0u);
              else
                tc_mma_nvf4(tmem, adesc + 2 * j, bdesc + 2 * j, idesc, sfa_t + 4 * j, sfb_t + 8 * j,
                            (kb | j) != 0 ? 1u : 0u);
            }
            if (kPair) {
              tc_commit_pair(cluster_addr(&sm.empty[stage], 0));
              tc_commit_pair(cluster_addr(&sm.empty[stage], 1));
            } else {
              tc_commit(&sm.empty[stage]);
            }
          }
          __syncwarp();
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (leader) {
          if (kPair) {
            tc_commit_pair(cluster_addr(&sm.accf, 0));
            tc_commit_pair(cluster_addr(&sm.accf, 1));
          } else {
            tc_commit(&sm.accf);
          }
        }
        __syncwarp();
      }
    mma_done:
      // whatever the exit, no MMA or scale copy of the issuing lane is still running when
      // the TMEM is freed (a bounded wait of its own, also after an abort)
      if (leader) {
        if (kPair) tc_commit_pair(cluster_addr(&sm.fin, 0));
        else tc_commit(&sm.fin);
        volatile int no_abort = 0;
        mbar_wait(&sm.fin, 0, g.status, &no_abort, 1000000000ull);
      }
      __syncwarp();
    } else if (kPair && lane == 0) {
      // CTA 1: each stage of this CTA that is full and whose scales are in its TMEM counts
      // as one arrival on CTA 0's full barrier (one cluster-scope arrival per stage: as
      // four, one per scale warp, they stretched a stage to ~1500 cycles)
      uint32_t stage = 0, phase = 0;
      const uint32_t full0 = cluster_addr(&sm.full[0], 0);
      for (int t = first; t < total; t += stride) {
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!wait(&sm.full[stage], phase) || !wait(&sm.sfready[stage], phase)) goto relay_done;
          mbar_arrive_cluster(full0 + stage * (uint32_t)sizeof(uint64_t));
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
    relay_done:;
    }
  } else if (warp >= kFirstEpiWarp + kEpiWarps) {
    // scale warps: the stage's A scales (four 512-byte blocks, one per MMA) go to columns
    // [0, 16) of the stage's scale slot, B's (two blocks per MMA: rows 0-127, then
    // 128-255) to [16, 48), block j at 4j / 16 + 8j (+4), each as 32 lanes x 16 bytes in
    // every lane quadrant.  A stage's slot is rewritten only after its scale barrier has
    // completed again, i.e. after the MMAs that read the previous contents (their commit
    // freed the stage before it was refilled).
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    uint32_t stage = 0, phase = 0;
    for (int t = first; t < total; t += stride) {
      const int kbt = kRagged ? tile_job<true>(g, sm.offsets, sm.rows, A, B, t, n_tiles, m_tiles, kblocks).kblocks
                              : kblocks;
      for (int kb = 0; kb < kbt; ++kb) {
        const bool ok = wait(&sm.sfull[stage], phase);
        if (!__all_sync(0xFFFFFFFFu, ok)) goto sf_done;
        const uint4* sfa = reinterpret_cast<const uint4*>(sm.stage[stage] + L::kSFA) + lane;
        const uint4* sfb = reinterpret_cast<const uint4*>(sm.stage[stage] + L::kSFB) + lane;
        uint32_t ra[16], rb[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 a = sfa[32 * j], b0 = sfb[32 * j], b1 = sfb[128 + 32 * j];
          ra[4 * j] = a.x, ra[4 * j + 1] = a.y, ra[4 * j + 2] = a.z, ra[4 * j + 3] = a.w;
          rb[8 * j] = b0.x, rb[8 * j + 1] = b0.y, rb[8 * j + 2] = b0.z, rb[8 * j + 3] = b0.w;
          rb[8 * j + 4] = b1.x, rb[8 * j + 5] = b1.y, rb[8 * j + 6] = b1.z, rb[8 * j + 7] = b1.w;
        }
        const uint32_t taddr = tmem + lane_base + kSFCol0 + stage * kSFStageCols;
        tmem_st_32x32b_x16(taddr, ra);
        tmem_st_32x32b_x32(taddr + 16, rb);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.sfready[stage]);   // (pair, CTA 1: relayed to CTA 0 by warp 2)
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  sf_done:;
  } else {
    // epilogue: TMEM lane quadrant q = warp % 4 (the lanes this warp may read), column
    // half of the tile = (warp - 3) / 4
    const int q = warp & 3;
    const int ew = warp - kFirstEpiWarp;
    const int half = kSwiGLU ? ew >> 3 : ew >> 2;        // 128-column half of the tile
    const int sub = kSwiGLU ? (ew >> 2) & 1 : 0;         // SwiGLU: 32-column slice of the half
    uint8_t* buf = sm.out + ew * (kOutBytes / kEpiWarps);
    const ff* silu_tab = static_cast<const ff*>(g.silu_tab);
    // SwiGLU: the values of a tile that the float32 path could not settle (one in about
    // 2000) are recorded during that pass -- the first two per lane in registers, any
    // further ones in a small per-lane array -- and evaluated exactly after the next tile's
    // accumulator has been drained and released, off the path accumulator -> drain ->
    // next MMA.  The fix-up is stored once the box holding the value has been written,
    // and joins the row max.
    uint32_t d_x2a = 0, d_x2b = 0, d_mask = 0;   // d_mask: columns (bits) still to settle
    int d_n = 0;
    uint32_t d_ovf[30];
    __nv_bfloat16* d_hp = nullptr;
    int64_t d_row = 0;
    auto flush_deferred = [&]() {
      if (!__any_sync(0xFFFFFFFFu, d_n != 0)) return;
      if (lane == 0) bulk_wait_all<0>();   // this warp's boxes have reached global memory
      fence_proxy_async_global();
      __syncwarp();
      for (int k = 0; __any_sync(0xFFFFFFFFu, d_n > k); ++k) {
        const bool has = d_n > k;
        uint32_t x2 = 0x3F803F80u;         // lanes with nothing left evaluate gate = up = 1
        if (has) x2 = k == 0 ? d_x2a : (k == 1 ? d_x2b : d_ovf[k - 2]);
        const uint32_t hb = swiglu_exact(silu_tab, __uint_as_float(x2 << 16), __uint_as_float(x2 & 0xFFFF0000u));
        if (has) {
          const int j = __ffs((int)d_mask) - 1;   // recorded in increasing column order
          d_mask &= d_mask - 1;
          *reinterpret_cast<uint16_t*>(d_hp + j) = (uint16_t)hb;
          const uint32_t mag = hb & 0x7FFFu;
          if (g.h_amax != nullptr && mag != 0u && mag <= 0x7F80u) atomicMax(g.h_amax + d_row, mag << 16);
        }
      }
      d_n = 0;
      d_mask = 0;
    };
    // the accumulator is drained: one lane per warp arrives (after the warp's loads have
    // completed) on its CTA's barrier, or, in a pair, on CTA 0's
    const uint32_t acce0 = kPair ? cluster_addr(&sm.acce, 0) : 0u;
    auto release_acc = [&]() {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (kPair) mbar_arrive_cluster(acce0);
        else mbar_arrive(&sm.acce);
      }
    };
    bool aborted = false;
    int it = 0;
    for (int t = first; t < total; t += stride, ++it) {
      const TileJob job = job_of(t);
      const int n_tile = job.n_tile, e = job.e;
      const int32_t row0 = job.row0, in_group = job.in_group;
      const bool valid = q * 32 + lane < in_group;
      const bool full_warp = q * 32 + 32 <= in_group;             // warp-uniform
      const int64_t row = (int64_t)row0 + q * 32 + lane;
      const float ga = kRagged ? g.ga[e] : (valid ? g.ga[row] : 0.0f);   // ragged: one scale per expert
      // every lane waits (bounded), then the warp leaves together if any lane gave up
      const bool acc_ready = wait(&sm.accf, it & 1);
      if (!__all_sync(0xFFFFFFFFu, acc_ready)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      const float scale = __fmul_rn(ga, sm.gb[e]);
      const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + half * 128;
      // Skip only warp-uniformly: every lane of a partial slab computes (whatever the
      // rows past the group hold, the arithmetic below ends), so the warp-wide votes and
      // syncs see all 32 lanes; only the row-by-row stores of a partial slab depend on
      // the lane.
      const bool skip = q * 32 >= in_group;
      const int32_t y = row0 + q * 32;
      if (kSwiGLU) {
        // Columns [0, 64) of this half are gate, [64, 128) up (64-row gate/up interleave
        // of W13); this warp takes gate columns sub*32 + [0, 32) and the matching up
        // columns, i.e. h columns n_tile*128 + half*64 + sub*32 + [0, 32).  All 32 values
        // take the branch-free float32 path first (independent chains the compiler can
        // interleave); the rare values it cannot settle are recorded for the next tile.
        // gu: BF16 gate | BF16 up << 16, one rounding instruction per pair.  The slice
        // comes out of TMEM in two halves of 16 columns, each packed before the next is
        // loaded, so that at most 48 of the accumulator's registers are live at once.
        uint32_t gu[32];
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t vg[16], vu[16];
          NVFP4_TMEM_LD_X16(taddr + 32 * sub + 16 * hh, vg);
          NVFP4_TMEM_LD_X16(taddr + 64 + 32 * sub + 16 * hh, vu);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const __nv_bfloat162 pr = __floats2bfloat162_rn(__fmul_rn(__uint_as_float(vg[i]), scale),
                                                            __fmul_rn(__uint_as_float(vu[i]), scale));
            gu[16 * hh + i] = *reinterpret_cast<const uint32_t*>(&pr);
          }
        }
        release_acc();
        flush_deferred();   // the previous tile's leftovers (its box is written by now)
        if (skip) continue;
        const int32_t x = n_tile * 128 + half * 64 + sub * 32;
        d_hp = g.h + row * g.I + x;
        d_row = row;
        uint32_t w[16];
#pragma unroll
        for (int p = 0; p < 16; ++p) {
          float hf[2];
#pragma unroll
          for (int s2 = 0; s2 < 2; ++s2) {
            const uint32_t x2 = gu[2 * p + s2];
            bool ok;
            hf[s2] = swiglu_fast_f32(__uint_as_float(x2 << 16), __uint_as_float(x2 & 0xFFFF0000u), ok);
            if (!ok && valid) {
              if (d_n == 0) d_x2a = x2;
              else if (d_n == 1) d_x2b = x2;
              else d_ovf[d_n - 2] = x2;
              ++d_n;
              d_mask |= 1u << (2 * p + s2);
            }
          }
          const __nv_bfloat162 hp = __floats2bfloat162_rn(hf[0], hf[1]);
          w[p] = *reinterpret_cast<const uint32_t*>(&hp);
        }
        if (full_warp) {
          // 32 rows x 64 bytes, 64-byte swizzled (16-byte chunk j of row r at
          // (j ^ ((r >> 1) & 3)) * 16, the TMA SWIZZLE_64B image), one TMA store
          if (lane == 0) bulk_wait_read<0>();   // the previous box has been read
          __syncwarp();
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(buf + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
                make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmd, buf, x, y);
            bulk_commit();
          }
        } else if (valid) {
          __nv_bfloat16* hp = g.h + row * g.I + x;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(hp + 8 * j) = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
        }
        if (g.h_amax != nullptr && valid) {
          // max |h| of the row's 32 values as BF16 magnitude bits (integers order like
          // the magnitudes; NaN patterns are ignored, as a float max would)
          // (deferred values join the max when they are settled)
          uint32_t m2 = 0;
#pragma unroll
          for (int j = 0; j < 16; ++j) m2 = __vmaxu2(m2, w[j] & 0x7FFF7FFFu);   // both halves at once
          uint32_t hmax = max(m2 & 0xFFFFu, m2 >> 16);
          if (d_mask != 0u || hmax > 0x7F80u) {
            // values still to be settled (they join when they are) or NaN patterns: the
            // element-wise max without them
            hmax = 0;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const uint32_t lo = (d_mask >> (2 * j)) & 1u ? 0u : w[j] & 0x7FFFu;
              const uint32_t hi = (d_mask >> (2 * j + 1)) & 1u ? 0u : (w[j] >> 16) & 0x7FFFu;
              hmax = max(hmax, max(lo <= 0x7F80u ? lo : 0u, hi <= 0x7F80u ? hi : 0u));
            }
          }
          if (hmax != 0u) atomicMax(g.h_amax + row, hmax << 16);
        }
      } else if (!g.out_f32) {
        // BF16: each pair of 32-column chunks is packed as soon as it is loaded (one paired
        // multiply and one paired conversion per column pair), so at most 64 accumulator
        // values are live next to the 64 packed words
        uint32_t w[2][32];
#pragma unroll
        for (int b2 = 0; b2 < 2; ++b2) {
          uint32_t v[2][32];
          NVFP4_TMEM_LD_X32(taddr + 64 * b2, v[0]);
          NVFP4_TMEM_LD_X32(taddr + 64 * b2 + 32, v[1]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int p = 0; p < 16; ++p) w[b2][16 * c + p] = bf16x2_scaled(v[c][2 * p], v[c][2 * p + 1], scale);
          }
        }
        release_acc();
        if (skip) continue;
#pragma unroll
        for (int b2 = 0; b2 < 2; ++b2) {
          const int32_t x = n_tile * kBN + half * 128 + 64 * b2;
          if (full_warp) {
            store_box(buf, w[b2], lane, &tmd, x, y);
          } else if (valid) {
            uint8_t* dp = static_cast<uint8_t*>(g.d) + (row * g.ldd + x) * 2;
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(dp + 16 * j) =
                  make_uint4(w[b2][4 * j], w[b2][4 * j + 1], w[b2][4 * j + 2], w[b2][4 * j + 3]);
          }
        }
      } else {
        // float32: the half's first 64 columns are stored before the last 64 are loaded,
        // so at most 64 accumulator values are live; the accumulator is released once the
        // last load has completed
#pragma unroll
        for (int b2 = 0; b2 < 2; ++b2) {
          uint32_t v[2][32];
          NVFP4_TMEM_LD_X32(taddr + 64 * b2, v[0]);
          NVFP4_TMEM_LD_X32(taddr + 64 * b2 + 32, v[1]);
          tmem_ld_wait();
          if (b2 == 1) release_acc();
          if (skip) continue;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[c][i] = __float_as_uint(__fmul_rn(__uint_as_float(v[c][i]), scale));
            const int32_t x = n_tile * kBN + half * 128 + 64 * b2 + 32 * c;
            if (full_warp) {
              store_box(buf, v[c], lane, &tmd, x, y);
            } else if (valid) {
              uint8_t* dp = static_cast<uint8_t*>(g.d) + (row * g.ldd + x) * 4;
#pragma unroll
              for (int j = 0; j < 8; ++j)
                *reinterpret_cast<uint4*>(dp + 16 * j) =
                    make_uint4(v[c][4 * j], v[c][4 * j + 1], v[c][4 * j + 2], v[c][4 * j + 3]);
            }
          }
        }
      }
    }
    if (kSwiGLU && !aborted) flush_deferred();
    if (lane == 0) bulk_wait_all<0>();   // the last boxes are read before the CTA exits
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (kPair) cluster_sync();   // no remote arrival or peer read is left in flight
  tc_fence_after();
  if (warp == 2) {
    if (kPair) tmem_dealloc_pair(tmem, kTmemCols);
    else tmem_dealloc(tmem, kTmemCols);
  }
}

template <int kMode>
static cudaError_t launch_tiled(const uint8_t* A, const uint8_t* B, const CUtensorMap& tmd, const GemmArgs& g,
                                int64_t tiles, cudaStream_t s, bool pdl = false) {
  if (kMode == 1 && g.silu_tab == nullptr) return cudaErrorInvalidValue;
  static std::atomic<bool> attr_set[64];   // the attribute is set once per device
  cudaError_t err = set_smem_attr_once(attr_set, (const void*)grouped_gemm_tiled_kernel<kMode, false>,
                                       (int)gt::smem_bytes<false>());
  if (err != cudaSuccess) return err;
  if (tiles == 0) return cudaSuccess;
  int grid = num_sms();
  if (tiles < grid) grid = (int)tiles;
  return launch_pdl(pdl, grouped_gemm_tiled_kernel<kMode, false>, dim3((unsigned)grid), dim3(gt::threads(kMode == 1, false)),
                    gt::smem_bytes<false>(), s, A, B, tmd, g);
}

// CTA-pair launch: clusters of two CTAs, as many clusters as fit on the device at once
// (one CTA per SM), each looping over pair tiles.  `tiles` bounds the pair tiles.
template <int kMode>
static cudaError_t launch_pair(const uint8_t* A, const uint8_t* B, const CUtensorMap& tmd, const GemmArgs& g,
                               int64_t tiles, cudaStream_t s) {
  if (kMode == 1 && g.silu_tab == nullptr) return cudaErrorInvalidValue;
  const void* fn = (const void*)grouped_gemm_tiled_kernel<kMode, true>;
  static std::atomic<bool> attr_set[64];
  cudaError_t err = set_smem_attr_once(attr_set, fn, (int)gt::smem_bytes<true>());
  if (err != cudaSuccess) return err;
  if (tiles == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(gt::threads(kMode == 1, true), 1, 1);
  cfg.dynamicSmemBytes = gt::smem_bytes<true>();
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static std::atomic<int> resident[64];   // clusters resident at once, per device (0: not known yet)
  int dev = 0;
  cudaGetDevice(&dev);
  int clusters = (dev >= 0 && dev < 64) ? resident[dev].load(std::memory_order_acquire) : 0;
  if (clusters <= 0) {
    cfg.gridDim = dim3(2 * (num_sms() / 2), 1, 1);
    err = cudaOccupancyMaxActiveClusters(&clusters, fn, &cfg);
    if (err != cudaSuccess) return err;
    if (clusters <= 0) return cudaErrorInvalidConfiguration;
    if (dev >= 0 && dev < 64) resident[dev].store(clusters, std::memory_order_release);
  }
  if (tiles < clusters) clusters = (int)tiles;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  return cudaLaunchKernelEx(&cfg, grouped_gemm_tiled_kernel<kMode, true>, A, B, tmd, g);
}

// The CTA-pair kernel runs the grouped-row modes when NVFP4_GEMM_CTA_PAIR=1 (measured
// slower than one CTA per tile on the forward's shapes, so not the default).
static bool pair_enabled() {
  const char* v = std::getenv("NVFP4_GEMM_CTA_PAIR");
  return v != nullptr && v[0] == '1';
}

cudaError_t launch_grouped_gemm_tiled(const uint8_t* A, const uint8_t* B, const CUtensorMap& tmd, const GemmArgs& g,
                                      int64_t max_m_tiles, bool swiglu, cudaStream_t s, bool pdl) {
  const int64_t tiles = max_m_tiles * (g.N / gt::kBN);
  if (pair_enabled())
    return swiglu ? launch_pair<1>(A, B, tmd, g, tiles, s) : launch_pair<0>(A, B, tmd, g, tiles, s);
  return swiglu ? launch_tiled<1>(A, B, tmd, g, tiles, s, pdl) : launch_tiled<0>(A, B, tmd, g, tiles, s, pdl);
}

cudaError_t launch_grouped_gemm_ragged_k(const uint8_t* A, const uint8_t* B, const CUtensorMap& tmd,
                                         const GemmArgs& g, cudaStream_t s) {
  if (g.m_rows <= 0 || g.m_rows % gt::kBM != 0) return cudaErrorInvalidValue;
  const int64_t tiles = (int64_t)g.E * (g.m_rows / gt::kBM) * (g.N / gt::kBN);
  return launch_tiled<2>(A, B, tmd, g, tiles, s);
}

int tiled_max_experts() { return gt::kMaxE; }

}  // namespace nvfp4

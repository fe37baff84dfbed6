// NVFP4 quantiser kernels: the scope amax pass and the row quantiser.
//
// "The 4-bitter Lesson: Balancing Stability and Performance in NVFP4 RL":
//   §Baseline -- E2M1 values, one E4M3 scale per 16 values, one FP32 global scale;
//   §"Why is the NVFP4 pretraining recipe not sufficient for RL?" -- one global scale
//   per weight tensor, one per token for activations, computed inside the fused
//   quantisation kernel, and stochastic rounding as the pretraining recipe's option.
//
// Layout of the work: one warp per input row.  Lane l owns the 16-byte chunks at
// columns 8l + 256i, so every load instruction of the warp reads 512 contiguous bytes
// and every code store writes 128 contiguous bytes.  The two lanes l, l^1 hold the two
// halves of one 16-value block; their shuffle gives the block max.  Lanes 8q gather the
// four scale bytes of a 64-column group into the one 32-bit word the tiled scale layout
// keeps contiguous.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "encode.cuh"
#include "launch.h"
#include "pdl.cuh"
#include "ptx.cuh"
#include "status.cuh"
#include "tiled.cuh"

namespace nvfp4 {

constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ int64_t sf_word_offset(int64_t r, int64_t w, int64_t sf_words) {
  return ((r >> 7) * sf_words + w) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4;
}
// The 32-bit word holding scale columns 4w .. 4w+3 of row r in the standalone output:
// the 128x4 tiled layout, or row-major [rows, cols/16] when a.sf_row_bytes > 0.
__device__ __forceinline__ uint32_t* sf_at(const QuantArgs& a, int64_t r, int64_t w) {
  return reinterpret_cast<uint32_t*>(a.sf + (a.sf_row_bytes ? r * a.sf_row_bytes + 4 * w
                                                              : sf_word_offset(r, w, a.sf_words)));
}

// Output addressing for both layouts: 8 bytes of codes at byte `b` of output row `orow`,
// and the 32-bit word holding scale columns 4w .. 4w+3.
__device__ __forceinline__ uint8_t* code_ptr(const QuantArgs& a, int64_t orow, int64_t b) {
  return a.tiled_R ? a.codes + tiled_code_offset(orow, b, a.kblocks, a.tiled_R) : a.codes + orow * a.codes_ld + b;
}
__device__ __forceinline__ uint8_t* sfw_ptr(const QuantArgs& a, int64_t orow, int64_t w) {
  return a.tiled_R ? a.codes + tiled_sf_offset(orow, 4 * w, a.kblocks, a.tiled_R)
                   : reinterpret_cast<uint8_t*>(sf_at(a, orow, w));
}

// Output addressing of one row, set up once per row so that each block's code and scale
// addresses are a few 32-bit operations.  Codes of block b (8 bytes) sit at
//   codes + (b >> 4) * code_outer + ((((b >> 1) & 7) ^ swz) << 4) + (b & 1) * 8
// (row-major: code_outer = 128, swz = 0; GEMM-tiled: code_outer = one K-block, swz = the
// row's swizzle), and scale word w (columns 4w .. 4w+3) at
//   sf + (w >> 2) * sf_outer + (w & 3) * sf_inner.
struct RowOut {
  uint8_t* codes;
  uint8_t* sf;
  uint32_t code_outer, swz, sf_outer, sf_inner;
};

__device__ __forceinline__ RowOut row_out(const QuantArgs& a, int64_t orow) {
  RowOut o;
  if (a.tiled_R) {
    const int lg = tiled_log2_rows(a.tiled_R);
    const int64_t blk = orow >> lg, rr = orow & (a.tiled_R - 1), r128 = rr & 127;
    const int64_t base = blk * a.kblocks * tiled_block_bytes(a.tiled_R);
    o.codes = a.codes + base + rr * 128;
    o.sf = a.codes + base + (int64_t)a.tiled_R * 128 + (rr >> 7) * 2048 + (r128 & 31) * 16 + (r128 >> 5) * 4;
    o.code_outer = o.sf_outer = (uint32_t)tiled_block_bytes(a.tiled_R);
    o.swz = (uint32_t)(rr & 7);
    o.sf_inner = 512;
  } else {
    o.codes = a.codes + orow * a.codes_ld;
    o.code_outer = 128;
    o.swz = 0;
    if (a.sf_row_bytes) {
      o.sf = a.sf + orow * a.sf_row_bytes;
      o.sf_outer = 16;
      o.sf_inner = 4;
    } else {
      o.sf = a.sf + ((orow >> 7) * a.sf_words) * 512 + (orow & 31) * 16 + ((orow >> 5) & 3) * 4;
      o.sf_outer = 2048;
      o.sf_inner = 512;
    }
  }
  return o;
}
__device__ __forceinline__ uint2* row_codes(const RowOut& o, uint32_t b) {
  return reinterpret_cast<uint2*>(o.codes + (b >> 4) * o.code_outer + ((((b >> 1) & 7u) ^ o.swz) << 4) +
                                  (b & 1u) * 8);
}
__device__ __forceinline__ uint32_t* row_sf_word(const RowOut& o, uint32_t w) {
  return reinterpret_cast<uint32_t*>(o.sf + (w >> 2) * o.sf_outer + (w & 3u) * o.sf_inner);
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

// ------------------------------------------------------------------ amax of each scope

// Zeroes the n scope words before an amax pass (a kernel rather than a memset, so that the
// amax kernel can be launched as its programmatic dependent).
__global__ void __launch_bounds__(256) zero_words_kernel(uint32_t* p, int64_t n) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    p[i] = 0u;
}

// Max |x| over the tensor (group_rows == 0) or over each group of group_rows rows.
// Results are float bit patterns combined with atomicMax, which for non-negative floats
// is the float maximum whatever the order: deterministic.
__global__ void __launch_bounds__(256) amax_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows, int64_t cols,
                                                   int64_t ld, int64_t group_rows, uint32_t* amax_bits) {
  grid_dep_sync();   // the scope words have been zeroed
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t nwarp = (int64_t)gridDim.x * 8;
  const int64_t per = (rows + nwarp - 1) / nwarp;
  const int64_t r0 = warp * per, r1 = min(rows, r0 + per);
  float m = 0.0f;
  int64_t grp = group_rows ? (r0 / group_rows) : 0;
  for (int64_t r = r0; r < r1; ++r) {
    if (group_rows && r / group_rows != grp) {
      m = warp_max(m);
      if (lane == 0 && m > 0.0f) atomicMax(&amax_bits[grp], __float_as_uint(m));
      m = 0.0f;
      grp = r / group_rows;
    }
    const __nv_bfloat16* xr = x + r * ld;
    for (int64_t c = 8 * lane; c < cols; c += 256) {
      float f[8];
      bf16x8_to_f32(ld_nc_v4(xr + c), f);
      m = fmaxf(m, absmax8(f));
    }
  }
  m = warp_max(m);
  if (group_rows) {
    if (lane == 0 && r0 < r1 && m > 0.0f) atomicMax(&amax_bits[grp], __float_as_uint(m));
    return;
  }
  __shared__ float sm[8];
  if (lane == 0) sm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = sm[0];
    for (int i = 1; i < 8; ++i) b = fmaxf(b, sm[i]);
    if (b > 0.0f) atomicMax(&amax_bits[0], __float_as_uint(b));
  }
}

// Max |x| of a contiguous tensor seen as n16 16-byte chunks: eight independent loads in
// flight per thread (up to 2048 threads per SM: ~256 KB in flight), one atomicMax per
// block.  Launched as a programmatic dependent of the kernel that zeroes the result word:
// the loads and the block's reduction overlap that kernel, and only the atomic waits for
// it; the encode kernel after it may be scheduled as soon as this grid is placed (every
// block fits at once) and waits for its completion before reading the result.
__global__ void __launch_bounds__(256) amax_flat_kernel(const uint4* __restrict__ x, int64_t n16,
                                                        uint32_t* amax_bits) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  constexpr int kU = 8;
  float m = 0.0f;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + (kU - 1) * stride < n16; i += kU * stride) {
    uint4 v[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) v[u] = ld_nc_v4(x + i + u * stride);
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      float f[8];
      bf16x8_to_f32(v[u], f);
      m = fmaxf(m, absmax8(f));
    }
  }
  for (; i < n16; i += stride) {
    float f[8];
    bf16x8_to_f32(ld_nc_v4(x + i), f);
    m = fmaxf(m, absmax8(f));
  }
  m = warp_max(m);
  __shared__ float sm[8];
  const int lane = threadIdx.x & 31;
  if (lane == 0) sm[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = sm[0];
    for (int k = 1; k < 8; ++k) b = fmaxf(b, sm[k]);
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the result word has been zeroed
    if (b > 0.0f) atomicMax(&amax_bits[0], __float_as_uint(b));
  }
}

// ------------------------------------------------------------------ row quantiser

__device__ __forceinline__ int64_t interleave_row(int64_t r, int64_t I) {
  const int64_t n2 = 2 * I, e = r / n2, rl = r - e * n2;
  int64_t o;
  if (rl < I) {
    o = (rl >> 6) * 128 + (rl & 63);
  } else {
    const int64_t u = rl - I;
    o = (u >> 6) * 128 + 64 + (u & 63);
  }
  return e * n2 + o;
}

// Encode one input row held in registers (lane l owns the 16-byte chunks at columns
// 8l + 256i) and write its codes, scale words and global scale to its output row.
template <int RND, int MAXC>
__device__ __forceinline__ void quantize_row(const QuantArgs& a, int64_t row, const uint4 (&q)[MAXC], int lane) {
  const int64_t data_words = (a.cols + 63) / 64;
  float bm[MAXC];
  float rmax = 0.0f;
#pragma unroll
  for (int i = 0; i < MAXC; ++i) {
    float f[8];
    bf16x8_to_f32(q[i], f);
    const float cm = absmax8(f);
    bm[i] = fmaxf(cm, __shfl_xor_sync(kFull, cm, 1));
    rmax = fmaxf(rmax, bm[i]);
  }
  float g;
  if (a.mode == kScopeRow) {
    rmax = warp_max(rmax);
    g = a.g_in ? a.g_in[row] : __fdiv_rn(rmax, kGlobalDivisor);
  } else if (a.mode == kScopeTensor) {
    g = a.g_in ? a.g_in[0] : __fdiv_rn(__uint_as_float(a.amax_bits[0]), kGlobalDivisor);
  } else {
    const int64_t gi = row / a.group_rows;
    g = a.g_in ? a.g_in[gi] : __fdiv_rn(__uint_as_float(a.amax_bits[gi]), kGlobalDivisor);
  }
  const float six_g = __fmul_rn(6.0f, g);

  const int64_t orow = a.map == kMapInterleave ? interleave_row(row, a.map_I) : row;

#pragma unroll
  for (int i = 0; i < MAXC; ++i) {
    const int64_t col = 8 * lane + 256 * i;
    const bool active = col < a.cols;
    const BlockScale bs = block_scale(bm[i], g, six_g);
    float f[8];
    bf16x8_to_f32(q[i], f);
    uint32_t word;
    if (RND == kRoundSR) {
      const uint64_t j = a.rng_offset + (uint64_t)(row * a.cols + col) / 8u;
      const uint4 rnd = philox4x32_10(make_uint4((uint32_t)j, (uint32_t)(j >> 32), 0u, 0u), (uint32_t)a.seed,
                                      (uint32_t)(a.seed >> 32));
      word = e2m1x8_sr(f, q[i], bs, rnd);
    } else {
      word = e2m1x8_rn(f, bs);
    }
    const uint32_t sfb = active ? bs.sf : 0u;
    const uint32_t s2 = __shfl_down_sync(kFull, sfb, 2);
    const uint32_t s4 = __shfl_down_sync(kFull, sfb, 4);
    const uint32_t s6 = __shfl_down_sync(kFull, sfb, 6);
    const uint32_t sfw = sfb | (s2 << 8) | (s4 << 16) | (s6 << 24);
    if (active) *reinterpret_cast<uint32_t*>(a.codes + orow * a.codes_ld + col / 2) = word;
    if ((lane & 7) == 0 && active)
      *sf_at(a, orow, 4 * i + lane / 8) = sfw;
  }
  for (int64_t w = data_words + lane; w < a.sf_words; w += 32)
    *sf_at(a, orow, w) = 0u;
  for (int64_t b = a.cols / 2 + 8 * lane; b < a.cols_pad / 2; b += 256)
    *reinterpret_cast<uint2*>(a.codes + orow * a.codes_ld + b) = make_uint2(0u, 0u);
  if (lane == 0 && a.g_out != nullptr) {
    if (a.mode == kScopeRow) a.g_out[row] = g;
    else if (a.mode == kScopeTensor && row == 0) a.g_out[0] = g;
    else if (a.mode == kScopeGroup && row % a.group_rows == 0) a.g_out[row / a.group_rows] = g;
  }
}

// Zero scale words of the tile-grid padding rows (rows .. rows_total - 1).
__device__ __forceinline__ void zero_pad_rows(const QuantArgs& a, int64_t warp, int64_t nwarp, int lane) {
  for (int64_t row = a.rows + warp; row < a.rows_total; row += nwarp)
    for (int64_t w = lane; w < a.sf_words; w += 32)
      *sf_at(a, row, w) = 0u;
}

// Register path (any width up to 8192 columns): the warp loads its row straight into
// registers.
template <int RND, int MAXC>
__global__ void __launch_bounds__(256) quantize_rows_kernel(QuantArgs a) {
  grid_dep_sync();   // (programmatic launch after the amax pass: its result is visible)
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t nwarp = (int64_t)gridDim.x * 8;
  for (int64_t row = warp; row < a.rows; row += nwarp) {
    uint4 q[MAXC];
    const __nv_bfloat16* xr = a.x + row * a.ld;
#pragma unroll
    for (int i = 0; i < MAXC; ++i) {
      const int64_t col = 8 * lane + 256 * i;
      q[i] = col < a.cols ? ld_nc_v4(xr + col) : make_uint4(0, 0, 0, 0);
    }
    quantize_row<RND, MAXC>(a, row, q, lane);
  }
  zero_pad_rows(a, warp, nwarp, lane);
}

// Streaming path (rows up to 2048 columns).  Every warp keeps a.q_stages rows in flight
// in a shared-memory ring filled by bulk async copies (cp.async.bulk, completion on an
// mbarrier), so HBM sees several rows per warp while the warp encodes the current one.
// The ring is sized to the row (stride a.q_stride bytes): short rows get more stages and
// more warps per SM, so that about 200 KB per SM are in flight whatever the width.
// Encoding works lane per 16-value block: block b of the row belongs to lane b % 32, so
// each lane computes its block scale once, stores 8 bytes of codes (a warp stores 256
// contiguous bytes) and four neighbouring lanes gather one 32-bit scale word.
constexpr int kQWarps = 8;
constexpr int kQMaxStages = 8;
constexpr int kQMaxSlots = 4;           // 16-value blocks per lane: rows of up to 2048 columns
constexpr size_t kQSmemMax = 200 * 1024;
__host__ __device__ constexpr size_t stream_smem_bytes(int stages, int stride) {
  return (size_t)kQWarps * stages * stride + (size_t)kQWarps * stages * sizeof(uint64_t) + 16;
}

// One 16-value block (two 16-byte chunks of BF16) -> its E4M3 scale byte and 8 bytes of
// codes, given the scope's g and 6g.
// amax_b < 0: the block max is computed here.
template <int RND>
__device__ __forceinline__ void encode_regs(const QuantArgs& a, int64_t row, int64_t blk, const uint4& q0,
                                            const uint4& q1, float g, float six_g, uint32_t& sf_out,
                                            uint2& codes_out, float amax_b = -1.0f) {
  float h0[8], h1[8];
  bf16x8_to_f32(q0, h0);
  bf16x8_to_f32(q1, h1);
  const BlockScale bs = block_scale(amax_b >= 0.0f ? amax_b : absmax16_bf16(q0, q1), g, six_g);
  if (RND == kRoundSR) {
    const uint64_t j = a.rng_offset + (uint64_t)(row * a.cols + blk * 16) / 8u;
    const uint32_t k0 = (uint32_t)a.seed, k1 = (uint32_t)(a.seed >> 32);
    codes_out.x = e2m1x8_sr(h0, q0, bs, philox4x32_10(make_uint4((uint32_t)j, (uint32_t)(j >> 32), 0u, 0u), k0, k1));
    codes_out.y = e2m1x8_sr(h1, q1, bs,
                            philox4x32_10(make_uint4((uint32_t)(j + 1), (uint32_t)((j + 1) >> 32), 0u, 0u), k0, k1));
  } else {
    codes_out = e2m1x16_rn(h0, h1, bs);
  }
  sf_out = bs.sf;
}

// Scopes whose global scale is known before encoding (per tensor, per group: after the
// amax pass, or given): every 64-value group of a row is independent.  One thread per
// group: 128 bytes in (eight 16-byte loads issued together), four blocks encoded, 8 bytes
// of codes per block and one 32-bit scale word out -- no row reduction, no cross-lane
// traffic.  The (row, group) position advances by the grid stride without divisions.
// Groups past the data (up to cols_pad) are written as zeros, and so are the scale words
// of rows .. rows_total-1.
template <int RND>
__global__ void __launch_bounds__(256) quantize_known_scale_kernel(QuantArgs a) {
  grid_dep_sync();
  const int64_t words = a.sf_words, nb = a.cols / 16, nb_pad = a.cols_pad / 16;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t s_row = stride / words, s_w = stride - s_row * words;
  int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int64_t row = i0 / words, w = i0 - row * words;
  float g0 = 0.0f;
  if (a.mode == kScopeTensor)
    g0 = a.g_in ? a.g_in[0] : __fdiv_rn(__uint_as_float(a.amax_bits[0]), kGlobalDivisor);
  for (; row < a.rows; row += s_row, w += s_w) {
    if (w >= words) {
      w -= words;
      if (++row >= a.rows) break;
    }
    const int64_t blk0 = 4 * w;
    uint4 q[8];
    const __nv_bfloat16* xr = a.x + row * a.ld + blk0 * 16;
#pragma unroll
    for (int j = 0; j < 8; ++j) q[j] = blk0 + j / 2 < nb ? ld_nc_v4(xr + 8 * j) : make_uint4(0u, 0u, 0u, 0u);
    float g = g0;
    int64_t gi = 0;
    if (a.mode != kScopeTensor) {
      gi = (int64_t)((uint32_t)row / (uint32_t)a.group_rows);
      g = a.g_in ? a.g_in[gi] : __fdiv_rn(__uint_as_float(a.amax_bits[gi]), kGlobalDivisor);
    }
    const float six_g = __fmul_rn(6.0f, g);
    uint32_t sfw = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      const int64_t blk = blk0 + b;
      uint32_t sf = 0;
      uint2 cw = make_uint2(0u, 0u);
      if (blk < nb) encode_regs<RND>(a, row, blk, q[2 * b], q[2 * b + 1], g, six_g, sf, cw);
      sfw |= sf << (8 * b);
      if (blk < nb_pad) *reinterpret_cast<uint2*>(code_ptr(a, row, blk * 8)) = cw;
    }
    *reinterpret_cast<uint32_t*>(sfw_ptr(a, row, w)) = sfw;
    if (w == 0 && a.g_out != nullptr && (a.mode == kScopeTensor ? row == 0 : row % a.group_rows == 0))
      a.g_out[gi] = g;
  }
  if (a.tiled_R == 0)
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (a.rows_total - a.rows) * words; i += stride)
      *sf_at(a, a.rows + i / words, i % words) = 0u;
}

// Known-scale scopes over row-major rows of a multiple of 64 columns: the same encoding
// with one 16-value block per lane, consecutive lanes on consecutive blocks.  Each load
// instruction of a warp reads 1 KB contiguous, each code store writes 256 B contiguous,
// and the scale arithmetic runs once per block.  Lanes 4q .. 4q+3 gather one 32-bit
// scale word.  Each warp loads kSlabs slabs of 32 blocks before encoding them, to keep
// 64 bytes per lane in flight.  Idx is the block index type (32-bit when every index
// fits).
template <int RND, typename Idx>
__global__ void __launch_bounds__(256) quantize_known_coalesced_kernel(QuantArgs a) {
  grid_dep_sync();
  constexpr int kSlabs = 2;
  const int lane = threadIdx.x & 31;
  const Idx bpr = (Idx)(a.cols / 16);
  const int64_t total = a.rows * (int64_t)bpr;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t wstride = ((int64_t)gridDim.x * blockDim.x) >> 5;
  float g0 = 0.0f;
  if (a.mode == kScopeTensor)
    g0 = a.g_in ? a.g_in[0] : __fdiv_rn(__uint_as_float(a.amax_bits[0]), kGlobalDivisor);
  const float six_g0 = __fmul_rn(6.0f, g0);
  // (row, block column) of this lane's block in slab 0, advanced without divisions: one
  // iteration moves by `step` blocks, slab s by 32 s more
  const int64_t step = wstride * 32 * kSlabs;
  const Idx step_r = (Idx)(step / (int64_t)bpr), step_c = (Idx)(step % (int64_t)bpr);
  int64_t base = warp0 * 32 * kSlabs;
  Idx r0 = (Idx)((base + lane) / (int64_t)bpr), c0 = (Idx)((base + lane) % (int64_t)bpr);
  for (; base < total; base += step) {
    uint4 v0[kSlabs], v1[kSlabs];
    Idx row[kSlabs], cb[kSlabs];
    bool live[kSlabs];
#pragma unroll
    for (int s2 = 0; s2 < kSlabs; ++s2) {
      Idx r = r0, c = c0 + 32 * s2;
      while (c >= bpr) {
        c -= bpr;
        ++r;
      }
      row[s2] = r;
      cb[s2] = c;
      live[s2] = base + 32 * s2 + lane < total;
      v0[s2] = v1[s2] = make_uint4(0u, 0u, 0u, 0u);
      if (live[s2]) {
        const __nv_bfloat16* src = a.x + (int64_t)r * a.ld + 16 * (int64_t)c;
        v0[s2] = ld_nc_v4(src);
        v1[s2] = ld_nc_v4(src + 8);
      }
    }
    c0 += step_c;
    r0 += step_r;
    if (c0 >= bpr) {
      c0 -= bpr;
      ++r0;
    }
#pragma unroll
    for (int s2 = 0; s2 < kSlabs; ++s2) {
      float g = g0, six_g = six_g0;
      int64_t gi = 0;
      if (a.mode != kScopeTensor) {
        gi = (int64_t)((uint64_t)row[s2] / (uint64_t)a.group_rows);
        g = a.g_in ? a.g_in[gi] : __fdiv_rn(__uint_as_float(a.amax_bits[gi]), kGlobalDivisor);
        six_g = __fmul_rn(6.0f, g);
      }
      uint32_t sf = 0;
      uint2 cw = make_uint2(0u, 0u);
      encode_regs<RND>(a, row[s2], cb[s2], v0[s2], v1[s2], g, six_g, sf, cw);
      if (live[s2]) *reinterpret_cast<uint2*>(a.codes + (int64_t)row[s2] * a.codes_ld + 8 * (int64_t)cb[s2]) = cw;
      // the scale word of this lane's 64-value group: block k of it sits at lane 4q + k
      const uint32_t s1 = __shfl_down_sync(kFull, sf, 1);
      const uint32_t s2w = __shfl_down_sync(kFull, sf, 2);
      const uint32_t s3 = __shfl_down_sync(kFull, sf, 3);
      if (live[s2] && (lane & 3) == 0) *sf_at(a, row[s2], cb[s2] / 4) = sf | (s1 << 8) | (s2w << 16) | (s3 << 24);
      if (live[s2] && cb[s2] == 0 && a.g_out != nullptr &&
          (a.mode == kScopeTensor ? row[s2] == 0 : (int64_t)row[s2] % a.group_rows == 0))
        a.g_out[gi] = g;
    }
  }
  const int64_t stride = (int64_t)gridDim.x * blockDim.x, words = a.sf_words;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < (a.rows_total - a.rows) * words; i += stride)
    *sf_at(a, a.rows + i / words, i % words) = 0u;
}

template <int RND>
__global__ void __launch_bounds__(kQWarps * 32, 3) quantize_rows_stream_kernel(QuantArgs a) {
  grid_dep_sync();
  extern __shared__ __align__(128) uint8_t qsm[];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int64_t warp = (int64_t)blockIdx.x * kQWarps + wib;
  const int64_t nwarp = (int64_t)gridDim.x * kQWarps;
  const int kQStages = a.q_stages, stride = a.q_stride;
  uint8_t* ring = qsm + (size_t)wib * kQStages * stride;
  uint64_t* bars = reinterpret_cast<uint64_t*>(qsm + (size_t)kQWarps * kQStages * stride) + wib * kQStages;
  volatile int* abort = reinterpret_cast<volatile int*>(qsm + (size_t)kQWarps * kQStages * stride +
                                                        (size_t)kQWarps * kQStages * sizeof(uint64_t));
  if (threadIdx.x == 0) *abort = 0;
  const uint32_t row_bytes = (uint32_t)(a.cols * 2);
  const int64_t nblk = a.cols / 16;
  const int64_t data_words = (a.cols + 63) / 64;
  int64_t nrows = a.rows;
  if (a.rows_dev != nullptr && (int64_t)*a.rows_dev < nrows) nrows = *a.rows_dev;
  if (lane == 0) {
    for (int s = 0; s < kQStages; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (lane == 0) {
    for (int s = 0; s < kQStages; ++s) {
      const int64_t r = warp + s * nwarp;
      if (r < nrows) {
        mbar_arrive_expect_tx(&bars[s], row_bytes);
        bulk_load(ring + s * stride, a.x + r * a.ld, row_bytes, &bars[s]);
      }
    }
  }
  uint32_t parity = 0;
  int s = 0;
  for (int64_t row = warp; row < nrows; row += nwarp) {
    if (!mbar_wait(&bars[s], (parity >> s) & 1u, a.status, abort)) break;
    parity ^= 1u << s;
    const uint8_t* buf = ring + s * stride;
    if (a.row_filter != nullptr && a.row_filter[row] < 0) {   // a padding slot: nothing to encode
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int64_t r2 = row + (int64_t)kQStages * nwarp;
        if (r2 < nrows) {
          mbar_arrive_expect_tx(&bars[s], row_bytes);
          bulk_load(ring + s * stride, a.x + r2 * a.ld, row_bytes, &bars[s]);
        }
      }
      s = s + 1 == kQStages ? 0 : s + 1;
      continue;
    }
    // block maxima of the row from the packed BF16 bits (block b of the row at lane b % 32,
    // slot b / 32; rows of up to 2048 columns), kept for the encode pass
    float bmax[kQMaxSlots];
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < kQMaxSlots; ++i) {
      const int64_t blk = lane + 32 * i;
      bmax[i] = 0.0f;
      if (blk < nblk) {
        bmax[i] = absmax16_bf16(*reinterpret_cast<const uint4*>(buf + blk * 32),
                                *reinterpret_cast<const uint4*>(buf + blk * 32 + 16));
        m = fmaxf(m, bmax[i]);
      }
    }
    float g;
    if (a.mode == kScopeRow) {
      m = warp_max(m);
      g = a.g_in ? a.g_in[row] : __fdiv_rn(m, kGlobalDivisor);
    } else if (a.mode == kScopeTensor) {
      g = a.g_in ? a.g_in[0] : __fdiv_rn(__uint_as_float(a.amax_bits[0]), kGlobalDivisor);
    } else {
      const int64_t gi = row / a.group_rows;
      g = a.g_in ? a.g_in[gi] : __fdiv_rn(__uint_as_float(a.amax_bits[gi]), kGlobalDivisor);
    }
    const float six_g = __fmul_rn(6.0f, g);
    const int64_t orow = a.map == kMapInterleave ? interleave_row(row, a.map_I) : row;
    const RowOut ro = row_out(a, orow);
    // stochastic rounding: one block at a time (the block max read again from shared
    // memory), so that three CTAs of its registers fit on an SM
    constexpr int kUnroll = RND == kRoundSR ? 1 : kQMaxSlots;
#pragma unroll kUnroll
    for (int i = 0; i < kQMaxSlots; ++i) {
      if (32 * i >= nblk) break;                       // warp-uniform
      const uint32_t blk = (uint32_t)lane + 32u * i;
      const bool active = blk < nblk;
      uint32_t sfb = 0;
      uint2 cw = make_uint2(0u, 0u);
      if (active) {
        const uint4 q0 = *reinterpret_cast<const uint4*>(buf + blk * 32);
        const uint4 q1 = *reinterpret_cast<const uint4*>(buf + blk * 32 + 16);
        encode_regs<RND>(a, row, blk, q0, q1, g, six_g, sfb, cw, RND == kRoundSR ? absmax16_bf16(q0, q1) : bmax[i]);
      }
      const uint32_t s1 = __shfl_down_sync(kFull, sfb, 1);
      const uint32_t s2 = __shfl_down_sync(kFull, sfb, 2);
      const uint32_t s3 = __shfl_down_sync(kFull, sfb, 3);
      const uint32_t sfw = sfb | (s1 << 8) | (s2 << 16) | (s3 << 24);
      if (active) *row_codes(ro, blk) = cw;
      if ((lane & 3) == 0 && active) *row_sf_word(ro, blk >> 2) = sfw;
    }
    fence_proxy_async_smem();   // this row's reads of the buffer precede the next bulk write
    __syncwarp();
    if (lane == 0) {
      const int64_t r2 = row + (int64_t)kQStages * nwarp;
      if (r2 < nrows) {
        mbar_arrive_expect_tx(&bars[s], row_bytes);
        bulk_load(ring + s * stride, a.x + r2 * a.ld, row_bytes, &bars[s]);
      }
    }
    for (int64_t w = data_words + lane; w < a.sf_words; w += 32) *row_sf_word(ro, (uint32_t)w) = 0u;
    for (int64_t b = nblk + lane; b < a.cols_pad / 16; b += 32) *row_codes(ro, (uint32_t)b) = make_uint2(0u, 0u);
    if (lane == 0 && a.g_out != nullptr) {
      if (a.mode == kScopeRow) a.g_out[row] = g;
      else if (a.mode == kScopeTensor && row == 0) a.g_out[0] = g;
      else if (a.mode == kScopeGroup && row % a.group_rows == 0) a.g_out[row / a.group_rows] = g;
    }
    s = s + 1 == kQStages ? 0 : s + 1;
  }
  if (a.tiled_R == 0) zero_pad_rows(a, warp, nwarp, lane);
}

// Per-row NVFP4 of rows whose max |x| is already known (the SwiGLU epilogue folds it
// into amax_bits while it writes h): no row-wide reduction is left, so every thread
// encodes two neighbouring 16-value blocks on its own -- 64 bytes in (four 16-byte loads
// issued before anything waits on them), 16 bytes of codes and two scale bytes out --
// and two neighbouring lanes (blocks 4w .. 4w+3 of a row) form the 32-bit scale word.
// Blocks past I (up to Ip) are written as zeros.
__device__ __forceinline__ void requant_block(const uint4& q0, const uint4& q1, float g, uint32_t& sf,
                                              uint32_t& c0, uint32_t& c1) {
  float v0[8], v1[8];
  bf16x8_to_f32(q0, v0);
  bf16x8_to_f32(q1, v1);
  const BlockScale bs = block_scale(absmax16_bf16(q0, q1), g, __fmul_rn(6.0f, g));
  sf = bs.sf;
  const uint2 c = e2m1x16_rn(v0, v1, bs);
  c0 = c.x;
  c1 = c.y;
}

// Idx: the index type of the unit and byte arithmetic (32-bit when every index fits).
template <typename Idx>
__global__ void __launch_bounds__(256) requant_tiled_kernel(const __nv_bfloat16* __restrict__ h,
                                                            const uint32_t* __restrict__ amax_bits,
                                                            const int32_t* __restrict__ perm,
                                                            const int32_t* __restrict__ n_rows_dev, int64_t max_rows,
                                                            int64_t I, int64_t Ip, uint8_t* __restrict__ out,
                                                            float* __restrict__ g_out) {
  grid_dep_sync();
  const int lane = threadIdx.x & 31;
  int64_t rows = *n_rows_dev;
  if (rows > max_rows) rows = max_rows;
  const Idx np = (Idx)(Ip / 32), np_data = (Idx)(I / 32), kblocks = (Idx)(Ip / 256);
  const int64_t total = rows * (int64_t)np;   // np % 2 == 0: lane pairs hold blocks 4w .. 4w+3 of one row
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < total; base += stride) {
    const Idx i = (Idx)(base + threadIdx.x);
    const bool in = base + threadIdx.x < total;
    const Idx row = in ? i / np : 0, pr = in ? i - row * np : 0;
    const bool data = in && pr < np_data;
    uint4 q[4] = {};
    if (data) {
      const __nv_bfloat16* src = h + (int64_t)row * I + pr * 32;
#pragma unroll
      for (int j = 0; j < 4; ++j) q[j] = ld_nc_v4(src + 8 * j);
    }
    const bool live = in && perm[row] >= 0;
    uint32_t sf2 = 0;
    uint4 cw = make_uint4(0u, 0u, 0u, 0u);
    if (live && data) {
      const float g = __fdiv_rn(__uint_as_float(amax_bits[row]), kGlobalDivisor);
      uint32_t sa, sb;
      requant_block(q[0], q[1], g, sa, cw.x, cw.y);
      requant_block(q[2], q[3], g, sb, cw.z, cw.w);
      sf2 = sa | (sb << 8);
      if (pr == 0) g_out[row] = g;
    }
    const uint32_t s1 = __shfl_down_sync(kFull, sf2, 1);
    if (live) {
      // the GEMM-tiled layout (128-row blocks) in Idx arithmetic: codes bytes 16 pr .. of the
      // row, scale columns 2 pr, 2 pr + 1
      const Idx blk = row >> 7, rr = row & 127, b = pr * 16, kb = b >> 7, bb = b & 127;
      *reinterpret_cast<uint4*>(out + (size_t)((blk * kblocks + kb) * (Idx)(128 * 144) + rr * 128 +
                                               (((bb >> 4) ^ (rr & 7)) << 4))) = cw;
      if ((lane & 1) == 0) {
        const Idx c = 2 * pr, kc = c >> 4, cc = c & 15;
        *reinterpret_cast<uint32_t*>(out + (size_t)((blk * kblocks + kc) * (Idx)(128 * 144) + 128 * 128 +
                                                    (cc >> 2) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + (cc & 3))) =
            sf2 | (s1 << 16);
      }
    }
  }
}

cudaError_t launch_requant_tiled(const __nv_bfloat16* h, const uint32_t* amax_bits, const int32_t* perm,
                                 const int32_t* n_rows_dev, int64_t max_rows, int64_t I, int64_t Ip, uint8_t* out,
                                 float* g_out, cudaStream_t s, bool pdl) {
  const int64_t total = max_rows * (Ip / 32);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 8 * (int64_t)num_sms()) blocks = 8 * (int64_t)num_sms();
  // 32-bit index arithmetic when the units and the output's bytes all fit
  if (total < ((int64_t)1 << 31) && tiled_bytes(max_rows, Ip, 128) < ((int64_t)1 << 31))
    return launch_pdl(pdl, requant_tiled_kernel<uint32_t>, dim3((unsigned)blocks), dim3(256), 0, s, h, amax_bits, perm,
                      n_rows_dev, max_rows, I, Ip, out, g_out);
  return launch_pdl(pdl, requant_tiled_kernel<int64_t>, dim3((unsigned)blocks), dim3(256), 0, s, h, amax_bits, perm,
                    n_rows_dev, max_rows, I, Ip, out, g_out);
}

template <int RND>
static cudaError_t launch_quant_rnd(const QuantArgs& a, int maxc, int grid, cudaStream_t s, bool pdl) {
  const dim3 g((unsigned)grid), b(256);
  switch (maxc) {
    case 1: return launch_pdl(pdl, quantize_rows_kernel<RND, 1>, g, b, 0, s, a);
    case 2: return launch_pdl(pdl, quantize_rows_kernel<RND, 2>, g, b, 0, s, a);
    case 4: return launch_pdl(pdl, quantize_rows_kernel<RND, 4>, g, b, 0, s, a);
    case 8: return launch_pdl(pdl, quantize_rows_kernel<RND, 8>, g, b, 0, s, a);
    case 16: return launch_pdl(pdl, quantize_rows_kernel<RND, 16>, g, b, 0, s, a);
    default: return launch_pdl(pdl, quantize_rows_kernel<RND, 32>, g, b, 0, s, a);
  }
}

template <int RND>
static cudaError_t launch_stream(const QuantArgs& a, int grid, size_t smem, cudaStream_t s, bool pdl) {
  static std::atomic<bool> attr_set[64];   // the attribute is set once per device
  {
    const cudaError_t err = set_smem_attr_once(attr_set, (const void*)quantize_rows_stream_kernel<RND>, (int)kQSmemMax + 4096);
    if (err != cudaSuccess) return err;
  }
  return launch_pdl(pdl, quantize_rows_stream_kernel<RND>, dim3((unsigned)grid), dim3(kQWarps * 32), smem, s, a);
}

cudaError_t launch_amax(const void* x, int64_t rows, int64_t cols, int64_t ld, int64_t group_rows,
                        uint32_t* amax_bits, int64_t n_scopes, cudaStream_t s) {
  if (n_scopes > 0) {
    int64_t zb = (n_scopes + 255) / 256;
    if (zb > 4 * (int64_t)num_sms()) zb = 4 * (int64_t)num_sms();
    const cudaError_t err = launch_pdl(false, zero_words_kernel, dim3((unsigned)zb), dim3(256), 0, s, amax_bits, n_scopes);
    if (err != cudaSuccess) return err;
  }
  if (rows == 0) return cudaSuccess;
  const int sms = num_sms();
  if (group_rows == 0 && ld == cols) {   // one scope over contiguous rows: flat pass
    const int64_t n16 = rows * cols / 8;
    int64_t blocks = (n16 + 255) / 256;
    if (blocks > 8 * sms) blocks = 8 * sms;
    return launch_pdl(true, amax_flat_kernel, dim3((unsigned)blocks), dim3(256), 0, s, static_cast<const uint4*>(x), n16,
                      amax_bits);
  }
  int64_t blocks = (rows + 7) / 8;
  if (blocks > 4 * sms) blocks = 4 * sms;
  return launch_pdl(true, amax_kernel, dim3((unsigned)blocks), dim3(256), 0, s, static_cast<const __nv_bfloat16*>(x),
                    rows, cols, ld, group_rows, amax_bits);
}

cudaError_t launch_quantize_rows(const QuantArgs& a, int rounding, cudaStream_t s, bool pdl) {
  if (a.rows_total == 0) return cudaSuccess;
  int maxc = 1;
  while (maxc * 256 < a.cols) maxc *= 2;
  const int sms = num_sms();
  int64_t blocks = (a.rows_total + 7) / 8;
  // rows of up to 2048 columns whose pitch keeps every row 16-byte aligned: streaming path
  // (the only one that writes the GEMM-tiled layout or takes a row filter / device count)
  const bool stream_ok = maxc <= 8 && (a.ld * 2) % 16 == 0;
  // per-tensor / per-group scopes in row order: the elementwise kernel
  if (a.mode != kScopeRow && a.map == kMapIdentity && a.row_filter == nullptr && a.rows_dev == nullptr &&
      (a.ld * 2) % 16 == 0 && reinterpret_cast<uintptr_t>(a.x) % 16 == 0) {
    if (a.tiled_R == 0 && a.cols % 64 == 0 && a.cols_pad == a.cols) {
      // row-major output, rows of whole 64-value groups: the lane-interleaved kernel
      const int64_t units = a.rows * (a.cols / 16);
      int64_t nb = (units + 511) / 512;     // 64 blocks per warp and iteration
      if (nb > 8 * (int64_t)sms) nb = 8 * (int64_t)sms;   // 8 CTAs of 8 warps per SM, several iterations each
      if (nb < 1) nb = 1;
      const bool i32 = units + 128 < ((int64_t)1 << 32);
      const dim3 g((unsigned)nb), b(256);
      if (rounding == kRoundSR)
        return i32 ? launch_pdl(pdl, quantize_known_coalesced_kernel<kRoundSR, uint32_t>, g, b, 0, s, a)
                   : launch_pdl(pdl, quantize_known_coalesced_kernel<kRoundSR, int64_t>, g, b, 0, s, a);
      return i32 ? launch_pdl(pdl, quantize_known_coalesced_kernel<kRoundRNE, uint32_t>, g, b, 0, s, a)
                 : launch_pdl(pdl, quantize_known_coalesced_kernel<kRoundRNE, int64_t>, g, b, 0, s, a);
    }
    const int64_t total = (a.rows > a.rows_total - a.rows ? a.rows : a.rows_total - a.rows) * a.sf_words;
    int64_t nb = (total + 255) / 256;
    if (nb > 8 * (int64_t)sms) nb = 8 * (int64_t)sms;
    if (nb < 1) nb = 1;
    return rounding == kRoundSR ? launch_pdl(pdl, quantize_known_scale_kernel<kRoundSR>, dim3((unsigned)nb), dim3(256), 0, s, a)
                                : launch_pdl(pdl, quantize_known_scale_kernel<kRoundRNE>, dim3((unsigned)nb), dim3(256), 0, s, a);
  }
  if (!stream_ok && (a.tiled_R != 0 || a.row_filter != nullptr || a.rows_dev != nullptr)) return cudaErrorInvalidValue;
  if (stream_ok) {
    // ring sizing: stride = the row rounded up to 128 bytes; up to 4 blocks (32 warps) per
    // SM (the register file's limit at 64 registers), at least 2 stages per warp, and as
    // many stages as keep the SM's ring near kQSmemMax
    QuantArgs b = a;
    b.q_stride = (int)((a.cols * 2 + 127) / 128 * 128);
    int blocks_per_sm = (int)(kQSmemMax / stream_smem_bytes(2, b.q_stride));
    if (blocks_per_sm > 4) blocks_per_sm = 4;
    if (blocks_per_sm < 1) blocks_per_sm = 1;
    int stages = (int)((kQSmemMax / blocks_per_sm - 16) / ((size_t)kQWarps * (b.q_stride + sizeof(uint64_t))));
    if (stages > kQMaxStages) stages = kQMaxStages;
    if (stages < 2) stages = 2;
    b.q_stages = stages;
    const size_t smem = stream_smem_bytes(stages, b.q_stride);
    int resident = 0;   // the registers of the rounding variant may allow fewer blocks
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident,
                                                      rounding == kRoundSR ? quantize_rows_stream_kernel<kRoundSR>
                                                                           : quantize_rows_stream_kernel<kRoundRNE>,
                                                      kQWarps * 32, smem) == cudaSuccess &&
        resident >= 1 && resident < blocks_per_sm)
      blocks_per_sm = resident;
    int64_t nb = (a.rows_total + kQWarps - 1) / kQWarps;
    if (nb > (int64_t)blocks_per_sm * sms) nb = (int64_t)blocks_per_sm * sms;
    return rounding == kRoundSR ? launch_stream<kRoundSR>(b, (int)nb, smem, s, pdl)
                                : launch_stream<kRoundRNE>(b, (int)nb, smem, s, pdl);
  }
  const int64_t cap = (int64_t)(maxc <= 8 ? 8 : 4) * sms;
  if (blocks > cap) blocks = cap;
  return rounding == kRoundSR ? launch_quant_rnd<kRoundSR>(a, maxc, (int)blocks, s, pdl)
                              : launch_quant_rnd<kRoundRNE>(a, maxc, (int)blocks, s, pdl);
}

}  // namespace nvfp4

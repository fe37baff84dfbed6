// Kernels of the expert block's W4A4 backward ("The 4-bitter Lesson: Balancing Stability
// and Performance in NVFP4 RL", §"Why is the NVFP4 pretraining recipe not sufficient for
// RL?": the pretraining recipe quantises the backward GEMMs too, with stochastic rounding
// of the gradients):
//   combine_backward_kernel   dy[slot(t,j)] = BF16(w[t,j] dout[t]) and dw[t,j] = <dout[t], y[slot]>
//   group_amax_kernel         max |x| over each expert's rows of a slot-ordered matrix
//   group_amax_g_kernel       the same maximum from the rows' own global scales, where the
//                             rows were already quantised per row
//   kofs_kernel               per-expert token counts -> 256-token K-block prefix sums
//   tquant_kernel             per-expert transposed NVFP4 (blocks of 16 tokens, one global
//                             scale per expert matrix) straight into the GEMM-tiled layout:
//                             the operands of the weight-gradient GEMMs, whose contraction
//                             runs over each expert's own (ragged) token count.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "encode.cuh"
#include "group.cuh"
#include "launch.h"
#include "ptx.cuh"
#include "status.cuh"
#include "tiled.cuh"

namespace nvfp4 {

namespace {
constexpr unsigned kAll = 0xFFFFFFFFu;

__device__ __forceinline__ uint4 ldg_nc(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

// BF16 (bits) of the exact product w * d, rounded once to nearest even, in float64: the
// product of a float32 and a BF16 value has at most 32 significant bits, so it is exact
// there; it is rounded at the spacing of its BF16 binade (2^-133 below 2^-126, where BF16
// values are subnormal).  The slow path of bf16_of_product.
__device__ __noinline__ uint32_t bf16_of_product_f64(float w, float d) {
  const double x = (double)w * (double)d;
  const double ax = fabs(x);
  int ex;
  frexp(ax, &ex);                                   // ax = m 2^ex, m in [0.5, 1)
  const int e = max(ex - 1, -126);                  // exponent of the BF16 binade
  const double r = rint(ldexp(ax, 7 - e));          // ax / spacing, to an integer, ties to even
  const float rf = (float)ldexp(r, e - 7);          // a BF16 value (or +inf past the range)
  return ((__float_as_uint(rf) >> 16) & 0x7FFFu) | (x < 0.0 ? 0x8000u : 0u);
}

// BF16 (bits) of the exact product w * d of a float32 and a BF16 value, rounded once to
// nearest even.  p = fl32(w d) rounded to BF16 is the rounding of the exact product
// unless p sits exactly on a BF16 midpoint (low half 0x8000): BF16 midpoints are float32
// values, so none lies strictly between the exact product and its nearest float32 p.  On
// a midpoint the exact product decides (bf16_of_product_f64; an FMA residual cannot: for
// products below about 2^-118 it may itself round to zero).
__device__ __forceinline__ uint32_t bf16_of_product(float w, float d) {
  const uint32_t b = __float_as_uint(__fmul_rn(w, d));
  if ((b & 0xFFFFu) == 0x8000u) return bf16_of_product_f64(w, d);
  const uint32_t lsb = (b >> 16) & 1u;
  return (b + 0x7FFFu + lsb) >> 16;   // round to nearest even (finite inputs)
}

// The same for two values at once, packed (w d0 in the low half): both float32 products
// by one paired multiply, both roundings to BF16 by one paired conversion (round to
// nearest even, subnormals kept); only a product that sits exactly on a BF16 midpoint
// -- where the float32 rounding may have decided the side -- goes through
// bf16_of_product.
__device__ __forceinline__ uint32_t bf16x2_of_products(float w, float d0, float d1) {
  float p0, p1;
  asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %4};\n"
      " mul.rn.f32x2 d, a, b;\n mov.b64 {%0, %1}, d;\n}"
      : "=f"(p0), "=f"(p1)
      : "f"(d0), "f"(d1), "f"(w));
  if ((__float_as_uint(p0) & 0xFFFFu) == 0x8000u || (__float_as_uint(p1) & 0xFFFFu) == 0x8000u)
    return bf16_of_product(w, d0) | (bf16_of_product(w, d1) << 16);
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(p1), "f"(p0));   // upper half from p1
  return r;
}
}  // namespace

// One warp per token: for each of its k slots, dy = BF16(w dout) and dw = sum_h dout y in
// float32 (each lane sums its columns in order with one rounding per term, then a
// fixed-shape butterfly over the lanes: the same order on every run); and dy's row of the
// slot layout quantised at once -- per-row scale, stochastic rounding with Philox key
// `key`, element index slot * H + column -- into the GEMM-tiled dyq (128-row blocks) with
// its global scale g_dy[slot], exactly as the row quantiser would from dy.  Lane l owns
// the 16-value blocks b = l + 32 i of the row, so each lane encodes whole blocks.  The
// row max needs no pass over dy: BF16 rounding is monotone, so max_h |BF16(w dout_h)| =
// BF16(|w| max_h |dout_h|), from the token's max |dout| taken once.
// Also (amax_bits != nullptr) the max |dy| of each expert's rows, for the transposed
// quantisation of dy: the slot's expert is the group holding it (starts [E+1]).
__global__ void __launch_bounds__(256, 3) combine_backward_kernel(const __nv_bfloat16* __restrict__ dout,
                                                                  const int32_t* __restrict__ inv,
                                                                  const float* __restrict__ w,
                                                                  const __nv_bfloat16* __restrict__ y, int64_t T,
                                                                  int k, int64_t H, __nv_bfloat16* __restrict__ dy,
                                                                  float* __restrict__ dw,
                                                                  const int32_t* __restrict__ starts, int E,
                                                                  uint32_t* __restrict__ amax_bits, uint8_t* dyq,
                                                                  float* __restrict__ g_dy, uint64_t key) {
  constexpr int kMaxSlots = 4;                  // 16-value blocks per lane: H <= 2048
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t nwarp = (int64_t)gridDim.x * 8;
  const int nb = (int)(H / 16);
  const int64_t kblocks = H / 256;
  const uint32_t k0 = (uint32_t)key, k1 = (uint32_t)(key >> 32);
  for (int64_t t = warp; t < T; t += nwarp) {
    // the token's max |dout| (its row is read again per slot, from L1)
    uint32_t dm = 0;
#pragma unroll
    for (int i = 0; i < kMaxSlots; ++i) {
      const int b = lane + 32 * i;
      if (b < nb)
        dm = max(dm, __float_as_uint(absmax16_bf16(ldg_nc(dout + t * H + 16 * b), ldg_nc(dout + t * H + 16 * b + 8))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dm = max(dm, __shfl_xor_sync(kAll, dm, o));
    for (int j = 0; j < k; ++j) {
      const int32_t slot = inv[t * k + j];
      if (slot < 0) continue;                   // warp-uniform
      const float wj = w[t * k + j];
      // the row's max |dy| (float bits of a BF16 value) and its global scale
      const uint32_t mb = bf16_of_product(fabsf(wj), __uint_as_float(dm)) << 16;
      const float g = __fdiv_rn(__uint_as_float(mb), kGlobalDivisor);
      const float six_g = __fmul_rn(6.0f, g);
      const int64_t rr = slot & 127;
      uint8_t* rcodes = dyq + (slot >> 7) * kblocks * tiled_block_bytes(128) + rr * 128;
      uint8_t* rsf = dyq + (slot >> 7) * kblocks * tiled_block_bytes(128) + 128 * 128 + (rr & 31) * 16 + (rr >> 5) * 4;
      float acc = 0.0f;
      // not unrolled: four copies of the block's products, Philox pair and SR encodes
      // outgrew the instruction cache (measured: the backward 5.89 ms unrolled, 5.74 rolled)
#pragma unroll 1
      for (int i = 0; i < kMaxSlots; ++i) {
        if (32 * i >= nb) break;                // warp-uniform
        const int b = lane + 32 * i;
        const bool active = b < nb;
        uint32_t o[8];
        uint32_t sfb = 0;
        uint2 cw = make_uint2(0u, 0u);
        if (active) {
          const uint4 y0 = ldg_nc(y + (int64_t)slot * H + 16 * b);
          const uint4 y1 = ldg_nc(y + (int64_t)slot * H + 16 * b + 8);
          const uint4 d0q = ldg_nc(dout + t * H + 16 * b), d1q = ldg_nc(dout + t * H + 16 * b + 8);
          const uint32_t dw8[8] = {d0q.x, d0q.y, d0q.z, d0q.w, d1q.x, d1q.y, d1q.z, d1q.w};
          const uint32_t yw8[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
          float lo8[8], hi8[8];
#pragma unroll
          for (int p = 0; p < 8; ++p) {
            const float d0 = __uint_as_float(dw8[p] << 16), d1 = __uint_as_float(dw8[p] & 0xFFFF0000u);
            const float y0f = __uint_as_float(yw8[p] << 16), y1f = __uint_as_float(yw8[p] & 0xFFFF0000u);
            o[p] = bf16x2_of_products(wj, d0, d1);
            acc = __fmaf_rn(d0, y0f, acc);
            acc = __fmaf_rn(d1, y1f, acc);
            float* dst = p < 4 ? lo8 : hi8;
            dst[2 * (p & 3)] = __uint_as_float(o[p] << 16);
            dst[2 * (p & 3) + 1] = __uint_as_float(o[p] & 0xFFFF0000u);
          }
          uint4* dyp = reinterpret_cast<uint4*>(dy + (int64_t)slot * H + 16 * b);
          dyp[0] = make_uint4(o[0], o[1], o[2], o[3]);
          dyp[1] = make_uint4(o[4], o[5], o[6], o[7]);
          const uint4 ow0 = make_uint4(o[0], o[1], o[2], o[3]), ow1 = make_uint4(o[4], o[5], o[6], o[7]);
          const BlockScale bs = block_scale(absmax16_bf16(ow0, ow1), g, six_g);
          const uint64_t jc = (uint64_t)(slot * H + 16 * b) / 8u;
          cw.x = e2m1x8_sr(lo8, ow0, bs, philox4x32_10(make_uint4((uint32_t)jc, (uint32_t)(jc >> 32), 0u, 0u), k0, k1));
          cw.y = e2m1x8_sr(hi8, ow1, bs,
                           philox4x32_10(make_uint4((uint32_t)(jc + 1), (uint32_t)((jc + 1) >> 32), 0u, 0u), k0, k1));
          sfb = bs.sf;
        }
        const uint32_t s1 = __shfl_down_sync(kAll, sfb, 1);
        const uint32_t s2 = __shfl_down_sync(kAll, sfb, 2);
        const uint32_t s3 = __shfl_down_sync(kAll, sfb, 3);
        if (active) {
          *reinterpret_cast<uint2*>(rcodes + (b >> 4) * tiled_block_bytes(128) + ((((b >> 1) & 7) ^ (rr & 7)) << 4) +
                                    (b & 1) * 8) = cw;
          const int wd = b >> 2;
          if ((lane & 3) == 0)
            *reinterpret_cast<uint32_t*>(rsf + (wd >> 2) * tiled_block_bytes(128) + (wd & 3) * 512) =
                sfb | (s1 << 8) | (s2 << 16) | (s3 << 24);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(kAll, acc, o));
      if (lane == 0) {
        dw[t * k + j] = acc;
        g_dy[slot] = g;
        if (amax_bits != nullptr && mb != 0u) atomicMax(amax_bits + find_group(starts, E, slot), mb);
      }
    }
  }
}

cudaError_t launch_combine_backward(const void* dout, const int32_t* inv, const float* w, const void* y, int64_t T,
                                    int k, int64_t H, void* dy, float* dw, const int32_t* starts, int E,
                                    uint32_t* amax_bits, uint8_t* dyq, float* g_dy, uint64_t key, cudaStream_t s) {
  if (H % 256 != 0 || H > 2048) return cudaErrorInvalidValue;
  if (amax_bits != nullptr) {
    const cudaError_t err = cudaMemsetAsync(amax_bits, 0, sizeof(uint32_t) * E, s);
    if (err != cudaSuccess) return err;
  }
  if (T == 0) return cudaSuccess;
  int64_t blocks = (T + 7) / 8;
  if (blocks > 16 * (int64_t)num_sms()) blocks = 16 * (int64_t)num_sms();
  combine_backward_kernel<<<(int)blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(dout), inv, w,
                                                      static_cast<const __nv_bfloat16*>(y), T, k, H,
                                                      static_cast<__nv_bfloat16*>(dy), dw, starts, E, amax_bits,
                                                      dyq, g_dy, key);
  return cudaGetLastError();
}

// amax_bits[e] = max |src[row(r), 0..F)| over the rows r of expert e's group (slots
// starts[e] .. starts[e] + counts[e] - 1), row(r) = rowmap[r] or r; float bits combined
// with atomicMax (order-free for non-negative floats).  One warp per slot row.  amax_bits
// must be zeroed first.
__global__ void __launch_bounds__(256) group_amax_kernel(const __nv_bfloat16* __restrict__ src, int64_t ld, int64_t F,
                                                         const int32_t* __restrict__ rowmap,
                                                         const int32_t* __restrict__ starts,
                                                         const int32_t* __restrict__ counts, int E, int64_t max_rows,
                                                         uint32_t* __restrict__ amax_bits) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t nwarp = (int64_t)gridDim.x * 8;
  int64_t rows = starts[E];
  if (rows > max_rows) rows = max_rows;
  for (int64_t r = warp; r < rows; r += nwarp) {
    const int e = find_group(starts, E, (int32_t)r);
    if (r - starts[e] >= counts[e]) continue;               // group padding (warp-uniform)
    const int64_t sr = rowmap != nullptr ? rowmap[r] : r;
    uint32_t m = 0;
    for (int64_t c = 8 * lane; c < F; c += 256) {
      const uint4 q = ldg_nc(src + sr * ld + c);
      const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) asm("max.u16x2 %0, %0, %1;" : "+r"(m) : "r"(wv[i] & 0x7FFF7FFFu));
    }
    uint32_t mb = max(m & 0xFFFFu, m >> 16) << 16;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mb = max(mb, __shfl_xor_sync(kAll, mb, o));
    if (lane == 0 && mb != 0u) atomicMax(amax_bits + e, mb);
  }
}

cudaError_t launch_group_amax(const void* src, int64_t ld, int64_t F, const int32_t* rowmap, const int32_t* starts,
                              const int32_t* counts, int E, int64_t max_rows, uint32_t* amax_bits, cudaStream_t s) {
  cudaError_t err = cudaMemsetAsync(amax_bits, 0, sizeof(uint32_t) * E, s);
  if (err != cudaSuccess || max_rows == 0) return err;
  int64_t blocks = (max_rows + 7) / 8;
  if (blocks > 8 * (int64_t)num_sms()) blocks = 8 * (int64_t)num_sms();
  group_amax_kernel<<<(int)blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(src), ld, F, rowmap, starts, counts,
                                                E, max_rows, amax_bits);
  return cudaGetLastError();
}

// amax_bits[e] = max |src[row(r), 0..F)| over the rows r of expert e's group, as
// group_amax_kernel, for rows that already carry a per-row global scale g_rows[r] =
// fl32(amax_r / 2688) (the forward's per-token and per-row scales, the backward's dD rows):
// amax_r is a BF16 value, and where g_rows[r] is a normal float32 (>= 2^-125), g * 2688 is
// within 2^-23 (relative) of it, so rounding that product to BF16 gives amax_r exactly;
// smaller non-zero scales (rows whose max is below about 2^-113) read the row.  One thread
// per row, the warp's rows combined per expert before one atomicMax each.  amax_bits must
// be zeroed first.
__global__ void __launch_bounds__(256) group_amax_g_kernel(const float* __restrict__ g_rows,
                                                           const __nv_bfloat16* __restrict__ src, int64_t ld,
                                                           int64_t F, const int32_t* __restrict__ rowmap,
                                                           const int32_t* __restrict__ starts,
                                                           const int32_t* __restrict__ counts, int E,
                                                           int64_t max_rows, uint32_t* __restrict__ amax_bits) {
  int64_t rows = starts[E];
  if (rows > max_rows) rows = max_rows;
  const int lane = threadIdx.x & 31;
  for (int64_t base = (int64_t)blockIdx.x * blockDim.x; base < rows; base += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = base + threadIdx.x;   // the loop is uniform over the block (votes below)
    int e = -1;
    uint32_t v = 0;
    if (r < rows) {
      e = find_group(starts, E, (int32_t)r);
      if (r - starts[e] < counts[e]) {
        const float g = g_rows[r];
        if (g >= 0x1p-125f) {
          const uint32_t b = __float_as_uint(__fmul_rn(g, 2688.0f));
          v = ((b + 0x7FFFu + ((b >> 16) & 1u)) >> 16) << 16;
        } else if (g > 0.0f) {
          const int64_t sr = rowmap != nullptr ? rowmap[r] : r;
          const uint16_t* q = reinterpret_cast<const uint16_t*>(src + sr * ld);
          uint32_t m = 0;
          for (int64_t c = 0; c < F; ++c) m = max(m, (uint32_t)(q[c] & 0x7FFFu));
          v = m << 16;
        }
      } else {
        e = -1;   // group padding
      }
    }
    const unsigned same = __match_any_sync(kAll, e);
    const uint32_t m = __reduce_max_sync(same, v);
    if (e >= 0 && m != 0u && lane == __ffs((int)same) - 1) atomicMax(amax_bits + e, m);
  }
}

cudaError_t launch_group_amax_g(const float* g_rows, const void* src, int64_t ld, int64_t F, const int32_t* rowmap,
                                const int32_t* starts, const int32_t* counts, int E, int64_t max_rows,
                                uint32_t* amax_bits, cudaStream_t s) {
  cudaError_t err = cudaMemsetAsync(amax_bits, 0, sizeof(uint32_t) * E, s);
  if (err != cudaSuccess || max_rows == 0) return err;
  int64_t blocks = (max_rows + 255) / 256;
  if (blocks > 2 * (int64_t)num_sms()) blocks = 2 * (int64_t)num_sms();
  group_amax_g_kernel<<<(int)blocks, 256, 0, s>>>(g_rows, static_cast<const __nv_bfloat16*>(src), ld, F, rowmap,
                                                  starts, counts, E, max_rows, amax_bits);
  return cudaGetLastError();
}

// kofs[e] = sum over e' < e of max(1, ceil(counts[e'] / 256)) (counts == nullptr: every
// group has `uniform` rows): the first 256-token K-block of each expert in the wgrad
// operands.  One block of 1024 threads.
__global__ void __launch_bounds__(1024) kofs_kernel(const int32_t* __restrict__ counts, int64_t uniform, int E,
                                                    int32_t* __restrict__ kofs) {
  __shared__ int32_t part[1024];
  const int per = (E + 1023) / 1024;
  const int e0 = threadIdx.x * per, e1 = min(E, e0 + per);
  int32_t local = 0;
  for (int e = e0; e < e1; ++e) {
    const int64_t n = counts != nullptr ? counts[e] : uniform;
    local += (int32_t)max((int64_t)1, (n + 255) / 256);
  }
  part[threadIdx.x] = local;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {   // inclusive scan
    const int32_t v = threadIdx.x >= o ? part[threadIdx.x - o] : 0;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  int32_t run = part[threadIdx.x] - local;
  for (int e = e0; e < e1; ++e) {
    kofs[e] = run;
    const int64_t n = counts != nullptr ? counts[e] : uniform;
    run += (int32_t)max((int64_t)1, (n + 255) / 256);
  }
  if (threadIdx.x == 1023) kofs[E] = part[1023];
}

cudaError_t launch_kofs(const int32_t* counts, int64_t uniform, int E, int32_t* kofs, cudaStream_t s) {
  kofs_kernel<<<1, 1024, 0, s>>>(counts, uniform, E, kofs);
  return cudaGetLastError();
}

// Per-expert transposed NVFP4 into the GEMM-tiled layout.  For expert e, the source rows
// are the expert's "tokens" t = 0 .. count_e - 1 (src row rowmap[start_e + t] or
// start_e + t; uniform groups: e * uniform + t) and the columns its features f < F; the
// quantised matrix is the transpose [Fp, tp_e] (tp_e = 256 * (kofs[e+1] - kofs[e]) tokens,
// zero beyond count_e; rows F .. Fp - 1 zero), blocks of 16 along the tokens, one global
// scale g_e = amax_e / 2688 for the matrix, RNE or stochastic rounding with key
// seed + (((stream << 10) + e) << 40) and element index f * tp_e + t.  Output: R-row
// blocks (128 or 256) by 256-token K-blocks; expert e's blocks start at block
// (Fp / R) * kofs[e], row-block-major.
//
// One CTA per (expert, 128 output rows, K-block) unit, two CTAs per SM: the 256 x 128 BF16
// source tile goes into shared memory with 16-byte asynchronous copies, each thread
// encodes pairs of features (4-byte column reads, conflict-free across a warp) for one
// 16-token block at a time, writes codes and scale bytes into the unit's 18 KB image (the
// 128-row block of the layout), and bulk stores write it: whole for R = 128, as the codes
// (16 KB) and scale (2 KB) halves of a 256-row block for R = 256.
struct TQuant {
  const __nv_bfloat16* src;
  int64_t ld;
  const int32_t* rowmap;     // nullable
  const int32_t* starts;     // nullable: uniform groups
  const int32_t* counts;     // nullable: uniform groups
  int64_t uniform;
  const int32_t* kofs;       // [E+1]
  int E, F, Fp, R;
  const uint32_t* amax_bits; // [E]
  float* g_out;              // [E]
  uint8_t* out;
  uint64_t seed;
  int stream;
};

constexpr int kTQRows = 128;                                  // output rows per unit
constexpr int kTQSmem = 256 * kTQRows * 2 + kTQRows * 144 + 256 * 8;   // source tile + image + rows

template <int RND>
__global__ void __launch_bounds__(256) tquant_kernel(const TQuant q) {
  extern __shared__ __align__(128) uint8_t tsm[];
  constexpr int R = kTQRows;
  uint8_t* tile = tsm;                                        // [256 tokens][128 features] BF16
  uint8_t* img = tsm + 256 * R * 2;                           // the unit's 18 KB image
  int64_t* srow = reinterpret_cast<int64_t*>(img + R * 144);  // source row of each tile token
  const uint32_t tile_s = smem_u32(tile);
  const int tid = threadIdx.x;
  const int rblocks = q.Fp / R;
  const int64_t units = (int64_t)q.kofs[q.E] * rblocks;
  for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
    const int32_t kg = (int32_t)(u / rblocks);
    const int rb = (int)(u - (int64_t)kg * rblocks);
    const int e = find_group(q.kofs, q.E, kg);
    const int kb = kg - q.kofs[e];
    const int64_t kbe = q.kofs[e + 1] - q.kofs[e];
    const int64_t tp = 256 * kbe;
    const int64_t start = q.starts != nullptr ? q.starts[e] : (int64_t)e * q.uniform;
    const int64_t count = q.counts != nullptr ? q.counts[e] : q.uniform;
    const int f0 = rb * R;
    // 1. the source tile: tokens kb*256 .. +255 of the expert, features f0 .. f0+127; the
    //    tile's 256 source rows are looked up once (one per thread) before the copies
    {
      const int64_t tok = (int64_t)kb * 256 + tid;
      const int64_t r = start + tok;
      srow[tid] = tok < count ? (q.rowmap != nullptr ? (int64_t)q.rowmap[r] : r) : -1;
    }
    __syncthreads();
    constexpr int kChunksPerRow = R * 2 / 16;
    for (int i = tid; i < 256 * kChunksPerRow; i += 256) {
      const int t = i / kChunksPerRow, ch = i - t * kChunksPerRow;
      const int f = f0 + ch * 8;
      const uint32_t dst = tile_s + (uint32_t)(t * R * 2 + ch * 16);
      const int64_t sr = srow[t];
      if (sr >= 0 && f < q.F) {
        cp_async_16(dst, q.src + sr * q.ld + f);
      } else {
        *reinterpret_cast<uint4*>(tile + t * R * 2 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    cp_async_wait_all();
    __syncthreads();
    // 2. encode: feature pair (2p, 2p+1) of the unit, 16-token block b
    const float g = __fdiv_rn(__uint_as_float(q.amax_bits[e]), kGlobalDivisor);
    const float six_g = __fmul_rn(6.0f, g);
    if (tid == 0 && kb == 0 && rb == 0) q.g_out[e] = g;
    const uint64_t key = q.seed + ((((uint64_t)q.stream << 10) + (uint64_t)e) << 40);
    for (int i = tid; i < (R / 2) * 16; i += 256) {
      const int p = i % (R / 2), b = i / (R / 2);
      float v[2][16];
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        const uint32_t pr = *reinterpret_cast<const uint32_t*>(tile + (b * 16 + t) * R * 2 + p * 4);
        v[0][t] = __uint_as_float(pr << 16);
        v[1][t] = __uint_as_float(pr & 0xFFFF0000u);
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int rr = 2 * p + h;                          // row of the image
        float am = 0.0f;
#pragma unroll
        for (int t = 0; t < 16; ++t) am = fmaxf(am, fabsf(v[h][t]));
        const BlockScale bs = block_scale(am, g, six_g);
        float lo8[8], hi8[8];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          lo8[t] = v[h][t];
          hi8[t] = v[h][8 + t];
        }
        uint2 cw;
        if (RND == kRoundSR) {
          const uint64_t j = ((uint64_t)(f0 + rr) * (uint64_t)tp + (uint64_t)kb * 256 + (uint64_t)b * 16) / 8u;
          const uint32_t k0 = (uint32_t)key, k1 = (uint32_t)(key >> 32);
          cw.x = e2m1x8_sr(lo8, bs, philox4x32_10(make_uint4((uint32_t)j, (uint32_t)(j >> 32), 0u, 0u), k0, k1));
          cw.y = e2m1x8_sr(hi8, bs, philox4x32_10(make_uint4((uint32_t)(j + 1), (uint32_t)((j + 1) >> 32), 0u, 0u),
                                                  k0, k1));
        } else {
          cw = e2m1x16_rn(lo8, hi8, bs);
        }
        // codes: K-byte 8b of row rr, 128-byte swizzled; scale (rr, b)
        *reinterpret_cast<uint2*>(img + rr * 128 + ((((b >> 1) ^ (rr & 7))) << 4) + (b & 1) * 8) = cw;
        img[R * 128 + (b >> 2) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + (b & 3)] = (uint8_t)bs.sf;
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      if (q.R == 128) {
        bulk_store(q.out + ((int64_t)rblocks * q.kofs[e] + (int64_t)rb * kbe + kb) * (128 * 144), img, 128 * 144);
      } else {   // one half of a 256-row block: its codes and its row group of scales
        const int64_t blk = (int64_t)(rblocks / 2) * q.kofs[e] + (int64_t)(rb >> 1) * kbe + kb;
        uint8_t* base = q.out + blk * (256 * 144);
        bulk_store(base + (rb & 1) * (128 * 128), img, 128 * 128);
        bulk_store(base + 256 * 128 + (rb & 1) * 2048, img + 128 * 128, 2048);
      }
      bulk_commit();
      bulk_wait_read<0>();     // the image is read before the next unit overwrites it
    }
    __syncthreads();
  }
  if (tid == 0) bulk_wait_all<0>();
}

template <int RND>
static cudaError_t launch_tq(const TQuant& q, int64_t max_units, cudaStream_t s) {
  static std::atomic<bool> attr_set[64];
  const cudaError_t err = set_smem_attr_once(attr_set, (const void*)tquant_kernel<RND>, kTQSmem);
  if (err != cudaSuccess) return err;
  int64_t grid = max_units;
  if (grid > 2 * (int64_t)num_sms()) grid = 2 * (int64_t)num_sms();
  if (grid < 1) grid = 1;
  tquant_kernel<RND><<<(int)grid, 256, kTQSmem, s>>>(q);
  return cudaGetLastError();
}

// max_kblocks: an upper bound on kofs[E] (the grid is sized from it; the kernel reads the
// exact count on the device).  R: 128 or 256 (the output layout's row blocks); Fp % R == 0.
cudaError_t launch_tquant(const void* src, int64_t ld, const int32_t* rowmap, const int32_t* starts,
                          const int32_t* counts, int64_t uniform, const int32_t* kofs, int E, int F, int Fp, int R,
                          const uint32_t* amax_bits, float* g_out, uint8_t* out, int rounding, uint64_t seed,
                          int stream_id, int64_t max_kblocks, cudaStream_t s) {
  if ((R != 128 && R != 256) || Fp % R != 0) return cudaErrorInvalidValue;
  TQuant q;
  q.src = static_cast<const __nv_bfloat16*>(src);
  q.ld = ld;
  q.rowmap = rowmap;
  q.starts = starts;
  q.counts = counts;
  q.uniform = uniform;
  q.kofs = kofs;
  q.E = E;
  q.F = F;
  q.Fp = Fp;
  q.R = R;
  q.amax_bits = amax_bits;
  q.g_out = g_out;
  q.out = out;
  q.seed = seed;
  q.stream = stream_id;
  const int64_t units = max_kblocks * (Fp / kTQRows);
  return rounding == kRoundSR ? launch_tq<kRoundSR>(q, units, s) : launch_tq<kRoundRNE>(q, units, s);
}

}  // namespace nvfp4

// NVFP4 -> BF16 / float32: DQ(Q(x)) = value(code) * decode(block scale) * global scale,
// the operand of the dequantised backward ("The 4-bitter Lesson: Balancing Stability and
// Performance in NVFP4 RL", §"Improving Gradient Stability", footnote 6: Q and DQ).
//
// The exact value has at most 2 + 4 + 24 significant bits: value(code) * decode(sf) is
// exact in float32, and the product with g is formed exactly as a float-float (product
// and its fma remainder), then rounded once to the output type: float32 by the product
// itself, BF16 by round-to-nearest-even of the product with the remainder breaking a tie
// at a BF16 midpoint.  Magnitudes below 2^-100 (where the remainder could underflow) take
// a float64 path.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "launch.h"
#include "swiglu.cuh"

namespace nvfp4 {

// value(code) * 2^-126: the code's 3 magnitude bits placed at float32 bits 22..24 (the
// exponent's low bits and the top mantissa bit) with its sign at bit 31 -- the E2M1
// subnormal 0.5 becomes the float32 subnormal 2^-127 -- so value(code) is this times
// 2^126, exactly.
__device__ __forceinline__ float e2m1_scaled(uint32_t code) {
  return __uint_as_float(((code & 7u) << 22) | ((code & 8u) << 28));
}

__device__ __forceinline__ float e4m3_value(uint32_t b) {
  const uint32_t e = (b >> 3) & 0xFu, m = b & 7u;
  return e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : __fmul_rn((float)m, 0.001953125f);
}

// BF16 rounding of the exact product p = a * g (a exact in float32).
__device__ __forceinline__ uint32_t dq_bf16_bits(float a, float g) {
  const float hi = __fmul_rn(a, g);
  if (hi == 0.0f) return __float_as_uint(hi) >> 16;            // exact zero (keeps its sign)
  const float ahi = fabsf(hi);
  if (!(ahi >= 0x1p-100f) || !(ahi <= 3.0e38f)) return f64_to_bf16_bits((double)a * (double)g);
  const float lo = __fmaf_rn(a, g, -hi);
  const uint32_t b = __float_as_uint(hi);
  if ((b & 0xFFFFu) != 0x8000u || lo == 0.0f) return f32_to_bf16_rne_bits(b);
  return ((lo > 0.0f) == (hi > 0.0f)) ? (b >> 16) + 1u : (b >> 16);
}

// One thread per 8 values (4 code bytes) of a row: 8 BF16 (16 bytes) or float32 (32
// bytes) out.  Each thread takes four such units per iteration and issues their loads
// (codes, scale byte, global scale) before any arithmetic.  Idx is the unit index type
// (32-bit when every index fits).
template <bool kF32, typename Idx>
__global__ void __launch_bounds__(256) dequantize_kernel(const uint8_t* __restrict__ codes,
                                                         const uint8_t* __restrict__ sf,
                                                         const float* __restrict__ g, int64_t rows, int64_t cols,
                                                         int mode, int64_t group_rows, void* __restrict__ out,
                                                         int64_t ldo) {
  constexpr int kU = 4;
  const int64_t chunks = cols / 8, total = rows * chunks, sf_words = (cols / 16 + 3) / 4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += kU * stride) {
    uint32_t word[kU], sfb[kU];
    float gs[kU];
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const int64_t i = i0 + j * stride;
      word[j] = 0u;
      sfb[j] = 0u;
      gs[j] = 0.0f;
      if (i < total) {
        const int64_t r = (int64_t)((Idx)i / (Idx)chunks), c8 = i - r * chunks, blk = c8 / 2;
        word[j] = __ldcs(reinterpret_cast<const uint32_t*>(codes + r * (cols / 2) + 4 * c8));
        sfb[j] = sf[((r >> 7) * sf_words + blk / 4) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (blk & 3)];
        gs[j] = g[mode == kScopeTensor ? 0 : (mode == kScopeRow ? r : (int64_t)((Idx)r / (Idx)group_rows))];
      }
    }
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const int64_t i = i0 + j * stride;
      if (i >= total) continue;
      const int64_t r = (int64_t)((Idx)i / (Idx)chunks), c8 = i - r * chunks;
      const float s = e4m3_value(sfb[j]);
      // value(code) * s, exact: (value * 2^-126) * s has at most 6 significant bits and stays
      // above 2^-142, and the power of two restores the value
      if (kF32) {
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          v[e] = __fmul_rn(__fmul_rn(__fmul_rn(e2m1_scaled(word[j] >> (4 * e)), s), 0x1p126f), gs[j]);
        float* o = static_cast<float*>(out) + r * ldo + 8 * c8;
        __stcs(reinterpret_cast<float4*>(o), make_float4(v[0], v[1], v[2], v[3]));
        __stcs(reinterpret_cast<float4*>(o + 4), make_float4(v[4], v[5], v[6], v[7]));
      } else {
        uint32_t h[8];
#pragma unroll
        for (int e = 0; e < 8; ++e)
          h[e] = dq_bf16_bits(__fmul_rn(__fmul_rn(e2m1_scaled(word[j] >> (4 * e)), s), 0x1p126f), gs[j]);
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out) + r * ldo + 8 * c8;
        __stcs(reinterpret_cast<uint4*>(o),
               make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16)));
      }
    }
  }
}

// BF16 output, one thread per 16-value block (8 code bytes, 1 scale byte).  The block's
// 8 magnitudes v * s * g (v = 0, 0.5, 1, 1.5, 2, 3, 4, 6) take 8 BF16 values: P = BF16(s g)
// and Q = BF16(1.5 s g) are rounded once each (dq_bf16_bits), and the others are P and Q
// times a power of two -- exact while every one of them stays a normal BF16 value, since
// scaling by a power of two commutes with the rounding there; otherwise each of the 7 is
// rounded on its own.  The 8 values sit as a byte table (low bytes, high bytes), and four
// codes at a time become four BF16 values by byte permutes indexed by their magnitude
// bits, the sign bit ORed in (a zero keeps the code's sign, as the exact product does).
template <typename Idx>
__global__ void __launch_bounds__(256) dequantize_bf16_kernel(const uint8_t* __restrict__ codes,
                                                              const uint8_t* __restrict__ sf,
                                                              const float* __restrict__ g, int64_t rows,
                                                              int64_t cols, int mode, int64_t group_rows,
                                                              __nv_bfloat16* __restrict__ out, int64_t ldo) {
  const Idx bpr = (Idx)(cols / 16);
  const int64_t total = rows * (int64_t)bpr, sf_words = (cols / 16 + 3) / 4;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += stride) {
    const Idx r = (Idx)i / bpr, b = (Idx)i - r * bpr;
    const uint2 cw = __ldcs(reinterpret_cast<const uint2*>(codes + (int64_t)r * (cols / 2) + 8 * (int64_t)b));
    const uint32_t sfb = sf[(((int64_t)r >> 7) * sf_words + b / 4) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (b & 3)];
    const float gs = g[mode == kScopeTensor ? 0 : (mode == kScopeRow ? (int64_t)r : (int64_t)r / group_rows)];
    const float s = e4m3_value(sfb);
    const uint32_t P = dq_bf16_bits(s, gs), Q = dq_bf16_bits(__fmul_rn(1.5f, s), gs);
    const uint32_t eP = (P >> 7) & 0xFFu, eQ = (Q >> 7) & 0xFFu;
    uint32_t t[8];
    t[0] = 0u;
    if (eP - 2u <= 250u && eQ - 1u <= 251u) {   // P/2 .. 4P and Q .. 4Q all normal BF16 values
      t[1] = P - 0x80u;
      t[2] = P;
      t[3] = Q;
      t[4] = P + 0x80u;
      t[5] = Q + 0x80u;
      t[6] = P + 0x100u;
      t[7] = Q + 0x100u;
    } else {
#pragma unroll
      for (int m = 1; m < 8; ++m)
        t[m] = dq_bf16_bits(__fmul_rn(__fmul_rn(e2m1_scaled((uint32_t)m), s), 0x1p126f), gs);
    }
    const uint32_t w0 = t[0] | (t[1] << 16), w1 = t[2] | (t[3] << 16), w2 = t[4] | (t[5] << 16),
                   w3 = t[6] | (t[7] << 16);
    const uint32_t lo0 = __byte_perm(w0, w1, 0x6420), lo1 = __byte_perm(w2, w3, 0x6420);   // low bytes of t[0..7]
    const uint32_t hi0 = __byte_perm(w0, w1, 0x7531), hi1 = __byte_perm(w2, w3, 0x7531);   // high bytes
    uint32_t o[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t c4 = ((q < 2 ? cw.x : cw.y) >> (16 * (q & 1))) & 0xFFFFu;   // codes 4q .. 4q+3
      const uint32_t sel = c4 & 0x7777u;                                         // their magnitudes
      const uint32_t lo = __byte_perm(lo0, lo1, sel), hi = __byte_perm(hi0, hi1, sel);
      o[2 * q] = __byte_perm(lo, hi, 0x5140) | ((c4 << 12) & 0x8000u) | ((c4 << 24) & 0x80000000u);
      o[2 * q + 1] = __byte_perm(lo, hi, 0x7362) | ((c4 << 4) & 0x8000u) | ((c4 << 16) & 0x80000000u);
    }
    __nv_bfloat16* op = out + (int64_t)r * ldo + 16 * (int64_t)b;
    __stcs(reinterpret_cast<uint4*>(op), make_uint4(o[0], o[1], o[2], o[3]));
    __stcs(reinterpret_cast<uint4*>(op + 8), make_uint4(o[4], o[5], o[6], o[7]));
  }
}

cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* sf, const float* g, int64_t rows, int64_t cols,
                              int mode, int64_t group_rows, void* out, bool out_f32, int64_t ldo, cudaStream_t s) {
  const int64_t total = rows * (cols / 8);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 1023) / 1024;   // 4 units per thread and iteration
  if (blocks > 64 * (int64_t)num_sms()) blocks = 64 * (int64_t)num_sms();
  const bool i32 = total < ((int64_t)1 << 32);
  if (out_f32 && i32)
    dequantize_kernel<true, uint32_t><<<(int)blocks, 256, 0, s>>>(codes, sf, g, rows, cols, mode, group_rows, out, ldo);
  else if (out_f32)
    dequantize_kernel<true, int64_t><<<(int)blocks, 256, 0, s>>>(codes, sf, g, rows, cols, mode, group_rows, out, ldo);
  else {
    const int64_t nblk = rows * (cols / 16);
    int64_t bb = (nblk + 255) / 256;
    if (bb > 16 * (int64_t)num_sms()) bb = 16 * (int64_t)num_sms();
    auto* o = static_cast<__nv_bfloat16*>(out);
    if (nblk < ((int64_t)1 << 32) && rows < ((int64_t)1 << 31))
      dequantize_bf16_kernel<uint32_t><<<(int)bb, 256, 0, s>>>(codes, sf, g, rows, cols, mode, group_rows, o, ldo);
    else
      dequantize_bf16_kernel<int64_t><<<(int)bb, 256, 0, s>>>(codes, sf, g, rows, cols, mode, group_rows, o, ldo);
  }
  return cudaGetLastError();
}

}  // namespace nvfp4

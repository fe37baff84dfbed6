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
  else if (i32)
    dequantize_kernel<false, uint32_t><<<(int)blocks, 256, 0, s>>>(codes, sf, g, rows, cols, mode, group_rows, out,
                                                                   ldo);
  else
    dequantize_kernel<false, int64_t><<<(int)blocks, 256, 0, s>>>(codes, sf, g, rows, cols, mode, group_rows, out,
                                                                  ldo);
  return cudaGetLastError();
}

}  // namespace nvfp4

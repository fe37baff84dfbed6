// MXFP8 quantiser and dequantiser: the format of the recipe's MXFP8 validation runs
// ("The 4-bitter Lesson: Balancing Stability and Performance in NVFP4 RL",
// §"Improving Gradient Stability", "Results Validation with MXFP8": quantised forward
// and backward, and quantised forward with a dequantised backward).  The pages name the
// format without defining it.  It is read as OCP MX v1.0 MXFP8:
//   * blocks of 32 values along a row;
//   * an E8M0 block scale b = max(floor(log2 amax) - 8 + 127, 0), so that 2^(b-127)
//     maps the block's amax into [256, 512);
//   * E4M3 elements x * 2^(127-b), rounded to nearest even with satfinite;
//   * a zero magnitude encoded as +0.
//
// For BF16 input, floor(log2 amax) + 127 is the exponent field of amax.  Subnormals
// and zero have field 0 and give b = 0.  So b = max(field(amax) - 8, 0).  The multiplier
// 2^(127-b) is a normal float32, and x * 2^(127-b) is exact wherever it can round to a
// non-zero E4M3 value.  E4M3 rounding is therefore the only rounding.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "launch.h"

namespace nvfp4 {

// One thread per 8 values (16 bytes of BF16); 4 threads per 32-value block; 16 threads
// per 4-block group, whose scale bytes form one 32-bit word of the 128x4 tiled layout.
// Rows rows..rows_pad-1 of the tile grid get zero scale words and no codes.
// A warp takes kSlabs 32-unit slabs (512 bytes of x each) per iteration, loads all of
// them, then encodes them, so that each thread keeps kSlabs 16-byte loads in flight.
__device__ __forceinline__ void mx_encode_unit(uint4 v, int lane, bool store, int64_t r, int64_t c8, int64_t cols,
                                               uint8_t* __restrict__ codes, uint8_t* __restrict__ sf) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  // amax as BF16 magnitude bits (finite inputs: integer order = magnitude order)
  uint32_t m = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) m = max(m, max(w[i] & 0x7FFFu, (w[i] >> 16) & 0x7FFFu));
  m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
  m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
  const uint32_t field = m >> 7;
  const uint32_t b = field > 8u ? field - 8u : 0u;                  // E8M0 byte, 0..246
  const float mult = __uint_as_float((254u - b) << 23);             // 2^(127 - b)
  uint32_t q[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint16_t p[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t pair = w[2 * h + i];
      const float lo = __fmul_rn(__uint_as_float(pair << 16), mult);
      const float hi = __fmul_rn(__uint_as_float(pair & 0xFFFF0000u), mult);
      asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(p[i]) : "f"(hi), "f"(lo));
    }
    const uint32_t c = (uint32_t)p[0] | ((uint32_t)p[1] << 16);
    // zero magnitudes as +0: keep a byte's sign bit only where its magnitude is non-zero
    const uint32_t mag = c & 0x7F7F7F7Fu;
    const uint32_t nz = (mag + 0x7F7F7F7Fu) & 0x80808080u;
    q[h] = mag | (c & nz);
  }
  if (store && r >= 0) *reinterpret_cast<uint2*>(codes + r * cols + 8 * c8) = make_uint2(q[0], q[1]);
  // scale word of this lane's 4-block group: bytes from lanes g, g+4, g+8, g+12
  const int g0 = lane & 16;
  uint32_t word = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) word |= __shfl_sync(0xFFFFFFFFu, b, g0 + 4 * j) << (8 * j);
  if (store && (lane & 15) == 0) {
    const int64_t rr = r >= 0 ? r : -r - 1;
    *reinterpret_cast<uint32_t*>(sf + ((rr >> 7) * (cols / 128) + c8 / 16) * 512 + (rr & 31) * 16 +
                                 ((rr >> 5) & 3) * 4) = word;
  }
}

// Idx: the type of the unit index (32-bit when every index fits, which keeps the
// per-unit row / column division short).
template <typename Idx>
__global__ void __launch_bounds__(256) mx_quantize_kernel(const __nv_bfloat16* __restrict__ x, int64_t rows,
                                                          int64_t cols, int64_t ld, int64_t rows_pad,
                                                          uint8_t* __restrict__ codes, uint8_t* __restrict__ sf) {
  const int lane = threadIdx.x & 31;
  const int64_t chunks = cols / 8, total = rows_pad * chunks;
  const int64_t warp0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t wstride = ((int64_t)gridDim.x * blockDim.x) >> 5;
  // Every lane of a warp runs every iteration (the shuffles take all 32 lanes); lanes
  // past the end compute on zeros and store nothing.
  constexpr int kSlabs = 4;
  for (int64_t base = warp0 * 32 * kSlabs; base < total; base += wstride * 32 * kSlabs) {
    uint4 v[kSlabs];
    int64_t r[kSlabs], c8[kSlabs];
    bool live[kSlabs];
#pragma unroll
    for (int s2 = 0; s2 < kSlabs; ++s2) {
      const int64_t u = base + 32 * s2 + lane;
      live[s2] = u < total;
      const Idx q = live[s2] ? (Idx)u / (Idx)chunks : (Idx)0;
      r[s2] = (int64_t)q;
      c8[s2] = live[s2] ? (int64_t)((Idx)u - q * (Idx)chunks) : 0;
      v[s2] = make_uint4(0u, 0u, 0u, 0u);
      if (live[s2] && r[s2] < rows) v[s2] = __ldcs(reinterpret_cast<const uint4*>(x + r[s2] * ld + 8 * c8[s2]));
    }
#pragma unroll
    for (int s2 = 0; s2 < kSlabs; ++s2)
      // padding rows are passed as -r-1: scale word only, no codes
      mx_encode_unit(v[s2], lane, live[s2], r[s2] < rows ? r[s2] : -r[s2] - 1, c8[s2], cols, codes, sf);
  }
}

// One thread per 8 values: 8 code bytes in, 8 BF16 (16 bytes) or float32 (32 bytes)
// out; each thread takes four such units per iteration, loads first.  value(code) *
// 2^(b-127) is exact in float32 (at most 4 significant bits, within [2^-136, 2^136)), so
// float32 output is exact and BF16 output is rounded once.
template <bool kF32, typename Idx>
__global__ void __launch_bounds__(256) mx_dequantize_kernel(const uint8_t* __restrict__ codes,
                                                            const uint8_t* __restrict__ sf, int64_t rows,
                                                            int64_t cols, void* __restrict__ out, int64_t ldo) {
  constexpr int kU = 4;
  const int64_t chunks = cols / 8, total = rows * chunks, tiles_per_row = cols / 128;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i0 < total; i0 += kU * stride) {
    uint2 cw[kU];
    uint32_t sb[kU];
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const int64_t i = i0 + j * stride;
      cw[j] = make_uint2(0u, 0u);
      sb[j] = 127u;
      if (i < total) {
        const int64_t r = (int64_t)((Idx)i / (Idx)chunks), c8 = i - r * chunks, blk = c8 / 4;
        cw[j] = __ldcs(reinterpret_cast<const uint2*>(codes + r * cols + 8 * c8));
        sb[j] = sf[((r >> 7) * tiles_per_row + blk / 4) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (blk & 3)];
      }
    }
#pragma unroll
    for (int j = 0; j < kU; ++j) {
      const int64_t i = i0 + j * stride;
      if (i >= total) continue;
      const int64_t r = (int64_t)((Idx)i / (Idx)chunks), c8 = i - r * chunks;
      const uint32_t b = sb[j];
      const float s = b == 0xFFu ? __int_as_float(0x7FC00000) : (b == 0u ? __uint_as_float(0x00400000u)
                                                                          : __uint_as_float(b << 23));
      // The 7 magnitude bits of an E4M3 code placed at float32 bits 20..26 give
      // value(code) * 2^-120 for normal and subnormal codes alike, so value(code) =
      // f * 2^120 exactly; times the block scale, exact as well (or Inf past the range).
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t c = ((e < 4 ? cw[j].x : cw[j].y) >> (8 * (e & 3))) & 0xFFu;
        const float f = __uint_as_float(((c & 0x7Fu) << 20) | ((c & 0x80u) << 24));
        const float val = (c & 0x7Fu) == 0x7Fu ? __int_as_float(0x7FC00000) : __fmul_rn(f, 0x1p120f);
        v[e] = __fmul_rn(val, s);
      }
      if (kF32) {
        float* o = static_cast<float*>(out) + r * ldo + 8 * c8;
        __stcs(reinterpret_cast<float4*>(o), make_float4(v[0], v[1], v[2], v[3]));
        __stcs(reinterpret_cast<float4*>(o + 4), make_float4(v[4], v[5], v[6], v[7]));
      } else {
        // one round-to-nearest-even conversion per pair (exact value in float32 -> BF16)
        uint32_t h[4];
#pragma unroll
        for (int p2 = 0; p2 < 4; ++p2) {
          const __nv_bfloat162 pr = __floats2bfloat162_rn(v[2 * p2], v[2 * p2 + 1]);
          h[p2] = *reinterpret_cast<const uint32_t*>(&pr);
        }
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out) + r * ldo + 8 * c8;
        __stcs(reinterpret_cast<uint4*>(o), make_uint4(h[0], h[1], h[2], h[3]));
      }
    }
  }
}

cudaError_t launch_mx_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* codes, uint8_t* sf,
                               cudaStream_t s) {
  const int64_t rows_pad = (rows + 127) / 128 * 128;
  const int64_t total = rows_pad * (cols / 8);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 1023) / 1024;               // 128 units per warp and iteration
  if (blocks > 64 * (int64_t)num_sms()) blocks = 64 * (int64_t)num_sms();
  if (total + 128 < ((int64_t)1 << 32))
    mx_quantize_kernel<uint32_t><<<(int)blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x), rows, cols, ld,
                                                             rows_pad, codes, sf);
  else
    mx_quantize_kernel<int64_t><<<(int)blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(x), rows, cols, ld,
                                                            rows_pad, codes, sf);
  return cudaGetLastError();
}

cudaError_t launch_mx_dequantize(const uint8_t* codes, const uint8_t* sf, int64_t rows, int64_t cols, void* out,
                                 bool out_f32, int64_t ldo, cudaStream_t s) {
  const int64_t total = rows * (cols / 8);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 1023) / 1024;               // 4 units per thread and iteration
  if (blocks > 64 * (int64_t)num_sms()) blocks = 64 * (int64_t)num_sms();
  // 32-bit unit indices when every index (including the unrolled look-ahead) fits
  const bool i32 = total + 4 * blocks * 256 < ((int64_t)1 << 32);
  if (out_f32 && i32)
    mx_dequantize_kernel<true, uint32_t><<<(int)blocks, 256, 0, s>>>(codes, sf, rows, cols, out, ldo);
  else if (out_f32)
    mx_dequantize_kernel<true, int64_t><<<(int)blocks, 256, 0, s>>>(codes, sf, rows, cols, out, ldo);
  else if (i32)
    mx_dequantize_kernel<false, uint32_t><<<(int)blocks, 256, 0, s>>>(codes, sf, rows, cols, out, ldo);
  else
    mx_dequantize_kernel<false, int64_t><<<(int)blocks, 256, 0, s>>>(codes, sf, rows, cols, out, ldo);
  return cudaGetLastError();
}

}  // namespace nvfp4

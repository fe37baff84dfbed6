// NVFP4 element and scale encoding on the device (sm_103a).
//
// Scale arithmetic ("The 4-bitter Lesson: Balancing Stability and Performance in NVFP4
// RL", §Baseline: E2M1 values, one E4M3 scale per 16 values, one FP32 global scale;
// footnote 6 of §"Improving Gradient Stability": Q = clip(round(x/s), qmin, qmax)),
// every step one IEEE float32 operation, round to nearest even, in this order:
//   g = amax / 2688;  sf = E4M3_rn_satfinite(amax_block / (6 g));  s = decode(sf) * g;
//   r = 1 / s;        code = E2M1(x * r)  (RNE, or stochastic rounding).
// All products / quotients use the explicit _rn intrinsics so that no FMA contraction or
// approximate division can change a bit.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

namespace nvfp4 {

constexpr float kGlobalDivisor = 2688.0f;   // 6 (E2M1 max) * 448 (E4M3 max)

// 8 BF16 values (one 16-byte load) -> float32
__device__ __forceinline__ void bf16x8_to_f32(const uint4& q, float (&f)[8]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ float absmax8(const float (&f)[8]) {
  float m = fabsf(f[0]);
#pragma unroll
  for (int i = 1; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
  return m;
}

// E4M3 byte -> float32 (exact; scales are non-negative so the sign bit is 0).
__device__ __forceinline__ float e4m3_decode(uint32_t b) {
  const uint32_t e = (b >> 3) & 0xFu, m = b & 7u;
  return e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : __fmul_rn((float)m, 0.001953125f);
}

// float32 (>= 0) -> E4M3 byte, round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t e4m3_encode(float t) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(0.0f), "f"(t));
  return d & 0xFFu;
}

struct BlockScale {
  uint32_t sf;  // E4M3 byte written to the scale tensor
  float r;      // encode multiplier 1/s, or 0 when the block decodes to zero
};

// Block scale of one 16-value block with max |x| = amax_b, given the scope's g and 6g.
__device__ __forceinline__ BlockScale block_scale(float amax_b, float g, float six_g) {
  BlockScale bs;
  if (!(g > 0.0f)) {
    bs.sf = 0;
    bs.r = 0.0f;
    return bs;
  }
  const float t = __fdiv_rn(amax_b, six_g);
  bs.sf = e4m3_encode(t);
  const float s = __fmul_rn(e4m3_decode(bs.sf), g);
  float r = 0.0f;
  if (s > 0.0f) {
    r = __frcp_rn(s);
    if (!(r <= 3.402823466e38f)) r = 0.0f;   // s below 2^-128: reciprocal not finite
  }
  bs.r = r;
  return bs;
}

// Clear the sign of every code whose magnitude is zero (zero always encodes as +0).
__device__ __forceinline__ uint32_t canonical_zero(uint32_t w) {
  const uint32_t nz = (w | (w >> 1) | (w >> 2)) & 0x11111111u;
  return w & (0x77777777u | (nz << 3));
}

// 8 scaled values -> 8 E2M1 codes (RNE, satfinite), element 2i in the low nibble of
// byte i, packed little-endian into 32 bits.
__device__ __forceinline__ uint32_t e2m1x8_rn(const float (&v)[8]) {
  uint32_t out;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(out)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return canonical_zero(out);
}

// Philox4x32-10 (Salmon et al., SC'11): 10 rounds of the Philox-4x32 bijection, key
// bumped by the Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// Stochastic rounding of one scaled value to E2M1: lo <= |v| < hi neighbouring grid
// magnitudes, p = (|v| - lo) / (hi - lo) (exact), round up iff r16 < p * 2^16;
// |v| >= 6 saturates.  Zero magnitude encodes as +0.
__device__ __forceinline__ uint32_t e2m1_sr(float v, uint32_t r16) {
  const float a = fabsf(v);
  const uint32_t c = (a >= 0.5f) + (a >= 1.0f) + (a >= 1.5f) + (a >= 2.0f) + (a >= 3.0f) + (a >= 4.0f) +
                     (a >= 6.0f);
  uint32_t code;
  if (c >= 7) {
    code = 7;
  } else {
    const float lo = c < 4 ? __fmul_rn((float)c, 0.5f) : (float)(c - 2);
    const float inv_gap = c < 4 ? 2.0f : (c < 6 ? 1.0f : 0.5f);
    const float p = __fmul_rn(__fsub_rn(a, lo), inv_gap);
    code = c + (((float)r16 < __fmul_rn(p, 65536.0f)) ? 1u : 0u);
  }
  return code | ((__float_as_uint(v) >> 31) && code ? 8u : 0u);
}

// 8 scaled values of one chunk with their Philox block output -> packed codes.
__device__ __forceinline__ uint32_t e2m1x8_sr(const float (&v)[8], uint4 rnd) {
  const uint32_t w[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
  uint32_t out = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const uint32_t r16 = (w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
    out |= e2m1_sr(v[e], r16) << (4 * e);
  }
  return out;
}

}  // namespace nvfp4

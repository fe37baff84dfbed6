// h = BF16(silu(gate) * up), the BF16 value nearest to the exact real number.
//
// The float32 evaluation h32 = (g * rcp(1 + expf(-g))) * u (expf within 2 ulp, four
// correctly rounded operations) has relative error below 2^-22 + 4 * 2^-24, i.e. under 8
// ulps of h32; when h32 lies within 16 ulps of a BF16 rounding midpoint, or outside the
// range where the bound holds, h is recomputed in float64 and rounded once to BF16
// through a round-to-odd float32 step.  The result equals the rounding of the exact
// value except when the exact value sits within ~1e-15 (relative) of a midpoint, which
// silu(g)*u with g != 0 never reaches exactly.
#pragma once
#include <cstdint>

namespace nvfp4 {

__device__ __forceinline__ uint32_t f32_to_bf16_rne_bits(uint32_t b) {
  return (b + 0x7FFFu + ((b >> 16) & 1u)) >> 16;
}

// float64 -> BF16 with a single rounding: round-to-odd into float32 (which keeps 16 more
// bits than BF16), then round-to-nearest-even into BF16.
__device__ __forceinline__ uint32_t f64_to_bf16_bits(double v) {
  float f = __double2float_rz(v);
  uint32_t b = __float_as_uint(f);
  if ((double)f != v) b |= 1u;
  return f32_to_bf16_rne_bits(b);
}

static __device__ __noinline__ uint32_t swiglu_f64(float g, float u) {
  const double gd = g, ud = u;
  const double sd = gd / (1.0 + exp(-gd));
  return f64_to_bf16_bits(sd * ud);
}

__device__ __forceinline__ uint32_t swiglu_bf16(float g, float u) {
  const float e = expf(-g);
  const float h = __fmul_rn(__fmul_rn(g, __frcp_rn(__fadd_rn(1.0f, e))), u);
  const uint32_t b = __float_as_uint(h);
  const uint32_t low = b & 0xFFFFu;
  const float ah = fabsf(h);
  const bool exact_zero = (g == 0.0f) || (u == 0.0f);
  const bool in_range = ah >= 1e-30f && ah <= 1e30f && e <= 3.0e38f;
  const bool near_mid = low >= 0x8000u - 16u && low <= 0x8000u + 16u;
  if (exact_zero || (in_range && !near_mid)) return f32_to_bf16_rne_bits(b);
  return swiglu_f64(g, u);
}

}  // namespace nvfp4

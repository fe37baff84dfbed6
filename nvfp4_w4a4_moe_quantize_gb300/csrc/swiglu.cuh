// h = BF16(silu(gate) * up), rounded once from silu computed in float64 as
// gate / (1 + exp(-gate)) and multiplied by up in float64 -- the value the oracle rounds.
//
// Fast path: h32 = (g * rcp(1 + expf(-g))) * u in float32 with expf within 2 ulp (CUDA's
// documented bound), rcp.approx within 1 ulp (PTX's documented bound) and three correctly
// rounded operations.  With unit roundoff eps = 2^-24 the relative error is at most
// 4eps (exp, damped by e/(1+e) <= 1) + eps (add) + 2eps (rcp) + 2eps (two products)
// = 9eps to first order, i.e. under 9 ulps of h32, while h32 and every intermediate stay
// normal or the sum 1 + e absorbs e.  So the BF16 rounding of h32 is the right one unless
// h32 lies within 16 ulps of a BF16 rounding midpoint (about 1 value in 2000) or outside
// [2^-100, 2^101) -- the cases handed to the exact path.
//
// Near a midpoint the value is recomputed in float-float arithmetic (pairs hi + lo of
// float32 values, about 46 significant bits), which runs on the float32 pipes: this GPU
// executes float64 at a small fraction of its float32 rate, and a float64 fallback
// inside the GEMM epilogue stalled whole warps.  exp is evaluated by Cody-Waite range
// reduction (t = k ln2 + r, ln2 split in three parts so that k ln2 is exact to ~2^-72)
// and the Taylor series of exp(r), |r| <= ln2/2, to degree 12.  The float-float result
// decides the rounding except where the exact value sits within ~2^-45 (relative) of a
// midpoint.  One structured family does: gate large and gate*up exactly a midpoint, where
// silu(gate)*up = gate*up*(1 - e) with e = exp(-gate) tiny.  The float64 reference rounds
// 1 + e to 1 when e <= 2^-53 (gate > 36.74) and then ties to even; for larger e it lands
// strictly below the midpoint.  The float-float path reproduces both cases by dropping e
// at the same threshold.  Inputs out of the float-float range (|gate| > 80, or |h| outside
// [2^-100, 2^100], where BF16 subnormals need care) take a float64 path.  The gate is a
// BF16 value, so silu(gate) as a float-float comes from a 65536-entry table built once per
// device with this arithmetic; the exact path is then one load and a float-float product.
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

__device__ __forceinline__ uint32_t swiglu_f64(float g, float u) {
  const double gd = g, ud = u;
  const double sd = gd / (1.0 + exp(-gd));
  return f64_to_bf16_bits(sd * ud);
}

// ---- float-float arithmetic: a value is hi + lo with |lo| <= ulp(hi) / 2.  Error-free
// transformations: Knuth's TwoSum, Dekker's FastTwoSum (|a| >= |b|), the fma product.
struct ff {
  float hi, lo;
};
__device__ __forceinline__ ff ff_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  return {s, __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb))};
}
__device__ __forceinline__ ff ff_fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ ff ff_two_prod(float a, float b) {
  const float p = __fmul_rn(a, b);
  return {p, __fmaf_rn(a, b, -p)};
}
__device__ __forceinline__ ff ff_mul(ff a, ff b) {
  const ff p = ff_two_prod(a.hi, b.hi);
  return ff_fast_two_sum(p.hi, __fadd_rn(p.lo, __fadd_rn(__fmul_rn(a.hi, b.lo), __fmul_rn(a.lo, b.hi))));
}
// Sum without heavy cancellation (|b| well above |a| in the Horner steps below).
__device__ __forceinline__ ff ff_add(ff a, ff b) {
  const ff s = ff_two_sum(a.hi, b.hi);
  return ff_fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}

// exp(t) as a float-float, |t| <= 80 (result a normal float32 up to ~2^-24 of its lo part).
__device__ __forceinline__ ff ff_exp(float t) {
  // ln2 = kLn2Hi + kLn2Mid + kLn2Lo: Hi has 15 significant bits and Mid 16, so k * Hi
  // and k * Mid are exact for |k| < 128; t - k * Hi is exact (Sterbenz).
  constexpr float kLog2e = 0x1.715476p+0f;
  constexpr float kLn2Hi = 0x1.62e4p-1f, kLn2Mid = 0x1.7f7ep-20f, kLn2Lo = -0x1.c610cap-37f;
  const float k = rintf(__fmul_rn(t, kLog2e));
  ff r = ff_two_sum(__fsub_rn(t, __fmul_rn(k, kLn2Hi)), -__fmul_rn(k, kLn2Mid));
  r = ff_fast_two_sum(r.hi, __fsub_rn(r.lo, __fmul_rn(k, kLn2Lo)));
  // exp(r) = sum_n r^n / n!: terms 8..12 in float32 (their sum is below 2^-27), then
  // Horner in float-float with 1/n! split into hi + lo.
  float tail = 0x1.1eed8ep-29f;
  tail = __fadd_rn(__fmul_rn(tail, r.hi), 0x1.ae6456p-26f);
  tail = __fadd_rn(__fmul_rn(tail, r.hi), 0x1.27e4fcp-22f);
  tail = __fadd_rn(__fmul_rn(tail, r.hi), 0x1.71de3ap-19f);
  tail = __fadd_rn(__fmul_rn(tail, r.hi), 0x1.a01a02p-16f);
  const ff c[8] = {{1.0f, 0.0f},
                   {1.0f, 0.0f},
                   {0.5f, 0.0f},
                   {0x1.555556p-3f, -0x1.555556p-28f},
                   {0x1.555556p-5f, -0x1.555556p-30f},
                   {0x1.111112p-7f, -0x1.dddddep-32f},
                   {0x1.6c16c2p-10f, -0x1.27d27ep-35f},
                   {0x1.a01a02p-13f, -0x1.7f97fap-39f}};
  ff p = {tail, 0.0f};
#pragma unroll
  for (int n = 7; n >= 0; --n) p = ff_add(ff_mul(p, r), c[n]);
  const float scale = __int_as_float(((int)k + 127) << 23);
  return {__fmul_rn(p.hi, scale), __fmul_rn(p.lo, scale)};
}

constexpr uint32_t kSwigluNeedF64 = 0xFFFFFFFFu;

// silu(g) = g / (1 + exp(-g)) as a float-float, |g| <= 80; a NaN hi part otherwise (the
// float64 path takes those).
__device__ __forceinline__ ff silu_ff(float g) {
  if (!(fabsf(g) <= 80.0f)) return {__int_as_float(0x7FC00000), 0.0f};
  const ff e = ff_exp(-g);
  ff d = {1.0f, 0.0f};                       // float64 rounds 1 + e to 1 for e <= 2^-53
  if (e.hi > 0x1p-53f) {
    d = ff_two_sum(1.0f, e.hi);
    d = ff_fast_two_sum(d.hi, __fadd_rn(d.lo, e.lo));
  }
  // s = g / d: quotient, exact remainder, correction
  const float q1 = __fdiv_rn(g, d.hi);
  const ff pq = ff_two_prod(q1, d.hi);
  float rem = __fsub_rn(__fsub_rn(g, pq.hi), pq.lo);
  rem = __fsub_rn(rem, __fmul_rn(q1, d.lo));
  return ff_fast_two_sum(q1, __fdiv_rn(rem, d.hi));
}

// BF16 rounding of s * u from the float-float s = silu(g); kSwigluNeedF64 when s is
// marked out of range or |s * u| is outside [2^-100, 2^100].
__device__ __forceinline__ uint32_t swiglu_finish(ff s, float u) {
  if (s.hi != s.hi) return kSwigluNeedF64;
  ff x = ff_two_prod(s.hi, u);
  x = ff_fast_two_sum(x.hi, __fadd_rn(x.lo, __fmul_rn(s.lo, u)));
  const float ax = fabsf(x.hi);
  if (!(ax >= 0x1p-100f && ax <= 0x1p100f)) return kSwigluNeedF64;
  const uint32_t b = __float_as_uint(x.hi);
  if ((b & 0xFFFFu) != 0x8000u || x.lo == 0.0f) return f32_to_bf16_rne_bits(b);
  // x.hi is a BF16 rounding midpoint: the sign of x.lo relative to x.hi decides
  return ((x.lo > 0.0f) == (x.hi > 0.0f)) ? (b >> 16) + 1u : (b >> 16);
}

// Gate values are BF16, so silu(g) takes 65536 values: the exact path reads its
// float-float silu from a table built once per device by silu_table_kernel (same
// arithmetic as silu_ff, entry i for the BF16 bit pattern i).
constexpr int kSiluTableSize = 65536;

__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// The float32 fast path, branch-free: the BF16 bits in `out`, and true when they are
// certainly the right rounding (false: the caller must take the exact path).
__device__ __forceinline__ bool swiglu_fast(float g, float u, uint32_t& out) {
  const float e = expf(-g);
  const float h = __fmul_rn(__fmul_rn(g, rcp_approx(__fadd_rn(1.0f, e))), u);
  const uint32_t b = __float_as_uint(h);
  const bool exact_zero = (g == 0.0f) | (u == 0.0f);
  const bool in_range = ((b >> 23) & 0xFFu) - 27u <= 200u;          // 2^-100 <= |h| < 2^101
  const bool near_mid = (b & 0xFFFFu) - (0x8000u - 16u) <= 32u;     // within 16 ulps
  out = f32_to_bf16_rne_bits(b);
  return exact_zero | (in_range & !near_mid);
}

// The same fast path returning the float32 h (the caller rounds pairs to BF16 with one
// conversion instruction, which is the same round-to-nearest-even for finite h).
__device__ __forceinline__ float swiglu_fast_f32(float g, float u, bool& ok) {
  const float e = expf(-g);
  const float h = __fmul_rn(__fmul_rn(g, rcp_approx(__fadd_rn(1.0f, e))), u);
  const uint32_t b = __float_as_uint(h);
  const bool exact_zero = (g == 0.0f) | (u == 0.0f);
  const bool in_range = ((b >> 23) & 0xFFu) - 27u <= 200u;          // 2^-100 <= |h| < 2^101
  const bool near_mid = (b & 0xFFFFu) - (0x8000u - 16u) <= 32u;     // within 16 ulps
  ok = exact_zero | (in_range & !near_mid);
  return h;
}

// The exact path for the values the fast path hands over, inlined at one warp-uniform
// site by its callers (a rarely taken call inside an unrolled epilogue loop cost far more
// than the work it did).  g must be a BF16 value; tab is the silu table.
__device__ __forceinline__ uint32_t swiglu_exact(const ff* __restrict__ tab, float g, float u) {
  const uint32_t r = swiglu_finish(tab[__float_as_uint(g) >> 16], u);
  return r != kSwigluNeedF64 ? r : swiglu_f64(g, u);
}
static __device__ __noinline__ uint32_t swiglu_slow(const ff* __restrict__ tab, float g, float u) {
  return swiglu_exact(tab, g, u);
}

__device__ __forceinline__ uint32_t swiglu_bf16(const ff* __restrict__ tab, float g, float u) {
  uint32_t b;
  return swiglu_fast(g, u, b) ? b : swiglu_slow(tab, g, u);
}

}  // namespace nvfp4

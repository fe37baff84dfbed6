// NVFP4 element and scale encoding on the device (sm_103a).
//
// Scale arithmetic ("The 4-bitter Lesson: Balancing Stability and Performance in NVFP4
// RL", §Baseline: E2M1 values, one E4M3 scale per 16 values, one FP32 global scale), every
// step one IEEE float32 operation, round to nearest even, in this order:
//   g = amax / 2688;  sf = E4M3_rn_satfinite(amax_block / (6 g));  s = decode(sf) * g.
// Element code (footnote 6 of §"Improving Gradient Stability": Q = clip(round(x/s), qmin,
// qmax)): round(x / s) of the exact quotient onto the E2M1 grid, ties to the even code,
// or stochastic rounding of that quotient.  The quotient is never rounded before the
// decision:
//   * fast path: two float32 products |x| * r_lo <= |x| / s <= |x| * r_hi, with r_lo and r_hi
//     bracketing 1/s; rounding is monotone, so where both round to the same code that is
//     the code of the exact quotient (one in about 10^4 blocks fails this test);
//   * exact path (the rest, and scales below 2^-60): the sign of |x| - m * s for each
//     decision threshold m, from one fused multiply-add -- exact, because the exact
//     difference is either zero or far above the smallest float32 subnormal.
// All products / quotients use the explicit _rn intrinsics so that no FMA contraction or
// approximate division can change a bit.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

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

// max |x| of 16 BF16 values (two 16-byte chunks), as a float: a tree of packed BF16
// maxima of magnitudes (max.xorsign.abs: the larger magnitude of each half, its sign the
// XOR of the two signs, cleared at the end); inputs are finite, so the result is exact.
__device__ __forceinline__ uint32_t maxabs_bf16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float absmax16_bf16(const uint4& q0, const uint4& q1) {
  const uint32_t m = maxabs_bf16x2(maxabs_bf16x2(maxabs_bf16x2(q0.x, q0.y), maxabs_bf16x2(q0.z, q0.w)),
                                   maxabs_bf16x2(maxabs_bf16x2(q1.x, q1.y), maxabs_bf16x2(q1.z, q1.w))) &
                     0x7FFF7FFFu;
  return __uint_as_float(max(m & 0xFFFFu, m >> 16) << 16);
}

__device__ __forceinline__ float absmax8(const float (&f)[8]) {
  float m = fabsf(f[0]);
#pragma unroll
  for (int i = 1; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
  return m;
}

// E4M3 byte -> float32 (exact; scales are non-negative so the sign bit is 0): the
// hardware E4M3 -> FP16 conversion (every E4M3 value, subnormals included, is an FP16
// value), then FP16 -> FP32.
__device__ __forceinline__ float e4m3_decode(uint32_t b) {
  uint32_t h2;
  asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}" : "=r"(h2) : "r"(b));
  return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// float32 (>= 0) -> E4M3 byte, round to nearest even, saturating at 448.
__device__ __forceinline__ uint32_t e4m3_encode(float t) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(0.0f), "f"(t));
  return d & 0xFFu;
}

constexpr float kTinyScale = 8.673617379884035e-19f;   // 2^-60

struct BlockScale {
  uint32_t sf;  // E4M3 byte written to the scale tensor
  float s;      // effective decode scale decode(sf) * g; 0 when the block decodes to zero
  float r_lo;   // fast path: 0 < r_lo * (1 + 2^-22) < 1/s < r_hi * (1 - 2^-22)  (0, 0 when s == 0)
  float r_hi;
  float r;      // the reciprocal itself, within 2^-22 of 1/s (0 when s == 0)
  bool exact_only;  // 0 < s < 2^-60: every element takes the exact path
};

// Block scale of one 16-value block with max |x| = amax_b, given the scope's g and 6g.
// The brackets come from the hardware reciprocal (rcp.approx.ftz.f32, at most one ulp from
// 1/s; s >= 2^-60 is a normal number, so flushing subnormals changes nothing): r * (1 -/+ 2^-18) leaves a margin of over 2^-19 on either side of 1/s, far more
// than the rounding of the reciprocal, of the bracket product and of |x| * r (2^-23 +
// 2 * 2^-24).
__device__ __forceinline__ BlockScale block_scale(float amax_b, float g, float six_g) {
  BlockScale bs;
  bs.exact_only = false;
  bs.r_lo = bs.r_hi = bs.r = 0.0f;
  if (!(g > 0.0f)) {
    bs.sf = 0;
    bs.s = 0.0f;
    return bs;
  }
  const float t = __fdiv_rn(amax_b, six_g);
  bs.sf = e4m3_encode(t);
  bs.s = __fmul_rn(e4m3_decode(bs.sf), g);
  if (bs.s >= kTinyScale) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(bs.s));
    bs.r = r;
    bs.r_lo = __fmul_rn(r, 0.99999618530273438f);   // 1 - 2^-18
    bs.r_hi = __fmul_rn(r, 1.0000038146972656f);    // 1 + 2^-18
  } else if (bs.s > 0.0f) {
    bs.exact_only = true;
  }
  return bs;
}

// Clear the sign of every code whose magnitude is zero (zero always encodes as +0).
__device__ __forceinline__ uint32_t canonical_zero(uint32_t w) {
  const uint32_t nz = (w | (w >> 1) | (w >> 2)) & 0x11111111u;
  return w & (0x77777777u | (nz << 3));
}

// 8 scaled values -> 8 E2M1 codes (RNE, satfinite), element 2i in the low nibble of
// byte i, packed little-endian into 32 bits; zero magnitudes keep their sign bit.
__device__ __forceinline__ uint32_t e2m1x8_raw(const float (&v)[8]) {
  uint32_t out;
  asm("{\n .reg .b8 b0, b1, b2, b3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      " cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      " mov.b32 %0, {b0, b1, b2, b3};\n}"
      : "=r"(out)
      : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
  return out;
}

// v = f * r for 8 values, two per instruction (mul.rn.f32x2: each lane one IEEE product).
__device__ __forceinline__ void scale8(const float (&f)[8], float r, float (&v)[8]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
    asm("{\n .reg .b64 a, b, d;\n mov.b64 a, {%2, %3};\n mov.b64 b, {%4, %4};\n"
        " mul.rn.f32x2 d, a, b;\n mov.b64 {%0, %1}, d;\n}"
        : "=f"(v[2 * i]), "=f"(v[2 * i + 1])
        : "f"(f[2 * i]), "f"(f[2 * i + 1]), "f"(r));
}

// |x| and s brought to where every product below stays exact in its sign: blocks with
// s < 2^-60 are scaled by 2^64 (exact; their elements are at most about 9 s).
__device__ __forceinline__ void exact_operands(float x, float s, float& a, float& t) {
  a = fabsf(x);
  t = s;
  if (s < kTinyScale) {
    a = __fmul_rn(a, 18446744073709551616.0f);   // 2^64
    t = __fmul_rn(s, 18446744073709551616.0f);
  }
}

// Exact round(|x| / s) (s > 0) onto the E2M1 grid, ties to the even code, saturating at 6:
// the number of midpoints m (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5) below the quotient, a
// tie at m counting when the code above it is even.  |x| - m s is formed exactly by the
// FMA and rounded once, which keeps its sign (zero only when it is exactly zero).
__device__ __forceinline__ uint32_t e2m1_exact_rn(float x, float s) {
  float a, t;
  exact_operands(x, s, a, t);
  const uint32_t c = (__fmaf_rn(-0.25f, t, a) > 0.0f) + (__fmaf_rn(-0.75f, t, a) >= 0.0f) +
                     (__fmaf_rn(-1.25f, t, a) > 0.0f) + (__fmaf_rn(-1.75f, t, a) >= 0.0f) +
                     (__fmaf_rn(-2.5f, t, a) > 0.0f) + (__fmaf_rn(-3.5f, t, a) >= 0.0f) +
                     (__fmaf_rn(-5.0f, t, a) > 0.0f);
  return c | ((__float_as_uint(x) >> 31) && c ? 8u : 0u);
}

// Element e of 8 values in registers (e is not a compile-time constant): a select tree,
// no local-memory array.
__device__ __forceinline__ float pick8(const float (&f)[8], uint32_t e) {
  const float a = (e & 1u) ? f[1] : f[0], b = (e & 1u) ? f[3] : f[2];
  const float c = (e & 1u) ? f[5] : f[4], d = (e & 1u) ? f[7] : f[6];
  const float ab = (e & 2u) ? b : a, cd = (e & 2u) ? d : c;
  return (e & 4u) ? cd : ab;
}

// E2M1 magnitude grid G and the midpoint between code c and c + 1 (c <= 6).
__device__ __forceinline__ float e2m1_grid(uint32_t c) {
  return c < 4u ? __fmul_rn((float)c, 0.5f) : (c < 6u ? (float)c - 2.0f : (c == 6u ? 4.0f : 6.0f));
}
__device__ __forceinline__ float e2m1_midpoint(uint32_t c) {
  return c < 4u ? __fmaf_rn(0.5f, (float)c, 0.25f) : (c == 6u ? 5.0f : (float)c - 1.5f);
}

// 8 values of one block -> 8 E2M1 codes of round(x / s), packed as e2m1x8_raw, zero
// magnitudes as +0.  The bracket codes lo (from |x| r_lo) and hi (|x| r_hi) differ only
// where the quotient lies within the bracket's width of a midpoint, and there by one step
// (midpoints are far apart relative to the bracket): those elements -- about 0.2% of
// Gaussian data, most of them structured ties that the rounded g creates -- are settled
// one at a time by the sign of |x| - m s for the one midpoint m between lo and hi.
__device__ __forceinline__ uint32_t e2m1x8_rn(const float (&f)[8], const BlockScale& bs) {
  if (!bs.exact_only) {
    float vl[8], vh[8];
    scale8(f, bs.r_lo, vl);
    scale8(f, bs.r_hi, vh);
    uint32_t lo = e2m1x8_raw(vl);
    uint32_t diff = lo ^ e2m1x8_raw(vh);
    while (diff != 0u) {
      const uint32_t sh = (uint32_t)(__ffs((int)diff) - 1) & ~3u;
      const uint32_t c = (lo >> sh) & 7u;                  // the lower candidate
      const float x = pick8(f, sh >> 2);
      const float d = __fmaf_rn(-e2m1_midpoint(c), bs.s, fabsf(x));
      const uint32_t cnew = (d > 0.0f || (d == 0.0f && (c & 1u))) ? c + 1u : c;   // a tie goes to the even code
      const uint32_t sign = cnew && (__float_as_uint(x) >> 31) ? 8u : 0u;
      lo = (lo & ~(0xFu << sh)) | ((cnew | sign) << sh);
      diff &= ~(0xFu << sh);
    }
    return canonical_zero(lo);
  }
  uint32_t out = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) out |= e2m1_exact_rn(f[e], bs.s) << (4 * e);
  return out;
}

// The exact path of a whole block (scales below 2^-60), out of line; the values are
// rebuilt from their BF16 words.
static __device__ __noinline__ uint2 e2m1x16_rn_exact_w(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3, uint32_t w4,
                                                       uint32_t w5, uint32_t w6, uint32_t w7, float s) {
  const uint32_t wv[8] = {w0, w1, w2, w3, w4, w5, w6, w7};
  uint32_t lo = 0, hi = 0;
#pragma unroll
  for (int e = 0; e < 16; ++e) {
    const float fe = __uint_as_float((e & 1) ? (wv[e >> 1] & 0xFFFF0000u) : (wv[e >> 1] << 16));
    const uint32_t c = e2m1_exact_rn(fe, s);
    if (e < 8) lo |= c << (4 * e); else hi |= c << (4 * (e - 8));
  }
  return make_uint2(lo, hi);
}
__device__ __forceinline__ uint2 e2m1x16_rn_exact(const float (&h0)[8], const float (&h1)[8], float s) {
  const auto pk = [](float a, float b) { return __byte_perm(__float_as_uint(a), __float_as_uint(b), 0x7632); };
  return e2m1x16_rn_exact_w(pk(h0[0], h0[1]), pk(h0[2], h0[3]), pk(h0[4], h0[5]), pk(h0[6], h0[7]), pk(h1[0], h1[1]),
                            pk(h1[2], h1[3]), pk(h1[4], h1[5]), pk(h1[6], h1[7]), s);
}

// One whole 16-value block (h0: values 0..7, h1: values 8..15) -> its 16 codes (x: 0..7,
// y: 8..15), as e2m1x8_rn on both halves but with one settling loop for the block.
__device__ __forceinline__ uint2 e2m1x16_rn(const float (&h0)[8], const float (&h1)[8], const BlockScale& bs) {
  if (bs.exact_only) return e2m1x16_rn_exact(h0, h1, bs.s);
  float vl[8], vh[8];
  scale8(h0, bs.r_lo, vl);
  scale8(h0, bs.r_hi, vh);
  const uint32_t l0 = e2m1x8_raw(vl), d0 = l0 ^ e2m1x8_raw(vh);
  scale8(h1, bs.r_lo, vl);
  scale8(h1, bs.r_hi, vh);
  const uint32_t l1 = e2m1x8_raw(vl), d1 = l1 ^ e2m1x8_raw(vh);
  uint64_t lo = ((uint64_t)l1 << 32) | l0;
  uint64_t diff = ((uint64_t)d1 << 32) | d0;
  while (diff != 0ull) {
    const uint32_t sh = (uint32_t)(__ffsll((long long)diff) - 1) & ~3u;
    const uint32_t c = (uint32_t)(lo >> sh) & 7u;        // the lower candidate
    const uint32_t e = sh >> 2;
    const float x = (e & 8u) ? pick8(h1, e & 7u) : pick8(h0, e & 7u);
    const float d = __fmaf_rn(-e2m1_midpoint(c), bs.s, fabsf(x));
    const uint32_t cnew = (d > 0.0f || (d == 0.0f && (c & 1u))) ? c + 1u : c;   // a tie goes to the even code
    const uint32_t sign = cnew && (__float_as_uint(x) >> 31) ? 8u : 0u;
    lo = (lo & ~(0xFull << sh)) | ((uint64_t)(cnew | sign) << sh);
    diff &= ~(0xFull << sh);
  }
  return make_uint2(canonical_zero((uint32_t)lo), canonical_zero((uint32_t)(lo >> 32)));
}

// The sign bits of 8 BF16 values (4 words, value 2i in the low half of word i) at bit
// 4e + 3 of a packed code word: a byte permute with sign replication turns the sign of
// each value into a 0x00 / 0xFF byte, two more interleave the even and odd values.
__device__ __forceinline__ uint32_t sign_nibbles(const uint4& w) {
  uint32_t lo, hi;
  asm("prmt.b32 %0, %1, %2, 0xFDB9;" : "=r"(lo) : "r"(w.x), "r"(w.y));   // values 0..3
  asm("prmt.b32 %0, %1, %2, 0xFDB9;" : "=r"(hi) : "r"(w.z), "r"(w.w));   // values 4..7
  return (__byte_perm(lo, hi, 0x6420) & 0x08080808u) | (__byte_perm(lo, hi, 0x7531) & 0x80808080u);
}

// The words of 8 floats that hold BF16 values, as BF16 pairs (value 2i in the low half of
// word i).
__device__ __forceinline__ uint4 bf16_words(const float (&f)[8]) {
  const auto hi16 = [](float a, float b) { return __byte_perm(__float_as_uint(a), __float_as_uint(b), 0x7632); };
  return make_uint4(hi16(f[0], f[1]), hi16(f[2], f[3]), hi16(f[4], f[5]), hi16(f[6], f[7]));
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

// Stochastic rounding (the reading): with lo <= q < hi the neighbouring grid magnitudes
// around the quotient q = |x|/s and p = (q - lo) / (hi - lo), round up iff r16 < p 2^16; q >= 6
// saturates; zero magnitude encodes as +0.  As a function of q this is the number of
// thresholds tau_j = G_{j-1} + r16 (G_j - G_{j-1}) / 2^16 (j = 1..7, G the grid) that q
// exceeds.
// Exact stochastic rounding of the quotient |x| / s (s > 0): the number of thresholds
// tau_j (above) with |x| > tau_j * s, each decided by the sign of one FMA (tau_j has at
// most 19 significant bits, so |x| - tau_j s is either zero or far from underflow).
__device__ __forceinline__ uint32_t e2m1_exact_sr(float x, float s, uint32_t r16) {
  float a, t;
  exact_operands(x, s, a, t);
  const float u = __fmul_rn((float)r16, 1.52587890625e-05f);   // r16 / 2^16, exact
  const float h = __fmul_rn(u, 0.5f);
  const uint32_t c = (__fmaf_rn(-h, t, a) > 0.0f) + (__fmaf_rn(-__fadd_rn(0.5f, h), t, a) > 0.0f) +
                     (__fmaf_rn(-__fadd_rn(1.0f, h), t, a) > 0.0f) +
                     (__fmaf_rn(-__fadd_rn(1.5f, h), t, a) > 0.0f) +
                     (__fmaf_rn(-__fadd_rn(2.0f, u), t, a) > 0.0f) +
                     (__fmaf_rn(-__fadd_rn(3.0f, u), t, a) > 0.0f) +
                     (__fmaf_rn(-__fadd_rn(4.0f, __fmul_rn(u, 2.0f)), t, a) > 0.0f);
  return c | ((__float_as_uint(x) >> 31) && c ? 8u : 0u);
}

// The rare paths of e2m1x8_sr, out of line (kept inline, they doubled the hot loop's code:
// measured, instruction-cache misses were the second stall reason of the SR quantiser, and
// out of line the row quantiser runs 52 instead of 61 us): the values are rebuilt from the
// BF16 words.  _settle: the exact stochastic rounding of every value whose grid
// coordinate sits within one unit of a threshold; _exact: every value (scales below 2^-60).
static __device__ __noinline__ uint32_t e2m1x8_sr_settle(uint4 words, float r, float s, uint4 rnd, uint32_t out) {
  const uint32_t wv[4] = {words.x, words.y, words.z, words.w};
  const uint32_t w[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float fe = __uint_as_float((e & 1) ? (wv[e >> 1] & 0xFFFF0000u) : (wv[e >> 1] << 16));
    const uint32_t vb = __float_as_uint(__fmul_rn(fabsf(fe), r));
    const uint32_t lin = __float_as_uint(__fmaf_rd(__uint_as_float(vb), 0x1p-124f, 0x1.ep-120f));
    const uint32_t x4 = vb < 0x3F800000u ? lin : (vb >> 4);
    const uint32_t r16 = (w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
    const uint32_t a = x4 - 4u * r16 + (0x3FFFFu - 0x3F00000u);
    if ((~a & 0x3FFFEu) == 0u) {
      const uint32_t c = e2m1_exact_sr(fe, s, r16);
      out = (out & ~(0xFu << (4 * e))) | (c << (4 * e));
    }
  }
  return out;
}

static __device__ __noinline__ uint32_t e2m1x8_sr_exact(uint4 words, float s, uint4 rnd) {
  const uint32_t wv[4] = {words.x, words.y, words.z, words.w};
  const uint32_t w[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
  uint32_t out = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const float fe = __uint_as_float((e & 1) ? (wv[e >> 1] & 0xFFFF0000u) : (wv[e >> 1] << 16));
    out |= e2m1_exact_sr(fe, s, (w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu) << (4 * e);
  }
  return out;
}

// 8 values of one chunk with their Philox block output -> packed codes of the
// stochastically rounded exact quotients.  One product v = |x| r per value (|v/q - 1| <=
// 2^-21 for the exact quotient q = |x|/s).  The rounding counts the thresholds
// tau_j = G_{j-1} + r16 (G_j - G_{j-1}) / 2^16 below q; on the grid coordinate
// X = 2^16 t (t = 2v below 2, v + 2 below 4, v/2 + 4 above, so that grid point G_i sits at
// X = 2^16 i) they are the integers T_j = 2^16 (j - 1) + r16, and the code is the number of
// T_j below X.  X4 = floor(4X) is formed without rounding: below v = 1 by one FMA rounded
// down (v 2^19 counted in units of the last place of a float whose bits are offset by
// 0x3F00000); from v = 1 on, t is linear within each binade of v with the binade's slope,
// so X4 = (bits(v) - 0x3F000000) / 16 exactly.  v's error moves X by at most 1/8, so the
// count is the exact quotient's unless X4 - 4 T_j is -1 or 0 for some j; those values --
// about one in 10^5 -- take the exact count of thresholds below q (e2m1_exact_sr).  The
// count from X4 is (X4 + 2^18 - 1 - 4 r16) / 2^18, saturated at 7.
// Codes are placed with integer multiply-adds (code * 16^e + out), which can run on the
// FMA pipe next to the ALU work; the eight signs come from the BF16 words w (value 2i in
// the low half of word i) by byte permutes.
__device__ __forceinline__ uint32_t e2m1x8_sr(const float (&f)[8], const uint4& words, const BlockScale& bs,
                                              uint4 rnd) {
  const uint32_t w[4] = {rnd.x, rnd.y, rnd.z, rnd.w};
  if (!(bs.s > 0.0f)) return 0u;
  if (!bs.exact_only) {
    uint32_t out = 0, near = 0xFFFFFFFFu;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float v = __fmul_rn(fabsf(f[e]), bs.r);
      const uint32_t vb = __float_as_uint(v);
      // bits of v 2^-124 + 2^-120 (1 + 0x700000 / 2^23), rounded down: 0x3F00000 + floor(v 2^19)
      const uint32_t lin = __float_as_uint(__fmaf_rd(v, 0x1p-124f, 0x1.ep-120f));
      const uint32_t x4 = vb < 0x3F800000u ? lin : (vb >> 4);          // X4 + 0x3F00000
      const uint32_t r16 = (w[e >> 1] >> (16 * (e & 1))) & 0xFFFFu;
      const uint32_t a = x4 - 4u * r16 + (0x3FFFFu - 0x3F00000u);      // X4 + 2^18 - 1 - 4 r16
      near = min(near, ~a & 0x3FFFEu);                                  // 0: X4 - 4 T_j in {-1, 0}
      out += min(a >> 18, 7u) * (1u << (4 * e));
    }
    out = canonical_zero(out | sign_nibbles(words));
    if (near == 0u) out = e2m1x8_sr_settle(words, bs.r, bs.s, rnd, out);
    return out;
  }
  return e2m1x8_sr_exact(words, bs.s, rnd);
}

// The same, for callers that hold only the floats.
__device__ __forceinline__ uint32_t e2m1x8_sr(const float (&f)[8], const BlockScale& bs, uint4 rnd) {
  return e2m1x8_sr(f, bf16_words(f), bs, rnd);
}

}  // namespace nvfp4

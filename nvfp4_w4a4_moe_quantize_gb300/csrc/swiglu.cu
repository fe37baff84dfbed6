// SwiGLU over the gate/up GEMM output, followed by per-row NVFP4 requantisation of h.
//
// The down projection's input is quantised the same way as the block's input: one FP32
// scale per routed row, E4M3 scales per 16 values, E2M1 codes ("The 4-bitter Lesson:
// Balancing Stability and Performance in NVFP4 RL", §"Why is the NVFP4 pretraining
// recipe not sufficient for RL?": per-token activation scales).
//
// h = BF16(silu(gate) * up) rounded as the float64 reference does (see swiglu.cuh).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "encode.cuh"
#include "launch.h"
#include "swiglu.cuh"

namespace nvfp4 {

constexpr unsigned kAll = 0xFFFFFFFFu;

// silu of every BF16 bit pattern as a float-float (swiglu.cuh), built on first use per
// device; every call shares it read-only.
static __device__ __align__(256) ff g_silu_tab[kSiluTableSize];

__global__ void __launch_bounds__(256) silu_table_kernel(ff* __restrict__ tab) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < kSiluTableSize) tab[i] = silu_ff(__uint_as_float((uint32_t)i << 16));
}

const void* silu_table(cudaStream_t s) {
  static const void* ptr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_silu_tab) != cudaSuccess) return nullptr;
    silu_table_kernel<<<kSiluTableSize / 256, 256, 0, s>>>(static_cast<ff*>(p));
    // wait once, so that calls on other streams never read a table still being built
    if (cudaGetLastError() != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) return nullptr;
    ptr[dev] = p;
  }
  return ptr[dev];
}

// One warp per routed row.  Lane l owns h columns 8l + 256i; gate of h column c sits at
// D column (c/64)*128 + c%64 and up at the same plus 64 (64-row interleave of W13).
template <int MAXC>
__global__ void __launch_bounds__(256) swiglu_quant_kernel(const __nv_bfloat16* __restrict__ d,
                                                           const int32_t* __restrict__ perm, int64_t rows,
                                                           const int32_t* __restrict__ nrows_dev, int64_t I,
                                                           int64_t Ip,
                                                           __nv_bfloat16* __restrict__ h_out,
                                                           uint8_t* __restrict__ hq, uint8_t* __restrict__ hsf,
                                                           float* __restrict__ gh, const ff* __restrict__ tab) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t nwarp = (int64_t)gridDim.x * 8;
  const int64_t sf_words = Ip / 64, data_words = (I + 63) / 64;
  if (nrows_dev != nullptr && (int64_t)*nrows_dev < rows) rows = *nrows_dev;
  for (int64_t r = warp; r < rows; r += nwarp) {
    if (perm[r] < 0) continue;
    const __nv_bfloat16* dr = d + r * (2 * I);
    uint4 hv[MAXC];
    float bm[MAXC];
    float rmax = 0.0f;
#pragma unroll
    for (int i = 0; i < MAXC; ++i) {
      const int64_t c = 8 * lane + 256 * i;
      hv[i] = make_uint4(0, 0, 0, 0);
      float cm = 0.0f;
      if (c < I) {
        const int64_t gc = (c >> 6) * 128 + (c & 63);
        const uint4 gq = *reinterpret_cast<const uint4*>(dr + gc);
        const uint4 uq = *reinterpret_cast<const uint4*>(dr + gc + 64);
        float gf[8], uf[8];
        bf16x8_to_f32(gq, gf);
        bf16x8_to_f32(uq, uf);
        uint32_t hb[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          hb[e] = swiglu_bf16(tab, gf[e], uf[e]);
          cm = fmaxf(cm, fabsf(__uint_as_float(hb[e] << 16)));
        }
        hv[i] = make_uint4(hb[0] | (hb[1] << 16), hb[2] | (hb[3] << 16), hb[4] | (hb[5] << 16),
                           hb[6] | (hb[7] << 16));
        if (h_out != nullptr) *reinterpret_cast<uint4*>(h_out + r * I + c) = hv[i];
      }
      bm[i] = fmaxf(cm, __shfl_xor_sync(kAll, cm, 1));
      rmax = fmaxf(rmax, bm[i]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) rmax = fmaxf(rmax, __shfl_xor_sync(kAll, rmax, o));
    const float g = __fdiv_rn(rmax, kGlobalDivisor);
    const float six_g = __fmul_rn(6.0f, g);
    uint8_t* qr = hq + r * (Ip / 2);
#pragma unroll
    for (int i = 0; i < MAXC; ++i) {
      const int64_t c = 8 * lane + 256 * i;
      const bool active = c < I;
      const BlockScale bs = block_scale(bm[i], g, six_g);
      float f[8];
      bf16x8_to_f32(hv[i], f);
      const uint32_t word = e2m1x8_rn(f, bs);
      const uint32_t sfb = active ? bs.sf : 0u;
      const uint32_t s2 = __shfl_down_sync(kAll, sfb, 2);
      const uint32_t s4 = __shfl_down_sync(kAll, sfb, 4);
      const uint32_t s6 = __shfl_down_sync(kAll, sfb, 6);
      if (active) {
        *reinterpret_cast<uint32_t*>(qr + c / 2) = word;
        if ((lane & 7) == 0) {
          const int64_t w = 4 * i + lane / 8;
          *reinterpret_cast<uint32_t*>(hsf + ((r >> 7) * sf_words + w) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4) =
              sfb | (s2 << 8) | (s4 << 16) | (s6 << 24);
        }
      }
    }
    for (int64_t w = data_words + lane; w < sf_words; w += 32)
      *reinterpret_cast<uint32_t*>(hsf + ((r >> 7) * sf_words + w) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4) = 0u;
    for (int64_t b = I / 2 + 8 * lane; b < Ip / 2; b += 256) *reinterpret_cast<uint2*>(qr + b) = make_uint2(0u, 0u);
    if (lane == 0) gh[r] = g;
  }
}

// SwiGLU backward: for h = silu(g) * u with s = sigmoid(g),
//     dgate = dh * u * s * (1 + g * (1 - s)),   dup = dh * g * s,
// each in float32 (s = 1 / (1 + e^-g) with expf and a correctly rounded division), rounded
// once to BF16.  One thread per 8 columns of a row: gate and up from [gate | up] rows of
// pitch 2I, dh from rows of pitch I, [dgate | dup] out like the input.
// gu_interleaved: gate/up columns in the 64-chunk interleave of the prepared W13 (gate
// column c at (c/64)*128 + c%64, up column c 64 further), as the gate/up GEMM writes D;
// otherwise [gate | up].  dh has row pitch dh_ld; dgu is always [dgate | dup].
__global__ void __launch_bounds__(256) swiglu_backward_kernel(const __nv_bfloat16* __restrict__ gu,
                                                              const __nv_bfloat16* __restrict__ dh, int64_t rows,
                                                              int64_t I, int gu_interleaved, int64_t dh_ld,
                                                              __nv_bfloat16* __restrict__ dgu) {
  const int64_t chunks = I / 8, total = rows * chunks;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / chunks, c = 8 * (i - r * chunks);
    const int64_t gcol = gu_interleaved ? (c >> 6) * 128 + (c & 63) : c;
    const int64_t ucol = gu_interleaved ? gcol + 64 : I + c;
    const uint4 gq = *reinterpret_cast<const uint4*>(gu + r * 2 * I + gcol);
    const uint4 uq = *reinterpret_cast<const uint4*>(gu + r * 2 * I + ucol);
    const uint4 hq = *reinterpret_cast<const uint4*>(dh + r * dh_ld + c);
    const uint32_t gw[4] = {gq.x, gq.y, gq.z, gq.w}, uw[4] = {uq.x, uq.y, uq.z, uq.w},
                   hw[4] = {hq.x, hq.y, hq.z, hq.w};
    uint32_t dg[4], du[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      float rg[2], ru[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float g = __uint_as_float(e ? gw[p] & 0xFFFF0000u : gw[p] << 16);
        const float u = __uint_as_float(e ? uw[p] & 0xFFFF0000u : uw[p] << 16);
        const float d = __uint_as_float(e ? hw[p] & 0xFFFF0000u : hw[p] << 16);
        const float sg = __fdiv_rn(1.0f, __fadd_rn(1.0f, expf(-g)));
        const float ds = __fmul_rn(sg, __fadd_rn(1.0f, __fmul_rn(g, __fsub_rn(1.0f, sg))));
        rg[e] = __fmul_rn(__fmul_rn(d, u), ds);
        ru[e] = __fmul_rn(d, __fmul_rn(g, sg));
      }
      const __nv_bfloat162 a = __floats2bfloat162_rn(rg[0], rg[1]);
      const __nv_bfloat162 b = __floats2bfloat162_rn(ru[0], ru[1]);
      dg[p] = *reinterpret_cast<const uint32_t*>(&a);
      du[p] = *reinterpret_cast<const uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(dgu + r * 2 * I + c) = make_uint4(dg[0], dg[1], dg[2], dg[3]);
    *reinterpret_cast<uint4*>(dgu + r * 2 * I + I + c) = make_uint4(du[0], du[1], du[2], du[3]);
  }
}

cudaError_t launch_swiglu_backward(const void* gu, const void* dh, int64_t rows, int64_t I, void* dgu,
                                   cudaStream_t s, bool gu_interleaved, int64_t dh_ld) {
  const int64_t total = rows * (I / 8);
  if (total == 0) return cudaSuccess;
  int64_t blocks = (total + 255) / 256;
  if (blocks > 16 * (int64_t)num_sms()) blocks = 16 * (int64_t)num_sms();
  swiglu_backward_kernel<<<(int)blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(gu),
                                                     static_cast<const __nv_bfloat16*>(dh), rows, I,
                                                     gu_interleaved ? 1 : 0, dh_ld > 0 ? dh_ld : I,
                                                     static_cast<__nv_bfloat16*>(dgu));
  return cudaGetLastError();
}

cudaError_t launch_swiglu_quant(const void* d, const int32_t* perm, int64_t rows, const int32_t* nrows_dev,
                                int64_t I, int64_t Ip, void* h_out, uint8_t* hq, uint8_t* hsf, float* gh,
                                cudaStream_t s) {
  const ff* tab = static_cast<const ff*>(silu_table(s));
  if (tab == nullptr) return cudaErrorUnknown;
  if (rows == 0) return cudaSuccess;
  int64_t blocks = (rows + 7) / 8;
  if (blocks > 8 * num_sms()) blocks = 8 * num_sms();
  const auto* dp = static_cast<const __nv_bfloat16*>(d);
  auto* hp = static_cast<__nv_bfloat16*>(h_out);
  if (I <= 256) swiglu_quant_kernel<1><<<(int)blocks, 256, 0, s>>>(dp, perm, rows, nrows_dev, I, Ip, hp, hq, hsf, gh, tab);
  else if (I <= 512) swiglu_quant_kernel<2><<<(int)blocks, 256, 0, s>>>(dp, perm, rows, nrows_dev, I, Ip, hp, hq, hsf, gh, tab);
  else if (I <= 768) swiglu_quant_kernel<3><<<(int)blocks, 256, 0, s>>>(dp, perm, rows, nrows_dev, I, Ip, hp, hq, hsf, gh, tab);
  else if (I <= 1024) swiglu_quant_kernel<4><<<(int)blocks, 256, 0, s>>>(dp, perm, rows, nrows_dev, I, Ip, hp, hq, hsf, gh, tab);
  else if (I <= 2048) swiglu_quant_kernel<8><<<(int)blocks, 256, 0, s>>>(dp, perm, rows, nrows_dev, I, Ip, hp, hq, hsf, gh, tab);
  else swiglu_quant_kernel<16><<<(int)blocks, 256, 0, s>>>(dp, perm, rows, nrows_dev, I, Ip, hp, hq, hsf, gh, tab);
  return cudaGetLastError();
}

}  // namespace nvfp4

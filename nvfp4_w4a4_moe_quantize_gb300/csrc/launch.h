// Internal launch interface between the C ABI (api.cu) and the kernel files.
#pragma once
#include <atomic>
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace nvfp4 {

enum : int { kScopeTensor = 0, kScopeRow = 1, kScopeGroup = 2 };
enum : int { kRoundRNE = 0, kRoundSR = 1 };
enum : int { kMapIdentity = 0, kMapInterleave = 1 };

struct QuantArgs {
  const __nv_bfloat16* x;  // input rows [rows, ld]
  int64_t rows, cols, ld;
  int mode;                // kScope*
  int64_t group_rows;
  const float* g_in;       // nullable: given global scales
  const uint32_t* amax_bits;  // tensor / group modes without g_in
  float* g_out;            // nullable
  uint8_t* codes;          // output codes, codes_ld bytes per output row
  int64_t codes_ld;
  uint8_t* sf;             // tiled scales (or row-major, see sf_row_bytes)
  int64_t sf_words;        // 4-scale words per row of the tile grid = ceil(cols_pad / 64)
  int64_t sf_row_bytes;    // > 0: row-major scales [rows, cols/16] (cols % 64 == 0, no padding
                           //      rows or words); 0: the 128x4 tiled layout
  int64_t cols_pad;        // stored columns (>= cols): codes / scales beyond cols are zero
  int64_t rows_total;      // rows visited; rows..rows_total-1 only get zero scales
  int map;                 // kMap*
  int64_t map_I;           // interleave: intermediate size I
  uint64_t seed, rng_offset;
  int* status;
  int tiled_R;             // 0: row-major codes + 128x4 scales; 128 / 256: GEMM-tiled output
                           //    (codes and scales both in `codes`, see tiled.cuh)
  int64_t kblocks;         // tiled: cols_pad / 256
  const int32_t* row_filter;  // nullable: rows with row_filter[row] < 0 are skipped
  const int32_t* rows_dev;    // nullable: device count capping `rows`
  int q_stages, q_stride;     // streaming path: ring stages per warp, bytes per stage (set by the launcher)
};

struct GemmArgs {
  const uint8_t* sfa;      // tiled scales of A (M_total rows)
  const uint8_t* sfb;      // tiled scales of B (E*N rows)
  const float* ga;         // [M_total]
  const float* gb;         // [E]
  const int32_t* offsets;  // [E+1] padded group starts
  const int32_t* rows;     // [E] valid rows per group
  int64_t m_total;         // rows of A, D (and ga): every group must lie inside [0, m_total)
                           // (ragged K: the K-blocks the operands hold)
  int32_t m_rows;          // ragged K: rows of A and of D per expert (a multiple of 128)
  int32_t E;
  int32_t N, K;
  void* d;
  int64_t ldd;
  int out_f32;
  int* status;
  __nv_bfloat16* h;        // SwiGLU epilogue: h [M, I]
  int64_t I;
  uint32_t* h_amax;        // SwiGLU epilogue, nullable: per-row max |h| (float bits), atomicMax-combined
  const void* silu_tab;    // SwiGLU epilogue: silu_table()
};

// Device address of the per-device silu table of the SwiGLU exact path (built by one
// kernel on stream s, waited for, on the first call per device); nullptr on failure.
const void* silu_table(cudaStream_t s);

int num_sms();
int* device_status_ptr();

// Sets a kernel's dynamic shared-memory limit once per device (flags: one per device,
// 64 devices).  Concurrent first calls may both set it, which is harmless.
inline cudaError_t set_smem_attr_once(std::atomic<bool>* flags, const void* func, int bytes) {
  int dev = 0;
  cudaGetDevice(&dev);
  const bool cached = dev >= 0 && dev < 64;
  if (cached && flags[dev].load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t err = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (err == cudaSuccess && cached) flags[dev].store(true, std::memory_order_release);
  return err;
}

cudaError_t launch_amax(const void* x, int64_t rows, int64_t cols, int64_t ld, int64_t group_rows,
                        uint32_t* amax_bits, int64_t n_scopes, cudaStream_t s);
// pdl: launched as a programmatic dependent of the kernel before it on the stream (the
// encode kernels wait for that grid's completion before reading anything it wrote).
cudaError_t launch_quantize_rows(const QuantArgs& a, int rounding, cudaStream_t s, bool pdl = false);

// Grouped GEMM: tensor maps are built by the caller (api.cu), all with 128-row boxes.
// The 128 x 256 tile kernel serves N % 256 == 0 and E <= 512; the 128 x 128
// kernel serves the rest.
bool n256_supported(const GemmArgs& g);
cudaError_t launch_grouped_gemm_n256(const CUtensorMap& tma, const CUtensorMap& tmb, const GemmArgs& g,
                                     int64_t max_m_tiles, cudaStream_t s);
// MXFP8 operands on the 128 x 256 tile kernel (N % 256 == 0, E <= 512).
cudaError_t launch_grouped_gemm_n256_mx(const CUtensorMap& tma, const CUtensorMap& tmb, const GemmArgs& g,
                                        int64_t max_m_tiles, cudaStream_t s);
cudaError_t launch_grouped_gemm(const CUtensorMap& tma, const CUtensorMap& tmb, const CUtensorMap& tmd,
                                const GemmArgs& g, int64_t max_m_tiles, cudaStream_t s);
// The same 128 x 128 tile kernel over MXFP8 operands (E4M3 codes [rows, K] bytes, E8M0
// scales per 32 values in the 128x4 tiled layout; g.ga / g.gb unused).  K % 128 == 0.
cudaError_t launch_grouped_gemm_mx(const CUtensorMap& tma, const CUtensorMap& tmb, const CUtensorMap& tmd,
                                   const GemmArgs& g, int64_t max_m_tiles, cudaStream_t s);
// BF16 grouped GEMM (the dequantised backward): A [M_total, K], B [E*N, K] BF16, both as
// byte maps with 128-byte boxes; g.sfa / g.sfb / g.ga / g.gb unused.  N % 128 == 0,
// K % 64 == 0.
cudaError_t launch_grouped_gemm_bf16(const CUtensorMap& tma, const CUtensorMap& tmb, const CUtensorMap& tmd,
                                     const GemmArgs& g, int64_t max_m_tiles, cudaStream_t s);
// MXFP8 quantiser: x BF16 [rows, ld] -> E4M3 codes [rows, cols] + E8M0 scales, 128x4 tiled
// for rows padded to 128 (padding words 0).  cols % 128 == 0.
cudaError_t launch_mx_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, uint8_t* codes, uint8_t* sf,
                               cudaStream_t s);
// MXFP8 DQ into BF16 or float32 rows of pitch ldo.  cols % 128 == 0.
cudaError_t launch_mx_dequantize(const uint8_t* codes, const uint8_t* sf, int64_t rows, int64_t cols, void* out,
                                 bool out_f32, int64_t ldo, cudaStream_t s);

// GEMM over GEMM-tiled operands (tiled.cuh): N % 256 == 0, K % 256 == 0, E <= 512.
// swiglu: the gate/up epilogue writes h = BF16(silu(gate) * up) to g.h instead of D.
// tmd: tensor map of the output, 32-row boxes: D with 128-byte boxes (128-byte swizzle),
// or h [M_total, N/2] BF16 with 64-byte boxes (64-byte swizzle).
cudaError_t launch_grouped_gemm_tiled(const uint8_t* A, const uint8_t* B, const CUtensorMap& tmd, const GemmArgs& g,
                                      int64_t max_m_tiles, bool swiglu, cudaStream_t s, bool pdl = false);
int tiled_max_experts();
// The same kernel over ragged K per expert (the weight-gradient GEMMs): g.offsets = the
// K-block prefix sums kofs [E+1], g.m_rows rows of A and D per expert, g.ga / g.gb one
// scale per expert, D [E * m_rows, N] through tmd (plain store).
cudaError_t launch_grouped_gemm_ragged_k(const uint8_t* A, const uint8_t* B, const CUtensorMap& tmd,
                                         const GemmArgs& g, cudaStream_t s);
// Backward kernels (backward.cu).
// amax_bits (nullable): zeroed, then the max |dy| of each expert's rows (starts: the
// padded group offsets [E+1]).  dy's rows are also quantised per row with stochastic
// rounding (Philox key `key`) into the GEMM-tiled dyq (128-row blocks, K = H) and g_dy.
// H % 256 == 0, H <= 2048.
cudaError_t launch_combine_backward(const void* dout, const int32_t* inv, const float* w, const void* y, int64_t T,
                                    int k, int64_t H, void* dy, float* dw, const int32_t* starts, int E,
                                    uint32_t* amax_bits, uint8_t* dyq, float* g_dy, uint64_t key, cudaStream_t s);
cudaError_t launch_group_amax(const void* src, int64_t ld, int64_t F, const int32_t* rowmap, const int32_t* starts,
                              const int32_t* counts, int E, int64_t max_rows, uint32_t* amax_bits, cudaStream_t s);
// The same maximum from per-row global scales g_rows = fl32(row max / 2688) (rows with a
// tiny non-zero scale are read).
cudaError_t launch_group_amax_g(const float* g_rows, const void* src, int64_t ld, int64_t F, const int32_t* rowmap,
                                const int32_t* starts, const int32_t* counts, int E, int64_t max_rows,
                                uint32_t* amax_bits, cudaStream_t s);
cudaError_t launch_kofs(const int32_t* counts, int64_t uniform, int E, int32_t* kofs, cudaStream_t s);
cudaError_t launch_tquant(const void* src, int64_t ld, const int32_t* rowmap, const int32_t* starts,
                          const int32_t* counts, int64_t uniform, const int32_t* kofs, int E, int F, int Fp, int R,
                          const uint32_t* amax_bits, float* g_out, uint8_t* out, int rounding, uint64_t seed,
                          int stream_id, int64_t max_kblocks, cudaStream_t s);
// Slot r (r < min(*n_rows_dev, max_rows), a multiple of 128) of the 128-row-block tiled
// `dst` gets token perm[r]'s row of the row-major per-token operand -- codes `src` [T, K/2],
// scales `src_sf` [T, K/16], both 16-byte aligned -- and dst_g[r] = src_g[perm[r]]; slots
// with perm[r] < 0 get zero codes and scales (dst_g[r] is not written).  K % 256 == 0.
// amax_zero (nullable): amax_zero[r] = 0 for every slot r < min(*n_rows_dev, max_rows).
cudaError_t launch_gather_tiled(const uint8_t* src, const uint8_t* src_sf, const float* src_g, const int32_t* perm,
                                const int32_t* n_rows_dev, int64_t max_rows, int64_t K, uint8_t* dst, float* dst_g,
                                uint32_t* amax_zero, cudaStream_t s);
// Per-row NVFP4 of h [rows, I] (BF16) whose row maxima |h| are already known (amax_bits,
// float bits): g[r] = amax / 2688, codes and scales into the GEMM-tiled layout with
// 128-row blocks and K = Ip (columns I .. Ip-1 zero).  Rows r < min(*n_rows_dev, max_rows)
// with perm[r] >= 0 are encoded; the others are not written.
// out[b*C + c, r] = x[b*R + r, c] (BF16, `batches` stacked [R, C] matrices of pitch ld).
cudaError_t launch_transpose_bf16(const void* x, int64_t batches, int64_t R, int64_t C, int64_t ld, void* out,
                                  cudaStream_t s);
// DQ of row-major codes + 128x4 tiled scales into BF16 or float32 rows of pitch ldo.
cudaError_t launch_dequantize(const uint8_t* codes, const uint8_t* sf, const float* g, int64_t rows, int64_t cols,
                              int mode, int64_t group_rows, void* out, bool out_f32, int64_t ldo, cudaStream_t s);
cudaError_t launch_requant_tiled(const __nv_bfloat16* h, const uint32_t* amax_bits, const int32_t* perm,
                                 const int32_t* n_rows_dev, int64_t max_rows, int64_t I, int64_t Ip, uint8_t* out,
                                 float* g_out, cudaStream_t s, bool pdl = false);
cudaError_t launch_pack_tiled(const uint8_t* codes, const uint8_t* sf, int64_t rows, int64_t K, int R,
                              uint8_t* out, cudaStream_t s);

// pdl (here and in the launchers below): a programmatic dependent launch (pdl.cuh), for
// decode-size batches.
cudaError_t launch_route_topk(const float* logits, int64_t T, int E, int k, int renorm, int32_t* ids,
                              float* w, cudaStream_t s, bool pdl = false);
// The forward's prologue for T*k <= 1024: the permutation (as launch_permute), each
// token's row of x quantised per row (RNE) straight into its k slots of the GEMM-tiled aq
// (128-row blocks, K = H), ga[slot] = the token's global scale, h_amax[slot] = 0.
// E <= 1024, H % 256 == 0, H <= 2048.
cudaError_t launch_prologue_small(const int32_t* ids, int64_t T, int k, int E, int32_t* counts, int32_t* offsets,
                                  int32_t* padded, int32_t* inv, int32_t* perm, int* status, const void* x, int64_t H,
                                  uint8_t* aq, float* ga, uint32_t* h_amax, cudaStream_t s);
cudaError_t launch_permute(const int32_t* ids, int64_t T, int k, int E, int32_t* counts, int32_t* offsets,
                           int32_t* padded, int32_t* inv, int32_t* perm, int32_t* hist, int64_t nchunks,
                           int* status, cudaStream_t s);
cudaError_t launch_combine(const void* y, const int32_t* inv, const float* w, int64_t T, int k, int64_t H,
                           void* out, cudaStream_t s, bool pdl = false);
// SwiGLU backward: [dgate | dup] (BF16 [rows, 2I]) from [gate | up] (BF16 [rows, 2I]) and dh
// (BF16 [rows, I]); I % 8 == 0.
// gu_interleaved: gu holds gate/up in the 64-chunk interleave of the prepared W13;
// dh_ld: row pitch of dh (0: I).
cudaError_t launch_swiglu_backward(const void* gu, const void* dh, int64_t rows, int64_t I, void* dgu,
                                   cudaStream_t s, bool gu_interleaved = false, int64_t dh_ld = 0);
// rows: rows of d to visit; nrows_dev (nullable): device count that caps rows.
cudaError_t launch_swiglu_quant(const void* d, const int32_t* perm, int64_t rows, const int32_t* nrows_dev,
                                int64_t I, int64_t Ip, void* h_out, uint8_t* hq, uint8_t* hsf, float* gh,
                                cudaStream_t s);

constexpr int64_t kPermuteChunk = 256;    // (token, j) entries per warp in the permute
inline int64_t permute_chunks(int64_t entries) { return (entries + kPermuteChunk - 1) / kPermuteChunk; }

}  // namespace nvfp4

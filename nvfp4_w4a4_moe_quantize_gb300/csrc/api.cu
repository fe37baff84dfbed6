// C ABI of the NVFP4 W4A4 MoE library: argument checks, workspace layouts, TMA tensor
// maps and the order of the kernels.  Every entry point only enqueues work on the
// caller's stream; nothing here allocates device memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "nvfp4moe.h"
#include "launch.h"
#include "status.cuh"
#include "tiled.cuh"

namespace nvfp4 {

__device__ int g_device_status;   // first error recorded by any kernel of this library

namespace {
constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices];
int* g_status_ptr[kMaxDevices];
std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device() {
  int d = 0;
  cudaGetDevice(&d);
  return d < 0 || d >= kMaxDevices ? 0 : d;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
inline int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }
inline size_t align256(size_t a) { return (a + 255) & ~size_t(255); }

nvfp4_status from_cuda(cudaError_t e) { return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_encode == nullptr) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

// 2-D map over a [rows, cols] matrix of `elt`-byte elements with row pitch `pitch_bytes`;
// box = 128 bytes x box_rows, 128-byte swizzle.
// 2-D tensor map with boxes of box_rows rows x box_bytes bytes (128: 128-byte swizzle,
// 64: 64-byte swizzle).
bool make_map(CUtensorMap* m, const void* base, int64_t rows, int64_t cols, int64_t pitch_bytes, uint32_t box_rows,
              CUtensorMapDataType dt, int elt, int box_bytes = 128) {
  auto enc = encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)pitch_bytes};
  cuuint32_t box[2] = {(cuuint32_t)(box_bytes / elt), box_rows};
  cuuint32_t es[2] = {1u, 1u};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             box_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct ForwardLayout {
  int64_t off[15];
};

// A side stream and a fork / join event pair per device, created on first use: work that
// does not depend on the caller's last operations overlaps them.  The mutex is held from
// the fork until the join is enqueued, so concurrent callers never interleave records.
struct SideStream {
  cudaStream_t stream = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};
static std::mutex g_side_mu;
static SideStream g_side[64];
static SideStream* side_stream_locked() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  SideStream& ss = g_side[dev];
  if (ss.stream == nullptr) {
    if (cudaStreamCreateWithFlags(&ss.stream, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess) {
      ss = SideStream{};
      return nullptr;
    }
  }
  return &ss;
}

// hist | counts | offsets | padded | inv | perm | Aq (tiled) | gA | h | hq (tiled) | gH | y
ForwardLayout forward_layout(int64_t T, int64_t k, int64_t E, int64_t H, int64_t I, size_t* hist_off,
                             size_t* hist_bytes) {
  ForwardLayout L;
  const int64_t Ip = round_up(I, 256);
  const int64_t mcap = round_up(T * k + E * 127, 128);
  const int64_t nchunks = permute_chunks(T * k);
  size_t p = 0;
  *hist_off = p;
  *hist_bytes = align256(sizeof(int32_t) * (size_t)(E * (nchunks > 0 ? nchunks : 1) + 1));
  p += *hist_bytes;
  auto take = [&](size_t bytes) {
    const size_t o = p;
    p += align256(bytes);
    return (int64_t)o;
  };
  L.off[0] = take(4 * E);
  L.off[1] = take(4 * (E + 1));
  L.off[2] = take(4 * (E + 1));
  L.off[3] = take(4 * T * k);
  L.off[4] = take(4 * mcap);
  L.off[5] = take((size_t)tiled_bytes(mcap, H, 128));
  L.off[6] = L.off[5];
  L.off[7] = take(4 * mcap);
  L.off[8] = take((size_t)mcap * I * 2);
  L.off[9] = take((size_t)tiled_bytes(mcap, Ip, 128));
  L.off[10] = L.off[9];
  L.off[11] = take(4 * mcap);
  L.off[12] = take((size_t)mcap * H * 2);
  L.off[13] = mcap;
  L.off[14] = (int64_t)p;
  return L;
}

struct BackwardLayout {
  int64_t off[18];
};

// dy | dyq (tiled, K = H) | g_dy | dh [M, Ip] | D [M, 2I] | dD [M, 2I] | dDq (tiled, K = 2I) |
// g_dD | dxs [M, H] | kofs | amax [4E] | g [4E] | wgrad operands: dy^T, h^T, dD^T, x^T
BackwardLayout backward_layout(int64_t T, int64_t k, int64_t E, int64_t H, int64_t I) {
  BackwardLayout L;
  const int64_t Ip = round_up(I, 256);
  const int64_t mcap = round_up(T * k + E * 127, 128);
  const int64_t kb = T * k / 256 + E + 1;        // >= sum over experts of max(1, ceil(count / 256))
  size_t p = 0;
  auto take = [&](size_t bytes) {
    const size_t o = p;
    p += align256(bytes);
    return (int64_t)o;
  };
  L.off[0] = take((size_t)mcap * H * 2);
  L.off[1] = take((size_t)tiled_bytes(mcap, H, 128));
  L.off[2] = take(4 * (size_t)mcap);
  L.off[3] = take((size_t)mcap * Ip * 2);
  L.off[4] = take((size_t)mcap * 2 * I * 2);
  L.off[5] = take((size_t)mcap * 2 * I * 2);
  L.off[6] = take((size_t)tiled_bytes(mcap, 2 * I, 128));
  L.off[7] = take(4 * (size_t)mcap);
  L.off[8] = take((size_t)mcap * H * 2);
  L.off[9] = take(4 * (size_t)(E + 1));
  L.off[10] = take(16 * (size_t)E);
  L.off[11] = take(16 * (size_t)E);
  L.off[12] = take((size_t)(H / 128) * kb * 128 * 144);
  L.off[13] = take((size_t)(Ip / 256) * kb * 256 * 144);
  L.off[14] = take((size_t)(2 * I / 128) * kb * 128 * 144);
  L.off[15] = take((size_t)(H / 256) * kb * 256 * 144);
  L.off[16] = kb;
  L.off[17] = (int64_t)p;
  return L;
}

nvfp4_status gemm(const uint8_t* A, const uint8_t* SFA, const float* gA, const uint8_t* B, const uint8_t* SFB,
                  const float* gB, const int32_t* offsets, const int32_t* rows, int64_t M_total, int64_t N, int64_t K,
                  int32_t E, void* D, int out_f32, int64_t ldd, cudaStream_t s) {
  GemmArgs g{};
  g.sfa = SFA;
  g.sfb = SFB;
  g.ga = gA;
  g.gb = gB;
  g.offsets = offsets;
  g.rows = rows;
  g.m_total = M_total;
  g.E = E;
  g.N = (int32_t)N;
  g.K = (int32_t)K;
  g.d = D;
  g.ldd = ldd;
  g.out_f32 = out_f32;
  g.status = device_status_ptr();
  const bool wide = n256_supported(g);   // its B map also has 128-row boxes (two per 256-row tile)
  CUtensorMap ma, mb, md;
  if (!make_map(&ma, A, M_total, K / 2, K / 2, 128, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1) ||
      !make_map(&mb, B, (int64_t)E * N, K / 2, K / 2, 128, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1))
    return NVFP4_ERR_CUDA;
  if (wide) return from_cuda(launch_grouped_gemm_n256(ma, mb, g, M_total / 128, s));
  if (!make_map(&md, D, M_total, N, ldd * (out_f32 ? 4 : 2), 32,
                out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out_f32 ? 4 : 2))
    return NVFP4_ERR_CUDA;
  return from_cuda(launch_grouped_gemm(ma, mb, md, g, M_total / 128, s));
}

}  // namespace

int num_sms() {
  const int d = current_device();
  if (g_sms[d] == 0) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, d);
    g_sms[d] = v > 0 ? v : 1;
  }
  return g_sms[d];
}

int* device_status_ptr() {
  const int d = current_device();
  if (g_status_ptr[d] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) == cudaSuccess) g_status_ptr[d] = static_cast<int*>(p);
  }
  return g_status_ptr[d];
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

size_t nvfp4_sf_bytes(int64_t rows, int64_t cols) {
  if (rows <= 0 || cols <= 0) return 0;
  return (size_t)((rows + 127) / 128) * (size_t)((cols + 63) / 64) * 512u;
}

nvfp4_status moe_weights_sizes(int32_t E, int64_t H, int64_t I, size_t sizes_out[4]) {
  if (E <= 0 || H <= 0 || I <= 0 || sizes_out == nullptr) return NVFP4_ERR_INVALID_ARG;
  const int64_t Ip = round_up(I, 256);
  sizes_out[0] = (size_t)tiled_bytes((int64_t)E * 2 * I, H, 256);
  sizes_out[1] = 4u * (size_t)E;
  sizes_out[2] = (size_t)tiled_bytes((int64_t)E * H, Ip, 256);
  sizes_out[3] = 4u * (size_t)E;
  return NVFP4_OK;
}

size_t nvfp4_tiled_bytes(int64_t rows, int64_t K, int32_t block_rows) {
  if (rows <= 0 || K <= 0 || K % 256 != 0 || (block_rows != 128 && block_rows != 256)) return 0;
  return (size_t)tiled_bytes(rows, K, block_rows);
}

size_t nvfp4_workspace_size(int op, int64_t a, int64_t b, int64_t E, int64_t H, int64_t I) {
  switch (op) {
    case NVFP4_OP_QUANTIZE:
      return align256(4u * (size_t)(a > 1 ? a : 1));
    case NVFP4_OP_PREPARE_WEIGHTS:
      return align256(8u * (size_t)(a > 1 ? a : 1));
    case NVFP4_OP_MOE_FORWARD: {
      size_t ho, hb;
      return (size_t)forward_layout(a, b, E, H, I, &ho, &hb).off[14];
    }
    case NVFP4_OP_MOE_PERMUTE: {
      const int64_t n = permute_chunks(a * b);
      return align256(4u * (size_t)(E * (n > 0 ? n : 1) + 1));   // chunk histograms + a completion counter
    }
    case NVFP4_OP_QUANTIZE_T:   // transposed BF16 copy [a, b] + amax scratch for up to a scopes
      return align256(2u * (size_t)a * (size_t)b) + align256(4u * (size_t)(a > 1 ? a : 1));
    case NVFP4_OP_MOE_BACKWARD:
      return (size_t)backward_layout(a, b, E, H, I).off[17];
    case NVFP4_OP_PREPARE_WEIGHTS_T:   // amax [2E] + K-block prefix sums [2(E+1)]
      return align256(8u * (size_t)(a > 1 ? a : 1)) + align256(8u * (size_t)((a > 1 ? a : 1) + 1));
    default:
      return 0;
  }
}

nvfp4_status moe_forward_workspace_layout(int64_t T, int32_t k, int32_t E, int64_t H, int64_t I,
                                          int64_t layout_out[15]) {
  if (T < 0 || k <= 0 || E <= 0 || H <= 0 || I <= 0 || layout_out == nullptr) return NVFP4_ERR_INVALID_ARG;
  size_t ho, hb;
  const ForwardLayout L = forward_layout(T, k, E, H, I, &ho, &hb);
  std::memcpy(layout_out, L.off, sizeof(L.off));
  return NVFP4_OK;
}

nvfp4_status nvfp4_status_check(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return NVFP4_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  if (v == kStatusTimeout) return NVFP4_ERR_TIMEOUT;
  if (v != 0) return NVFP4_ERR_DEVICE_STATUS;
  return NVFP4_OK;
}

const char* nvfp4_status_string(nvfp4_status s) {
  switch (s) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4_ERR_UNSUPPORTED: return "unsupported shape";
    case NVFP4_ERR_WORKSPACE: return "workspace too small";
    case NVFP4_ERR_CUDA: return "CUDA error";
    case NVFP4_ERR_DEVICE_STATUS: return "device reported invalid input";
    case NVFP4_ERR_TIMEOUT: return "device-side wait timed out";
    default: return "unknown status";
  }
}

nvfp4_status nvfp4_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld, nvfp4_scale_mode mode,
                            int64_t group_rows, nvfp4_rounding rounding, uint64_t seed, uint64_t rng_offset,
                            const float* g_in, float* g_out, uint8_t* codes, uint8_t* sf,
                            nvfp4_sf_layout sf_layout, void* ws, size_t ws_bytes, void* stream) {
  if (rows < 0 || cols <= 0 || cols % 16 != 0 || ld < cols || ld % 8 != 0) return NVFP4_ERR_INVALID_ARG;
  if (sf_layout != NVFP4_SF_SWIZZLED_128x4 && sf_layout != NVFP4_SF_ROWMAJOR) return NVFP4_ERR_INVALID_ARG;
  if (cols > 8192 || (sf_layout == NVFP4_SF_ROWMAJOR && cols % 64 != 0)) return NVFP4_ERR_UNSUPPORTED;
  if (mode < NVFP4_SCALE_PER_TENSOR || mode > NVFP4_SCALE_PER_GROUP) return NVFP4_ERR_INVALID_ARG;
  if (rounding != NVFP4_ROUND_RNE && rounding != NVFP4_ROUND_STOCHASTIC) return NVFP4_ERR_INVALID_ARG;
  if (mode == NVFP4_SCALE_PER_GROUP && (group_rows <= 0 || rows % group_rows != 0)) return NVFP4_ERR_INVALID_ARG;
  if (rows == 0) return NVFP4_OK;
  if (!x || !codes || !sf || !aligned16(x) || !aligned16(codes) || !aligned16(sf)) return NVFP4_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t n_scopes = mode == NVFP4_SCALE_PER_TENSOR ? 1 : (mode == NVFP4_SCALE_PER_GROUP ? rows / group_rows : rows);
  uint32_t* amax = nullptr;
  if (mode != NVFP4_SCALE_PER_ROW && g_in == nullptr) {
    if (ws == nullptr || ws_bytes < 4u * (size_t)n_scopes || !aligned16(ws)) return NVFP4_ERR_WORKSPACE;
    amax = static_cast<uint32_t*>(ws);
    cudaError_t e = launch_amax(x, rows, cols, ld, mode == NVFP4_SCALE_PER_GROUP ? group_rows : 0, amax, n_scopes, s);
    if (e != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  QuantArgs a{};
  a.x = static_cast<const __nv_bfloat16*>(x);
  a.rows = rows;
  a.cols = cols;
  a.ld = ld;
  a.mode = mode;
  a.group_rows = group_rows;
  a.g_in = g_in;
  a.amax_bits = amax;
  a.g_out = g_out;
  a.codes = codes;
  a.codes_ld = cols / 2;
  a.sf = sf;
  a.sf_words = (cols + 63) / 64;
  a.sf_row_bytes = sf_layout == NVFP4_SF_ROWMAJOR ? cols / 16 : 0;
  a.cols_pad = cols;
  a.rows_total = sf_layout == NVFP4_SF_ROWMAJOR ? rows : round_up(rows, 128);
  a.map = kMapIdentity;
  a.seed = seed;
  a.rng_offset = rng_offset;
  a.status = device_status_ptr();
  // after an amax pass the encode is its programmatic dependent (its launch overlaps the
  // pass's tail)
  return from_cuda(launch_quantize_rows(a, rounding, s, amax != nullptr));
}

nvfp4_status nvfp4_quantize_transposed(const void* x, int64_t batches, int64_t R, int64_t C, int64_t ld,
                                       nvfp4_scale_mode mode, int64_t group_rows, nvfp4_rounding rounding,
                                       uint64_t seed, uint64_t rng_offset, const float* g_in, float* g_out,
                                       uint8_t* codes, uint8_t* sf, void* ws, size_t ws_bytes, void* stream) {
  if (batches < 0 || R <= 0 || C <= 0 || R % 16 != 0 || ld < C || ld % 8 != 0) return NVFP4_ERR_INVALID_ARG;
  if (R > 8192) return NVFP4_ERR_UNSUPPORTED;
  if (batches == 0) return NVFP4_OK;
  if (!x || !aligned16(x)) return NVFP4_ERR_INVALID_ARG;
  const int64_t rows_t = batches * C;
  const size_t t_bytes = align256(2u * (size_t)rows_t * (size_t)R);
  if (ws == nullptr || !aligned16(ws) || ws_bytes < nvfp4_workspace_size(NVFP4_OP_QUANTIZE_T, rows_t, R, 0, 0, 0))
    return NVFP4_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_transpose_bf16(x, batches, R, C, ld, ws, s) != cudaSuccess) return NVFP4_ERR_CUDA;
  return nvfp4_quantize(ws, rows_t, R, R, mode, group_rows, rounding, seed, rng_offset, g_in, g_out, codes, sf,
                        NVFP4_SF_SWIZZLED_128x4, static_cast<uint8_t*>(ws) + t_bytes, ws_bytes - t_bytes, stream);
}

nvfp4_status nvfp4_dequantize(const uint8_t* codes, const uint8_t* sf, const float* g, int64_t rows, int64_t cols,
                              nvfp4_scale_mode mode, int64_t group_rows, void* out, nvfp4_out_dtype out_dtype,
                              int64_t ldo, void* stream) {
  if (rows < 0 || cols <= 0 || cols % 16 != 0 || ldo < cols || ldo % 8 != 0) return NVFP4_ERR_INVALID_ARG;
  if (mode < NVFP4_SCALE_PER_TENSOR || mode > NVFP4_SCALE_PER_GROUP) return NVFP4_ERR_INVALID_ARG;
  if (mode == NVFP4_SCALE_PER_GROUP && (group_rows <= 0 || rows % group_rows != 0)) return NVFP4_ERR_INVALID_ARG;
  if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_F32) return NVFP4_ERR_INVALID_ARG;
  if (rows == 0) return NVFP4_OK;
  if (!codes || !sf || !g || !out || !aligned16(codes) || !aligned16(sf) || !aligned16(out) || !aligned4(g))
    return NVFP4_ERR_INVALID_ARG;
  return from_cuda(launch_dequantize(codes, sf, g, rows, cols, mode, group_rows, out, out_dtype == NVFP4_OUT_F32, ldo,
                                     static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_grouped_gemm(const uint8_t* A, const uint8_t* SFA, const float* gA, const uint8_t* B,
                                const uint8_t* SFB, const float* gB, const int32_t* group_offsets,
                                const int32_t* group_rows, int64_t M_total, int64_t N, int64_t K, int32_t E,
                                void* D, nvfp4_out_dtype out_dtype, int64_t ldd, void* stream) {
  if (E <= 0 || E > 1024 || N <= 0 || K <= 0 || M_total < 0 || M_total % 128 != 0) return NVFP4_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 256 != 0) return NVFP4_ERR_UNSUPPORTED;
  if ((int64_t)E * N >= (int64_t)1 << 31 || M_total >= (int64_t)1 << 31 || K >= (int64_t)1 << 20)
    return NVFP4_ERR_UNSUPPORTED;
  if (ldd < N || ldd % 8 != 0) return NVFP4_ERR_INVALID_ARG;
  if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_F32) return NVFP4_ERR_INVALID_ARG;
  if (M_total == 0) return NVFP4_OK;
  const void* ptrs[] = {A, SFA, B, SFB, D};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return NVFP4_ERR_INVALID_ARG;
  if (!aligned4(gA) || !aligned4(gB) || !aligned4(group_offsets) || !aligned4(group_rows))
    return NVFP4_ERR_INVALID_ARG;
  return gemm(A, SFA, gA, B, SFB, gB, group_offsets, group_rows, M_total, N, K, E, D,
              out_dtype == NVFP4_OUT_F32, ldd, static_cast<cudaStream_t>(stream));
}

size_t mxfp8_sf_bytes(int64_t rows, int64_t cols) {
  if (rows <= 0 || cols <= 0) return 0;
  return (size_t)((rows + 127) / 128) * (size_t)((cols + 127) / 128) * 512u;
}

nvfp4_status mxfp8_quantize(const void* x, int64_t rows, int64_t cols, int64_t ld_elems, uint8_t* codes_out,
                            uint8_t* sf_out, void* stream) {
  if (rows < 0 || cols <= 0 || ld_elems < cols || ld_elems % 8 != 0) return NVFP4_ERR_INVALID_ARG;
  if (cols % 128 != 0) return NVFP4_ERR_UNSUPPORTED;
  if (rows == 0) return NVFP4_OK;
  if (!x || !codes_out || !sf_out || !aligned16(x) || !aligned16(codes_out) || !aligned16(sf_out))
    return NVFP4_ERR_INVALID_ARG;
  return from_cuda(launch_mx_quantize(x, rows, cols, ld_elems, codes_out, sf_out, static_cast<cudaStream_t>(stream)));
}

nvfp4_status mxfp8_dequantize(const uint8_t* codes, const uint8_t* sf, int64_t rows, int64_t cols, void* out,
                              nvfp4_out_dtype out_dtype, int64_t ldo, void* stream) {
  if (rows < 0 || cols <= 0 || ldo < cols || ldo % 8 != 0) return NVFP4_ERR_INVALID_ARG;
  if (cols % 128 != 0) return NVFP4_ERR_UNSUPPORTED;
  if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_F32) return NVFP4_ERR_INVALID_ARG;
  if (rows == 0) return NVFP4_OK;
  if (!codes || !sf || !out || !aligned16(codes) || !aligned16(sf) || !aligned16(out)) return NVFP4_ERR_INVALID_ARG;
  return from_cuda(launch_mx_dequantize(codes, sf, rows, cols, out, out_dtype == NVFP4_OUT_F32, ldo,
                                        static_cast<cudaStream_t>(stream)));
}

nvfp4_status mxfp8_grouped_gemm(const uint8_t* A, const uint8_t* SFA, const uint8_t* B, const uint8_t* SFB,
                                const int32_t* group_offsets, const int32_t* group_rows, int64_t M_total, int64_t N,
                                int64_t K, int32_t E, void* D, nvfp4_out_dtype out_dtype, int64_t ldd,
                                void* stream) {
  if (E <= 0 || E > 1024 || N <= 0 || K <= 0 || M_total < 0 || M_total % 128 != 0) return NVFP4_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 128 != 0) return NVFP4_ERR_UNSUPPORTED;
  if ((int64_t)E * N >= (int64_t)1 << 31 || M_total >= (int64_t)1 << 31 || K >= (int64_t)1 << 20)
    return NVFP4_ERR_UNSUPPORTED;
  if (ldd < N || ldd % 8 != 0) return NVFP4_ERR_INVALID_ARG;
  if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_F32) return NVFP4_ERR_INVALID_ARG;
  if (M_total == 0) return NVFP4_OK;
  const void* ptrs[] = {A, SFA, B, SFB, D};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return NVFP4_ERR_INVALID_ARG;
  if (!aligned4(group_offsets) || !aligned4(group_rows)) return NVFP4_ERR_INVALID_ARG;
  const bool out_f32 = out_dtype == NVFP4_OUT_F32;
  GemmArgs g{};
  g.sfa = SFA;
  g.sfb = SFB;
  g.offsets = group_offsets;
  g.rows = group_rows;
  g.m_total = M_total;
  g.E = E;
  g.N = (int32_t)N;
  g.K = (int32_t)K;
  g.d = D;
  g.ldd = ldd;
  g.out_f32 = out_f32;
  g.status = device_status_ptr();
  CUtensorMap ma, mb, md;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!make_map(&ma, A, M_total, K, K, 128, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1) ||
      !make_map(&mb, B, (int64_t)E * N, K, K, 128, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1))
    return NVFP4_ERR_CUDA;
  // N % 256 == 0: 128 x 256 tiles; else 128 x 128
  if (n256_supported(g)) return from_cuda(launch_grouped_gemm_n256_mx(ma, mb, g, M_total / 128, s));
  if (!make_map(&md, D, M_total, N, ldd * (out_f32 ? 4 : 2), 32,
                out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out_f32 ? 4 : 2))
    return NVFP4_ERR_CUDA;
  return from_cuda(launch_grouped_gemm_mx(ma, mb, md, g, M_total / 128, s));
}

nvfp4_status bf16_grouped_gemm(const void* A, const void* B, const int32_t* group_offsets,
                               const int32_t* group_rows, int64_t M_total, int64_t N, int64_t K, int32_t E, void* D,
                               nvfp4_out_dtype out_dtype, int64_t ldd, void* stream) {
  if (E <= 0 || E > 1024 || N <= 0 || K <= 0 || M_total < 0 || M_total % 128 != 0) return NVFP4_ERR_INVALID_ARG;
  if (N % 128 != 0 || K % 64 != 0) return NVFP4_ERR_UNSUPPORTED;
  if ((int64_t)E * N >= (int64_t)1 << 31 || M_total >= (int64_t)1 << 31 || K >= (int64_t)1 << 20)
    return NVFP4_ERR_UNSUPPORTED;
  if (ldd < N || ldd % 8 != 0) return NVFP4_ERR_INVALID_ARG;
  if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_F32) return NVFP4_ERR_INVALID_ARG;
  if (M_total == 0) return NVFP4_OK;
  const void* ptrs[] = {A, B, D};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return NVFP4_ERR_INVALID_ARG;
  if (!aligned4(group_offsets) || !aligned4(group_rows)) return NVFP4_ERR_INVALID_ARG;
  const bool out_f32 = out_dtype == NVFP4_OUT_F32;
  GemmArgs g{};
  g.offsets = group_offsets;
  g.rows = group_rows;
  g.m_total = M_total;
  g.E = E;
  g.N = (int32_t)N;
  g.K = (int32_t)K;
  g.d = D;
  g.ldd = ldd;
  g.out_f32 = out_f32;
  g.status = device_status_ptr();
  // the BF16 operands as byte matrices: 128-byte boxes are 64 values of K
  CUtensorMap ma, mb, md;
  if (!make_map(&ma, A, M_total, 2 * K, 2 * K, 128, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1) ||
      !make_map(&mb, B, (int64_t)E * N, 2 * K, 2 * K, 128, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1) ||
      !make_map(&md, D, M_total, N, ldd * (out_f32 ? 4 : 2), 32,
                out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, out_f32 ? 4 : 2))
    return NVFP4_ERR_CUDA;
  return from_cuda(launch_grouped_gemm_bf16(ma, mb, md, g, M_total / 128, static_cast<cudaStream_t>(stream)));
}

nvfp4_status moe_swiglu_backward(const void* gu, const void* dh, int64_t rows, int64_t I, void* dgu,
                                 void* stream) {
  if (rows < 0 || I <= 0 || I % 8 != 0) return NVFP4_ERR_INVALID_ARG;
  if (rows == 0) return NVFP4_OK;
  if (!gu || !dh || !dgu || !aligned16(gu) || !aligned16(dh) || !aligned16(dgu)) return NVFP4_ERR_INVALID_ARG;
  return from_cuda(launch_swiglu_backward(gu, dh, rows, I, dgu, static_cast<cudaStream_t>(stream)));
}

nvfp4_status bf16_transpose(const void* x, int64_t batches, int64_t R, int64_t C, int64_t ld, void* out,
                            void* stream) {
  if (batches < 0 || R < 0 || C < 0 || ld < C) return NVFP4_ERR_INVALID_ARG;
  if (batches == 0 || R == 0 || C == 0) return NVFP4_OK;
  if (x == nullptr || out == nullptr || !aligned4(x) || !aligned4(out)) return NVFP4_ERR_INVALID_ARG;
  return from_cuda(launch_transpose_bf16(x, batches, R, C, ld, out, static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_grouped_gemm_tiled(const uint8_t* A, const float* gA, const uint8_t* B, const float* gB,
                                      const int32_t* group_offsets, const int32_t* group_rows, int64_t M_total,
                                      int64_t N, int64_t K, int32_t E, void* D, nvfp4_out_dtype out_dtype,
                                      int64_t ldd, int32_t epilogue, void* stream) {
  if (E <= 0 || E > tiled_max_experts() || N <= 0 || K <= 0 || M_total < 0 || M_total % 128 != 0)
    return NVFP4_ERR_INVALID_ARG;
  if (N % 256 != 0 || K % 256 != 0) return NVFP4_ERR_UNSUPPORTED;
  if ((int64_t)E * N >= (int64_t)1 << 31 || M_total >= (int64_t)1 << 31 || K >= (int64_t)1 << 20)
    return NVFP4_ERR_UNSUPPORTED;
  if (epilogue != NVFP4_EPILOGUE_STORE && epilogue != NVFP4_EPILOGUE_SWIGLU) return NVFP4_ERR_INVALID_ARG;
  if (epilogue == NVFP4_EPILOGUE_STORE) {
    if (ldd < N || ldd % 8 != 0) return NVFP4_ERR_INVALID_ARG;
    if (out_dtype != NVFP4_OUT_BF16 && out_dtype != NVFP4_OUT_F32) return NVFP4_ERR_INVALID_ARG;
  }
  if (M_total == 0) return NVFP4_OK;
  const void* ptrs[] = {A, B, D};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return NVFP4_ERR_INVALID_ARG;
  if (!aligned4(gA) || !aligned4(gB) || !aligned4(group_offsets) || !aligned4(group_rows))
    return NVFP4_ERR_INVALID_ARG;
  GemmArgs g{};
  g.ga = gA;
  g.gb = gB;
  g.offsets = group_offsets;
  g.rows = group_rows;
  g.m_total = M_total;
  g.E = E;
  g.N = (int32_t)N;
  g.K = (int32_t)K;
  g.d = D;
  g.ldd = ldd;
  g.out_f32 = out_dtype == NVFP4_OUT_F32;
  g.status = device_status_ptr();
  g.h = static_cast<__nv_bfloat16*>(D);
  g.I = N / 2;
  const bool swiglu = epilogue == NVFP4_EPILOGUE_SWIGLU;
  if (swiglu && (g.silu_tab = silu_table(static_cast<cudaStream_t>(stream))) == nullptr) return NVFP4_ERR_CUDA;
  CUtensorMap md;
  const bool ok = swiglu ? make_map(&md, D, M_total, N / 2, N, 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64)
                         : make_map(&md, D, M_total, N, ldd * (g.out_f32 ? 4 : 2), 32,
                                    g.out_f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                                    g.out_f32 ? 4 : 2);
  if (!ok) return NVFP4_ERR_CUDA;
  return from_cuda(launch_grouped_gemm_tiled(A, B, md, g, M_total / 128, swiglu, static_cast<cudaStream_t>(stream)));
}

nvfp4_status nvfp4_pack_tiled(const uint8_t* codes, const uint8_t* sf, int64_t rows, int64_t K, int32_t block_rows,
                              uint8_t* out, void* stream) {
  if (rows < 0 || K <= 0 || K % 256 != 0 || (block_rows != 128 && block_rows != 256)) return NVFP4_ERR_INVALID_ARG;
  if (rows == 0) return NVFP4_OK;
  if (!codes || !sf || !out || !aligned16(codes) || !aligned16(sf) || !aligned16(out)) return NVFP4_ERR_INVALID_ARG;
  return from_cuda(launch_pack_tiled(codes, sf, rows, K, block_rows, out, static_cast<cudaStream_t>(stream)));
}

nvfp4_status moe_route_topk(const float* logits, int64_t T, int32_t E, int32_t k, int renormalize, int32_t* ids,
                            float* weights, void* stream) {
  if (T < 0 || E <= 0 || E > 1024 || k <= 0 || k > 32 || k > E) return NVFP4_ERR_INVALID_ARG;
  if (T == 0) return NVFP4_OK;
  if (!logits || !ids || !weights) return NVFP4_ERR_INVALID_ARG;
  // decode-size batches: a programmatic dependent launch (as the expert block's kernels)
  return from_cuda(launch_route_topk(logits, T, E, k, renormalize, ids, weights, static_cast<cudaStream_t>(stream),
                                     T * k <= 1024));
}

nvfp4_status moe_permute(const int32_t* ids, int64_t T, int32_t k, int32_t E, int32_t* counts, int32_t* offsets,
                         int32_t* padded_offsets, int32_t* inv, int32_t* perm, void* ws, size_t ws_bytes,
                         void* stream) {
  if (T < 0 || k <= 0 || k > 32 || E <= 0 || E > 1024 || T * k >= ((int64_t)1 << 31) - (int64_t)E * 128)
    return NVFP4_ERR_INVALID_ARG;
  if (!counts || !offsets || !padded_offsets || (T > 0 && (!ids || !inv))) return NVFP4_ERR_INVALID_ARG;
  const size_t need = nvfp4_workspace_size(NVFP4_OP_MOE_PERMUTE, T, k, E, 0, 0);
  if (ws == nullptr || ws_bytes < need) return NVFP4_ERR_WORKSPACE;
  return from_cuda(launch_permute(ids, T, k, E, counts, offsets, padded_offsets, inv, perm,
                                  static_cast<int32_t*>(ws), permute_chunks(T * k), device_status_ptr(),
                                  static_cast<cudaStream_t>(stream)));
}

nvfp4_status moe_combine(const void* y, const int32_t* inv, const float* w, int64_t T, int32_t k, int64_t H,
                         void* out, void* stream) {
  if (T < 0 || k <= 0 || k > 32 || H <= 0 || H % 8 != 0) return NVFP4_ERR_INVALID_ARG;
  if (T == 0) return NVFP4_OK;
  if (!y || !inv || !w || !out || !aligned16(y) || !aligned16(out)) return NVFP4_ERR_INVALID_ARG;
  return from_cuda(launch_combine(y, inv, w, T, k, H, out, static_cast<cudaStream_t>(stream)));
}

nvfp4_status moe_swiglu_quantize(const void* d, const int32_t* perm, int64_t rows, int64_t I, void* h_out,
                                 uint8_t* hq, uint8_t* hsf, float* gh, void* stream) {
  if (rows < 0 || I <= 0 || I % 64 != 0 || I > 4096) return NVFP4_ERR_INVALID_ARG;
  if (rows == 0) return NVFP4_OK;
  if (!d || !perm || !hq || !hsf || !gh || !aligned16(d) || !aligned16(hq) || !aligned16(hsf))
    return NVFP4_ERR_INVALID_ARG;
  if (h_out != nullptr && !aligned16(h_out)) return NVFP4_ERR_INVALID_ARG;
  return from_cuda(launch_swiglu_quant(d, perm, rows, nullptr, I, round_up(I, 256), h_out, hq, hsf, gh,
                                       static_cast<cudaStream_t>(stream)));
}

nvfp4_status moe_prepare_weights(const void* w13, const void* w2, int32_t E, int64_t H, int64_t I,
                                 const nvfp4_moe_weights* out, void* ws, size_t ws_bytes, void* stream) {
  if (E <= 0 || H <= 0 || I <= 0 || out == nullptr) return NVFP4_ERR_INVALID_ARG;
  if (E > tiled_max_experts() || H % 256 != 0 || I % 128 != 0 || H > 2048 || I > 2048) return NVFP4_ERR_UNSUPPORTED;
  if (out->E != E || out->H != H || out->I != I) return NVFP4_ERR_INVALID_ARG;
  const void* ptrs[] = {w13, w2, out->w13, out->w13_g, out->w2, out->w2_g};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return NVFP4_ERR_INVALID_ARG;
  if (ws == nullptr || ws_bytes < nvfp4_workspace_size(NVFP4_OP_PREPARE_WEIGHTS, E, 0, 0, 0, 0) || !aligned16(ws))
    return NVFP4_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t Ip = round_up(I, 256);
  uint32_t* amax = static_cast<uint32_t*>(ws);
  cudaError_t e = launch_amax(w13, (int64_t)E * 2 * I, H, H, 2 * I, amax, E, s);
  if (e != cudaSuccess) return NVFP4_ERR_CUDA;
  QuantArgs a{};
  a.x = static_cast<const __nv_bfloat16*>(w13);
  a.rows = (int64_t)E * 2 * I;
  a.cols = H;
  a.ld = H;
  a.mode = kScopeGroup;
  a.group_rows = 2 * I;
  a.amax_bits = amax;
  a.g_out = out->w13_g;
  a.codes = out->w13;
  a.sf_words = H / 64;
  a.cols_pad = H;
  a.rows_total = a.rows;
  a.map = kMapInterleave;
  a.map_I = I;
  a.status = device_status_ptr();
  a.tiled_R = 256;
  a.kblocks = H / 256;
  e = launch_quantize_rows(a, kRoundRNE, s);
  if (e != cudaSuccess) return NVFP4_ERR_CUDA;
  uint32_t* amax2 = amax + E;
  e = launch_amax(w2, (int64_t)E * H, I, I, H, amax2, E, s);
  if (e != cudaSuccess) return NVFP4_ERR_CUDA;
  QuantArgs b{};
  b.x = static_cast<const __nv_bfloat16*>(w2);
  b.rows = (int64_t)E * H;
  b.cols = I;
  b.ld = I;
  b.mode = kScopeGroup;
  b.group_rows = H;
  b.amax_bits = amax2;
  b.g_out = out->w2_g;
  b.codes = out->w2;
  b.sf_words = Ip / 64;
  b.cols_pad = Ip;
  b.rows_total = b.rows;
  b.map = kMapIdentity;
  b.status = device_status_ptr();
  b.tiled_R = 256;
  b.kblocks = Ip / 256;
  return from_cuda(launch_quantize_rows(b, kRoundRNE, s));
}

nvfp4_status moe_expert_forward(const void* x, const int32_t* ids, const float* w, int64_t T, int32_t k,
                                const nvfp4_moe_weights* wt, void* out, void* ws, size_t ws_bytes, void* stream) {
  if (wt == nullptr || T < 0 || k <= 0 || k > 32) return NVFP4_ERR_INVALID_ARG;
  const int32_t E = wt->E;
  const int64_t H = wt->H, I = wt->I;
  if (E <= 0 || E > tiled_max_experts() || k > E) return NVFP4_ERR_INVALID_ARG;
  if (H % 256 != 0 || I % 128 != 0 || H > 2048 || I > 2048) return NVFP4_ERR_UNSUPPORTED;
  if (T * k >= ((int64_t)1 << 31) - (int64_t)E * 128) return NVFP4_ERR_UNSUPPORTED;
  if (T == 0) return NVFP4_OK;
  const void* ptrs[] = {x, out, ws, wt->w13, wt->w13_g, wt->w2, wt->w2_g};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return NVFP4_ERR_INVALID_ARG;
  if (!aligned4(ids) || !aligned4(w)) return NVFP4_ERR_INVALID_ARG;   // read element by element
  size_t hist_off, hist_bytes;
  const ForwardLayout L = forward_layout(T, k, E, H, I, &hist_off, &hist_bytes);
  if (ws_bytes < (size_t)L.off[14]) return NVFP4_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* base = static_cast<uint8_t*>(ws);
  auto at = [&](int i) { return base + L.off[i]; };
  int32_t* counts = reinterpret_cast<int32_t*>(at(0));
  int32_t* offsets = reinterpret_cast<int32_t*>(at(1));
  int32_t* padded = reinterpret_cast<int32_t*>(at(2));
  int32_t* inv = reinterpret_cast<int32_t*>(at(3));
  int32_t* perm = reinterpret_cast<int32_t*>(at(4));
  uint8_t* aq = at(5);
  float* ga = reinterpret_cast<float*>(at(7));
  __nv_bfloat16* hbuf = reinterpret_cast<__nv_bfloat16*>(at(8));
  uint8_t* hq = at(9);
  float* gh = reinterpret_cast<float*>(at(11));
  void* ybuf = at(12);
  const int64_t mcap = L.off[13];
  const int64_t Ip = round_up(I, 256);
  int* status = device_status_ptr();

  // per-token operand -- row-major codes [T, H/2], then row-major scales [T, H/16] -- and
  // its global scales (parked in y's region, free until the down GEMM; the reservation is
  // that of the tiled form, which is no smaller), then the per-row max |h| that the
  // gate/up epilogue accumulates
  uint8_t* xq = static_cast<uint8_t*>(ybuf);
  float* gx = reinterpret_cast<float*>(xq + align256(tiled_bytes(T, H, 128)));
  uint32_t* h_amax = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(gx) + align256(sizeof(float) * T));
  cudaError_t e;
  // decode-size batches: one prologue launch, and every kernel of the chain a programmatic
  // dependent launch (its launch overlaps the previous kernel's tail)
  const bool small = T * k <= 1024 && E <= 1024;
  if (small) {
    // 1-2. decode-size batches: grouping, per-token NVFP4 of x and its placement in every
    //      routed slot in one launch (one CTA per token)
    e = launch_prologue_small(ids, T, k, E, counts, offsets, padded, inv, perm, status, x, H, aq, ga, h_amax, s);
    if (e != cudaSuccess) return NVFP4_ERR_CUDA;
  } else {
    // 1-2. expert grouping on the caller's stream and, forked onto a side stream at the same
    //      point, the per-token NVFP4 of x into a token-ordered row-major operand (it does
    //      not depend on the grouping); then, joined, the gather into every routed slot
    //      of the GEMM-tiled operand with the token's global scale (padding slots zero,
    //      h_amax zero).  Row-major scales make a slot's 16 scale bytes of a K block one
    //      read (measured: forward 697 vs 700 us with the tiled per-token operand)
    std::lock_guard<std::mutex> lk(g_side_mu);
    SideStream* ss = side_stream_locked();
    if (ss == nullptr) return NVFP4_ERR_CUDA;
    if (cudaEventRecord(ss->fork, s) != cudaSuccess || cudaStreamWaitEvent(ss->stream, ss->fork, 0) != cudaSuccess)
      return NVFP4_ERR_CUDA;
    QuantArgs a{};
    a.x = static_cast<const __nv_bfloat16*>(x);
    a.rows = T;
    a.cols = H;
    a.ld = H;
    a.mode = kScopeRow;
    a.g_out = gx;
    a.codes = xq;
    a.sf_words = H / 64;
    a.cols_pad = H;
    a.rows_total = T;
    a.map = kMapIdentity;
    a.status = status;
    a.codes_ld = H / 2;
    a.sf = xq + T * H / 2;
    a.sf_row_bytes = H / 16;
    // (measured: enqueueing the grouping first gained nothing; this order hides 6 us)
    const cudaError_t eq = launch_quantize_rows(a, kRoundRNE, ss->stream);
    const cudaError_t ep = launch_permute(ids, T, k, E, counts, offsets, padded, inv, perm,
                                          reinterpret_cast<int32_t*>(base + hist_off), permute_chunks(T * k), status, s);
    // the join is enqueued whatever happened, so that the caller's stream (or a capture of
    // it) never keeps an unjoined fork
    const cudaError_t er = cudaEventRecord(ss->join, ss->stream);
    const cudaError_t ew = cudaStreamWaitEvent(s, ss->join, 0);
    if (eq != cudaSuccess || ep != cudaSuccess || er != cudaSuccess || ew != cudaSuccess) return NVFP4_ERR_CUDA;
    e = launch_gather_tiled(xq, xq + T * H / 2, gx, perm, padded + E, mcap, H, aq, ga, h_amax, s);
    if (e != cudaSuccess) return NVFP4_ERR_CUDA;
  }

  // 3. gate/up GEMM with the SwiGLU epilogue: h = BF16(silu(gate) * up)
  GemmArgs g1{};
  g1.ga = ga;
  g1.gb = wt->w13_g;
  g1.offsets = padded;
  g1.rows = counts;
  g1.m_total = mcap;
  g1.E = E;
  g1.N = (int32_t)(2 * I);
  g1.K = (int32_t)H;
  g1.status = status;
  g1.h = hbuf;
  g1.I = I;
  g1.h_amax = h_amax;
  g1.silu_tab = silu_table(s);
  if (g1.silu_tab == nullptr) return NVFP4_ERR_CUDA;
  CUtensorMap mh, my;
  if (!make_map(&mh, hbuf, mcap, I, I * 2, 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64) ||
      !make_map(&my, ybuf, mcap, H, H * 2, 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2))
    return NVFP4_ERR_CUDA;
  e = launch_grouped_gemm_tiled(aq, wt->w13, mh, g1, mcap / 128, true, s, small);
  if (e != cudaSuccess) return NVFP4_ERR_CUDA;

  // 4. per-row NVFP4 of h (routed rows only), K zero-padded to Ip, GEMM-tiled, with the
  //    row maxima the epilogue gathered
  e = launch_requant_tiled(hbuf, h_amax, perm, padded + E, mcap, I, Ip, hq, gh, s, small);
  if (e != cudaSuccess) return NVFP4_ERR_CUDA;

  // 5. down GEMM -> y (BF16)
  GemmArgs g2{};
  g2.ga = gh;
  g2.gb = wt->w2_g;
  g2.offsets = padded;
  g2.rows = counts;
  g2.m_total = mcap;
  g2.E = E;
  g2.N = (int32_t)H;
  g2.K = (int32_t)Ip;
  g2.d = ybuf;
  g2.ldd = H;
  g2.out_f32 = 0;
  g2.status = status;
  e = launch_grouped_gemm_tiled(hq, wt->w2, my, g2, mcap / 128, false, s, small);
  if (e != cudaSuccess) return NVFP4_ERR_CUDA;

  // 6. weighted un-permute
  return from_cuda(launch_combine(ybuf, inv, w, T, k, H, out, s, small));
}

nvfp4_status moe_weights_t_sizes(int32_t E, int64_t H, int64_t I, size_t sizes_out[4]) {
  if (E <= 0 || H <= 0 || I <= 0 || sizes_out == nullptr) return NVFP4_ERR_INVALID_ARG;
  const int64_t Ip = round_up(I, 256);
  sizes_out[0] = (size_t)tiled_bytes((int64_t)E * H, 2 * I, 256);
  sizes_out[1] = 4u * (size_t)E;
  sizes_out[2] = (size_t)tiled_bytes((int64_t)E * Ip, H, 256);
  sizes_out[3] = 4u * (size_t)E;
  return NVFP4_OK;
}

nvfp4_status moe_prepare_weights_backward(const void* w13, const void* w2, int32_t E, int64_t H, int64_t I,
                                          const nvfp4_moe_weights_t* out, void* ws, size_t ws_bytes, void* stream) {
  if (E <= 0 || H <= 0 || I <= 0 || out == nullptr) return NVFP4_ERR_INVALID_ARG;
  if (E > tiled_max_experts() || H % 256 != 0 || I % 128 != 0 || H > 8192 || I > 4096) return NVFP4_ERR_UNSUPPORTED;
  if (out->E != E || out->H != H || out->I != I) return NVFP4_ERR_INVALID_ARG;
  const void* ptrs[] = {w13, w2, out->w13t, out->w13t_g, out->w2t, out->w2t_g};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return NVFP4_ERR_INVALID_ARG;
  if (ws == nullptr || ws_bytes < nvfp4_workspace_size(NVFP4_OP_PREPARE_WEIGHTS_T, E, 0, 0, 0, 0) || !aligned16(ws))
    return NVFP4_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t Ip = round_up(I, 256);
  uint32_t* amax = static_cast<uint32_t*>(ws);
  int32_t* kofs = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(ws) + align256(8u * (size_t)E));
  // W13_e [2I, H] -> W13_e^T [H, 2I]: the 2I rows of each expert are its "tokens"
  if (launch_amax(w13, (int64_t)E * 2 * I, H, H, 2 * I, amax, E, s) != cudaSuccess ||
      launch_kofs(nullptr, 2 * I, E, kofs, s) != cudaSuccess ||
      launch_tquant(w13, H, nullptr, nullptr, nullptr, 2 * I, kofs, E, (int)H, (int)H, 256, amax, out->w13t_g,
                    out->w13t, kRoundRNE, 0, 0, (int64_t)E * (2 * I / 256), s) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  // W2_e [H, I] -> W2_e^T [I, H], rows I .. Ip-1 zero
  uint32_t* amax2 = amax + E;
  int32_t* kofs2 = kofs + E + 1;
  if (launch_amax(w2, (int64_t)E * H, I, I, H, amax2, E, s) != cudaSuccess ||
      launch_kofs(nullptr, H, E, kofs2, s) != cudaSuccess ||
      launch_tquant(w2, I, nullptr, nullptr, nullptr, H, kofs2, E, (int)I, (int)Ip, 256, amax2, out->w2t_g, out->w2t,
                    kRoundRNE, 0, 0, (int64_t)E * (H / 256), s) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}

nvfp4_status moe_backward_workspace_layout(int64_t T, int32_t k, int32_t E, int64_t H, int64_t I,
                                           int64_t layout_out[18]) {
  if (T < 0 || k <= 0 || E <= 0 || H <= 0 || I <= 0 || layout_out == nullptr) return NVFP4_ERR_INVALID_ARG;
  const BackwardLayout L = backward_layout(T, k, E, H, I);
  std::memcpy(layout_out, L.off, sizeof(L.off));
  return NVFP4_OK;
}

nvfp4_status moe_expert_backward(const void* dout, const void* x, const float* w, int64_t T, int32_t k,
                                 const nvfp4_moe_weights* wt, const nvfp4_moe_weights_t* wtt, const void* fwd_ws,
                                 size_t fwd_ws_bytes, uint64_t seed, void* dx, float* dw, float* dw13, float* dw2,
                                 void* ws, size_t ws_bytes, void* stream) {
  if (wt == nullptr || wtt == nullptr || T < 0 || k <= 0 || k > 32) return NVFP4_ERR_INVALID_ARG;
  const int32_t E = wt->E;
  const int64_t H = wt->H, I = wt->I;
  if (wtt->E != E || wtt->H != H || wtt->I != I) return NVFP4_ERR_INVALID_ARG;
  if (E <= 0 || E > tiled_max_experts() || k > E) return NVFP4_ERR_INVALID_ARG;
  if (H % 256 != 0 || I % 128 != 0 || H > 2048 || I > 1024) return NVFP4_ERR_UNSUPPORTED;
  if (T * k >= ((int64_t)1 << 31) - (int64_t)E * 128) return NVFP4_ERR_UNSUPPORTED;
  if (T == 0) return NVFP4_OK;
  const void* ptrs[] = {dout, x, dx, dw13, dw2, ws, fwd_ws, wt->w13, wt->w13_g, wtt->w13t, wtt->w13t_g, wtt->w2t,
                        wtt->w2t_g};
  for (const void* p : ptrs)
    if (p == nullptr || !aligned16(p)) return NVFP4_ERR_INVALID_ARG;
  if (!aligned4(w) || !aligned4(dw)) return NVFP4_ERR_INVALID_ARG;
  size_t hist_off, hist_bytes;
  const ForwardLayout F = forward_layout(T, k, E, H, I, &hist_off, &hist_bytes);
  if (fwd_ws_bytes < (size_t)F.off[14]) return NVFP4_ERR_WORKSPACE;
  const BackwardLayout L = backward_layout(T, k, E, H, I);
  if (ws_bytes < (size_t)L.off[17]) return NVFP4_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint8_t* fb = static_cast<const uint8_t*>(fwd_ws);
  const int32_t* counts = reinterpret_cast<const int32_t*>(fb + F.off[0]);
  const int32_t* padded = reinterpret_cast<const int32_t*>(fb + F.off[2]);
  const int32_t* inv = reinterpret_cast<const int32_t*>(fb + F.off[3]);
  const int32_t* perm = reinterpret_cast<const int32_t*>(fb + F.off[4]);
  const uint8_t* aq = fb + F.off[5];
  const float* ga = reinterpret_cast<const float*>(fb + F.off[7]);
  const void* hbuf = fb + F.off[8];
  const void* ybuf = fb + F.off[12];
  const int64_t mcap = F.off[13];
  const int64_t Ip = round_up(I, 256);
  uint8_t* b = static_cast<uint8_t*>(ws);
  auto at = [&](int i) { return b + L.off[i]; };
  void* dy = at(0);
  uint8_t* dyq = at(1);
  float* g_dy = reinterpret_cast<float*>(at(2));
  void* dh = at(3);
  void* dbuf = at(4);
  void* dD = at(5);
  uint8_t* dDq = at(6);
  float* g_dD = reinterpret_cast<float*>(at(7));
  void* dxs = at(8);
  int32_t* kofs = reinterpret_cast<int32_t*>(at(9));
  uint32_t* amax = reinterpret_cast<uint32_t*>(at(10));
  float* gexp = reinterpret_cast<float*>(at(11));
  const int64_t kb_cap = L.off[16];
  int* status = device_status_ptr();
  auto fail = [](cudaError_t e) { return e != cudaSuccess; };

  auto key = [&](int stream_id) { return seed + ((uint64_t)stream_id << 50); };   // expert 0's key of the stream
  // 1. weighted un-permute backward: dy per slot, dw per (token, j), and dy's rows
  //    quantised (per row, stochastic rounding) into the dgrad's A operand
  if (fail(launch_combine_backward(dout, inv, w, ybuf, T, k, H, dy, dw, padded, E, amax, dyq, g_dy, key(0), s)))
    return NVFP4_ERR_CUDA;

  // row quantisation of a slot-ordered gradient (per row, stochastic rounding) into the
  // GEMM-tiled A operand; padding slots are skipped
  auto quant_rows = [&](const void* src, int64_t cols, uint8_t* out, float* g_out, uint64_t key) {
    QuantArgs a{};
    a.x = static_cast<const __nv_bfloat16*>(src);
    a.rows = mcap;
    a.cols = cols;
    a.ld = cols;
    a.mode = kScopeRow;
    a.g_out = g_out;
    a.codes = out;
    a.sf_words = cols / 64;
    a.cols_pad = cols;
    a.rows_total = mcap;
    a.map = kMapIdentity;
    a.seed = key;
    a.status = status;
    a.tiled_R = 128;
    a.kblocks = cols / 256;
    a.row_filter = perm;
    a.rows_dev = padded + E;
    return launch_quantize_rows(a, kRoundSR, s);
  };
  // grouped GEMM over GEMM-tiled operands with a plain BF16 store into [mcap, N] (pitch ld)
  auto dgrad = [&](const uint8_t* A, const float* gA, const uint8_t* B, const float* gB, int64_t N, int64_t K,
                   void* out, int64_t ld_cols, int64_t store_cols) {
    GemmArgs g{};
    g.ga = gA;
    g.gb = gB;
    g.offsets = padded;
    g.rows = counts;
    g.m_total = mcap;
    g.E = E;
    g.N = (int32_t)N;
    g.K = (int32_t)K;
    g.d = out;
    g.ldd = ld_cols;
    g.status = status;
    CUtensorMap md;
    if (!make_map(&md, out, mcap, store_cols, ld_cols * 2, 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2))
      return cudaErrorInvalidValue;
    return launch_grouped_gemm_tiled(A, B, md, g, mcap / 128, false, s);
  };

  // 2. dgrad of the down projection: dh = Q(dy) Q(W2^T), dh [mcap, Ip]
  if (fail(dgrad(dyq, g_dy, wtt->w2t, wtt->w2t_g, Ip, H, dh, Ip, Ip)))
    return NVFP4_ERR_CUDA;
  // 3. the gate/up output D again (the fused forward keeps only h), then the SwiGLU backward
  //    into the canonical [dgate | dup]
  if (fail(dgrad(aq, ga, wt->w13, wt->w13_g, 2 * I, H, dbuf, 2 * I, 2 * I)) ||
      fail(launch_swiglu_backward(dbuf, dh, mcap, I, dD, s, true, Ip)))
    return NVFP4_ERR_CUDA;
  // 4. dgrad of gate/up: dxs = Q(dD) Q(W13^T), then dx = sum over each token's slots
  if (fail(quant_rows(dD, 2 * I, dDq, g_dD, key(2))) ||
      fail(dgrad(dDq, g_dD, wtt->w13t, wtt->w13t_g, H, 2 * I, dxs, H, H)) ||
      fail(launch_combine(dxs, inv, nullptr, T, k, H, dx, s)))
    return NVFP4_ERR_CUDA;

  // 5. weight gradients: per-expert transposed quantisation along the tokens, then the
  //    ragged-K grouped GEMM (float32 out)
  if (fail(launch_kofs(counts, 0, E, kofs, s))) return NVFP4_ERR_CUDA;
  // the per-expert maxima of the wgrad operands: dy's from the combine backward; dD's, h's
  // and x's from the per-row global scales their row quantisations left (g_dD, the
  // forward's gH and the per-slot token scales gA), without another pass over the rows
  auto wgrad = [&](const void* gsrc, int64_t Fa, const float* g_gsrc, const void* asrc, int64_t ld_a,
                   const float* g_asrc, const int32_t* rowmap, int64_t Fb, int64_t Fbp, int stream_id, int slot,
                   uint8_t* Aw, uint8_t* Bw, float* out) {
    uint32_t* am = amax + 2 * slot * E;
    float* gg = gexp + 2 * slot * E;
    if ((g_gsrc != nullptr &&
         fail(launch_group_amax_g(g_gsrc, gsrc, Fa, Fa, nullptr, padded, counts, E, mcap, am, s))) ||
        fail(launch_group_amax_g(g_asrc, asrc, ld_a, Fb, rowmap, padded, counts, E, mcap, am + E, s)) ||
        fail(launch_tquant(gsrc, Fa, nullptr, padded, counts, 0, kofs, E, (int)Fa, (int)Fa, 128, am, gg, Aw, kRoundSR,
                           seed, stream_id, kb_cap, s)) ||
        fail(launch_tquant(asrc, ld_a, rowmap, padded, counts, 0, kofs, E, (int)Fb, (int)Fbp, 256, am + E, gg + E, Bw,
                           kRoundRNE, 0, 0, kb_cap, s)))
      return cudaErrorUnknown;
    GemmArgs g{};
    g.ga = gg;
    g.gb = gg + E;
    g.offsets = kofs;
    g.m_total = kb_cap;
    g.m_rows = (int32_t)Fa;
    g.E = E;
    g.N = (int32_t)Fbp;
    g.K = 256;
    g.d = out;
    g.ldd = Fb;
    g.out_f32 = 1;
    g.status = status;
    CUtensorMap md;
    if (!make_map(&md, out, (int64_t)E * Fa, Fb, Fb * 4, 32, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4))
      return cudaErrorInvalidValue;
    return launch_grouped_gemm_ragged_k(Aw, Bw, md, g, s);
  };
  const float* gh = reinterpret_cast<const float*>(fb + F.off[11]);
  if (fail(wgrad(dy, H, nullptr, hbuf, I, gh, nullptr, I, Ip, 1, 0, at(12), at(13), dw2)) ||
      fail(wgrad(dD, 2 * I, g_dD, x, H, ga, perm, H, H, 3, 1, at(14), at(15), dw13)))
    return NVFP4_ERR_CUDA;
  return NVFP4_OK;
}

}  // extern "C"

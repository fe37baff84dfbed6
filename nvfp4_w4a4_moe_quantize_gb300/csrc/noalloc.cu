// NVFP4 quantisation for callers that cannot allocate device memory.
//
// nvfp4_quantize needs a small workspace (one 32-bit amax word per scale scope) in the
// per-tensor and per-group modes.  Some callers have no way to provide it: code running
// where no allocator is reachable (a host plug-in handed only the tensors it must read
// and write, or a runtime whose memory pool may not be touched from this call).  This
// entry point keeps that scratch in a fixed device array owned by the library instead.
//
// The array is a file-scope __device__ object, so every GPU that loads the library holds
// it (16 KB) until the process exits.  Host code cannot use the array's name as a device
// address; the first call on each device resolves the address with
// cudaGetSymbolAddress (with that device current) and keeps it.  The kernels are the
// ones nvfp4_quantize launches; only the place of the scratch differs.
#include <cuda_runtime.h>

#include <mutex>

#include "launch.h"
#include "nvfp4moe.h"

namespace nvfp4 {

constexpr int64_t kNoAllocMaxScopes = 4096;   // amax words: per-tensor 1, per-group rows/group_rows

static __device__ __align__(256) uint32_t g_noalloc_amax[kNoAllocMaxScopes];

namespace {
constexpr int kMaxDev = 64;
uint32_t* g_noalloc_addr[kMaxDev];
std::mutex g_noalloc_mu;

// Device address of g_noalloc_amax on the current device (resolved once per device).
uint32_t* noalloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_amax) != cudaSuccess) return nullptr;
    g_noalloc_addr[dev] = static_cast<uint32_t*>(p);
  }
  return g_noalloc_addr[dev];
}
}  // namespace

}  // namespace nvfp4

extern "C" nvfp4_status nvfp4_quantize_noalloc(const void* x, int64_t rows, int64_t cols, int64_t ld_elems,
                                               nvfp4_scale_mode mode, int64_t group_rows,
                                               nvfp4_rounding rounding, uint64_t seed, uint64_t rng_offset,
                                               const float* global_scale_in, float* global_scale_out,
                                               uint8_t* codes_out, uint8_t* sf_out, void* stream) {
  using namespace nvfp4;
  if (mode == NVFP4_SCALE_PER_GROUP && (group_rows <= 0 || rows % group_rows != 0)) return NVFP4_ERR_INVALID_ARG;
  const int64_t n_scopes = mode == NVFP4_SCALE_PER_TENSOR ? 1
                           : mode == NVFP4_SCALE_PER_GROUP ? (rows > 0 ? rows / group_rows : 0) : 0;
  if (n_scopes > kNoAllocMaxScopes && global_scale_in == nullptr) return NVFP4_ERR_UNSUPPORTED;
  uint32_t* scratch = noalloc_scratch();
  if (scratch == nullptr) return NVFP4_ERR_CUDA;
  return nvfp4_quantize(x, rows, cols, ld_elems, mode, group_rows, rounding, seed, rng_offset, global_scale_in,
                        global_scale_out, codes_out, sf_out, NVFP4_SF_SWIZZLED_128x4, scratch,
                        sizeof(uint32_t) * kNoAllocMaxScopes, stream);
}

// Routing, expert grouping and the weighted un-permute of the MoE expert block.
//
// Top-k routing and the grouping of (token, slot) pairs by expert are the "token permute
// by router top-k" around the expert GEMMs; the weighted un-permute returns every
// token's k expert outputs to its row.  Slot order: experts ascending, tokens ascending
// inside an expert (a stable counting sort), each expert's group starting at a multiple
// of 128 rows -- deterministic and independent of thread timing, so that a token's
// output bits never depend on the batch ("Low-Bit Precision Training Is Ready for
// Production...", §"The Cross-Engine Alignment Problem").
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "encode.cuh"
#include "launch.h"
#include "pdl.cuh"
#include "status.cuh"
#include "tiled.cuh"

namespace nvfp4 {

constexpr unsigned kFullMask = 0xFFFFFFFFu;

// ------------------------------------------------------------------ top-k routing

// Float bits -> a key whose unsigned order is the float order (-0 is folded onto +0 so the
// two compare equal, as floats do; NaN sorts below every number).
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(__fadd_rn(v, 0.0f));
  if (v != v) return 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// One warp per token.  Lane l holds experts l, l+32, ...; k rounds of a warp arg-max
// with (larger logit, then lower id) as the order: each round one warp max-reduction of
// the order keys (redux.sync) and one min-reduction of the expert ids holding that key.
// Weights: expf relative to the top logit, then divided by the sum over the chosen k (or
// over all experts).
template <int EPL>
__global__ void __launch_bounds__(256) route_topk_kernel(const float* __restrict__ logits, int64_t T, int E, int k,
                                                         int renorm, int32_t* __restrict__ ids,
                                                         float* __restrict__ w) {
  grid_dep_sync();
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t nwarp = (int64_t)gridDim.x * 8;
  for (int64_t t = warp; t < T; t += nwarp) {
    float v[EPL];
    uint32_t key[EPL];
    const float* lr = logits + t * E;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      v[i] = e < E ? lr[e] : -INFINITY;
    }
    uint32_t live = 0;   // bit i: expert lane + 32 i exists and is not taken yet
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      key[i] = order_key(v[i]);
      if (lane + 32 * i < E) live |= 1u << i;
    }
    int my_id = 0;
    float my_v = 0.0f;
    for (int j = 0; j < k; ++j) {
      uint32_t best = 0;
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if ((live >> i) & 1u) best = max(best, key[i]);
      const uint32_t wbest = __reduce_max_sync(kFullMask, best);
      uint32_t cand = 0xFFFFFFFFu;
#pragma unroll
      for (int i = EPL - 1; i >= 0; --i)
        if (((live >> i) & 1u) && key[i] == wbest) cand = (uint32_t)(lane + 32 * i);
      const uint32_t bi = __reduce_min_sync(kFullMask, cand);
      float bv = 0.0f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) bv = (uint32_t)(lane + 32 * i) == bi ? v[i] : bv;
      if ((int)(bi & 31u) == lane) live &= ~(1u << (bi >> 5));
      bv = __shfl_sync(kFullMask, bv, (int)(bi & 31u));
      if (lane == j) {
        my_id = (int)bi;
        my_v = bv;
      }
    }
    const float top = __shfl_sync(kFullMask, my_v, 0);
    const float ex = lane < k ? expf(my_v - top) : 0.0f;
    float den;
    if (renorm) {
      den = ex;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(kFullMask, den, o);
    } else {
      den = 0.0f;
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (lane + 32 * i < E) den += expf(v[i] - top);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(kFullMask, den, o);
    }
    if (lane < k) {
      ids[t * k + lane] = my_id;
      w[t * k + lane] = __fdiv_rn(ex, den);
    }
  }
}

// The same routing for E <= 32 * EPL with EPL <= 4: each lane first sorts its EPL
// (key, expert id) pairs by (larger key, then lower id) with a small comparator network,
// so a round compares only the 32 list heads: one max-reduction of the head keys, one
// min-reduction of the ids whose head holds that key, and the owning lane pops its head.
// Experts past E have key 0 and id 0xFFFFFFFF, below every real expert.
__device__ __forceinline__ void route_ce(uint32_t& ka, uint32_t& ia, float& va, uint32_t& kb, uint32_t& ib,
                                         float& vb) {
  const bool sw = kb > ka || (kb == ka && ib < ia);
  const uint32_t tk = sw ? kb : ka, ti = sw ? ib : ia;
  const float tv = sw ? vb : va;
  kb = sw ? ka : kb;
  ib = sw ? ia : ib;
  vb = sw ? va : vb;
  ka = tk;
  ia = ti;
  va = tv;
}

template <int EPL>
__global__ void __launch_bounds__(256) route_topk_sorted_kernel(const float* __restrict__ logits, int64_t T, int E,
                                                                int k, int renorm, int32_t* __restrict__ ids,
                                                                float* __restrict__ w) {
  grid_dep_sync();
  static_assert(EPL == 1 || EPL == 2 || EPL == 4, "lists of 1, 2 or 4");
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t nwarp = (int64_t)gridDim.x * 8;
  for (int64_t t = warp; t < T; t += nwarp) {
    float v[EPL], sv[EPL];
    uint32_t key[EPL], id[EPL];
    const float* lr = logits + t * E;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      v[i] = e < E ? lr[e] : -INFINITY;
      sv[i] = v[i];
      key[i] = e < E ? order_key(v[i]) : 0u;
      id[i] = e < E ? (uint32_t)e : 0xFFFFFFFFu;
    }
    if (EPL >= 2) route_ce(key[0], id[0], sv[0], key[1 % EPL], id[1 % EPL], sv[1 % EPL]);
    if (EPL == 4) {
      route_ce(key[2 % EPL], id[2 % EPL], sv[2 % EPL], key[3 % EPL], id[3 % EPL], sv[3 % EPL]);
      route_ce(key[0], id[0], sv[0], key[2 % EPL], id[2 % EPL], sv[2 % EPL]);
      route_ce(key[1 % EPL], id[1 % EPL], sv[1 % EPL], key[3 % EPL], id[3 % EPL], sv[3 % EPL]);
      route_ce(key[1 % EPL], id[1 % EPL], sv[1 % EPL], key[2 % EPL], id[2 % EPL], sv[2 % EPL]);
    }
    int my_id = 0;
    float my_v = 0.0f;
    for (int j = 0; j < k; ++j) {
      const uint32_t wbest = __reduce_max_sync(kFullMask, key[0]);
      const uint32_t bi = __reduce_min_sync(kFullMask, key[0] == wbest ? id[0] : 0xFFFFFFFFu);
      const float bv = __shfl_sync(kFullMask, sv[0], (int)(bi & 31u));
      if (id[0] == bi) {   // pop this lane's head
#pragma unroll
        for (int i = 0; i + 1 < EPL; ++i) {
          key[i] = key[i + 1];
          id[i] = id[i + 1];
          sv[i] = sv[i + 1];
        }
        key[EPL - 1] = 0u;
        id[EPL - 1] = 0xFFFFFFFFu;
      }
      if (lane == j) {
        my_id = (int)bi;
        my_v = bv;
      }
    }
    const float top = __shfl_sync(kFullMask, my_v, 0);
    const float ex = lane < k ? expf(my_v - top) : 0.0f;
    float den;
    if (renorm) {
      den = ex;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(kFullMask, den, o);
    } else {
      den = 0.0f;
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (lane + 32 * i < E) den += expf(v[i] - top);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(kFullMask, den, o);
    }
    if (lane < k) {
      ids[t * k + lane] = my_id;
      w[t * k + lane] = __fdiv_rn(ex, den);
    }
  }
}

cudaError_t launch_route_topk(const float* logits, int64_t T, int E, int k, int renorm, int32_t* ids, float* w,
                              cudaStream_t s, bool pdl) {
  if (T == 0) return cudaSuccess;
  int64_t blocks = (T + 7) / 8;
  if (blocks > 16 * num_sms()) blocks = 16 * num_sms();
  const int epl = (E + 31) / 32;
#define NVFP4_ROUTE(N) \
  launch_pdl(pdl, route_topk_kernel<N>, dim3((unsigned)blocks), dim3(256), 0, s, logits, T, E, k, renorm, ids, w)
#define NVFP4_ROUTE_SORTED(N) \
  launch_pdl(pdl, route_topk_sorted_kernel<N>, dim3((unsigned)blocks), dim3(256), 0, s, logits, T, E, k, renorm, ids, w)
  cudaError_t err;
  if (epl <= 1) err = NVFP4_ROUTE_SORTED(1);
  else if (epl <= 2) err = NVFP4_ROUTE_SORTED(2);
  else if (epl <= 4) err = NVFP4_ROUTE_SORTED(4);
  else if (epl <= 8) err = NVFP4_ROUTE(8);
  else if (epl <= 16) err = NVFP4_ROUTE(16);
  else err = NVFP4_ROUTE(32);
#undef NVFP4_ROUTE
#undef NVFP4_ROUTE_SORTED
  return err;
}

// ------------------------------------------------------------------ expert grouping

// Pass 1: per chunk of kPermuteChunk flattened entries (one warp each), the count of
// entries per expert.  hist is [E][nchunks].  The warp loads its whole chunk first (one
// round trip), then finds matching lanes with __match_any_sync; the lowest lane of each
// match group adds the group's size.  Block 0 also clears the completion counter that
// pass 2 uses (hist[E * nchunks]).
constexpr int kPermuteSteps = kPermuteChunk / 32;
__global__ void __launch_bounds__(256) permute_hist_kernel(const int32_t* __restrict__ ids, int64_t n, int E,
                                                           int64_t nchunks, int32_t* __restrict__ hist,
                                                           int* status) {
  grid_dep_sync();
  extern __shared__ int32_t sh[];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  if (blockIdx.x == 0 && threadIdx.x == 0) hist[(int64_t)E * nchunks] = 0;
  const int64_t c = (int64_t)blockIdx.x * 8 + wib;
  if (c >= nchunks) return;
  int32_t* cnt = sh + wib * E;
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  const int64_t begin = c * kPermuteChunk;
  int ev[kPermuteSteps];
#pragma unroll
  for (int u = 0; u < kPermuteSteps; ++u) {
    const int64_t i = begin + 32 * u + lane;
    ev[u] = i < n ? ids[i] : -1;
  }
  __syncwarp();
#pragma unroll
  for (int u = 0; u < kPermuteSteps; ++u) {
    const int64_t i = begin + 32 * u + lane;
    int e = ev[u];
    if (i < n && (e < 0 || e >= E)) {
      set_status(status, kStatusBadInput);
      e = -1;
    }
    const unsigned peers = __match_any_sync(kFullMask, e);
    if (e >= 0 && lane == __ffs(peers) - 1) cnt[e] += __popc(peers);
    __syncwarp();
  }
  for (int e = lane; e < E; e += 32) hist[(int64_t)e * nchunks + c] = cnt[e];
}

// Pass 2: one warp per expert scans that expert's chunk counts in place (exclusive) and
// writes its total.  The last block to finish -- a completion counter, no block waits
// for another -- runs the unpadded and 128-padded exclusive scans over the experts
// (E <= 1024) and writes -1 into the padding slots of perm.
__global__ void __launch_bounds__(1024) permute_scan_kernel(int32_t* __restrict__ hist, int64_t nchunks, int E,
                                                            int32_t* __restrict__ counts,
                                                            int32_t* __restrict__ offsets,
                                                            int32_t* __restrict__ padded,
                                                            int32_t* __restrict__ perm) {
  grid_dep_sync();
  __shared__ int32_t s_cnt[1024];
  __shared__ int32_t s_pad[1025];
  __shared__ int32_t s_wsum[2][32];
  __shared__ int s_last;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = blockDim.x >> 5;
  constexpr int kVec = 8;
  for (int e = blockIdx.x * nw + wid; e < E; e += gridDim.x * nw) {
    int32_t* h = hist + (int64_t)e * nchunks;
    int32_t carry = 0;
    for (int64_t c0 = 0; c0 < nchunks; c0 += 32 * kVec) {
      int32_t v[kVec];
#pragma unroll
      for (int u = 0; u < kVec; ++u) {
        const int64_t c = c0 + 32 * u + lane;
        v[u] = c < nchunks ? h[c] : 0;
      }
#pragma unroll
      for (int u = 0; u < kVec; ++u) {
        int32_t x = v[u];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int32_t y = __shfl_up_sync(kFullMask, x, o);
          if (lane >= o) x += y;
        }
        const int64_t c = c0 + 32 * u + lane;
        if (c < nchunks) h[c] = carry + x - v[u];
        carry += __shfl_sync(kFullMask, x, 31);
      }
    }
    if (lane == 0) counts[e] = carry;
  }
  // completion: the last block sees every count
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    int* done = hist + (int64_t)E * nchunks;
    if (gridDim.x == 1) {
      s_last = 1;                     // a single block needs no counter
    } else {
      s_last = atomicAdd(done, 1) == (int)gridDim.x - 1;
      if (s_last) *done = 0;
    }
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int e = threadIdx.x;
  const int32_t cnt = e < E ? *reinterpret_cast<volatile int32_t*>(counts + e) : 0;
  if (e < E) s_cnt[e] = cnt;
  const int32_t pc = (cnt + 127) / 128 * 128;
  int32_t x0 = cnt, x1 = pc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t y0 = __shfl_up_sync(kFullMask, x0, o);
    const int32_t y1 = __shfl_up_sync(kFullMask, x1, o);
    if (lane >= o) {
      x0 += y0;
      x1 += y1;
    }
  }
  if (lane == 31) {
    s_wsum[0][wid] = x0;
    s_wsum[1][wid] = x1;
  }
  __syncthreads();
  if (wid == 0) {
    int32_t a0 = s_wsum[0][lane], a1 = s_wsum[1][lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t y0 = __shfl_up_sync(kFullMask, a0, o);
      const int32_t y1 = __shfl_up_sync(kFullMask, a1, o);
      if (lane >= o) {
        a0 += y0;
        a1 += y1;
      }
    }
    s_wsum[0][lane] = a0 - s_wsum[0][lane];
    s_wsum[1][lane] = a1 - s_wsum[1][lane];
  }
  __syncthreads();
  const int32_t excl0 = x0 - cnt + s_wsum[0][wid];
  const int32_t excl1 = x1 - pc + s_wsum[1][wid];
  if (e < E) {
    offsets[e] = excl0;
    padded[e] = excl1;
    s_pad[e] = excl1;
    if (e == E - 1) {
      offsets[E] = excl0 + cnt;
      padded[E] = excl1 + pc;
      s_pad[E] = excl1 + pc;
    }
  }
  __syncthreads();
  if (perm != nullptr) {
    for (int ee = wid; ee < E; ee += 32) {
      const int32_t lo = s_pad[ee] + s_cnt[ee], hi = s_pad[ee + 1];
      for (int32_t r = lo + lane; r < hi; r += 32) perm[r] = -1;
    }
  }
}

// Pass 3: the slot of every entry.  Inside a chunk the warp walks 32 entries at a time
// in order; an entry's rank among equal experts is the count of matching lower lanes
// plus the running count of that expert, which starts at the chunk's exclusive prefix.
__global__ void __launch_bounds__(256) permute_rank_kernel(const int32_t* __restrict__ ids, int64_t n, int k,
                                                           int E, int64_t nchunks,
                                                           const int32_t* __restrict__ hist,
                                                           const int32_t* __restrict__ padded,
                                                           int32_t* __restrict__ inv, int32_t* __restrict__ perm) {
  grid_dep_sync();
  extern __shared__ int32_t sh[];
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  int32_t* s_pad = sh;                 // E
  int32_t* run = sh + E + wib * E;     // E per warp
  for (int e = threadIdx.x; e < E; e += blockDim.x) s_pad[e] = padded[e];
  __syncthreads();
  const int64_t c = (int64_t)blockIdx.x * 8 + wib;
  if (c >= nchunks) return;
  for (int e = lane; e < E; e += 32) run[e] = hist[(int64_t)e * nchunks + c];
  __syncwarp();
  const unsigned lt = (1u << lane) - 1u;
  const int64_t begin = c * kPermuteChunk, end = min(n, (c + 1) * kPermuteChunk);
  int ev[kPermuteSteps];   // the whole chunk first: one round trip
#pragma unroll
  for (int u = 0; u < kPermuteSteps; ++u) {
    const int64_t i = begin + 32 * u + lane;
    ev[u] = i < end ? ids[i] : -1;
  }
#pragma unroll
  for (int u = 0; u < kPermuteSteps; ++u) {
    const int64_t i = begin + 32 * u + lane;
    int e = ev[u];
    if (e >= E) e = -1;
    const unsigned peers = __match_any_sync(kFullMask, e);
    if (e >= 0) {
      const int32_t slot = s_pad[e] + run[e] + __popc(peers & lt);
      inv[i] = slot;
      if (perm != nullptr) perm[slot] = (int32_t)(i / k);
    } else if (i < end) {
      inv[i] = -1;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) run[e] += __popc(peers);
    __syncwarp();
  }
}

// Small batches (n = T*k <= 1024 entries: decode-shaped launches): the three passes in
// one block of 1024 threads -- per-expert counts in shared memory, the unpadded and
// 128-padded exclusive scans, and each entry's rank among the earlier entries of its
// expert (a scan over at most n - 1 ids in shared memory): the same stable slot order.
// s_inv receives every entry's slot (-1 for an id out of range).  `write`: this block
// also stores counts, offsets, padded, inv and perm, and flags bad ids.
struct PermuteSmem {
  int32_t id[1024], cnt[1024], wsum[2][32], off[1025], pad[1025], inv[1024];
};

__device__ __forceinline__ void permute_small_block(const int32_t* __restrict__ ids, int n, int k, int E, bool write,
                                                    int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                                                    int32_t* __restrict__ padded, int32_t* __restrict__ inv,
                                                    int32_t* __restrict__ perm, int* status, PermuteSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  sm.cnt[tid] = 0;
  int e = -1;
  if (tid < n) {
    e = ids[tid];
    if (e < 0 || e >= E) {
      if (write) set_status(status, kStatusBadInput);
      e = -1;
    }
  }
  sm.id[tid] = e;
  __syncthreads();
  if (e >= 0) atomicAdd(&sm.cnt[e], 1);
  __syncthreads();
  // inclusive scans of the counts and of the 128-padded counts over the experts
  const int32_t c = tid < E ? sm.cnt[tid] : 0;
  int32_t a = c, b = (c + 127) / 128 * 128;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t ya = __shfl_up_sync(kFullMask, a, o), yb = __shfl_up_sync(kFullMask, b, o);
    if (lane >= o) {
      a += ya;
      b += yb;
    }
  }
  if (lane == 31) {
    sm.wsum[0][wid] = a;
    sm.wsum[1][wid] = b;
  }
  __syncthreads();
  if (wid == 0) {
    int32_t wa = sm.wsum[0][lane], wb = sm.wsum[1][lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int32_t ya = __shfl_up_sync(kFullMask, wa, o), yb = __shfl_up_sync(kFullMask, wb, o);
      if (lane >= o) {
        wa += ya;
        wb += yb;
      }
    }
    sm.wsum[0][lane] = wa;
    sm.wsum[1][lane] = wb;
  }
  __syncthreads();
  const int32_t base_a = wid ? sm.wsum[0][wid - 1] : 0, base_b = wid ? sm.wsum[1][wid - 1] : 0;
  const int32_t inc_a = a + base_a, inc_b = b + base_b;
  if (tid < E) {
    sm.off[tid + 1] = inc_a;
    sm.pad[tid + 1] = inc_b;
    if (write) {
      counts[tid] = c;
      offsets[tid + 1] = inc_a;
      padded[tid + 1] = inc_b;
    }
  }
  if (tid == 0) {
    sm.off[0] = sm.pad[0] = 0;
    if (write) offsets[0] = padded[0] = 0;
  }
  __syncthreads();
  const int32_t total_pad = sm.pad[E];
  if (write && perm != nullptr)
    for (int32_t slot = tid; slot < total_pad; slot += blockDim.x) perm[slot] = -1;
  __syncthreads();
  if (tid < n) {
    int32_t slot = -1;
    if (e >= 0) {
      int32_t rank = 0;
      for (int i = 0; i < tid; ++i) rank += sm.id[i] == e;
      slot = sm.pad[e] + rank;
      if (write && perm != nullptr) perm[slot] = tid / k;
    }
    sm.inv[tid] = slot;
    if (write) inv[tid] = slot;
  }
}

__global__ void __launch_bounds__(1024) permute_small_kernel(const int32_t* __restrict__ ids, int n, int k, int E,
                                                             int32_t* __restrict__ counts,
                                                             int32_t* __restrict__ offsets,
                                                             int32_t* __restrict__ padded,
                                                             int32_t* __restrict__ inv, int32_t* __restrict__ perm,
                                                             int* status) {
  grid_dep_sync();
  __shared__ PermuteSmem sm;
  permute_small_block(ids, n, k, E, true, counts, offsets, padded, inv, perm, status, sm);
}

// The forward's whole prologue for small batches (n = T*k <= 1024): one CTA per token.
// Every CTA forms the same slot order (permute_small_block; CTA 0 stores it), then its
// warp 0 quantises the token's row of x (per-row scale, round to nearest: the row
// quantiser's arithmetic) and writes it into each of the token's k slots of the
// GEMM-tiled operand aq (128-row blocks, K = H), with the token's global scale in ga and
// a zero in h_amax.  This replaces the permutation, the token-order quantisation and the
// slot gather (three to five launches) for decode-size batches; slots of group padding
// are left as they are (no kernel stores their results).
__global__ void __launch_bounds__(1024) moe_prologue_small_kernel(
    const int32_t* __restrict__ ids, int n, int k, int E, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ padded, int32_t* __restrict__ inv,
    int32_t* __restrict__ perm, int* status, const __nv_bfloat16* __restrict__ x, int64_t H, uint8_t* aq,
    float* __restrict__ ga, uint32_t* __restrict__ h_amax) {
  grid_dep_sync();
  __shared__ PermuteSmem sm;
  permute_small_block(ids, n, k, E, blockIdx.x == 0, counts, offsets, padded, inv, perm, status, sm);
  __syncthreads();
  if (threadIdx.x >= 32) return;
  constexpr int kMaxSlots = 4;                  // 16-value blocks per lane: H <= 2048
  const int lane = threadIdx.x;
  const int64_t t = blockIdx.x;
  const int nb = (int)(H / 16);
  const int64_t kblocks = H / 256;
  uint4 q[kMaxSlots][2];
  float bm[kMaxSlots];
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < kMaxSlots; ++i) {
    const int b = lane + 32 * i;
    q[i][0] = q[i][1] = make_uint4(0u, 0u, 0u, 0u);
    bm[i] = 0.0f;
    if (b < nb) {
      q[i][0] = *reinterpret_cast<const uint4*>(x + t * H + 16 * b);
      q[i][1] = *reinterpret_cast<const uint4*>(x + t * H + 16 * b + 8);
      bm[i] = absmax16_bf16(q[i][0], q[i][1]);
      m = fmaxf(m, bm[i]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFullMask, m, o));
  const float g = __fdiv_rn(m, kGlobalDivisor);
  const float six_g = __fmul_rn(6.0f, g);
  uint2 cw[kMaxSlots];
  uint32_t sfw[kMaxSlots];
#pragma unroll
  for (int i = 0; i < kMaxSlots; ++i) {
    const int b = lane + 32 * i;
    uint32_t sfb = 0;
    cw[i] = make_uint2(0u, 0u);
    if (b < nb) {
      float h0[8], h1[8];
      bf16x8_to_f32(q[i][0], h0);
      bf16x8_to_f32(q[i][1], h1);
      const BlockScale bs = block_scale(bm[i], g, six_g);
      cw[i] = e2m1x16_rn(h0, h1, bs);
      sfb = bs.sf;
    }
    const uint32_t s1 = __shfl_down_sync(kFullMask, sfb, 1);
    const uint32_t s2 = __shfl_down_sync(kFullMask, sfb, 2);
    const uint32_t s3 = __shfl_down_sync(kFullMask, sfb, 3);
    sfw[i] = sfb | (s1 << 8) | (s2 << 16) | (s3 << 24);
  }
  for (int j = 0; j < k; ++j) {
    const int32_t slot = sm.inv[t * k + j];
    if (slot < 0) continue;                     // an id out of range: counted nowhere
    const int64_t rr = slot & 127;
    uint8_t* blk0 = aq + (int64_t)(slot >> 7) * kblocks * tiled_block_bytes(128);
#pragma unroll
    for (int i = 0; i < kMaxSlots; ++i) {
      const int b = lane + 32 * i;
      if (b >= nb) continue;
      *reinterpret_cast<uint2*>(blk0 + (b >> 4) * tiled_block_bytes(128) + rr * 128 +
                                ((((b >> 1) & 7) ^ (rr & 7)) << 4) + (b & 1) * 8) = cw[i];
      const int wd = b >> 2;
      if ((lane & 3) == 0)
        *reinterpret_cast<uint32_t*>(blk0 + (wd >> 2) * tiled_block_bytes(128) + 128 * 128 + (wd & 3) * 512 +
                                     (rr & 31) * 16 + (rr >> 5) * 4) = sfw[i];
    }
    if (lane == 0) {
      ga[slot] = g;
      h_amax[slot] = 0u;
    }
  }
}

cudaError_t launch_prologue_small(const int32_t* ids, int64_t T, int k, int E, int32_t* counts, int32_t* offsets,
                                  int32_t* padded, int32_t* inv, int32_t* perm, int* status, const void* x, int64_t H,
                                  uint8_t* aq, float* ga, uint32_t* h_amax, cudaStream_t s) {
  if (T * k > 1024 || E > 1024 || H % 256 != 0 || H > 2048) return cudaErrorInvalidValue;
  if (T == 0) return cudaSuccess;
  return launch_pdl(true, moe_prologue_small_kernel, dim3((unsigned)T), dim3(1024), 0, s, ids, (int)(T * k), k, E, counts,
                    offsets, padded, inv, perm, status, static_cast<const __nv_bfloat16*>(x), H, aq, ga, h_amax);
}

cudaError_t launch_permute(const int32_t* ids, int64_t T, int k, int E, int32_t* counts, int32_t* offsets,
                           int32_t* padded, int32_t* inv, int32_t* perm, int32_t* hist, int64_t nchunks,
                           int* status, cudaStream_t s) {
  const int64_t n = T * k;
  if (n > 0 && n <= 1024 && E <= 1024) {
    return launch_pdl(false, permute_small_kernel, dim3(1), dim3(1024), 0, s, ids, (int)n, k, E, counts, offsets, padded, inv,
                      perm, status);
  }
  const int blocks = (int)((nchunks + 7) / 8);
  if (nchunks > 0) {
    cudaError_t err = launch_pdl(false, permute_hist_kernel, dim3(blocks), dim3(256), 8 * E * sizeof(int32_t), s, ids, n, E,
                                 nchunks, hist, status);
    if (err != cudaSuccess) return err;
  }
  // no entries: the scan still writes counts / offsets (one block)
  cudaError_t err = launch_pdl(false, permute_scan_kernel, dim3(nchunks == 0 ? 1u : (unsigned)((E + 31) / 32)), dim3(1024), 0,
                               s, hist, nchunks, E, counts, offsets, padded, perm);
  if (err != cudaSuccess || nchunks == 0) return err;
  return launch_pdl(false, permute_rank_kernel, dim3(blocks), dim3(256), 9 * E * sizeof(int32_t), s, ids, n, k, E, nchunks,
                    hist, padded, inv, perm);
}

// ------------------------------------------------------------------ weighted un-permute

// One warp per token; lane l owns columns 8l + 256i.  out = BF16 of the float32 sum, in
// order j = 0..k-1, of float32 products w[t, j] * y[slot]; a slot of -1 (an entry whose
// expert id was rejected) contributes nothing.  For k <= KM the k slot rows of a column
// chunk are loaded before any is summed (k loads in flight per lane); a missing slot
// loads zeros with weight 0, whose +0 product leaves the (never -0) sum unchanged.
template <int KM>
__global__ void __launch_bounds__(256) combine_kernel(const __nv_bfloat16* __restrict__ y,
                                                      const int32_t* __restrict__ inv,
                                                      const float* __restrict__ w, int64_t T, int k, int64_t H,
                                                      __nv_bfloat16* __restrict__ out) {
  grid_dep_sync();
  // one warp per (token, 256-column chunk): small batches still spread over the GPU
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int64_t nwarp = (int64_t)gridDim.x * 8;
  const int64_t nch = (H + 255) / 256;
  for (int64_t item = warp; item < T * nch; item += nwarp) {
    const int64_t t = item / nch, c0 = (item - t * nch) * 256;
    int32_t my_slot = -1;
    float my_w = 0.0f;
    if (lane < k) {
      my_slot = inv[t * k + lane];
      my_w = w != nullptr ? w[t * k + lane] : 1.0f;   // no weights: the plain sum (exact products)
    }
    if (my_slot < 0) my_w = 0.0f;
    for (int64_t c = c0 + 8 * lane; c < min(H, c0 + 256); c += 256) {
      float acc[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = 0.0f;
      if constexpr (KM > 0) {
        uint4 q[KM];
#pragma unroll
        for (int j = 0; j < KM; ++j) {
          const int32_t sl = __shfl_sync(kFullMask, my_slot, j);
          q[j] = j < k && sl >= 0 ? *reinterpret_cast<const uint4*>(y + (int64_t)sl * H + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < KM; ++j) {
          if (j >= k) break;
          const float wj = __shfl_sync(kFullMask, my_w, j);
          const uint32_t wd[4] = {q[j].x, q[j].y, q[j].z, q[j].w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[2 * e] = __fadd_rn(acc[2 * e], __fmul_rn(wj, __uint_as_float(wd[e] << 16)));
            acc[2 * e + 1] = __fadd_rn(acc[2 * e + 1], __fmul_rn(wj, __uint_as_float(wd[e] & 0xFFFF0000u)));
          }
        }
      } else {
        for (int j = 0; j < k; ++j) {
          const int32_t sl = __shfl_sync(kFullMask, my_slot, j);
          const float wj = __shfl_sync(kFullMask, my_w, j);
          if (sl < 0) continue;
          const uint4 q = *reinterpret_cast<const uint4*>(y + (int64_t)sl * H + c);
          const uint32_t wd[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[2 * e] = __fadd_rn(acc[2 * e], __fmul_rn(wj, __uint_as_float(wd[e] << 16)));
            acc[2 * e + 1] = __fadd_rn(acc[2 * e + 1], __fmul_rn(wj, __uint_as_float(wd[e] & 0xFFFF0000u)));
          }
        }
      }
      uint4 o;
      uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 p = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
        ow[e] = *reinterpret_cast<const uint32_t*>(&p);
      }
      *reinterpret_cast<uint4*>(out + t * H + c) = o;
    }
  }
}

cudaError_t launch_combine(const void* y, const int32_t* inv, const float* w, int64_t T, int k, int64_t H, void* out,
                           cudaStream_t s, bool pdl) {
  if (T == 0) return cudaSuccess;
  int64_t blocks = (T * ((H + 255) / 256) + 7) / 8;
  if (blocks > 16 * num_sms()) blocks = 16 * num_sms();
  const auto* yp = static_cast<const __nv_bfloat16*>(y);
  auto* op = static_cast<__nv_bfloat16*>(out);
  return k <= 8 ? launch_pdl(pdl, combine_kernel<8>, dim3((unsigned)blocks), dim3(256), 0, s, yp, inv, w, T, k, H, op)
                : launch_pdl(pdl, combine_kernel<0>, dim3((unsigned)blocks), dim3(256), 0, s, yp, inv, w, T, k, H, op);
}

}  // namespace nvfp4

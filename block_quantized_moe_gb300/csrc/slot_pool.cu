// Device-side expert-slot pool with least-recently-used victims, one decode step per call:
// the contract of the hybrid expert cache's victim selection on the FreeToken cache page (the
// pull request that speeds up victim selection in its ensure-experts kernel):
//   1. the slot of every requested expert that is resident is marked used in this step, which
//      makes it the most recently used slot of the pool (Change, first point);
//   2. the distinct missing experts, in order of first appearance among the routes and up to
//      the step's fetch budget, each take the least recently used slot not used in this step,
//      ties to the lowest slot (Change, second point), evicting its previous expert; the copy
//      plan lists (slot, expert);
//   3. every route's expert id is rewritten to its slot, or -1 if the expert is not resident --
//      only after every route has been read (Fix: the in-place rewrite raced with later loads).
// One CTA owns the whole pool for the step, so the pool state needs no atomics beyond the
// first-appearance claims; every other write happens between block barriers.
#include <limits.h>

#include "common.cuh"
#include "internal.h"

namespace ftmoe {

constexpr int kPoolThreads = 1024;
constexpr int kPoolWarps = kPoolThreads / 32;

__device__ __forceinline__ void argmin_pair(long long& u, int& s, long long ou, int os) {
  if (ou < u || (ou == u && os < s)) {
    u = ou;
    s = os;
  }
}

__global__ void __launch_bounds__(kPoolThreads, 1)
    slot_pool_kernel(int32_t* __restrict__ ids, int R, int32_t* __restrict__ slot_expert,
                     long long* __restrict__ usage, int S, int32_t* __restrict__ expert_slot, int E, long long step,
                     int max_fetch, int32_t* __restrict__ plan, int32_t* __restrict__ n_fetch) {
  extern __shared__ int pool_smem[];
  int* rid = pool_smem;          // [R] each route's expert, -1 if inactive or out of range
  int* claim = rid + R;          // [E] the first route asking for expert e
  int* miss = claim + E;         // [min(max_fetch, R)] missing experts by rank
  __shared__ int s_scan[kPoolWarps + 1];
  __shared__ long long s_wu[kPoolWarps];
  __shared__ int s_ws[kPoolWarps];
  __shared__ int s_stop;
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  for (int e = tid; e < E; e += kPoolThreads) claim[e] = INT_MAX;
  // every route is read before any is rewritten
  for (int r = tid; r < R; r += kPoolThreads) {
    int v = ids[r];
    if (v >= E) {
      raise_error(FTMOE_ERR_EXPERT_ID_RANGE);
      v = -1;
    }
    rid[r] = v < 0 ? -1 : v;
  }
  __syncthreads();
  for (int r = tid; r < R; r += kPoolThreads)
    if (rid[r] >= 0) atomicMin(&claim[rid[r]], r);
  __syncthreads();
  // 1. hits; first appearances of missing experts counted over contiguous runs of routes
  const int per = (R + kPoolThreads - 1) / kPoolThreads;
  const int r0 = tid * per, r1 = r0 + per < R ? r0 + per : R;
  int cnt = 0;
  for (int r = r0; r < r1; ++r) {
    const int e = rid[r];
    if (e < 0 || claim[e] != r) continue;  // the first route of the expert decides
    const int s = expert_slot[e];
    if (s >= 0)
      usage[s] = step;
    else
      ++cnt;
  }
  // ranks of the missing experts in route order (block exclusive scan)
  int inc = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) s_scan[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    const int w = s_scan[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    s_scan[lane] = wi - w;
    if (lane == 31) s_scan[kPoolWarps] = wi;
  }
  __syncthreads();
  const int nmiss = s_scan[kPoolWarps];
  int k = s_scan[warp] + inc - cnt;
  for (int r = r0; r < r1; ++r) {
    const int e = rid[r];
    if (e < 0 || claim[e] != r || expert_slot[e] >= 0) continue;
    if (k < max_fetch) miss[k] = e;
    ++k;
  }
  __syncthreads();
  // 2. fetches, one after another: the least recently used slot not used in this step
  const int nf = nmiss < max_fetch ? nmiss : max_fetch;
  int fetched = 0;
  for (int f = 0; f < nf; ++f) {
    long long bu = LLONG_MAX;
    int bs = INT_MAX;
    for (int s = tid; s < S; s += kPoolThreads) {
      const long long u = usage[s];
      if (u < step) argmin_pair(bu, bs, u, s);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      argmin_pair(bu, bs, __shfl_xor_sync(0xffffffffu, bu, o), __shfl_xor_sync(0xffffffffu, bs, o));
    if (lane == 0) {
      s_wu[warp] = bu;
      s_ws[warp] = bs;
    }
    __syncthreads();
    if (warp == 0) {
      bu = s_wu[lane];
      bs = s_ws[lane];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
        argmin_pair(bu, bs, __shfl_xor_sync(0xffffffffu, bu, o), __shfl_xor_sync(0xffffffffu, bs, o));
      if (lane == 0) {
        s_stop = bs == INT_MAX;  // every slot was used in this step
        if (!s_stop) {
          const int e = miss[f];
          const int old = slot_expert[bs];
          if (old >= 0) expert_slot[old] = -1;
          slot_expert[bs] = e;
          expert_slot[e] = bs;
          usage[bs] = step;
          plan[2 * f] = bs;
          plan[2 * f + 1] = e;
        }
      }
    }
    __syncthreads();
    if (s_stop) break;
    ++fetched;
  }
  if (tid == 0) *n_fetch = fetched;
  // 3. routes to slots, after every fetch
  for (int r = tid; r < R; r += kPoolThreads) {
    const int e = rid[r];
    ids[r] = e >= 0 ? expert_slot[e] : -1;
  }
}

FTMOE_DEFINE_ERR_READER(read_err_slots)

}  // namespace ftmoe

extern "C" ftmoe_status ftmoe_expert_slots(int32_t* expert_ids, int64_t routes, int32_t* slot_expert,
                                           int64_t* slot_usage, int32_t num_slots, int32_t* expert_slot,
                                           int32_t num_experts, int64_t step, int32_t max_fetch, int32_t* fetch_plan,
                                           int32_t* n_fetch, void* stream) {
  using namespace ftmoe;
  if (routes < 0 || routes > kSlotPoolMaxRoutes || num_slots <= 0 || num_experts <= 0 ||
      num_experts > kSlotPoolMaxExperts || max_fetch < 0)
    return FTMOE_INVALID_ARG;
  if (!slot_expert || !slot_usage || !expert_slot || !n_fetch || (routes > 0 && !expert_ids) ||
      (max_fetch > 0 && !fetch_plan))
    return FTMOE_INVALID_ARG;
  const int64_t nmiss_store = max_fetch < routes ? max_fetch : routes;
  const size_t smem = (size_t)(routes + num_experts + nmiss_store) * 4;
  static size_t granted[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || smem > granted[dev]) {
    if (cudaFuncSetAttribute(slot_pool_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return FTMOE_CUDA_ERROR;
    if (dev >= 0 && dev < 64) granted[dev] = smem;
  }
  const cudaError_t e =
      launch_kernel(slot_pool_kernel, dim3(1), dim3(kPoolThreads), smem, reinterpret_cast<cudaStream_t>(stream),
                    false, expert_ids, (int)routes, slot_expert, reinterpret_cast<long long*>(slot_usage),
                    (int)num_slots, expert_slot, (int)num_experts, (long long)step, (int)nmiss_store, fetch_plan,
                    n_fetch);
  return e == cudaSuccess ? FTMOE_OK : FTMOE_CUDA_ERROR;
}

// Expert segmenter: per-expert row counts and offsets, the dst2src map the gather walks
// ("m * topk entries", SGLang gather page, Motivation) and route2dst for the combine.
//
// One CTA per expert e. Each thread owns a contiguous run of routes, so route order
// inside an expert (stability) follows from an exclusive scan of per-thread match
// counts. The CTA also counts the active routes of lower experts for its own offset.
// No atomics: every output is a deterministic function of expert_ids.
#include "common.cuh"
#include "internal.h"

namespace ftmoe {

constexpr int kSegThreads = 512;

__device__ __forceinline__ int block_exclusive_scan(int v, int* total, int* sh /*[32]*/) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int inc = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) sh[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int w = lane < (int)(blockDim.x >> 5) ? sh[lane] : 0;
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += t;
    }
    sh[lane] = wi - w;  // exclusive prefix of warp totals
    if (lane == 31) sh[32] = wi;
  }
  __syncthreads();
  const int res = sh[warp] + inc - v;
  *total = sh[32];
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(kSegThreads) segment_kernel(
    const int32_t* __restrict__ ids, int64_t routes, int32_t topk, int32_t E,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ dst2src,
    int32_t* __restrict__ route2dst) {
  pdl_wait();  // the predecessor's outputs are complete from here on
  pdl_trigger();
  __shared__ int sh[33];
  const int e = blockIdx.x;
  const int64_t per = (routes + blockDim.x - 1) / blockDim.x;
  const int64_t r0 = (int64_t)threadIdx.x * per;
  const int64_t r1 = r0 + per < routes ? r0 + per : routes;

  int below = 0, mine = 0;
  for (int64_t r = r0; r < r1; ++r) {
    const int id = ids[r];
    below += (id >= 0 && id < e);
    mine += (id == e);
    if (e == 0 && id >= E) raise_error(FTMOE_ERR_EXPERT_ID_RANGE);
  }
  int below_total, mine_total;
  (void)block_exclusive_scan(below, &below_total, sh);
  const int my_base = block_exclusive_scan(mine, &mine_total, sh);
  const int off = below_total;
  if (threadIdx.x == 0) {
    counts[e] = mine_total;
    offsets[e] = off;
    if (e == E - 1) offsets[E] = off + mine_total;
  }
  int d = off + my_base;
  for (int64_t r = r0; r < r1; ++r) {
    const int id = ids[r];
    if (id == e) {
      dst2src[d] = (int32_t)(r / topk);
      route2dst[r] = d;
      ++d;
    } else if (e == 0 && (id < 0 || id >= E)) {
      route2dst[r] = -1;  // inactive (or out-of-range, reported above) routes
    }
  }
}

cudaError_t launch_segment(const int32_t* ids, int64_t routes, int32_t topk, int32_t E,
                           int32_t* counts, int32_t* offsets, int32_t* dst2src,
                           int32_t* route2dst, cudaStream_t st) {
  return launch_kernel(segment_kernel, dim3(E), dim3(kSegThreads), 0, st, true, ids, routes, topk, E, counts, offsets,
                       dst2src, route2dst);
}

FTMOE_DEFINE_ERR_READER(read_err_segment)

}  // namespace ftmoe

// Expert segmenter: per-expert row counts and offsets, the dst2src map the gather walks
// ("m * topk entries", SGLang gather page, Motivation) and route2dst for the combine.
//
// One CTA per expert e. The routes are walked in chunks of the block size, one id per
// thread, so route order inside an expert (stability) follows from an exclusive scan of
// the matches in each chunk. The CTA also counts the active routes of lower experts for
// its own offset. No atomics: every output is a deterministic function of expert_ids.
#include "common.cuh"
#include "internal.h"
#include "rowquant.cuh"

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

// Segments of expert e, by one CTA of kSegThreads threads. Pass 1 counts the active
// routes of lower experts (this expert's offset) and of this expert; pass 2 walks the
// routes in chunks of blockDim.x, one coalesced id per thread, and gives each matching
// route its row by an exclusive scan of the chunk, so rows follow route order.
__device__ __forceinline__ void segment_expert(const int32_t* __restrict__ ids, int64_t routes, int32_t topk,
                                               int32_t E, int32_t* __restrict__ counts,
                                               int32_t* __restrict__ offsets, int32_t* __restrict__ dst2src,
                                               int32_t* __restrict__ route2dst, int e, int* sh) {
  int below = 0, mine = 0;
  for (int64_t r = threadIdx.x; r < routes; r += blockDim.x) {
    const int id = ids[r];
    below += (id >= 0 && id < e);
    mine += (id == e);
    if (e == 0 && id >= E) raise_error(FTMOE_ERR_EXPERT_ID_RANGE);
  }
  int below_total, mine_total;
  (void)block_exclusive_scan(below, &below_total, sh);
  (void)block_exclusive_scan(mine, &mine_total, sh);
  const int off = below_total;
  if (threadIdx.x == 0) {
    counts[e] = mine_total;
    offsets[e] = off;
    if (e == E - 1) offsets[E] = off + mine_total;
  }
  int base = off;
  for (int64_t c0 = 0; c0 < routes; c0 += blockDim.x) {
    const int64_t r = c0 + threadIdx.x;
    const int id = r < routes ? ids[r] : -1;
    int chunk_total;
    const int pos = block_exclusive_scan(id == e ? 1 : 0, &chunk_total, sh);
    if (id == e) {
      const int d = base + pos;
      dst2src[d] = (int32_t)(r / topk);
      route2dst[r] = d;
    } else if (e == 0 && r < routes && (id < 0 || id >= E)) {
      route2dst[r] = -1;  // inactive (or out-of-range, reported above) routes
    }
    base += chunk_total;
  }
}

__global__ void __launch_bounds__(kSegThreads) segment_kernel(
    const int32_t* __restrict__ ids, int64_t routes, int32_t topk, int32_t E,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ dst2src,
    int32_t* __restrict__ route2dst) {
  pdl_wait();  // the predecessor's outputs are complete from here on
  pdl_trigger();
  __shared__ int sh[33];
  segment_expert(ids, routes, topk, E, counts, offsets, dst2src, route2dst, blockIdx.x, sh);
}

// The fused forward's first launch: FP8 quantization of the token rows and the expert
// segmenter are independent steps, so one grid runs both -- blocks [0, E) segment one
// expert each (first, as they take longest), blocks [E, E + qblocks) quantize (one warp
// per 1x128 group).
template <bool kVec>
__global__ void __launch_bounds__(kSegThreads) prep_fp8_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t k, int64_t ld_x, uint8_t* __restrict__ q,
    float* __restrict__ s, int64_t ng, int qblocks, const int32_t* __restrict__ ids, int64_t routes, int32_t topk,
    int32_t E, int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ dst2src,
    int32_t* __restrict__ route2dst) {
  pdl_wait();  // the predecessor's outputs are complete from here on
  pdl_trigger();
  __shared__ int sh[33];
  if ((int)blockIdx.x < E) {
    segment_expert(ids, routes, topk, E, counts, offsets, dst2src, route2dst, (int)blockIdx.x, sh);
  } else {
    const int qb = (int)blockIdx.x - E;
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)qblocks * (blockDim.x >> 5);
    for (int64_t w = (int64_t)qb * (blockDim.x >> 5) + (threadIdx.x >> 5); w < rows * ng; w += nwarps) {
      const int64_t row = w / ng, g = w - row * ng;
      quantize_fp8_group<kVec>(x, k, ld_x, q, s, ng, row, g, lane);
    }
  }
}

cudaError_t launch_segment(const int32_t* ids, int64_t routes, int32_t topk, int32_t E,
                           int32_t* counts, int32_t* offsets, int32_t* dst2src,
                           int32_t* route2dst, cudaStream_t st) {
  return launch_kernel(segment_kernel, dim3(E), dim3(kSegThreads), 0, st, true, ids, routes, topk, E, counts, offsets,
                       dst2src, route2dst);
}

cudaError_t launch_prep_fp8(const uint16_t* x, int64_t rows, int64_t k, int64_t ld_x, uint8_t* q, float* scales,
                            const int32_t* ids, int64_t routes, int32_t topk, int32_t E, int32_t* counts,
                            int32_t* offsets, int32_t* dst2src, int32_t* route2dst, cudaStream_t st) {
  const int64_t ng = cdiv(k, kGroup);
  const int64_t warps = rows * ng;
  int64_t qb = cdiv(warps, kSegThreads / 32);
  if (qb > 152 * 16) qb = 152 * 16;  // grid-stride beyond this
  if (qb < 1) qb = 1;
  const bool vec = quantize_fp8_vec_ok(x, ld_x, q, k);
  return launch_kernel(vec ? prep_fp8_kernel<true> : prep_fp8_kernel<false>, dim3((unsigned)qb + E),
                       dim3(kSegThreads), 0, st, true, x, rows, k, ld_x, q, scales, ng, (int)qb, ids, routes, topk, E,
                       counts, offsets, dst2src, route2dst);
}

FTMOE_DEFINE_ERR_READER(read_err_segment)

}  // namespace ftmoe

// Expert segmenter: per-expert row counts and offsets, the dst2src map the gather walks
// ("m * topk entries", SGLang gather page, Motivation) and route2dst for the combine.
//
// One CTA per expert e. Each warp of the CTA owns a contiguous range of routes and walks it
// 32 ids at a time (coalesced); a ballot and a population count give each matching route
// its place inside the warp's range, and one scan of the warps' totals gives each range its
// first row, so rows follow route order (stability). The CTA also counts the active routes
// of lower experts for its own offset. No atomics: every output is a deterministic function
// of expert_ids.
#include "common.cuh"
#include "internal.h"
#include "rowquant.cuh"

namespace ftmoe {

constexpr int kSegThreads = 512;
constexpr int kSegBatch = 8;  // 32-id steps whose loads a warp issues together

// Segments of expert e, by one CTA of kSegThreads threads (sh: 2 * kSegThreads / 32 ints).
// Pass 1: every warp counts, over its own range, the active routes of lower experts and
// the routes of expert e. The warps' counts are combined once. Pass 2: every warp walks its
// range again and writes its matches from its first row on.
__device__ __forceinline__ void segment_expert(const int32_t* __restrict__ ids, int64_t routes, int32_t topk,
                                               int32_t E, int32_t* __restrict__ counts,
                                               int32_t* __restrict__ offsets, int32_t* __restrict__ dst2src,
                                               int32_t* __restrict__ route2dst, int e, int* sh) {
  constexpr int kWarps = kSegThreads / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // the warp's range [r0, r1), a whole number of 32-id steps. Range ri goes to warp
  // (ri - e) mod 16: every CTA reads all of the ids at the same time, and the rotation spreads
  // their first reads over 16 places instead of one
  const int ri = (warp + e) % kWarps;
  const int64_t span = ((routes + kWarps - 1) / kWarps + 31) / 32 * 32;
  const int64_t r0 = span * ri;
  const int64_t r1 = r0 + span < routes ? r0 + span : routes;
  // (the ids of a chunk of kSegBatch steps are loaded together: the walk is a chain of L2
  // round trips otherwise)
  int below = 0, mine = 0;
  for (int64_t c0 = r0; c0 < r1; c0 += 32 * kSegBatch) {
    int v[kSegBatch];
#pragma unroll
    for (int u = 0; u < kSegBatch; ++u) {
      const int64_t r = c0 + 32 * u + lane;
      v[u] = r < r1 ? ids[r] : -1;
    }
#pragma unroll
    for (int u = 0; u < kSegBatch; ++u) {
      below += (v[u] >= 0 && v[u] < e);
      mine += (v[u] == e);
      if (e == 0 && v[u] >= E) raise_error(FTMOE_ERR_EXPERT_ID_RANGE);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    below += __shfl_xor_sync(0xffffffffu, below, o);
    mine += __shfl_xor_sync(0xffffffffu, mine, o);
  }
  if (lane == 0) {
    sh[ri] = mine;
    sh[kWarps + ri] = below;
  }
  __syncthreads();
  int first = 0, off = 0, total = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    first += w < ri ? sh[w] : 0;
    total += sh[w];
    off += sh[kWarps + w];
  }
  if (threadIdx.x == 0) {
    counts[e] = total;
    offsets[e] = off;
    if (e == E - 1) offsets[E] = off + total;
  }
  int base = off + first;
  const uint32_t lower = (1u << lane) - 1u;
  for (int64_t c0 = r0; c0 < r1; c0 += 32 * kSegBatch) {
    int v[kSegBatch];
#pragma unroll
    for (int u = 0; u < kSegBatch; ++u) {
      const int64_t r = c0 + 32 * u + lane;
      v[u] = r < r1 ? ids[r] : -1;
    }
#pragma unroll
    for (int u = 0; u < kSegBatch; ++u) {
      const int64_t r = c0 + 32 * u + lane;
      const int id = v[u];
      const uint32_t m = __ballot_sync(0xffffffffu, id == e);
      if (id == e) {
        const int d = base + __popc(m & lower);
        dst2src[d] = (int32_t)(r / topk);
        route2dst[r] = d;
      } else if (e == 0 && r < r1 && (id < 0 || id >= E)) {
        route2dst[r] = -1;  // inactive (or out-of-range, reported above) routes
      }
      base += __popc(m);
    }
  }
}

__global__ void __launch_bounds__(kSegThreads) segment_kernel(
    const int32_t* __restrict__ ids, int64_t routes, int32_t topk, int32_t E,
    int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ dst2src,
    int32_t* __restrict__ route2dst) {
  pdl_wait();  // the predecessor's outputs are complete from here on
  pdl_trigger();
  __shared__ int sh[2 * (kSegThreads / 32)];
  segment_expert(ids, routes, topk, E, counts, offsets, dst2src, route2dst, blockIdx.x, sh);
}

// The fused forward's first launch: FP8 quantization of the token rows and the expert
// segmenter are independent steps, so one grid runs both -- blocks [0, E) segment one
// expert each (first, as they take longest), blocks [E, E + qblocks) quantize (a half-warp
// per 1x128 group). With the down GEMM's fused combine the quantizing blocks also zero its
// arrival counters and write the zero output rows of tokens that have no active route (the
// combine inside the GEMM only reaches tokens with at least one).
template <bool kVec>
__global__ void __launch_bounds__(kSegThreads) prep_fp8_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t k, int64_t ld_x, uint8_t* __restrict__ q,
    float* __restrict__ s, int64_t ng, int qblocks, const int32_t* __restrict__ ids, int64_t routes, int32_t topk,
    int32_t E, int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ dst2src,
    int32_t* __restrict__ route2dst, PrepCombine pc) {
  pdl_wait();  // the predecessor's outputs are complete from here on
  pdl_trigger();
  __shared__ int sh[2 * (kSegThreads / 32)];
  if ((int)blockIdx.x < E) {
    segment_expert(ids, routes, topk, E, counts, offsets, dst2src, route2dst, (int)blockIdx.x, sh);
  } else {
    const int qb = (int)blockIdx.x - E;
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)qblocks * (blockDim.x >> 5);
    const int64_t gwarp = (int64_t)qb * (blockDim.x >> 5) + (threadIdx.x >> 5);
    quantize_fp8_rows_hw<kVec>(x, k, ld_x, q, s, ng, rows * ng, gwarp, nwarps, lane);
    if (pc.zero_words != nullptr) {
      for (int64_t i = gwarp * 32 + lane; i < pc.n_zero_words; i += nwarps * 32) pc.zero_words[i] = 0u;
    }
    if (pc.out_rows != nullptr) {
      // (rows of hidden * out_bytes bytes, a multiple of 16, at 16-byte aligned starts)
      const int64_t row_bytes = pc.hidden * pc.out_bytes, ld_bytes = pc.ld_out * pc.out_bytes;
      for (int64_t t = gwarp; t < rows; t += nwarps) {
        bool any = false;
        for (int64_t j = lane; j < topk; j += 32) {
          const int id = ids[t * topk + j];
          any = any || (id >= 0 && id < E);
        }
        if (__any_sync(0xffffffffu, any)) continue;
        uint8_t* o = static_cast<uint8_t*>(pc.out_rows) + t * ld_bytes;
        for (int64_t b = (int64_t)lane * 16; b < row_bytes; b += 32 * 16)
          *reinterpret_cast<uint4*>(o + b) = make_uint4(0u, 0u, 0u, 0u);
      }
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
                            int32_t* offsets, int32_t* dst2src, int32_t* route2dst, const PrepCombine& pc,
                            cudaStream_t st) {
  const int64_t ng = cdiv(k, kGroup);
  const int64_t warps = cdiv(rows * ng, 2 * kHwBatch);
  int64_t qb = cdiv(warps, kSegThreads / 32);
  if (qb > 152 * 2) qb = 152 * 2;  // two resident CTAs per SM; the warps stride over the rest
  if (qb < 1) qb = 1;
  const bool vec = quantize_fp8_vec16_ok(x, ld_x, q, k);
  return launch_kernel(vec ? prep_fp8_kernel<true> : prep_fp8_kernel<false>, dim3((unsigned)qb + E),
                       dim3(kSegThreads), 0, st, true, x, rows, k, ld_x, q, scales, ng, (int)qb, ids, routes, topk, E,
                       counts, offsets, dst2src, route2dst, pc);
}

FTMOE_DEFINE_ERR_READER(read_err_segment)

}  // namespace ftmoe

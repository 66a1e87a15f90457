// Fused FP8 row + scale gather (SGLang "Gather the cutlass MoE activation and its scales
// in one launch", Modifications): one walk of dst2src writes both the row bytes and the
// row's scales; the unit of work that owns column 0 of a row also carries its scale row.
// Bytes are copied, never decoded. Row bases are 64-bit. Tails are masked, so any row width
// and any scale-row width (e.g. k = 896, 7 scales) works.
//
// One warp per (destination row, column tile): a row is split into as many tiles as it
// takes to give every SM several warps when rows are few, and is one tile when they are
// many. Each lane issues all of its 16-byte loads of a pass (up to kVecPerLane vectors)
// before its stores, and the map entry of the warp's next row is read while the current
// row is copied, so the map-then-row latency chain overlaps across rows.
#include "common.cuh"
#include "internal.h"

namespace ftmoe {

constexpr int kGatherThreads = 256;
constexpr int kGatherWarps = kGatherThreads / 32;
constexpr int kVecPerLane = 8;          // 16-byte vectors in flight per lane and pass
constexpr int kGatherCtasPerSm = 4;

// The row's scales, copied by the lanes of the warp that owns column 0.
__device__ __forceinline__ void copy_scale_row(const uint8_t* ss, uint8_t* ds, int64_t scale_bytes, int scale_mode,
                                               int lane) {
  if (scale_mode == 2) {
    for (int64_t c = (int64_t)lane * 16; c < scale_bytes; c += 32 * 16)
      *reinterpret_cast<uint4*>(ds + c) = *reinterpret_cast<const uint4*>(ss + c);
  } else if (scale_mode == 1) {
    for (int64_t c = (int64_t)lane * 4; c < scale_bytes; c += 32 * 4)
      *reinterpret_cast<uint32_t*>(ds + c) = *reinterpret_cast<const uint32_t*>(ss + c);
  } else {
    for (int64_t c = lane; c < scale_bytes; c += 32) ds[c] = ss[c];
  }
}

template <bool kVec>
__global__ void __launch_bounds__(kGatherThreads) gather_kernel(
    const uint8_t* __restrict__ src, const uint8_t* __restrict__ src_s, int64_t n_src, int64_t row_bytes,
    int64_t scale_bytes, const int32_t* __restrict__ map, int64_t n_dst, const int32_t* __restrict__ n_dst_dev,
    uint8_t* __restrict__ dst, uint8_t* __restrict__ dst_s, int wpr, int64_t tile_bytes, int scale_mode) {
  pdl_wait();  // the predecessor's outputs are complete from here on
  pdl_trigger();
  int64_t limit = n_dst;
  if (n_dst_dev != nullptr) {
    const int64_t d = *n_dst_dev;
    limit = d < limit ? d : limit;
  }
  const int lane = threadIdx.x & 31;
  const int64_t nw = (int64_t)gridDim.x * kGatherWarps;
  const int64_t items = limit * wpr;
  int64_t w = (int64_t)blockIdx.x * kGatherWarps + (threadIdx.x >> 5);
  int32_t m_next = w < items ? __ldg(map + w / wpr) : 0;
  for (; w < items; w += nw) {
    const int64_t r = w / wpr;
    const int tile = (int)(w - r * wpr);
    const int32_t m = m_next;
    if (w + nw < items) m_next = __ldg(map + (w + nw) / wpr);  // the next row's entry, in flight now
    const bool ok = m >= 0 && (int64_t)m < n_src;
    if (!ok) {
      if (tile == 0 && lane == 0) raise_error(FTMOE_ERR_MAP_RANGE);
      continue;
    }
    const int64_t c_begin = (int64_t)tile * tile_bytes;
    const int64_t c_end = c_begin + tile_bytes < row_bytes ? c_begin + tile_bytes : row_bytes;
    const uint8_t* s = src + (int64_t)m * row_bytes;
    uint8_t* d = dst + r * row_bytes;
    if (kVec) {
      for (int64_t cb = c_begin + (int64_t)lane * 16; cb < c_end; cb += 32 * 16 * kVecPerLane) {
        uint4 v[kVecPerLane];
#pragma unroll
        for (int u = 0; u < kVecPerLane; ++u) {
          const int64_t c = cb + (int64_t)u * 32 * 16;
          if (c < c_end) v[u] = __ldg(reinterpret_cast<const uint4*>(s + c));
        }
#pragma unroll
        for (int u = 0; u < kVecPerLane; ++u) {
          const int64_t c = cb + (int64_t)u * 32 * 16;
          if (c < c_end) *reinterpret_cast<uint4*>(d + c) = v[u];
        }
      }
    } else {
      for (int64_t c = c_begin + lane; c < c_end; c += 32) d[c] = s[c];
    }
    if (tile == 0 && scale_bytes > 0)
      copy_scale_row(src_s + (int64_t)m * scale_bytes, dst_s + r * scale_bytes, scale_bytes, scale_mode, lane);
  }
}

cudaError_t launch_gather(const uint8_t* src, const uint8_t* src_scales, int64_t n_src,
                          int64_t row_bytes, int64_t scale_bytes, const int32_t* dst2src,
                          int64_t n_dst, const int32_t* n_dst_dev, uint8_t* dst,
                          uint8_t* dst_scales, cudaStream_t st) {
  const bool vec = (row_bytes % 16 == 0) && ((uintptr_t)src % 16 == 0) && ((uintptr_t)dst % 16 == 0);
  int scale_mode = 0;
  if (scale_bytes % 16 == 0 && (uintptr_t)src_scales % 16 == 0 && (uintptr_t)dst_scales % 16 == 0)
    scale_mode = 2;
  else if (scale_bytes % 4 == 0 && (uintptr_t)src_scales % 4 == 0 && (uintptr_t)dst_scales % 4 == 0)
    scale_mode = 1;
  // Column tiles per row: enough warps to fill the GPU when rows are few (a tile is at
  // least one pass of 32 lanes x 16 bytes), one tile per row when they are many.
  const int64_t sms = sm_count();
  const int64_t target_warps = sms * kGatherCtasPerSm * kGatherWarps;
  const int64_t max_tiles = cdiv(row_bytes, 32 * 16) > 0 ? cdiv(row_bytes, 32 * 16) : 1;
  int64_t wpr = cdiv(target_warps, n_dst > 0 ? n_dst : 1);
  if (wpr > max_tiles) wpr = max_tiles;
  if (wpr < 1) wpr = 1;
  int64_t tile_bytes = cdiv(cdiv(row_bytes, wpr), 16) * 16;
  wpr = cdiv(row_bytes, tile_bytes);
  const int64_t items = n_dst * wpr;
  int64_t blocks = cdiv(items, kGatherWarps);
  if (blocks > sms * kGatherCtasPerSm) blocks = sms * kGatherCtasPerSm;  // warps stride over the rest
  if (blocks < 1) blocks = 1;
  return launch_kernel(vec ? gather_kernel<true> : gather_kernel<false>, dim3((unsigned)blocks), dim3(kGatherThreads),
                       0, st, true, src, src_scales, n_src, row_bytes, scale_bytes, dst2src, n_dst, n_dst_dev, dst,
                       dst_scales, (int)wpr, tile_bytes, scale_mode);
}

FTMOE_DEFINE_ERR_READER(read_err_gather)

}  // namespace ftmoe

// Fused FP8 row + scale gather (SGLang "Gather the cutlass MoE activation and its scales
// in one launch", Modifications): one walk of dst2src writes both the row bytes and the
// row's scales; the CTA that owns column 0 of a row also carries its scale row. Bytes are
// copied, never decoded. Row bases are 64-bit. Tails are masked, so any row width and any
// scale-row width (e.g. k = 896, 7 scales) works.
//
// Grid: x = column tile of a row, y = destination row (grid-stride over rows). 16-byte
// vector loads/stores when the widths and pointers allow, otherwise byte copies.
#include "common.cuh"
#include "internal.h"

namespace ftmoe {

constexpr int kGatherThreads = 128;
constexpr int kChunks = 4;  // 16-byte loads per thread and row issued before any store

// The row's scales: copied by the CTA that owns column 0 of the row.
__device__ __forceinline__ void copy_scale_row(const uint8_t* ss, uint8_t* ds, int64_t scale_bytes, int scale_mode) {
  if (scale_mode == 2) {
    for (int64_t c = (int64_t)threadIdx.x * 16; c < scale_bytes; c += kGatherThreads * 16)
      *reinterpret_cast<uint4*>(ds + c) = *reinterpret_cast<const uint4*>(ss + c);
  } else if (scale_mode == 1) {
    for (int64_t c = (int64_t)threadIdx.x * 4; c < scale_bytes; c += kGatherThreads * 4)
      *reinterpret_cast<uint32_t*>(ds + c) = *reinterpret_cast<const uint32_t*>(ss + c);
  } else {
    for (int64_t c = threadIdx.x; c < scale_bytes; c += kGatherThreads) ds[c] = ss[c];
  }
}

// Each CTA copies one column tile of two destination rows per iteration (rows y and
// y + gridDim.y, grid-stride over pairs), issuing all of a thread's loads for both rows
// before its stores so that the latency of the source rows overlaps.
template <bool kVec>
__global__ void __launch_bounds__(kGatherThreads) gather_kernel(
    const uint8_t* __restrict__ src, const uint8_t* __restrict__ src_s, int64_t n_src,
    int64_t row_bytes, int64_t scale_bytes, const int32_t* __restrict__ map, int64_t n_dst,
    const int32_t* __restrict__ n_dst_dev, uint8_t* __restrict__ dst, uint8_t* __restrict__ dst_s,
    int64_t tile_bytes, int scale_mode /*0 bytes, 1 words, 2 vec16*/) {
  pdl_wait();  // the predecessor's outputs are complete from here on
  pdl_trigger();
  int64_t limit = n_dst;
  if (n_dst_dev != nullptr) {
    const int64_t d = *n_dst_dev;
    limit = d < limit ? d : limit;
  }
  const int64_t c_begin = (int64_t)blockIdx.x * tile_bytes;
  int64_t c_end = c_begin + tile_bytes;
  if (c_end > row_bytes) c_end = row_bytes;
  const int64_t stride = gridDim.y;
  for (int64_t r0 = blockIdx.y; r0 < limit; r0 += 2 * stride) {
    const int64_t r1 = r0 + stride;
    const int32_t m0 = map[r0];
    const int32_t m1 = r1 < limit ? map[r1] : -1;
    const bool ok0 = m0 >= 0 && (int64_t)m0 < n_src;
    const bool ok1 = r1 < limit && m1 >= 0 && (int64_t)m1 < n_src;
    if (blockIdx.x == 0 && threadIdx.x == 0 && (!ok0 || (r1 < limit && !ok1))) raise_error(FTMOE_ERR_MAP_RANGE);
    const uint8_t* s0 = src + (int64_t)(ok0 ? m0 : 0) * row_bytes;
    const uint8_t* s1 = src + (int64_t)(ok1 ? m1 : 0) * row_bytes;
    uint8_t* d0 = dst + r0 * row_bytes;
    uint8_t* d1 = dst + r1 * row_bytes;
    if (kVec) {
      for (int64_t cb = c_begin + (int64_t)threadIdx.x * 16; cb < c_end; cb += kGatherThreads * 16 * kChunks) {
        uint4 v0[kChunks], v1[kChunks];
#pragma unroll
        for (int u = 0; u < kChunks; ++u) {
          const int64_t c = cb + (int64_t)u * kGatherThreads * 16;
          if (c < c_end) {
            if (ok0) v0[u] = __ldg(reinterpret_cast<const uint4*>(s0 + c));
            if (ok1) v1[u] = __ldg(reinterpret_cast<const uint4*>(s1 + c));
          }
        }
#pragma unroll
        for (int u = 0; u < kChunks; ++u) {
          const int64_t c = cb + (int64_t)u * kGatherThreads * 16;
          if (c < c_end) {
            if (ok0) *reinterpret_cast<uint4*>(d0 + c) = v0[u];
            if (ok1) *reinterpret_cast<uint4*>(d1 + c) = v1[u];
          }
        }
      }
    } else {
      for (int64_t c = c_begin + threadIdx.x; c < c_end; c += kGatherThreads) {
        if (ok0) d0[c] = s0[c];
        if (ok1) d1[c] = s1[c];
      }
    }
    if (blockIdx.x == 0 && scale_bytes > 0) {
      if (ok0) copy_scale_row(src_s + (int64_t)m0 * scale_bytes, dst_s + r0 * scale_bytes, scale_bytes, scale_mode);
      if (ok1) copy_scale_row(src_s + (int64_t)m1 * scale_bytes, dst_s + r1 * scale_bytes, scale_bytes, scale_mode);
    }
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
  // Column tiles: enough CTAs to cover the SMs at small row counts, whole rows (up to
  // 8 KiB per CTA) at large ones.
  const int64_t min_tile = kGatherThreads * 16;  // 2 KiB
  int64_t tiles = cdiv(row_bytes, 4 * min_tile);
  const int64_t want = cdiv(2 * 152, n_dst > 1 ? cdiv(n_dst, 2) : 1);  // CTAs per row pair
  if (tiles < want) tiles = want;
  const int64_t max_tiles = cdiv(row_bytes, min_tile);
  if (tiles > max_tiles) tiles = max_tiles;
  if (tiles < 1) tiles = 1;
  int64_t tile_bytes = cdiv(row_bytes, tiles);
  tile_bytes = cdiv(tile_bytes, 16) * 16;
  tiles = cdiv(row_bytes, tile_bytes);
  if (tiles < 1) tiles = 1;
  const int64_t pairs = cdiv(n_dst, 2);  // two rows per CTA iteration
  const int64_t rows_grid = pairs < 65535 ? pairs : 65535;
  dim3 grid((unsigned)tiles, (unsigned)(rows_grid > 0 ? rows_grid : 1));
  return launch_kernel(vec ? gather_kernel<true> : gather_kernel<false>, grid, dim3(kGatherThreads), 0, st, true, src,
                       src_scales, n_src, row_bytes, scale_bytes, dst2src, n_dst, n_dst_dev, dst, dst_scales,
                       tile_bytes, scale_mode);
}

FTMOE_DEFINE_ERR_READER(read_err_gather)

}  // namespace ftmoe

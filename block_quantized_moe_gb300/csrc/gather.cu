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
  for (int64_t row = blockIdx.y; row < limit; row += gridDim.y) {
    const int32_t m = map[row];
    if (m < 0 || (int64_t)m >= n_src) {
      if (blockIdx.x == 0 && threadIdx.x == 0) raise_error(FTMOE_ERR_MAP_RANGE);
      continue;
    }
    const uint8_t* s_row = src + (int64_t)m * row_bytes;
    uint8_t* d_row = dst + row * row_bytes;
    if (kVec) {
      for (int64_t c = c_begin + (int64_t)threadIdx.x * 16; c < c_end; c += kGatherThreads * 16)
        *reinterpret_cast<uint4*>(d_row + c) = __ldg(reinterpret_cast<const uint4*>(s_row + c));
    } else {
      for (int64_t c = c_begin + threadIdx.x; c < c_end; c += kGatherThreads) d_row[c] = s_row[c];
    }
    if (blockIdx.x == 0 && scale_bytes > 0) {
      const uint8_t* ss = src_s + (int64_t)m * scale_bytes;
      uint8_t* ds = dst_s + row * scale_bytes;
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
  const int64_t want = cdiv(2 * 152, n_dst > 0 ? n_dst : 1);
  if (tiles < want) tiles = want;
  const int64_t max_tiles = cdiv(row_bytes, min_tile);
  if (tiles > max_tiles) tiles = max_tiles;
  if (tiles < 1) tiles = 1;
  int64_t tile_bytes = cdiv(row_bytes, tiles);
  tile_bytes = cdiv(tile_bytes, 16) * 16;
  tiles = cdiv(row_bytes, tile_bytes);
  if (tiles < 1) tiles = 1;
  const int64_t rows_grid = n_dst < 65535 ? n_dst : 65535;
  dim3 grid((unsigned)tiles, (unsigned)(rows_grid > 0 ? rows_grid : 1));
  return launch_kernel(vec ? gather_kernel<true> : gather_kernel<false>, grid, dim3(kGatherThreads), 0, st, true, src,
                       src_scales, n_src, row_bytes, scale_bytes, dst2src, n_dst, n_dst_dev, dst, dst_scales,
                       tile_bytes, scale_mode);
}

FTMOE_DEFINE_ERR_READER(read_err_gather)

}  // namespace ftmoe

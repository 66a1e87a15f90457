// FP8 activation quantization of one 1x128 group by one warp (each lane owns 4 consecutive
// columns), shared by the quantizer kernel and the forward's prep kernel so both run the
// same arithmetic: amax = max|x| over the group, s = amax / 448 (IEEE fp32),
// code = e4m3_rne_satfinite(x / s); amax = 0 gives s = 0 and all-zero codes (SGLang
// "Gather the cutlass MoE activation and its scales in one launch", Motivation).
#pragma once

#include "common.cuh"

namespace ftmoe {

template <bool kVec>
__device__ __forceinline__ void quantize_fp8_group(const uint16_t* __restrict__ x, int64_t k, int64_t ld_x,
                                                   uint8_t* __restrict__ q, float* __restrict__ s, int64_t ng,
                                                   int64_t row, int64_t g, int lane) {
  const int64_t c0 = g * kGroup + lane * 4;
  const uint16_t* xr = x + row * ld_x;
  float v[4];
  const bool full = c0 + 4 <= k;
  if (kVec && full) {
    const uint2 p = *reinterpret_cast<const uint2*>(xr + c0);
    v[0] = bf16_bits_to_f(p.x & 0xffffu);
    v[1] = bf16_bits_to_f(p.x >> 16);
    v[2] = bf16_bits_to_f(p.y & 0xffffu);
    v[3] = bf16_bits_to_f(p.y >> 16);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = (c0 + i < k) ? bf16_bits_to_f(xr[c0 + i]) : 0.0f;
  }
  float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
  amax = warp_max(amax);
  const float sc = div_rn(amax, kE4M3Max);
  uint32_t codes = 0;
  if (amax > 0.0f) {
    codes = (uint32_t)f2_to_e4m3x2(div_rn(v[0], sc), div_rn(v[1], sc)) |
            ((uint32_t)f2_to_e4m3x2(div_rn(v[2], sc), div_rn(v[3], sc)) << 16);
  }
  uint8_t* qr = q + row * k;
  if (kVec && full) {
    *reinterpret_cast<uint32_t*>(qr + c0) = codes;
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (c0 + i < k) qr[c0 + i] = (uint8_t)(codes >> (8 * i));
  }
  if (lane == 0) s[row * ng + g] = sc;
}

// whether the vector form of quantize_fp8_group may be used for these pointers and sizes
inline bool quantize_fp8_vec_ok(const void* x, int64_t ld_x, const void* q, int64_t k) {
  return ((uintptr_t)x % 8 == 0) && (ld_x % 4 == 0) && ((uintptr_t)q % 4 == 0) && (k % 4 == 0);
}

// The same quantization of one 1x128 group by one half-warp: lane hl (0..15) of the half owns
// 8 consecutive columns, loaded as one 16-byte vector. The load and the rest are separate
// steps so that a loop can put several groups' loads in flight before it finishes any (the
// one-warp form keeps 8 bytes per lane in flight, too few to cover the memory latency).
// Both halves of the warp must call quantize_fp8_hw_finish together (the maximum takes
// shuffles within each half); a half with no group passes live = false.
template <bool kVec>
__device__ __forceinline__ uint4 quantize_fp8_hw_load(const uint16_t* __restrict__ x, int64_t k, int64_t ld_x,
                                                      int64_t row, int64_t g, int hl, bool live) {
  // the lane's 8 bf16 values as raw bits (zero past the row's end)
  const int64_t c0 = g * kGroup + hl * 8;
  const uint16_t* xr = x + row * ld_x;
  if (kVec && live && c0 + 8 <= k) return *reinterpret_cast<const uint4*>(xr + c0);
  uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (live && c0 + i < k) w[i >> 1] |= (uint32_t)xr[c0 + i] << (16 * (i & 1));
  return make_uint4(w[0], w[1], w[2], w[3]);
}

template <bool kVec>
__device__ __forceinline__ void quantize_fp8_hw_finish(uint4 raw, int64_t k, uint8_t* __restrict__ q,
                                                       float* __restrict__ s, int64_t ng, int64_t row, int64_t g,
                                                       int hl, bool live) {
  const int64_t c0 = g * kGroup + hl * 8;
  float v[8];
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = bf16_bits_to_f(w[i] & 0xffffu);
    v[2 * i + 1] = bf16_bits_to_f(w[i] >> 16);
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float sc = div_rn(amax, kE4M3Max);
  uint32_t codes[2] = {0u, 0u};
  if (amax > 0.0f) {
    const SharedDivisor ds(sc);  // x / sc as IEEE division rounds it
#pragma unroll
    for (int h = 0; h < 2; ++h)
      codes[h] = (uint32_t)f2_to_e4m3x2(ds.div(v[4 * h]), ds.div(v[4 * h + 1])) |
                 ((uint32_t)f2_to_e4m3x2(ds.div(v[4 * h + 2]), ds.div(v[4 * h + 3])) << 16);
  }
  if (!live) return;
  uint8_t* qr = q + row * k;
  if (kVec && c0 + 8 <= k) {
    *reinterpret_cast<uint2*>(qr + c0) = make_uint2(codes[0], codes[1]);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (c0 + i < k) qr[c0 + i] = (uint8_t)(codes[i >> 2] >> (8 * (i & 3)));
  }
  if (hl == 0) s[row * ng + g] = sc;
}

// The (row, group) units [0, units) of rows x ng groups, by the warps gwarp, gwarp + nwarps,
// ...: each warp takes kHwBatch pairs of units per pass (one unit per half-warp in each), all
// their loads issued before any is finished. The loop bound is uniform over the warp.
constexpr int kHwBatch = 4;
template <bool kVec>
__device__ __forceinline__ void quantize_fp8_rows_hw(const uint16_t* __restrict__ x, int64_t k, int64_t ld_x,
                                                     uint8_t* __restrict__ q, float* __restrict__ s, int64_t ng,
                                                     int64_t units, int64_t gwarp, int64_t nwarps, int lane) {
  const int half = lane >> 4, hl = lane & 15;
  auto load_batch = [&](int64_t w0, uint4 (&raw)[kHwBatch]) {
#pragma unroll
    for (int b = 0; b < kHwBatch; ++b) {
      const int64_t unit = 2 * (w0 + b * nwarps) + half;
      const bool live = unit < units;
      const int64_t row = live ? unit / ng : 0, g = live ? unit - row * ng : 0;
      raw[b] = quantize_fp8_hw_load<kVec>(x, k, ld_x, row, g, hl, live);
    }
  };
  // software pipeline: the next batch's loads are in flight while this batch is finished
  uint4 cur[kHwBatch];
  if (2 * gwarp < units) load_batch(gwarp, cur);
  for (int64_t w0 = gwarp; 2 * w0 < units; w0 += kHwBatch * nwarps) {
    uint4 nxt[kHwBatch];
    const int64_t w1 = w0 + kHwBatch * nwarps;
    if (2 * w1 < units) load_batch(w1, nxt);
#pragma unroll
    for (int b = 0; b < kHwBatch; ++b) {
      const int64_t unit = 2 * (w0 + b * nwarps) + half;
      const bool live = unit < units;
      const int64_t row = live ? unit / ng : 0, g = live ? unit - row * ng : 0;
      quantize_fp8_hw_finish<kVec>(cur[b], k, q, s, ng, row, g, hl, live);
    }
#pragma unroll
    for (int b = 0; b < kHwBatch; ++b) cur[b] = nxt[b];
  }
}

// whether the vector forms of quantize_fp8_hw_load / _finish may be used
inline bool quantize_fp8_vec16_ok(const void* x, int64_t ld_x, const void* q, int64_t k) {
  return ((uintptr_t)x % 16 == 0) && (ld_x % 8 == 0) && ((uintptr_t)q % 8 == 0) && (k % 8 == 0);
}

}  // namespace ftmoe

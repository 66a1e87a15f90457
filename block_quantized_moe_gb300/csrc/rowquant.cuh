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

}  // namespace ftmoe

// MXFP8 quantization: e4m3 codes with one power-of-two scale (an E8M0 byte) per 32
// consecutive elements of a row.
//
// The SGLang gather page (Modifications) names the mxfp8 branch of the blockwise MoE: a
// ue8m0 scale per 32 elements, and a bf16 activation that is gathered first and quantized
// after the gather. The recipe is the OCP Microscaling one: for each block of 32,
//   shared = floor(log2(amax)) - 8   (8: the exponent of E4M3's largest power of two),
//            clamped to [-127, 127]; scale byte = shared + 127;
//   code   = e4m3_rne_satfinite(x * 2^-shared).
// floor(log2(amax)) is read off the fp32 exponent field (zero and subnormal amax give
// -127), and multiplying by a power of two is exact here, so every code follows from the
// inputs alone: the kernels and any other implementation of the recipe agree bit for bit.
//
// Four threads share a 32-element block (eight elements each, one 16- or 32-byte load);
// the block maximum takes two shuffles.
#include "common.cuh"
#include "internal.h"

namespace ftmoe {

namespace mx {

constexpr int kPer = 8;  // elements per thread

__device__ __forceinline__ int shared_exp(float amax) {
  const int ef = (int)((__float_as_uint(amax) >> 23) & 0xFF);
  if (ef == 0) return -127;  // zero or subnormal maximum
  const int s = ef - 127 - 8;
  return s < -127 ? -127 : s;  // ef <= 255 keeps s <= 120
}

// 2^-s as fp32 for s in [-127, 120]: exponent field 127 - s in [7, 254]
__device__ __forceinline__ float pow2_neg(int s) { return __uint_as_float((uint32_t)(127 - s) << 23); }

// The block maximum of |v| over the four threads of a block (lanes 4b .. 4b + 3), then the
// eight codes of this thread; returns the shared exponent.
__device__ __forceinline__ int quantize8(const float (&v)[kPer], uint2& codes) {
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < kPer; ++i) m = fmaxf(m, fabsf(v[i]));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
  m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
  const int s = shared_exp(m);
  const float f = pow2_neg(s);
  codes.x = (uint32_t)f2_to_e4m3x2(v[0] * f, v[1] * f) | ((uint32_t)f2_to_e4m3x2(v[2] * f, v[3] * f) << 16);
  codes.y = (uint32_t)f2_to_e4m3x2(v[4] * f, v[5] * f) | ((uint32_t)f2_to_e4m3x2(v[6] * f, v[7] * f) << 16);
  return s;
}

template <typename In>
__device__ __forceinline__ void load8(const In* p, bool vec, float (&v)[kPer]);

template <>
__device__ __forceinline__ void load8<uint16_t>(const uint16_t* p, bool vec, float (&v)[kPer]) {
  if (vec) {
    const uint4 r = *reinterpret_cast<const uint4*>(p);
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = bf16_bits_to_f((uint16_t)(w[i] & 0xFFFF));
      v[2 * i + 1] = bf16_bits_to_f((uint16_t)(w[i] >> 16));
    }
  } else {
#pragma unroll
    for (int i = 0; i < kPer; ++i) v[i] = bf16_bits_to_f(p[i]);
  }
}

template <>
__device__ __forceinline__ void load8<float>(const float* p, bool vec, float (&v)[kPer]) {
  if (vec) {
    const float4 a = *reinterpret_cast<const float4*>(p);
    const float4 b = *reinterpret_cast<const float4*>(p + 4);
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
  } else {
#pragma unroll
    for (int i = 0; i < kPer; ++i) v[i] = p[i];
  }
}

__device__ __forceinline__ void store8(uint8_t* q, uint2 codes, bool vec) {
  if (vec) {
    *reinterpret_cast<uint2*>(q) = codes;
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      q[i] = (uint8_t)(codes.x >> (8 * i));
      q[4 + i] = (uint8_t)(codes.y >> (8 * i));
    }
  }
}

// Rows of x (bf16 or fp32) -> codes q [rows][k] and scale bytes s [rows][k / 32]; with a
// map, destination row d reads source row map[d] (the gather of the bf16 activation), an
// entry outside [0, n_src) raises FTMOE_ERR_MAP_RANGE and leaves the row untouched.
// n_dev (optional): device count of destination rows to write. k % 32 == 0.
template <typename In>
__global__ void __launch_bounds__(256) quant_rows_kernel(const In* __restrict__ x, int64_t ld_x, int64_t k,
                                                         int64_t rows, const int32_t* __restrict__ map, int64_t n_src,
                                                         const int32_t* __restrict__ n_dev, uint8_t* __restrict__ q,
                                                         uint8_t* __restrict__ s, bool vec_in, bool vec_out) {
  pdl_wait();
  pdl_trigger();
  int64_t limit = rows;
  if (n_dev != nullptr) {
    const int64_t d = *n_dev;
    limit = d < limit ? d : limit;
  }
  const int64_t per_row = k / kPer;
  const int64_t total = limit * per_row;
  const int lane = threadIdx.x & 31;
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  // a warp's 32 units are 8 whole blocks (per_row is a multiple of 4); the loop bound is
  // uniform over the warp, so the shuffles always see all of it
  for (int64_t base = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) - lane; base < total; base += nthreads) {
    const int64_t unit = base + lane;
    const bool live = unit < total;
    int64_t row = 0, c = 0, src = 0;
    bool ok = live;
    if (live) {
      row = unit / per_row;
      c = unit - row * per_row;
      src = row;
      if (map != nullptr) {
        src = map[row];
        if (src < 0 || src >= n_src) {
          if ((c & 3) == 0) raise_error(FTMOE_ERR_MAP_RANGE);
          ok = false;
        }
      }
    }
    float v[kPer];
    if (ok) {
      load8<In>(x + src * ld_x + c * kPer, vec_in, v);
    } else {
#pragma unroll
      for (int i = 0; i < kPer; ++i) v[i] = 0.0f;
    }
    uint2 codes;
    const int sh = quantize8(v, codes);
    if (ok) {
      store8(q + row * k + c * kPer, codes, vec_out);
      if ((c & 3) == 0) s[row * (k / 32) + c / 4] = (uint8_t)(sh + 127);
    }
  }
}

// SiLU-and-mul of fp32 gate/up rows (g = columns [0, inter), u = [inter, 2 inter)), the
// same fp32 expression as the FP8 kernel, then MXFP8 quantization of the product.
__global__ void __launch_bounds__(256) silu_mul_kernel(const float* __restrict__ gu, int64_t rows, int64_t inter,
                                                       int64_t ld, const int32_t* __restrict__ rows_dev,
                                                       uint8_t* __restrict__ q, uint8_t* __restrict__ s, bool vec_in,
                                                       bool vec_out) {
  // as in the FP8 kernel: the next GEMM reads nothing of this kernel's predecessor before
  // its own wait, so it may start streaming weights now
  pdl_trigger();
  pdl_wait();
  int64_t limit = rows;
  if (rows_dev != nullptr) {
    const int64_t d = *rows_dev;
    limit = d < limit ? d : limit;
  }
  const int64_t per_row = inter / kPer;
  const int64_t total = limit * per_row;
  const int lane = threadIdx.x & 31;
  const int64_t nthreads = (int64_t)gridDim.x * blockDim.x;
  for (int64_t base = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) - lane; base < total; base += nthreads) {
    const int64_t unit = base + lane;
    const bool live = unit < total;
    const int64_t row = live ? unit / per_row : 0, c = live ? unit - row * per_row : 0;
    float v[kPer];
    if (live) {
      float g[kPer], u[kPer];
      load8<float>(gu + row * ld + c * kPer, vec_in, g);
      load8<float>(gu + row * ld + inter + c * kPer, vec_in, u);
#pragma unroll
      for (int i = 0; i < kPer; ++i) v[i] = silu_mul_1(g[i], u[i]);
    } else {
#pragma unroll
      for (int i = 0; i < kPer; ++i) v[i] = 0.0f;
    }
    uint2 codes;
    const int sh = quantize8(v, codes);
    if (live) {
      store8(q + row * inter + c * kPer, codes, vec_out);
      if ((c & 3) == 0) s[row * (inter / 32) + c / 4] = (uint8_t)(sh + 127);
    }
  }
}

static int grid_for(int64_t units) {
  int64_t b = (units + 255) / 256;
  const int64_t cap = 152 * 16;
  if (b > cap) b = cap;
  return (int)(b < 1 ? 1 : b);
}

static bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace mx

cudaError_t launch_mxfp8_quant_bf16(const uint16_t* x, int64_t rows, int64_t k, int64_t ld_x, const int32_t* map,
                                    int64_t n_src, const int32_t* n_dev, uint8_t* q, uint8_t* s, cudaStream_t st) {
  const bool vin = mx::aligned(x, 16) && ld_x % 8 == 0, vout = mx::aligned(q, 8);
  return launch_kernel(mx::quant_rows_kernel<uint16_t>, dim3(mx::grid_for(rows * (k / mx::kPer))), dim3(256), 0, st,
                       true, x, ld_x, k, rows, map, n_src, n_dev, q, s, vin, vout);
}

cudaError_t launch_mxfp8_quant_f32(const float* x, int64_t rows, int64_t k, int64_t ld_x, uint8_t* q, uint8_t* s,
                                   cudaStream_t st) {
  const bool vin = mx::aligned(x, 16) && ld_x % 4 == 0, vout = mx::aligned(q, 8);
  return launch_kernel(mx::quant_rows_kernel<float>, dim3(mx::grid_for(rows * (k / mx::kPer))), dim3(256), 0, st, false,
                       x, ld_x, k, rows, static_cast<const int32_t*>(nullptr), rows,
                       static_cast<const int32_t*>(nullptr), q, s, vin, vout);
}

cudaError_t launch_silu_mul_mxfp8(const float* gu, int64_t rows, int64_t inter, int64_t ld_gu, const int32_t* rows_dev,
                                  uint8_t* q, uint8_t* s, cudaStream_t st) {
  const bool vin = mx::aligned(gu, 16) && ld_gu % 4 == 0 && inter % 4 == 0, vout = mx::aligned(q, 8);
  return launch_kernel(mx::silu_mul_kernel, dim3(mx::grid_for(rows * (inter / mx::kPer))), dim3(256), 0, st, true, gu,
                       rows, inter, ld_gu, rows_dev, q, s, vin, vout);
}

FTMOE_DEFINE_ERR_READER(read_err_mxfp8)

}  // namespace ftmoe

// Device helpers shared by the libftmoe kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_fp4.h>
#include <stdint.h>

#include "../../include/ftmoe.h"

namespace ftmoe {

constexpr int kGroup = 128;        // activation group width = weight block edge
constexpr float kE4M3Max = 448.0f;
constexpr float kE2M1Max = 6.0f;
constexpr int kNvfp4Block = 16;
constexpr int kMxBlock = 32;    // elements per E8M0 scale (MXFP8)

// Each translation unit keeps its own device error word; the host reads all of them.
// An index read on the device that is out of range is skipped and reported here.
static __device__ unsigned int g_err_word;

__device__ __forceinline__ void raise_error(unsigned int bit) { atomicOr(&g_err_word, bit); }

// Programmatic dependent launch. Inside the fused forward a kernel may start while its
// predecessor is still running; it waits here before it reads anything the predecessor
// writes (or writes anything it reads), and only then lets its own dependent start. So when
// a kernel starts, every kernel two or more launches earlier has completed -- with one
// exception: the FP8 SiLU-and-mul kernel lets the down GEMM start first, and the down GEMM
// reads nothing the gate/up GEMM writes before its own wait. Outside such a launch both are
// no-ops.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

#define FTMOE_DEFINE_ERR_READER(fname)                                                \
  uint32_t fname() {                                                                  \
    unsigned int v = 0, zero = 0;                                                     \
    if (cudaMemcpyFromSymbol(&v, ftmoe::g_err_word, sizeof(v)) != cudaSuccess) return 0; \
    cudaMemcpyToSymbol(ftmoe::g_err_word, &zero, sizeof(zero));                       \
    return v;                                                                         \
  }

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Two floats -> two e4m3 codes (round to nearest even, saturate to +-448), packed with
// the first value in the low byte. Uses the cuda_fp8.h conversion.
__device__ __forceinline__ uint16_t f2_to_e4m3x2(float a, float b) {
  return (uint16_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ uint8_t f_to_e4m3(float a) {
  return (uint8_t)__nv_cvt_float_to_fp8(a, __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float e4m3_to_f(uint8_t c) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)c, __NV_E4M3);
  return __half2float(__half(h));
}

// Two floats -> two e2m1 codes in one byte (first value in the low nibble), round to
// nearest even with saturation to +-6 (cuda_fp4.h conversion).
__device__ __forceinline__ uint8_t f2_to_e2m1x2(float a, float b) {
  return (uint8_t)__nv_cvt_float2_to_fp4x2(make_float2(a, b), __NV_E2M1, cudaRoundNearest);
}

__device__ __forceinline__ float bf16_bits_to_f(uint16_t b) {
  return __uint_as_float(((uint32_t)b) << 16);
}

// IEEE single-precision quotient, round to nearest (the build never uses fast math; the
// explicit intrinsic documents that the quantization decision depends on it).
__device__ __forceinline__ float div_rn(float a, float b) { return __fdiv_rn(a, b); }

// Many dividends over one divisor d, each quotient rounded to nearest even exactly as IEEE
// division rounds it. Markstein's theorem (P. W. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Develop. 34(1), 1990): with
// y = RN(1/d), q0 = RN(x*y) and the residual r = x - q0*d (exact with a fused multiply-add),
// RN(q0 + r*y) is the correctly rounded x/d, as long as nothing leaves the normal range. The
// reciprocal takes one IEEE division per divisor instead of one per element. A divisor far
// from 1 (outside [2^-100, 2^100], or not finite) keeps the IEEE division per element, and an
// exact q0 (r = 0) is kept as it is, so that a zero quotient keeps its sign. Quotients so small
// that they are subnormal round to zero codes in every format here either way.
struct SharedDivisor {
  float d, y;
  bool fast;
  __device__ __forceinline__ explicit SharedDivisor(float d_) : d(d_) {
    const float ad = fabsf(d_);
    fast = ad >= 0x1p-100f && ad <= 0x1p100f;
    y = fast ? __fdiv_rn(1.0f, d_) : 0.0f;
  }
  __device__ __forceinline__ float div(float x) const {
    if (!fast) return __fdiv_rn(x, d);
    const float q0 = __fmul_rn(x, y);
    const float r = __fmaf_rn(-q0, d, x);
    return r == 0.0f ? q0 : __fmaf_rn(r, y, q0);
  }
};

// silu(g) * u in fp32, the one expression every SiLU-and-mul of the library evaluates (the
// separate kernel and the gate/up GEMM epilogue give bit-identical results).
__device__ __forceinline__ float silu_mul_1(float g, float u) { return g / (1.0f + expf(-g)) * u; }

// Output element types of the combine: bf16 and fp16 (one round to nearest even of the fp32
// sum) or fp32. The separate combine kernel and the down GEMM's fused combine both use these.
struct OutBf16 {
  using T = uint16_t;
  static __device__ __forceinline__ uint16_t cvt(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }
};
struct OutF16 {
  using T = uint16_t;
  static __device__ __forceinline__ uint16_t cvt(float v) { return __half_as_ushort(__float2half_rn(v)); }
};
struct OutF32 {
  using T = float;
  static __device__ __forceinline__ float cvt(float v) { return v; }
};

// four outputs of one row, one vector store (8-byte aligned for 16-bit outputs, 16-byte for fp32)
__device__ __forceinline__ void store4(uint16_t* o, const uint16_t* b) {
  *reinterpret_cast<uint2*>(o) = make_uint2((uint32_t)b[0] | ((uint32_t)b[1] << 16), (uint32_t)b[2] | ((uint32_t)b[3] << 16));
}
__device__ __forceinline__ void store4(float* o, const float* b) {
  *reinterpret_cast<float4*>(o) = make_float4(b[0], b[1], b[2], b[3]);
}

// Positive floats order like their bit patterns, so a max over |x| can use atomicMax on
// the bits of a zero-initialised word.
__device__ __forceinline__ void atomic_max_pos(float* addr, float v) {
  atomicMax(reinterpret_cast<unsigned int*>(addr), __float_as_uint(v));
}

}  // namespace ftmoe

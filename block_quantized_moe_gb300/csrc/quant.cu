// Activation and weight quantizers.
//
// FP8 (SGLang "Gather the cutlass MoE activation and its scales in one launch",
// Motivation; FreeToken "perf(moe): skip inactive block-fp8 decode routes"): one fp32
// scale per 1x128 activation group and per 128x128 weight block, s = amax / 448 in IEEE
// fp32, code = e4m3_rne_satfinite(x / s), amax = 0 -> s = 0 and all-zero codes.
// NVFP4: fp32 tensor scale g = amax / (448 * 6), e4m3 block scale per 16 elements
// sb = e4m3(amax_block / (6 g)), code = e2m1_rne(x / (sb * g)).
#include "common.cuh"
#include "internal.h"
#include "rowquant.cuh"

namespace ftmoe {

// One warp per (row, 128-group); each lane owns 4 consecutive columns.
template <bool kVec>
__global__ void __launch_bounds__(256) quantize_act_fp8_kernel(
    const uint16_t* __restrict__ x, int64_t rows, int64_t k, int64_t ld_x,
    uint8_t* __restrict__ q, float* __restrict__ s, int64_t ng) {
  pdl_wait();  // the predecessor's outputs are complete from here on
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  quantize_fp8_rows_hw<kVec>(x, k, ld_x, q, s, ng, rows * ng,
                             (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5), nwarps, lane);
}

static int grid_for(int64_t work_items, int per_block) {
  int64_t b = cdiv(work_items, per_block);
  const int64_t cap = 152 * 32;  // grid-stride beyond this
  if (b > cap) b = cap;
  return (int)(b < 1 ? 1 : b);
}

cudaError_t launch_quantize_act_fp8(const uint16_t* x, int64_t rows, int64_t k, int64_t ld_x,
                                    uint8_t* q, float* scales, cudaStream_t st) {
  const int64_t ng = cdiv(k, kGroup);
  const bool vec = quantize_fp8_vec16_ok(x, ld_x, q, k);
  // (at most four resident CTAs per SM: each warp then runs several batches, the next one's
  // loads in flight while it finishes the current one)
  int grid = grid_for(rows * ng, 16 * kHwBatch);
  if (grid > 152 * 4) grid = 152 * 4;
  return launch_kernel(vec ? quantize_act_fp8_kernel<true> : quantize_act_fp8_kernel<false>, dim3(grid), dim3(256), 0,
                       st, true, x, rows, k, ld_x, q, scales, ng);
}

// ---------------------------------------------------------------------------------
// NVFP4 activation: (1) tensor amax, (2) per-16 block quantization, (3) amax -> g.
// ---------------------------------------------------------------------------------

template <typename T>
__device__ __forceinline__ float load_as_f(const T* p);
template <>
__device__ __forceinline__ float load_as_f<uint16_t>(const uint16_t* p) { return bf16_bits_to_f(*p); }
template <>
__device__ __forceinline__ float load_as_f<float>(const float* p) { return *p; }

// amax of |x| over rows x k (row stride ld) into *amax_bits (zeroed beforehand).
template <typename T>
__global__ void __launch_bounds__(256) tensor_amax_kernel(const T* __restrict__ x, int64_t rows,
                                                          int64_t k, int64_t ld,
                                                          int64_t matrix_stride,
                                                          float* __restrict__ amax_out) {
  pdl_wait();  // the predecessor's outputs are complete from here on
  pdl_trigger();
  // blockIdx.y selects a matrix (experts of a weight bank); one amax word per matrix
  const T* xm = x + (int64_t)blockIdx.y * matrix_stride;
  float m = 0.0f;
  const int64_t total = rows * k;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / k, c = i - r * k;
    m = fmaxf(m, fabsf(load_as_f<T>(xm + r * ld + c)));
  }
  m = warp_max(m);
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
    m = warp_max(m);
    if (threadIdx.x == 0 && m > 0.0f) atomic_max_pos(amax_out + blockIdx.y, m);
  }
}

// One thread per 16-element block. amax_in holds the tensor amax (per matrix).
template <typename T>
__global__ void __launch_bounds__(256) quantize_nvfp4_kernel(
    const T* __restrict__ x, int64_t rows, int64_t k, int64_t ld, int64_t matrix_stride,
    const float* __restrict__ amax_in, uint8_t* __restrict__ q, uint8_t* __restrict__ sb) {
  pdl_wait();  // the predecessor's outputs are complete from here on
  pdl_trigger();
  const int64_t nblk = k / kNvfp4Block;
  const int64_t mat = blockIdx.y;
  const T* xm = x + mat * matrix_stride;
  uint8_t* qm = q + mat * rows * (k / 2);
  uint8_t* sm = sb + mat * rows * nblk;
  const float g = div_rn(amax_in[mat], kE4M3Max * kE2M1Max);
  const float six_g = kE2M1Max * g;
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < rows * nblk;
       b += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = b / nblk, c0 = (b - r * nblk) * kNvfp4Block;
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = load_as_f<T>(xm + r * ld + c0 + i);
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(v[i]));
    uint8_t code_s = 0;
    float eff = 0.0f;
    if (g > 0.0f) {
      code_s = f_to_e4m3(div_rn(am, six_g));
      eff = e4m3_to_f(code_s) * g;
    }
    uint32_t lo = 0, hi = 0;
    if (eff != 0.0f) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        lo |= (uint32_t)f2_to_e2m1x2(div_rn(v[2 * i], eff), div_rn(v[2 * i + 1], eff)) << (8 * i);
        hi |= (uint32_t)f2_to_e2m1x2(div_rn(v[8 + 2 * i], eff), div_rn(v[8 + 2 * i + 1], eff)) << (8 * i);
      }
    }
    *reinterpret_cast<uint2*>(qm + r * (k / 2) + c0 / 2) = make_uint2(lo, hi);
    sm[r * nblk + c0 / kNvfp4Block] = code_s;
  }
}

__global__ void amax_to_global_scale_kernel(float* g, int n) {
  pdl_wait();  // the predecessor's outputs are complete from here on
  pdl_trigger();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) g[i] = div_rn(g[i], kE4M3Max * kE2M1Max);
}

cudaError_t launch_quantize_act_nvfp4(const uint16_t* x, int64_t rows, int64_t k, int64_t ld_x,
                                      uint8_t* q, uint8_t* scales, float* gscale,
                                      cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(gscale, 0, sizeof(float), st);
  if (e != cudaSuccess) return e;
  // the first kernel follows the memset, which takes part in no overlap
  e = launch_kernel(tensor_amax_kernel<uint16_t>, dim3(grid_for(rows * k, 256 * 8), 1), dim3(256), 0, st, false, x,
                    rows, k, ld_x, 0, gscale);
  if (e != cudaSuccess) return e;
  e = launch_kernel(quantize_nvfp4_kernel<uint16_t>, dim3(grid_for(rows * k / kNvfp4Block, 256), 1), dim3(256), 0,
                    st, true, x, rows, k, ld_x, 0, gscale, q, scales);
  return launch_kernel(amax_to_global_scale_kernel, dim3(1), dim3(32), 0, st, true, gscale, 1);
}

// ---------------------------------------------------------------------------------
// FP8 weight bank: one CTA per 128x128 block.
// ---------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) quantize_weights_fp8_kernel(
    const float* __restrict__ w, int64_t n, int64_t k, uint8_t* __restrict__ q,
    float* __restrict__ s, int64_t nb, int64_t kb) {
  const int64_t e = blockIdx.z, bn = blockIdx.y, bk = blockIdx.x;
  const float* we = w + e * n * k;
  uint8_t* qe = q + e * n * k;
  const int64_t r0 = bn * kGroup, c0 = bk * kGroup;
  const int tid = threadIdx.x;
  const int col = c0 + (tid & 127);      // one column per thread, 2 rows per step
  const int rsub = tid >> 7;              // 0 or 1
  float m = 0.0f;
  for (int i = rsub; i < kGroup; i += 2) {
    const int64_t r = r0 + i;
    if (r < n && col < k) m = fmaxf(m, fabsf(we[r * k + col]));
  }
  m = warp_max(m);
  __shared__ float red[8];
  __shared__ float sc_sh;
  if ((tid & 31) == 0) red[tid >> 5] = m;
  __syncthreads();
  if (tid == 0) {
    float a = red[0];
    for (int i = 1; i < 8; ++i) a = fmaxf(a, red[i]);
    sc_sh = div_rn(a, kE4M3Max);
    s[(e * nb + bn) * kb + bk] = sc_sh;
  }
  __syncthreads();
  const float sc = sc_sh;
  for (int i = rsub; i < kGroup; i += 2) {
    const int64_t r = r0 + i;
    if (r < n && col < k) {
      const float v = we[r * k + col];
      qe[r * k + col] = sc > 0.0f ? f_to_e4m3(div_rn(v, sc)) : (uint8_t)0;
    }
  }
}

cudaError_t launch_quantize_weights_fp8(const float* w, int32_t E, int64_t n, int64_t k,
                                        uint8_t* q, float* scales, cudaStream_t st) {
  const int64_t nb = cdiv(n, kGroup), kb = cdiv(k, kGroup);
  if (nb > 65535 || E > 65535) return cudaErrorInvalidValue;
  quantize_weights_fp8_kernel<<<dim3((unsigned)kb, (unsigned)nb, (unsigned)E), 256, 0, st>>>(
      w, n, k, q, scales, nb, kb);
  return cudaGetLastError();
}

cudaError_t launch_quantize_weights_nvfp4(const float* w, int32_t E, int64_t n, int64_t k,
                                          uint8_t* q, uint8_t* scales, float* gscale,
                                          cudaStream_t st) {
  if (E > 65535) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(gscale, 0, sizeof(float) * E, st);
  if (e != cudaSuccess) return e;
  tensor_amax_kernel<float><<<dim3(grid_for(n * k, 256 * 16) / 4 + 1, E), 256, 0, st>>>(
      w, n, k, k, n * k, gscale);
  quantize_nvfp4_kernel<float><<<dim3(grid_for(n * k / kNvfp4Block, 256) / 4 + 1, E), 256, 0, st>>>(
      w, n, k, k, n * k, gscale, q, scales);
  amax_to_global_scale_kernel<<<(unsigned)cdiv(E, 256), 256, 0, st>>>(gscale, E);
  return cudaGetLastError();
}

FTMOE_DEFINE_ERR_READER(read_err_quant)

}  // namespace ftmoe

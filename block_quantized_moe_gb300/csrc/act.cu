// SiLU-and-mul with re-quantization, and the routing-weighted top-k combine.
//
// The FreeToken decode page ("perf(moe): skip inactive block-fp8 decode routes") has the
// activation and the reduction read the whole gate/up and down buffers, including the
// zero tiles of inactive routes; zero rows here give scale 0 and zero codes, and the
// combine skips inactive slots without reading their routing weight.
#include "common.cuh"
#include "internal.h"

namespace ftmoe {

// One half-warp per (row, 128 outputs); a lane owns 8 consecutive outputs, so a warp keeps
// two groups' gate and up loads (four 16-byte loads a lane) in flight before any arithmetic.
template <bool kVec>
__global__ void __launch_bounds__(256) silu_mul_fp8_kernel(
    const float* __restrict__ gu, int64_t rows, int64_t inter, int64_t ld,
    const int32_t* __restrict__ rows_dev, uint8_t* __restrict__ q, float* __restrict__ s,
    int64_t ng) {
  // The down GEMM that follows reads nothing before its own wait that the gate/up GEMM
  // writes (only the segment offsets, complete long before), so it may start -- and begin
  // streaming its weights -- while this kernel still waits for the gate/up GEMM to finish.
  pdl_trigger();
  pdl_wait();  // the predecessor's outputs are complete from here on
  int64_t limit = rows;
  if (rows_dev != nullptr) {
    const int64_t d = *rows_dev;
    limit = d < limit ? d : limit;
  }
  const int lane = threadIdx.x & 31, hl = lane & 15;
  const int64_t units = limit * ng;  // (row, group) pairs
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  // the loop bound is uniform over the warp, so every shuffle sees all 32 lanes
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); 2 * w < units; w += nwarps) {
    const int64_t unit = 2 * w + (lane >> 4);
    const bool live = unit < units;
    const int64_t row = live ? unit / ng : 0, g = live ? unit - row * ng : 0;
    const int64_t c0 = g * kGroup + hl * 8;
    const float* gr = gu + row * ld;
    float a[8];
    const bool full = live && c0 + 8 <= inter;
    if (kVec && full) {
      const float4 g0 = *reinterpret_cast<const float4*>(gr + c0);
      const float4 g1 = *reinterpret_cast<const float4*>(gr + c0 + 4);
      const float4 u0 = *reinterpret_cast<const float4*>(gr + inter + c0);
      const float4 u1 = *reinterpret_cast<const float4*>(gr + inter + c0 + 4);
      a[0] = silu_mul_1(g0.x, u0.x);
      a[1] = silu_mul_1(g0.y, u0.y);
      a[2] = silu_mul_1(g0.z, u0.z);
      a[3] = silu_mul_1(g0.w, u0.w);
      a[4] = silu_mul_1(g1.x, u1.x);
      a[5] = silu_mul_1(g1.y, u1.y);
      a[6] = silu_mul_1(g1.z, u1.z);
      a[7] = silu_mul_1(g1.w, u1.w);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i)
        a[i] = (live && c0 + i < inter) ? silu_mul_1(gr[c0 + i], gr[inter + c0 + i]) : 0.0f;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(a[i]));
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sc = div_rn(amax, kE4M3Max);
    uint32_t codes[2] = {0u, 0u};
    if (amax > 0.0f) {
      const SharedDivisor ds(sc);  // a / sc as IEEE division rounds it
#pragma unroll
      for (int h = 0; h < 2; ++h)
        codes[h] = (uint32_t)f2_to_e4m3x2(ds.div(a[4 * h]), ds.div(a[4 * h + 1])) |
                   ((uint32_t)f2_to_e4m3x2(ds.div(a[4 * h + 2]), ds.div(a[4 * h + 3])) << 16);
    }
    if (live) {
      uint8_t* qr = q + row * inter;
      if (kVec && full) {
        *reinterpret_cast<uint32_t*>(qr + c0) = codes[0];
        *reinterpret_cast<uint32_t*>(qr + c0 + 4) = codes[1];
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (c0 + i < inter) qr[c0 + i] = (uint8_t)(codes[i >> 2] >> (8 * (i & 3)));
      }
      if (hl == 0) s[row * ng + g] = sc;
    }
  }
}

static int grid_cap(int64_t blocks) {
  const int64_t cap = 152 * 32;
  if (blocks > cap) blocks = cap;
  return (int)(blocks < 1 ? 1 : blocks);
}

cudaError_t launch_silu_mul_fp8(const float* gu, int64_t rows, int64_t inter, int64_t ld_gu,
                                const int32_t* rows_dev, uint8_t* q, float* scales,
                                cudaStream_t st) {
  const int64_t ng = cdiv(inter, kGroup);
  const bool vec = (ld_gu % 4 == 0) && (inter % 4 == 0) && ((uintptr_t)gu % 16 == 0) &&
                   ((uintptr_t)q % 4 == 0);
  const int grid = grid_cap(cdiv(rows * ng, 16));
  return launch_kernel(vec ? silu_mul_fp8_kernel<true> : silu_mul_fp8_kernel<false>, dim3(grid), dim3(256), 0, st,
                       true, gu, rows, inter, ld_gu, rows_dev, q, scales, ng);
}

// ---- NVFP4: pass 1 amax of a over the valid rows, pass 2 quantize, pass 3 amax -> g ----
__global__ void __launch_bounds__(256) silu_amax_kernel(const float* __restrict__ gu, int64_t rows,
                                                        int64_t inter, int64_t ld,
                                                        const int32_t* __restrict__ rows_dev,
                                                        float* __restrict__ amax_out) {
  pdl_wait();  // the predecessor's outputs are complete from here on
  pdl_trigger();
  int64_t limit = rows;
  if (rows_dev != nullptr) {
    const int64_t d = *rows_dev;
    limit = d < limit ? d : limit;
  }
  float m = 0.0f;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < limit * inter;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / inter, c = i - r * inter;
    m = fmaxf(m, fabsf(silu_mul_1(gu[r * ld + c], gu[r * ld + inter + c])));
  }
  m = warp_max(m);
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    m = threadIdx.x < 8 ? red[threadIdx.x] : 0.0f;
    m = warp_max(m);
    if (threadIdx.x == 0 && m > 0.0f) atomic_max_pos(amax_out, m);
  }
}

__global__ void __launch_bounds__(256) silu_quant_nvfp4_kernel(
    const float* __restrict__ gu, int64_t rows, int64_t inter, int64_t ld,
    const int32_t* __restrict__ rows_dev, const float* __restrict__ amax_in,
    uint8_t* __restrict__ q, uint8_t* __restrict__ sb) {
  pdl_wait();  // the predecessor's outputs are complete from here on
  pdl_trigger();
  int64_t limit = rows;
  if (rows_dev != nullptr) {
    const int64_t d = *rows_dev;
    limit = d < limit ? d : limit;
  }
  const int64_t nblk = inter / kNvfp4Block;
  const float g = div_rn(amax_in[0], kE4M3Max * kE2M1Max);
  const float six_g = kE2M1Max * g;
  for (int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; b < limit * nblk;
       b += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = b / nblk, c0 = (b - r * nblk) * kNvfp4Block;
    float v[16];
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      v[i] = silu_mul_1(gu[r * ld + c0 + i], gu[r * ld + inter + c0 + i]);
      am = fmaxf(am, fabsf(v[i]));
    }
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
    *reinterpret_cast<uint2*>(q + r * (inter / 2) + c0 / 2) = make_uint2(lo, hi);
    sb[r * nblk + c0 / kNvfp4Block] = code_s;
  }
}

__global__ void amax_to_gscale_1(float* g) {
  pdl_wait();
  pdl_trigger();
  g[0] = div_rn(g[0], kE4M3Max * kE2M1Max);
}

cudaError_t launch_silu_mul_nvfp4(const float* gu, int64_t rows, int64_t inter, int64_t ld_gu,
                                  const int32_t* rows_dev, uint8_t* q, uint8_t* scales,
                                  float* gscale, cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(gscale, 0, sizeof(float), st);
  if (e != cudaSuccess) return e;
  // the first kernel follows the memset, which takes part in no overlap
  e = launch_kernel(silu_amax_kernel, dim3(grid_cap(cdiv(rows * inter, 256 * 8))), dim3(256), 0, st, false, gu, rows,
                    inter, ld_gu, rows_dev, gscale);
  if (e != cudaSuccess) return e;
  e = launch_kernel(silu_quant_nvfp4_kernel, dim3(grid_cap(cdiv(rows * inter / kNvfp4Block, 256))), dim3(256), 0, st,
                    true, gu, rows, inter, ld_gu, rows_dev, gscale, q, scales);
  if (e != cudaSuccess) return e;
  return launch_kernel(amax_to_gscale_1, dim3(1), dim3(1), 0, st, true, gscale);
}

// ---- combine: out[t, h] = round( sum_j w[t,j] * y[row(t,j), h] ), active j ascending ----
// (output conversions OutBf16 / OutF16 / OutF32 and store4: common.cuh)
// The slot ids, weights and rows of a token are loaded six slots at a time with
// independent loads, then accumulated in ascending slot order.
template <bool kVec, typename Out>
__global__ void __launch_bounds__(128) combine_kernel(
    const float* __restrict__ y, int64_t ld_y, const int32_t* __restrict__ route2dst,
    const int32_t* __restrict__ ids, const float* __restrict__ w, int64_t tokens, int32_t topk,
    int64_t hidden, typename Out::T* __restrict__ out, int64_t ld_out) {
  pdl_wait();  // the predecessor's outputs are complete from here on
  pdl_trigger();
  const int64_t t = blockIdx.y;
  // eight outputs per thread, two runs of four: every slot's two row loads are in flight
  // together, and a slot's row index is loaded beside its id (the id only decides whether
  // the weight and the row are read)
  const int64_t h0 = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (h0 >= hidden) return;
  float acc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
  for (int j0 = 0; j0 < topk; j0 += 6) {
    constexpr int kS = 6;  // slots per batch
    int idv[kS];
    int64_t dst[kS];
#pragma unroll
    for (int u = 0; u < kS; ++u) {
      const int j = j0 + u;
      const int64_t r = t * topk + j;
      idv[u] = j < topk ? ids[r] : -1;
      dst[u] = (j < topk && route2dst != nullptr) ? (int64_t)route2dst[r] : r;
    }
    int64_t row[kS];
    float wt[kS];
#pragma unroll
    for (int u = 0; u < kS; ++u) {
      row[u] = -1;
      wt[u] = 0.0f;
      if (idv[u] >= 0) {  // inactive: neither the weight nor the row is read
        wt[u] = w[t * topk + j0 + u];
        row[u] = dst[u];
      }
    }
    float4 v[kS][2];
#pragma unroll
    for (int u = 0; u < kS; ++u) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        v[u][h] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        const int64_t c = h0 + 4 * h;
        if (row[u] >= 0 && c < hidden) {
          const float* yr = y + row[u] * ld_y + c;
          if (kVec && c + 4 <= hidden) {
            v[u][h] = *reinterpret_cast<const float4*>(yr);
          } else {
            v[u][h].x = yr[0];
            if (c + 1 < hidden) v[u][h].y = yr[1];
            if (c + 2 < hidden) v[u][h].z = yr[2];
            if (c + 3 < hidden) v[u][h].w = yr[3];
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kS; ++u) {
      if (row[u] >= 0) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          acc[h][0] = fmaf(wt[u], v[u][h].x, acc[h][0]);
          acc[h][1] = fmaf(wt[u], v[u][h].y, acc[h][1]);
          acc[h][2] = fmaf(wt[u], v[u][h].z, acc[h][2]);
          acc[h][3] = fmaf(wt[u], v[u][h].w, acc[h][3]);
        }
      }
    }
  }
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int64_t c = h0 + 4 * h;
    if (c >= hidden) break;
    typename Out::T b[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) b[i] = Out::cvt(acc[h][i]);
    typename Out::T* o = out + t * ld_out + c;
    if (kVec && c + 4 <= hidden) {
      store4(o, b);
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (c + i < hidden) o[i] = b[i];
    }
  }
}

template <typename Out>
static cudaError_t launch_combine_t(const float* y, int64_t ld_y, const int32_t* route2dst, const int32_t* ids,
                                   const float* w, int64_t tokens, int32_t topk, int64_t hidden,
                                   typename Out::T* out, int64_t ld_out, cudaStream_t st) {
  if (tokens > 65535) {
    // one launch per 65535-token slab keeps grid.y in range
    for (int64_t t0 = 0; t0 < tokens; t0 += 65535) {
      const int64_t tn = tokens - t0 < 65535 ? tokens - t0 : 65535;
      cudaError_t e = launch_combine_t<Out>(y, ld_y, route2dst ? route2dst + t0 * topk : nullptr, ids + t0 * topk,
                                            w + t0 * topk, tn, topk, hidden, out + t0 * ld_out, ld_out, st);
      if (e != cudaSuccess) return e;
      if (route2dst == nullptr) y += tn * topk * ld_y;
    }
    return cudaSuccess;
  }
  constexpr int kOutBytes = (int)sizeof(typename Out::T);
  const bool vec = (hidden % 4 == 0) && (ld_y % 4 == 0) && ((uintptr_t)y % 16 == 0) && (ld_out % 4 == 0) &&
                   ((uintptr_t)out % (4 * kOutBytes) == 0);
  dim3 grid((unsigned)cdiv(hidden, 8 * 128), (unsigned)tokens);
  return launch_kernel(vec ? combine_kernel<true, Out> : combine_kernel<false, Out>, grid, dim3(128), 0, st, true, y,
                       ld_y, route2dst, ids, w, tokens, topk, hidden, out, ld_out);
}

cudaError_t launch_combine(const float* y, int64_t ld_y, const int32_t* route2dst,
                           const int32_t* ids, const float* w, int64_t tokens, int32_t topk,
                           int64_t hidden, int32_t out_dtype, void* out, int64_t ld_out, cudaStream_t st) {
  switch (out_dtype) {
    case FTMOE_OUT_BF16:
      return launch_combine_t<OutBf16>(y, ld_y, route2dst, ids, w, tokens, topk, hidden,
                                       static_cast<uint16_t*>(out), ld_out, st);
    case FTMOE_OUT_FP16:
      return launch_combine_t<OutF16>(y, ld_y, route2dst, ids, w, tokens, topk, hidden,
                                      static_cast<uint16_t*>(out), ld_out, st);
    case FTMOE_OUT_FP32:
      return launch_combine_t<OutF32>(y, ld_y, route2dst, ids, w, tokens, topk, hidden, static_cast<float*>(out),
                                      ld_out, st);
    default:
      return cudaErrorInvalidValue;
  }
}

FTMOE_DEFINE_ERR_READER(read_err_act)

}  // namespace ftmoe

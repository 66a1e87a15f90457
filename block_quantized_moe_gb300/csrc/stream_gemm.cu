// HBM-streaming block-FP8 GEMM on CUDA cores, for decode batches (1-8 tokens).
//
// The FreeToken page "perf(moe): skip inactive block-fp8 decode routes" describes one
// shared decode kernel serving both the gate/up and the down GEMM, launched with fixed
// shapes, in which a negative expert slot writes a zero output tile and returns before
// reading activations, weights, scales or routing weights. This kernel keeps that
// contract and streams each active expert's weight rows once:
//
// * grid.x tiles the weight rows (kNT per CTA); grid.y is the route (SLOTS) or the
//   expert (GROUPED). Launch shapes depend only on (n, routes or E).
// * SLOTS: the CTA of the first route of an expert (in route order) is its leader and
//   computes that expert for every route that selected it, so each expert's weights
//   cross HBM once per step; later routes of the same expert exit at once.
// * Each warp owns weight rows; lanes read 16 consecutive bytes (coalesced 512 B per
//   warp load), convert e4m3 -> fp32 and multiply against the activation rows staged
//   in shared memory as fp32 values already multiplied by their 1x128 scales. Each
//   16-byte slice lies inside one 128-wide K block, so the lane applies that block's
//   weight scale before the cross-lane (warp shuffle) reduction. No MMA tile, so no
//   padding rows are ever computed.
#include "common.cuh"
#include "internal.h"

namespace ftmoe {

constexpr int kNT = 32;       // weight rows per CTA
constexpr int kSWarps = 8;
constexpr int kKC = 1024;     // K chunk of the activations staged in shared memory
constexpr int kMaxM = 8;      // activation rows per pass

template <bool kVec>
__global__ void __launch_bounds__(kSWarps * 32) stream_gemm_kernel(StreamGemmArgs a) {
  __shared__ __align__(16) float xs[kMaxM][kKC];
  __shared__ float acc[kNT][kMaxM];
  __shared__ int64_t arow[kMaxM], orow[kMaxM];
  __shared__ int s_nm, s_scan, s_done;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t n0 = (int64_t)blockIdx.x * kNT;
  const int64_t N = a.n, K = a.k;
  const int64_t kb_count = (K + kGroup - 1) / kGroup;
  const int64_t nb_count = (N + kGroup - 1) / kGroup;

  int e;
  int64_t seg_begin = 0, seg_end = 0;
  if (a.grouped) {
    e = blockIdx.y;
    // device-side offsets are clamped to the buffers, so bad offsets cannot reach
    // memory outside them
    seg_begin = a.offsets[e];
    seg_end = a.offsets[e + 1];
    if (seg_begin < 0) seg_begin = 0;
    if (seg_end > a.a_rows) seg_end = a.a_rows;
    if (seg_end <= seg_begin) return;
  } else {
    const int64_t r = blockIdx.y;
    e = a.slots[r];
    if (e < 0 || e >= a.E) {
      // inactive route: exact-zero output tile, nothing else of the route is read
      if (e >= a.E && tid == 0 && blockIdx.x == 0) raise_error(FTMOE_ERR_EXPERT_ID_RANGE);
      for (int i = tid; i < kNT; i += blockDim.x)
        if (n0 + i < N) a.out[r * a.ld_out + n0 + i] = 0.0f;
      return;
    }
    // leader test: an earlier route with the same expert does the work
    int earlier = 0;
    for (int64_t r2 = tid; r2 < r; r2 += blockDim.x) earlier |= (a.slots[r2] == e);
    if (__syncthreads_or(earlier)) return;
  }

  const uint8_t* wq = a.w_q + (int64_t)e * N * K;
  const float* ws = a.w_s + (int64_t)e * nb_count * kb_count;
  if (tid == 0) {
    s_scan = a.grouped ? 0 : (int)blockIdx.y;
    s_done = 0;
  }
  __syncthreads();

  while (true) {
    // ---- next batch of up to kMaxM member rows ----
    if (tid == 0) {
      int nm = 0;
      if (a.grouped) {
        int64_t i = seg_begin + s_scan;
        for (; nm < kMaxM && i < seg_end; ++i, ++nm) { arow[nm] = i; orow[nm] = i; }
        s_scan = (int)(i - seg_begin);
        s_done = (i >= seg_end);
      } else {
        int64_t r2 = s_scan;
        for (; nm < kMaxM && r2 < a.routes; ++r2) {
          if (a.slots[r2] == e) {
            arow[nm] = r2 / a.act_div;
            orow[nm] = r2;
            ++nm;
          }
        }
        s_scan = (int)r2;
        s_done = (r2 >= a.routes);
      }
      s_nm = nm;
    }
    __syncthreads();
    // read the batch bookkeeping now: thread 0 rewrites it once every thread has passed
    // the barrier at the end of this batch
    const int nm = s_nm;
    const int done = s_done;
    if (nm == 0) break;
    for (int i = tid; i < kNT * kMaxM; i += blockDim.x) (&acc[0][0])[i] = 0.0f;

    for (int64_t kc0 = 0; kc0 < K; kc0 += kKC) {
      const int kc_len = (int)((K - kc0) < kKC ? (K - kc0) : kKC);
      __syncthreads();
      // stage the dequantized activation chunk: xs[m][c] = code * scale
      for (int i = tid; i < kMaxM * kKC; i += blockDim.x) {
        const int m = i / kKC, c = i - m * kKC;
        float v = 0.0f;
        if (m < nm && c < kc_len) {
          const int64_t col = kc0 + c;
          v = e4m3_to_f(a.a_q[arow[m] * K + col]) * a.a_s[arow[m] * kb_count + col / kGroup];
        }
        xs[m][c] = v;
      }
      __syncthreads();
      for (int rr = warp; rr < kNT; rr += kSWarps) {
        const int64_t n = n0 + rr;
        if (n >= N) break;
        const uint8_t* wrow = wq + n * K + kc0;
        const float* wsrow = ws + (n / kGroup) * kb_count + kc0 / kGroup;
        float p[kMaxM];
#pragma unroll
        for (int m = 0; m < kMaxM; ++m) p[m] = 0.0f;
        for (int c = lane * 16; c < kc_len; c += 32 * 16) {
          uint32_t wv[4];
          if (kVec && c + 16 <= kc_len) {
            const uint4 t = __ldg(reinterpret_cast<const uint4*>(wrow + c));
            wv[0] = t.x; wv[1] = t.y; wv[2] = t.z; wv[3] = t.w;
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t word = 0;
#pragma unroll
              for (int b = 0; b < 4; ++b) {
                const int cc = c + 4 * j + b;
                if (cc < kc_len) word |= (uint32_t)wrow[cc] << (8 * b);
              }
              wv[j] = word;
            }
          }
          float wf[16];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 lo = e4m3x2_to_f2((uint16_t)(wv[j] & 0xffffu));
            const float2 hi = e4m3x2_to_f2((uint16_t)(wv[j] >> 16));
            wf[4 * j + 0] = lo.x; wf[4 * j + 1] = lo.y;
            wf[4 * j + 2] = hi.x; wf[4 * j + 3] = hi.y;
          }
          const float sw = wsrow[c / kGroup];
#pragma unroll
          for (int m = 0; m < kMaxM; ++m) {
            if (m < nm) {
              const float4* xv = reinterpret_cast<const float4*>(&xs[m][c]);
              float d = 0.0f;
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float4 x4 = xv[j];
                d = fmaf(wf[4 * j + 0], x4.x, d);
                d = fmaf(wf[4 * j + 1], x4.y, d);
                d = fmaf(wf[4 * j + 2], x4.z, d);
                d = fmaf(wf[4 * j + 3], x4.w, d);
              }
              p[m] = fmaf(sw, d, p[m]);
            }
          }
        }
#pragma unroll
        for (int m = 0; m < kMaxM; ++m) {
          if (m < nm) {
            const float v = warp_sum(p[m]);
            if (lane == 0) acc[rr][m] += v;
          }
        }
      }
    }
    __syncthreads();
    for (int i = tid; i < kNT * nm; i += blockDim.x) {
      const int m = i / kNT, rr = i - m * kNT;
      if (n0 + rr < N) a.out[orow[m] * a.ld_out + n0 + rr] = acc[rr][m];
    }
    __syncthreads();
    if (done) break;
  }
}

cudaError_t launch_stream_gemm(const StreamGemmArgs& a, cudaStream_t st) {
  const int64_t tiles = cdiv(a.n, kNT);
  const int64_t ys = a.grouped ? a.E : a.routes;
  if (ys <= 0 || tiles <= 0) return cudaSuccess;
  if (ys > 65535 || tiles > 0x7fffffff) return cudaErrorInvalidValue;
  const bool vec = (a.k % 16 == 0) && ((uintptr_t)a.w_q % 16 == 0);
  dim3 grid((unsigned)tiles, (unsigned)ys);
  if (vec)
    stream_gemm_kernel<true><<<grid, kSWarps * 32, 0, st>>>(a);
  else
    stream_gemm_kernel<false><<<grid, kSWarps * 32, 0, st>>>(a);
  return cudaGetLastError();
}

FTMOE_DEFINE_ERR_READER(read_err_stream_gemm)

}  // namespace ftmoe

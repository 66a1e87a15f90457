// HBM-streaming block-FP8 GEMM on CUDA cores, for decode batches (1-8 tokens).
//
// The FreeToken page "perf(moe): skip inactive block-fp8 decode routes" describes one
// shared decode kernel serving both the gate/up and the down GEMM, launched with fixed
// shapes, in which a negative expert slot writes a zero output tile and returns before
// reading activations, weights, scales or routing weights. This kernel keeps that
// contract and streams each active expert's weight rows from HBM once per call:
//
// * Work items are (expert, 64-row weight tile). In route-slot mode the expert of an
//   item is that of a "leader" route -- the first route (in route order) that selected
//   it -- and the item computes the tile for every route that selected the expert, so a
//   weight tile crosses HBM once. In grouped mode the expert's rows are a segment of the
//   activation buffer. Rows of routes with a negative slot are written as zeros first and
//   nothing else of those routes is read.
// * Persistent CTAs (two per SM). Warp 0 is a TMA producer keeping a ring of 64-row x
//   128-byte weight tiles (one 128-wide K block each, 128-byte swizzle) in flight; the
//   eight other warps consume it. Consumer thread (g, l) owns rows g and g+32 of the tile
//   and the 16-byte lane l of each K block (conflict-free reads through the swizzle).
//   e4m3 codes become fp16 exactly (one conversion per two values); the member
//   activation codes are staged once per expert in shared memory as fp16 too, and the
//   products run as fp16 x fp16 -> fp32 fused multiply-adds (exact products, fp32
//   accumulation) -- the fp16 -> fp32 conversion that would otherwise bound the kernel is
//   never executed. Each 16-byte slice lies in one K block, so the lane scales its
//   partial dot product by weight_scale * act_scale of that block and accumulates in
//   registers over all of K; one warp-shuffle reduction over the eight K lanes per tile.
// * No MMA tile, so no padding rows are computed. Every pipeline wait is bounded.
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace ftmoe {

namespace st {

constexpr int kRows = 64;          // weight rows per item
constexpr int kConsumers = 256;    // 32 row groups x 8 K lanes
constexpr int kThreads = kConsumers + 32;
constexpr int kMaxStages = 16;
constexpr int kTile = kRows * kGroup;  // 8 KiB per stage
constexpr size_t kCtaSmem = 110 * 1024;  // per-CTA budget that keeps two CTAs on an SM
constexpr int kMaxList = 1024;     // leaders (slot mode) or experts (grouped mode) per launch
constexpr int kMaxMembers = 8;     // activation rows staged per pass (upper bound)
constexpr size_t kStageBudget = 64 * 1024;  // bytes of staged activation codes (fp16) per CTA
constexpr int kMaxKB = 64;         // K blocks of a staged row (K <= 8192)

struct Params {
  const uint8_t* a_q;   // [rows][k]
  const float* a_s;     // [rows][kb]
  const float* w_s;     // [E][nb][kb]
  float* out;
  int64_t ld_out;
  int64_t a_rows;
  int64_t kp;           // K rounded up to 128: pitch of a staged activation row (fp16 codes)
  int n, k, E, KB, NB, n_tiles, mb, stages;
  int grouped;
  const int32_t* offsets;  // grouped: offsets of experts e0 .. e0+E (E+1 entries)
  int e0;                  // grouped: first expert of this launch
  const int32_t* slots;    // slots: [routes]
  int routes;
  int act_div;
};

// 16 e4m3 codes -> 8 packed f16x2 (exact: every e4m3 value is an fp16 value).
__device__ __forceinline__ void e4m3x16_to_h2(const uint4 w, uint32_t* h) {
  const uint32_t v[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const uint16_t lo = (uint16_t)(v[j] & 0xffffu), hi = (uint16_t)(v[j] >> 16);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h[2 * j]) : "h"(lo));
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h[2 * j + 1]) : "h"(hi));
  }
}

// a_lo += w.lo * x.lo; a_hi += w.hi * x.hi with fp16 operands and fp32 accumulation
// (products of two e4m3 values are exact in fp32).
__device__ __forceinline__ void fma_h2(float& a_lo, float& a_hi, uint32_t w2, uint32_t x2) {
  asm("{\n .reg .f16 wl, wh, xl, xh;\n mov.b32 {wl, wh}, %2;\n mov.b32 {xl, xh}, %3;\n"
      " fma.rn.f32.f16 %0, wl, xl, %0;\n fma.rn.f32.f16 %1, wh, xh, %1;\n}"
      : "+f"(a_lo), "+f"(a_hi)
      : "r"(w2), "r"(x2));
}

// Dot product of 16 weight values (8 f16x2) with the staged activation codes of the same
// 16 K positions. Staged codes are permuted inside each 128-wide K block so that the
// eight K lanes of a row group read one contiguous 128-byte line per instruction:
// halves [8*jj, 8*jj+8) of lane l's 16 sit at 64*jj + 8*l (fp16 units).
__device__ __forceinline__ float dot16h(const uint32_t* w, const __half* xl /* block base + 8*l */) {
  const uint4 x0 = *reinterpret_cast<const uint4*>(xl);
  const uint4 x1 = *reinterpret_cast<const uint4*>(xl + 64);
  float a = 0.0f, b = 0.0f, c = 0.0f, d = 0.0f;
  fma_h2(a, b, w[0], x0.x);
  fma_h2(c, d, w[1], x0.y);
  fma_h2(a, b, w[2], x0.z);
  fma_h2(c, d, w[3], x0.w);
  fma_h2(a, b, w[4], x1.x);
  fma_h2(c, d, w[5], x1.y);
  fma_h2(a, b, w[6], x1.z);
  fma_h2(c, d, w[7], x1.w);
  return (a + b) + (c + d);
}

// Expert and member range of list entry j. Slot mode: members are the routes from the
// leader on that selected the same expert; grouped mode: the rows of the segment.
struct Item {
  int e;
  int64_t first, end;
};

__device__ __forceinline__ Item item_of(const Params& p, const int* list, int j) {
  Item it;
  if (p.grouped) {
    it.e = list[j];
    int64_t lo = p.offsets[it.e - p.e0], hi = p.offsets[it.e - p.e0 + 1];
    if (lo < 0) lo = 0;
    if (hi > p.a_rows) hi = p.a_rows;
    it.first = lo;
    it.end = hi > lo ? hi : lo;
  } else {
    it.first = list[j];
    it.e = p.slots[it.first];
    it.end = p.routes;
  }
  return it;
}

__device__ __forceinline__ int member_count(const Params& p, const Item& it) {
  if (p.grouped) return (int)(it.end - it.first);
  int m = 0;
  for (int64_t r = it.first; r < p.routes; ++r) m += (p.slots[r] == it.e);
  return m;
}

__global__ void __launch_bounds__(kThreads) stream_gemm_kernel(const __grid_constant__ CUtensorMap map_w, Params p) {
  pdl_wait();  // the predecessor's outputs are complete from here on
  pdl_trigger();
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int kStages = p.stages;
  __half* xs = reinterpret_cast<__half*>(ring + kStages * kTile);  // [mb][kp] activation codes
  int* list = reinterpret_cast<int*>(xs + (size_t)p.mb * p.kp);    // [kMaxList]
  float* wsc = reinterpret_cast<float*>(list + kMaxList);           // [kMaxKB] weight scales of the tile
  float* asc = wsc + kMaxKB;                                        // [mb][kMaxKB] activation scales
  uint64_t* full = reinterpret_cast<uint64_t*>(asc + kMaxMembers * kMaxKB);
  uint64_t* empty = full + kStages;
  __shared__ int s_count;
  __shared__ volatile int s_abort;
  __shared__ int64_t s_arow[kMaxMembers], s_orow[kMaxMembers];
  __shared__ int s_nm, s_more;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t N = p.n, K = p.k;
  const int count_limit = p.grouped ? p.E : p.routes;

  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), kConsumers / 32);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // ---- zero rows of inactive routes (slot mode): written first, nothing else is read ----
  if (!p.grouped) {
    const int64_t total = (int64_t)p.routes * N;
    for (int64_t i = (int64_t)blockIdx.x * kThreads + tid; i < total; i += (int64_t)gridDim.x * kThreads) {
      const int64_t r = i / N, n = i - r * N;
      const int e = p.slots[r];
      if (e < 0 || e >= p.E) {
        p.out[r * p.ld_out + n] = 0.0f;
        if (e >= p.E && n == 0) raise_error(FTMOE_ERR_EXPERT_ID_RANGE);
      }
    }
  }
  // ---- the work list, in the same deterministic order in every CTA ----
  if (warp == 0) {
    int cnt = 0;
    for (int base = 0; base < count_limit; base += 32) {
      const int idx = base + lane;
      bool take = false;
      if (idx < count_limit) {
        if (p.grouped) {
          int64_t lo = p.offsets[idx], hi = p.offsets[idx + 1];
          if (lo < 0) lo = 0;
          if (hi > p.a_rows) hi = p.a_rows;
          take = hi > lo;
        } else {
          const int e = p.slots[idx];
          take = e >= 0 && e < p.E;
          for (int r2 = 0; take && r2 < idx; ++r2) take = (p.slots[r2] != e);
        }
      }
      const unsigned m = __ballot_sync(0xffffffffu, take);
      const int pos = cnt + __popc(m & ((1u << lane) - 1));
      if (take && pos < kMaxList) list[pos] = p.grouped ? idx + p.e0 : idx;
      cnt += __popc(m);
    }
    if (lane == 0) s_count = cnt < kMaxList ? cnt : kMaxList;
  }
  __syncthreads();
  const int n_items = s_count * p.n_tiles;
  // each CTA takes a contiguous range of items, so consecutive items mostly share an
  // expert and its staged activations
  const int i_begin = (int)(((int64_t)blockIdx.x * n_items) / gridDim.x);
  const int i_end = (int)(((int64_t)(blockIdx.x + 1) * n_items) / gridDim.x);

  if (warp == 0) {
    // ------------------------------- TMA producer -------------------------------
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first();  // the weight stream is read once
      uint32_t it = 0;
      bool ok = true;
      for (int i = i_begin; i < i_end && ok && !s_abort; ++i) {
        const Item itm = item_of(p, list, i / p.n_tiles);
        const int n0 = (i % p.n_tiles) * kRows;
        const int passes = (member_count(p, itm) + p.mb - 1) / p.mb;
        for (int pass = 0; pass < passes && ok; ++pass) {
          for (int kb = 0; kb < p.KB; ++kb, ++it) {
            const int s = it % kStages;
            if (!mbar_wait(smem_u32(&empty[s]), ((it / kStages) & 1) ^ 1, &s_abort)) { ok = false; break; }
            const uint32_t fb = smem_u32(&full[s]);
            mbar_expect_tx(fb, kTile);
            if (passes == 1)
              tma_load_3d_hint(smem_u32(ring + s * kTile), &map_w, fb, kb * kGroup, n0, itm.e, pol_w);
            else  // the tile is read again by the next pass
              tma_load_3d(smem_u32(ring + s * kTile), &map_w, fb, kb * kGroup, n0, itm.e);
          }
        }
      }
      // wait (bounded) for loads still in flight before the CTA may exit
      for (uint32_t s = 0; s < (uint32_t)kStages && s < it; ++s) {
        const uint32_t last = it - 1 - ((it - 1 - s) % kStages);
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&full[s]), (last / kStages) & 1) && globaltimer() - t0 < kTimeoutNs) {
        }
      }
    }
  } else {
    // --------------------------------- consumers ---------------------------------
    // Consumers leave their loops only through barriers whose outcome is uniform over all
    // consumer warps (bar.red.or on the abort flag, or the shared batch size), so no warp
    // can be left waiting at a named barrier.
    const int ct = tid - 32;
    const int rg = ct >> 3, kl = ct & 7;
    const uint32_t sw_chunk = (uint32_t)((kl ^ (rg & 7)) << 4);  // 128-byte swizzle (same for rg+32)
    uint32_t it = 0;
    bool aborted = false;
    int staged_j = -1;  // list entry whose members xs holds (single-pass items only)
    for (int i = i_begin; i < i_end && !aborted; ++i) {
      if (named_bar_or(1, kConsumers, s_abort)) break;
      const int j = i / p.n_tiles;
      const Item itm = item_of(p, list, j);
      const int64_t n0 = (int64_t)(i % p.n_tiles) * kRows;
      const int64_t row0 = n0 + rg, row1 = n0 + rg + 32;
      const float* wsr = p.w_s + ((int64_t)itm.e * p.NB + n0 / kGroup) * p.KB;
      for (int q = ct; q < p.KB; q += kConsumers) wsc[q] = wsr[q];
      int64_t scan = itm.first;  // meaningful in consumer thread 0 only
      int pass = 0;
      while (true) {
        if (ct == 0) {
          int nm = 0;
          if (p.grouped) {
            for (; nm < p.mb && scan < itm.end; ++scan, ++nm) { s_arow[nm] = scan; s_orow[nm] = scan; }
          } else {
            for (; nm < p.mb && scan < p.routes; ++scan) {
              if (p.slots[scan] == itm.e) {
                s_arow[nm] = scan / p.act_div;
                s_orow[nm] = scan;
                ++nm;
              }
            }
          }
          s_nm = nm;
          s_more = p.grouped ? (scan < itm.end) : (scan < p.routes);
        }
        named_bar(1, kConsumers);
        const int nm = s_nm;
        if (nm == 0) break;  // same value in every consumer thread
        // a single-pass item whose members are already staged keeps them
        const bool single = (pass == 0) && !s_more;
        if (!(single && staged_j == j)) {
          const int chunks = (int)(p.kp / 16);
          for (int q = ct; q < nm * chunks; q += kConsumers) {
            const int m = q / chunks, c16 = q - m * chunks;
            const int64_t c = (int64_t)c16 * 16;
            uint32_t h[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            if (c < K) e4m3x16_to_h2(__ldg(reinterpret_cast<const uint4*>(p.a_q + s_arow[m] * K + c)), h);
            // permuted position of lane l's halves [8*jj, 8*jj+8): kb*128 + 64*jj + 8*l
            const int64_t kb = c / kGroup;
            const int l = (int)((c % kGroup) / 16);
            __half* dst = xs + m * p.kp + kb * kGroup + 8 * l;
            *reinterpret_cast<uint4*>(dst) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(dst + 64) = make_uint4(h[4], h[5], h[6], h[7]);
          }
          for (int q = ct; q < nm * p.KB; q += kConsumers) {
            const int m = q / p.KB, kb = q - m * p.KB;
            asc[m * kMaxKB + kb] = p.a_s[s_arow[m] * p.KB + kb];
          }
          staged_j = single ? j : -1;
        }
        named_bar(1, kConsumers);
        float acc0[kMaxMembers], acc1[kMaxMembers];
#pragma unroll
        for (int m = 0; m < kMaxMembers; ++m) acc0[m] = acc1[m] = 0.0f;
        bool ok = true;
        for (int kb = 0; kb < p.KB; ++kb, ++it) {
          const int s = it % kStages;
          const int got = mbar_wait(smem_u32(&full[s]), (it / kStages) & 1, &s_abort) ? 1 : 0;
          if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
          const uint8_t* tile = ring + s * kTile;
          const uint4 wa = *reinterpret_cast<const uint4*>(tile + rg * kGroup + sw_chunk);
          const uint4 wb = *reinterpret_cast<const uint4*>(tile + (rg + 32) * kGroup + sw_chunk);
          uint32_t ha[8], hb[8];
          e4m3x16_to_h2(wa, ha);
          e4m3x16_to_h2(wb, hb);
          // release the slot only after the warp has consumed what it read from it (the
          // producer's next TMA write may otherwise land before a pending shared load)
          __syncwarp();
          if (lane == 0) mbar_arrive_after(smem_u32(&empty[s]), __uint_as_float(ha[0]), __uint_as_float(hb[0]));
          const int64_t off = (int64_t)kb * kGroup + 16 * kl;
          if (off >= K) continue;
          const float sw = wsc[kb];
          const __half* xl = xs + (int64_t)kb * kGroup + 8 * kl;
#pragma unroll
          for (int m = 0; m < kMaxMembers; ++m) {
            if (m < nm) {
              const float f = sw * asc[m * kMaxKB + kb];
              acc0[m] = fmaf(f, dot16h(ha, xl + m * p.kp), acc0[m]);
              acc1[m] = fmaf(f, dot16h(hb, xl + m * p.kp), acc1[m]);
            }
          }
        }
        if (ok) {
#pragma unroll
          for (int m = 0; m < kMaxMembers; ++m) {
#pragma unroll
            for (int o = 1; o < 8; o <<= 1) {
              acc0[m] += __shfl_xor_sync(0xffffffffu, acc0[m], o);
              acc1[m] += __shfl_xor_sync(0xffffffffu, acc1[m], o);
            }
          }
          if (kl == 0) {
#pragma unroll
            for (int m = 0; m < kMaxMembers; ++m) {
              if (m < nm) {
                if (row0 < N) p.out[s_orow[m] * p.ld_out + row0] = acc0[m];
                if (row1 < N) p.out[s_orow[m] * p.ld_out + row1] = acc1[m];
              }
            }
          }
        }
        ++pass;
        // orders this batch's reads of the staged rows and scales before they are rewritten
        if (named_bar_or(1, kConsumers, s_abort)) { aborted = true; break; }
      }
    }
  }
  __syncthreads();
}

}  // namespace st

static cudaError_t launch_part(const StreamGemmArgs& a, const CUtensorMap& map, int E, int e0,
                               const int32_t* offsets, const int32_t* slots, int routes, cudaStream_t stream) {
  st::Params p;
  p.a_q = a.a_q;
  p.a_s = a.a_s;
  p.w_s = a.w_s;
  p.out = a.out;
  p.ld_out = a.ld_out;
  p.a_rows = a.a_rows;
  p.kp = cdiv(a.k, kGroup) * kGroup;
  p.n = (int)a.n;
  p.k = (int)a.k;
  p.E = E;
  p.KB = (int)cdiv(a.k, kGroup);
  p.NB = (int)cdiv(a.n, kGroup);
  p.n_tiles = (int)cdiv(a.n, st::kRows);
  p.grouped = a.grouped;
  p.offsets = offsets;
  p.e0 = e0;
  p.slots = slots;
  p.routes = routes;
  p.act_div = a.act_div;
  // members staged per pass: no more than one route per token can pick an expert in slot
  // mode, so small batches stage fewer rows and leave the shared memory to the ring
  // members staged per pass. In slot mode an expert has at most one route per token (with
  // distinct ids per token), and with top-k routing over many experts more than four
  // tokens rarely share one; those rare experts take a second pass over L2-resident
  // weights, and the shared memory goes to the weight ring instead.
  int mb = st::kMaxMembers;
  if (!a.grouped) {
    const int64_t toks = a.topk > 0 ? routes / a.topk : routes;
    mb = (int)(toks < 4 ? (toks > 0 ? toks : 1) : 4);
  }
  while (mb > 1 && (size_t)mb * p.kp * 2 > st::kStageBudget) mb >>= 1;
  p.mb = mb;
  const size_t fixed = 1024 + (size_t)mb * p.kp * 2 + st::kMaxList * 4 + st::kMaxKB * 4 +
                       st::kMaxMembers * st::kMaxKB * 4;
  int stages = st::kMaxStages;
  while (stages > 2 && fixed + (size_t)stages * (st::kTile + 16) > st::kCtaSmem) --stages;
  p.stages = stages;
  const size_t smem = fixed + (size_t)stages * st::kTile + 2 * stages * 8;
  const int64_t max_items = (int64_t)(a.grouped ? E : (routes < a.E ? routes : a.E)) * p.n_tiles;
  int64_t grid = 2 * (int64_t)sm_count();
  if (grid > max_items) grid = max_items;
  if (!a.grouped && grid < 8) grid = 8;  // the zero rows of inactive routes
  if (grid < 1) grid = 1;
  int dev = 0;
  cudaGetDevice(&dev);
  static size_t granted[64] = {};  // per device: the largest limit set so far
  if (dev < 0 || dev >= 64 || smem > granted[dev]) {
    cudaError_t e = cudaFuncSetAttribute(st::stream_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) granted[dev] = smem;
  }
  return launch_kernel(st::stream_gemm_kernel, dim3((unsigned)grid), dim3(st::kThreads), smem, stream, true, map, p);
}

cudaError_t launch_stream_gemm(const StreamGemmArgs& a, cudaStream_t stream) {
  if (a.n <= 0 || a.k <= 0) return cudaSuccess;
  // TMA needs 16-byte aligned rows; a staged activation row must fit the staging budget
  if (a.k % 16 != 0 || (uintptr_t)a.w_q % 16 != 0 || (uintptr_t)a.a_q % 16 != 0 || a.n > (1 << 30) ||
      (size_t)cdiv(a.k, kGroup) * kGroup * 2 > st::kStageBudget || cdiv(a.k, kGroup) > st::kMaxKB)
    return cudaErrorInvalidValue;
  CUtensorMap map;
  const uint64_t dims[3] = {(uint64_t)a.k, (uint64_t)a.n, (uint64_t)a.E};
  const uint64_t strides[2] = {(uint64_t)a.k, (uint64_t)a.k * (uint64_t)a.n};
  const uint32_t box[3] = {(uint32_t)kGroup, (uint32_t)st::kRows, 1};
  if (!encode_u8_tmap(&map, a.w_q, 3, dims, strides, box)) return cudaErrorInvalidValue;
  if (a.grouped) {
    for (int e0 = 0; e0 < a.E; e0 += st::kMaxList) {
      const int En = a.E - e0 < st::kMaxList ? a.E - e0 : st::kMaxList;
      cudaError_t e = launch_part(a, map, En, e0, a.offsets + e0, nullptr, 0, stream);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
  // route-slot mode: one launch per chunk of whole tokens, at most kMaxList routes
  const int64_t topk = a.topk > 0 ? a.topk : 1;
  const int64_t chunk = (st::kMaxList / topk) * topk;
  if (chunk <= 0) return cudaErrorInvalidValue;
  for (int64_t r0 = 0; r0 < a.routes; r0 += chunk) {
    const int64_t rn = a.routes - r0 < chunk ? a.routes - r0 : chunk;
    StreamGemmArgs b = a;
    b.out = a.out + r0 * a.ld_out;
    // activation rows: token rows (gate/up) move by whole tokens, route rows by routes
    b.a_q = a.a_q + (r0 / a.act_div) * a.k;
    b.a_s = a.a_s + (r0 / a.act_div) * cdiv(a.k, kGroup);
    b.a_rows = a.a_rows - r0 / a.act_div;
    cudaError_t e = launch_part(b, map, a.E, 0, nullptr, a.slots + r0, (int)rn, stream);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

FTMOE_DEFINE_ERR_READER(read_err_stream_gemm)

}  // namespace ftmoe

// Fused decode forward for a few tokens (T <= 8): gate/up GEMM, SiLU-and-mul with FP8
// re-quantization, down GEMM and the routing-weighted combine in ONE persistent tcgen05
// kernel, after a small prep launch that quantizes the token rows.
//
// The FreeToken decode page ("perf(moe): skip inactive block-fp8 decode routes") runs one
// shared block-FP8 decode kernel for gate/up and for down, with the activation and the
// reduction as launches of their own, under CUDA graphs; at batch 1 its table scales with
// the active routes. At a few tokens the weights are the whole cost (each active expert's
// gate/up and down matrices cross HBM once) and launch gaps dominate what is left, so here
// the whole FFN after quantization is one launch whose work is spread evenly over the SMs:
//
//   * Tables. Every CTA derives the same tables from expert_ids: the distinct active
//     experts in ascending order (slot s), the tokens of each (one row per (token, expert),
//     in the slot of the token's first listing of the expert), and the distinct active
//     experts of each token. An inactive route (negative slot) appears in none of them: no
//     weight, activation, scale or routing weight of it is ever read.
//   * Gate/up, split evenly ("stream-K"). The 128-row weight blocks of all active experts
//     (gate block j and up block j adjacent) are cut into a fixed number of chunks of whole
//     TMA stages (chosen from the shape alone), and CTA c takes chunks [c * KU / G,
//     (c + 1) * KU / G) of the KU chunks. Each chunk is promoted per K block like the grouped
//     GEMM (act_scale x weight_scale on CUDA cores), from zero, and stored as fp32 partial
//     sums of the 8 token columns. The last CTA to arrive for a (gate block j, up block j)
//     pair -- a counter per pair -- adds the chunks of each block in K order, forms
//     silu(g) * u for the expert's routes, re-quantizes each route's 1x128 group to FP8 with
//     its scale amax / 448, and counts the pair done for the expert. Since the chunking and
//     the order of the sums depend on the shape only, a route's result does not depend on
//     which other experts the batch activates or on how the chunks fell to the CTAs.
//   * Down, whole blocks. CTA c takes a contiguous range of the (expert, 128-row block of
//     H) blocks. The weights stream as soon as the ring has room; the B operand (the
//     expert's intermediate rows, written by other CTAs) is staged by a loader warp once the
//     expert's pairs are all done (a bounded wait on the expert's counter).
//   * Combine. Each down block writes its routes' fp32 rows of y and counts them per
//     (token, block of H); the last arrival for a token reduces that token's active routes
//     in ascending slot order (fp32, from zero) and writes the output elements.
//
// The results differ from the separate kernels only in the order of the fp32 sums of a
// gate/up element (chunks are added after they are formed); the SiLU, quantization, down
// GEMM and combine arithmetic is the same expression.
//
// Roles: warp 0 TMA producer, warp 1 MMA issuer (and TMEM owner), warp 2 B loader for the
// down blocks, warp 3 scale-product tables (one item ahead), warps 4-7 promotion (warp w
// reads TMEM lanes 32 (w % 4) ..), warps 8-11 finishers (counters, pair finishing, combine),
// fed through a queue of mbarriers so that no wait on another CTA stalls the weight stream.
// MMA: tcgen05.mma kind::f8f6f4, M = 128 weight rows, N = 16 token (or route) columns,
// K = 32, four per 128-wide K block into a fresh TMEM accumulator; 16 accumulators rotate.
// Every wait is bounded: on timeout the kernel raises FTMOE_ERR_WAIT_TIMEOUT, stops all
// roles, lets its own TMA loads and MMAs drain, frees TMEM and returns.
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"
#include "rowquant.cuh"

namespace ftmoe {

namespace dk {

constexpr int kBM = 128;            // weight rows per block (MMA M)
constexpr int kBK = 128;            // K bytes per K block (one scale block)
constexpr int kN = 16;              // MMA N: token columns (gate/up) or route columns (down)
constexpr int kMaxRoutes = kDecodeMaxRoutes;
constexpr int kMaxRowsPerExpert = 16;
constexpr int kAcc = 16;            // TMEM accumulators of kN columns in rotation
constexpr int kTmemCols = kAcc * kN;
constexpr int kThreads = 384;
constexpr int kScaleWarp = 3;       // builds each item's scale-product table ahead of use
constexpr int kEpiWarp0 = 4;        // warps 4-7: promotion (one TMEM lane quarter each)
constexpr int kEpiThreads = 128;
constexpr int kFinWarp0 = 8;        // warps 8-11: counters, pair finishing, combine
constexpr int kFinThreads = 128;
constexpr int kQueue = 4;           // items the promoters may run ahead of the finishers
constexpr int kPartCols = kDecodeMaxTokens;  // partial sums keep the token columns
constexpr int kSubW = kBM * kBK;    // 16 KiB: one K block of one weight block
constexpr int kSubX = kN * kBK;     // 2 KiB: one K block of 16 token rows
constexpr int kMaxStages = 8;
constexpr int kFinBar = 2;          // named barrier of the finisher warpgroup

__device__ __forceinline__ uint32_t idesc_f8_n16() {
  return (1u << 4)                       // D format f32
         | ((uint32_t)(kN >> 3) << 17)   // N >> 3
         | ((uint32_t)(kBM >> 4) << 24); // M >> 4 (A = B = e4m3, both K-major)
}

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Bounded wait until *ctr >= target, polling with a short sleep between reads; false on
// timeout (raising FTMOE_ERR_WAIT_TIMEOUT and the abort flag) or when another role aborted.
__device__ __forceinline__ bool wait_count(const uint32_t* ctr, uint32_t target, volatile int* abort_flag) {
  if (ld_acquire_u32(ctr) >= target) return true;
  const unsigned long long t0 = globaltimer();
  while (ld_acquire_u32(ctr) < target) {
    if (*abort_flag) return false;
    if (globaltimer() - t0 > kTimeoutNs) {
      raise_error(FTMOE_ERR_WAIT_TIMEOUT);
      *abort_flag = 1;
      return false;
    }
    __nanosleep(128);
  }
  return true;
}

// Release/acquire fence at GPU scope: orders this thread's (and, through the barriers it
// took part in, its CTA's) global writes before a counter update, and the reads after an
// observed count after it.
__device__ __forceinline__ void fence_acq_rel_gpu() { asm volatile("fence.acq_rel.gpu;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

struct Params {
  const int32_t* ids;      // [T * topk]
  const float* rw;         // [T * topk]
  const float* x_s;        // [16][KB] (rows >= T are zero)
  const uint8_t* act_q_in; // == act_q (read by the B loader)
  const float* wg_s;       // [E][NB][KB]
  const float* wd_s;       // [E][HB][KB2]
  uint8_t* act_q;          // [R][I]
  float* act_s;            // [R][NJ]
  float* y;                // [R][H]
  float* part;             // [gate/up chunks][128 rows][kPartCols], chunk = block * kch + chunk in block
  uint32_t* cnt;           // pairs [u_max * NJ], experts [u_max], tokens [T * HB]
  void* out;
  int64_t ld_out;
  int out_dtype;
  int T, topk, E, H, I;
  int KB, KB2, NJ, NB, HB;
  int kbs_g, kbs_d, stages;
  int kch, ckb, u_max;     // chunks per gate/up block, K blocks per chunk, most distinct experts
};

// Shared-memory tables every role reads (built by all threads at the start).
struct Tables {
  int ids[kMaxRoutes];          // valid expert id of each route, or -1
  uint32_t bm[32];              // bitmap of active experts (E <= 1024)
  int pre[32];                  // distinct experts in lower bitmap words
  int canon[kMaxRoutes];        // first route of the same (token, expert): the row it shares
  int ex[kMaxRoutes];           // expert of slot s
  int m[kMaxRoutes];            // tokens of slot s (at most T)
  int rt[kMaxRoutes][kMaxRowsPerExpert];  // canonical route of each token of slot s, ascending
  int nact[kDecodeMaxTokens];   // distinct active experts per token
  int U;                        // distinct active experts
};

// The CTA's work, in the order every role walks it: gate/up segments, then down blocks.
struct Sched {
  int64_t KU;      // gate/up chunks of all active blocks
  int Gg;          // CTAs with gate/up work (min(grid, KU))
  int64_t u_lo, u_hi;  // this CTA's chunk range
  int d_lo, d_hi;      // this CTA's down blocks
  int KCH;             // chunks per gate/up block
};

__device__ __forceinline__ int64_t chunk_lo(int64_t c, int64_t KU, int Gg) { return c * KU / Gg; }
// the CTA whose chunk range holds chunk u (max c with chunk_lo(c) <= u)
__device__ __forceinline__ int cta_of(int64_t u, int64_t KU, int Gg) { return (int)(((u + 1) * Gg - 1) / KU); }

__global__ void __launch_bounds__(kThreads, 1)
    decode_fused_kernel(const __grid_constant__ CUtensorMap map_wg, const __grid_constant__ CUtensorMap map_wd,
                        const __grid_constant__ CUtensorMap map_x, Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int S = p.stages;
  const int stage_bytes = p.kbs_g * (kSubW + kSubX);
  uint8_t* ring = smem;
  uint8_t* bbuf = ring + (size_t)S * stage_bytes;              // two B buffers of [KB2][16 rows][128 B]
  const int bbuf_bytes = p.KB2 * kSubX;
  const int prod_kb = p.KB > p.KB2 ? p.KB : p.KB2;
  float* prod = reinterpret_cast<float*>(bbuf + 2 * bbuf_bytes);  // [2][max(KB, KB2)][kN]
  float* red = prod + 2 * prod_kb * kN;                         // [4 finisher warps][kMaxRowsPerExpert]
  uint64_t* bars = reinterpret_cast<uint64_t*>(red + 4 * kMaxRowsPerExpert);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tfull = bars + 2 * S;
  uint64_t* tempty = tfull + kAcc;
  uint64_t* bfull = tempty + kAcc;
  uint64_t* bempty = bfull + 2;
  uint64_t* pfull = bempty + 2;    // scale-product table i & 1 ready (32 arrivals: the scale warp)
  uint64_t* pempty = pfull + 2;    // ... read by the promoters (4 arrivals)
  uint64_t* qdone = pempty + 2;    // item promoted, its rows written (4 arrivals: promoter warps)
  uint64_t* qfree = qdone + kQueue;  // item finished (4 arrivals: finisher warps)
  __shared__ Tables tb;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  __shared__ int s_last;
  __shared__ int s_mark[kMaxRowsPerExpert];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = p.T * p.topk;

  // ---- tables from expert_ids (an input of the forward: safe to read before the wait) ----
  if (tid < 32) tb.bm[tid] = 0u;
  if (tid == 0) {
    s_abort = 0;
    for (int i = 0; i < S; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    for (int i = 0; i < kAcc; ++i) {
      mbar_init(smem_u32(&tfull[i]), 1);
      mbar_init(smem_u32(&tempty[i]), kEpiThreads / 32);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bfull[i]), 1);
      mbar_init(smem_u32(&bempty[i]), 1);
      mbar_init(smem_u32(&pfull[i]), 32);
      mbar_init(smem_u32(&pempty[i]), kEpiThreads / 32);
    }
    for (int i = 0; i < kQueue; ++i) {
      mbar_init(smem_u32(&qdone[i]), kEpiThreads / 32);
      mbar_init(smem_u32(&qfree[i]), kFinThreads / 32);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (tid < R) {
    const int id = p.ids[tid];
    const bool valid = id >= 0 && id < p.E;
    if (id >= p.E && blockIdx.x == 0) raise_error(FTMOE_ERR_EXPERT_ID_RANGE);
    tb.ids[tid] = valid ? id : -1;
    if (valid) atomicOr(&tb.bm[id >> 5], 1u << (id & 31));
  }
  __syncthreads();
  if (warp == 0) {
    const int c = __popc(tb.bm[lane]);
    int inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += t;
    }
    tb.pre[lane] = inc - c;
    if (lane == 31) tb.U = inc;
  }
  __syncthreads();
  // A token that lists one expert more than once has one intermediate row and one down row
  // for that expert, in the slot of its first listing (the canonical route); every listing
  // reads that row in the combine, with its own routing weight.
  if (tid < R) {
    const int id = tb.ids[tid];
    int c = tid;
    if (id >= 0)
      for (int j = (tid / p.topk) * p.topk; j < tid; ++j)
        if (tb.ids[j] == id) {
          c = j;
          break;
        }
    tb.canon[tid] = c;
  }
  __syncthreads();
  if (tid < R && tb.ids[tid] >= 0 && tb.canon[tid] == tid) {
    const int id = tb.ids[tid];
    const int s = tb.pre[id >> 5] + __popc(tb.bm[id >> 5] & ((1u << (id & 31)) - 1u));
    int pos = 0, count = 0;
    for (int j = 0; j < R; ++j) {
      const bool same = tb.ids[j] == id && tb.canon[j] == j;
      pos += (same && j < tid) ? 1 : 0;
      count += same ? 1 : 0;
    }
    tb.rt[s][pos] = tid;  // pos < count <= T <= kMaxRowsPerExpert
    if (pos == 0) {
      tb.ex[s] = id;
      tb.m[s] = count;
    }
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                 "n"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_before();
  __syncthreads();
  fence_after();
  if (tid < p.T) {  // distinct active experts per token: the arrivals its combine waits for
    int n = 0;
    for (int j = 0; j < p.topk; ++j) {
      const int r = tid * p.topk + j;
      n += (tb.ids[r] >= 0 && tb.canon[r] == r) ? 1 : 0;
    }
    tb.nact[tid] = n;
  }
  __syncthreads();

  const int U = tb.U;
  const int G = gridDim.x;
  Sched sc;
  sc.KCH = p.kch;
  sc.KU = (int64_t)U * p.NB * sc.KCH;
  sc.Gg = sc.KU < G ? (int)sc.KU : G;
  if ((int)blockIdx.x < sc.Gg) {
    sc.u_lo = chunk_lo(blockIdx.x, sc.KU, sc.Gg);
    sc.u_hi = chunk_lo(blockIdx.x + 1, sc.KU, sc.Gg);
  } else {
    sc.u_lo = sc.u_hi = 0;
  }
  const int ND = U * p.HB;
  sc.d_lo = (int)(((int64_t)blockIdx.x * ND) / G);
  sc.d_hi = (int)(((int64_t)(blockIdx.x + 1) * ND) / G);
  const int NJ = p.NJ, HB = p.HB;
  uint32_t* cnt_pair = p.cnt;
  uint32_t* cnt_exp = p.cnt + (size_t)p.u_max * NJ;
  uint32_t* cnt_tok = cnt_exp + p.u_max;
  const uint32_t tmem_base = s_tmem;

  // gate/up block b = (s * NJ + j) * 2 + half: expert slot s, pair j, half 0 gate / 1 up;
  // its weight rows are block j (gate) or block NJ + j (up) of the expert's 2I rows
  auto wrow_block = [&](int b) { const int j = (b >> 1) % NJ; return (b & 1) ? NJ + j : j; };
  auto slot_of_block = [&](int b) { return (b >> 1) / NJ; };

  if (warp == 0) {
    // ------------------------------- TMA producer -------------------------------
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first(), pol_x = l2_policy_evict_last();
      uint32_t it = 0;
      int pre_st[kMaxStages], pre_kb[kMaxStages];
      int npre = 0;
      bool waited = false;
      // one stage: the weights of K blocks [kb0, kb0 + kbs) of a weight block (+ the token
      // tile for gate/up stages); the first pass over the ring goes out before the wait on
      // the prep launch, whose token rows the gate/up stages also need
      auto issue = [&](bool gu, int e, int wrb, int kb0) -> bool {
        const int st = it % S;
        if (it >= (uint32_t)S) {
          if (!waited) {
            pdl_wait();
            waited = true;
            for (int i = 0; i < npre; ++i)
              tma_load_3d_hint(smem_u32(ring + (size_t)pre_st[i] * stage_bytes + p.kbs_g * kSubW), &map_x,
                               smem_u32(&full[pre_st[i]]), 0, 0, pre_kb[i], pol_x);
          }
          if (!mbar_wait(smem_u32(&empty[st]), ((it / S) & 1) ^ 1, &s_abort)) return false;
        }
        uint8_t* sw = ring + (size_t)st * stage_bytes;
        const uint32_t fb = smem_u32(&full[st]);
        if (gu) {
          mbar_expect_tx(fb, p.kbs_g * (kSubW + kSubX));
          tma_load_4d_hint(smem_u32(sw), &map_wg, fb, 0, wrb * kBM, kb0, e, pol_w);
          if (waited) {
            tma_load_3d_hint(smem_u32(sw + p.kbs_g * kSubW), &map_x, fb, 0, 0, kb0, pol_x);
          } else {
            pre_st[npre] = st;
            pre_kb[npre] = kb0;
            ++npre;
          }
        } else {
          mbar_expect_tx(fb, p.kbs_d * kSubW);
          tma_load_4d_hint(smem_u32(sw), &map_wd, fb, 0, wrb * kBM, kb0, e, pol_w);
        }
        ++it;
        return true;
      };
      // one walk over the CTA's stages (gate/up chunks, then down blocks), one call site: the
      // down phase runs the code the gate/up phase already brought into the instruction cache
      bool ok = true;
      int64_t u = sc.u_lo;
      int d = sc.d_lo, sub = 0;
      while (ok && !s_abort) {
        if (u < sc.u_hi) {
          const int b = (int)(u / sc.KCH), ch = (int)(u % sc.KCH);
          ok = issue(true, tb.ex[slot_of_block(b)], wrow_block(b), ch * p.ckb + sub * p.kbs_g);
          if (++sub == p.ckb / p.kbs_g) sub = 0, ++u;
        } else if (d < sc.d_hi) {
          ok = issue(false, tb.ex[d / HB], d % HB, sub * p.kbs_d);
          if (++sub == p.KB2 / p.kbs_d) sub = 0, ++d;
        } else {
          break;
        }
      }
      if (!waited) {
        pdl_wait();
        for (int i = 0; i < npre; ++i)
          tma_load_3d_hint(smem_u32(ring + (size_t)pre_st[i] * stage_bytes + p.kbs_g * kSubW), &map_x,
                           smem_u32(&full[pre_st[i]]), 0, 0, pre_kb[i], pol_x);
      }
      pdl_trigger();
      // loads still in flight complete on their full barrier (bounded wait)
      for (int st = 0; st < S && (uint32_t)st < it; ++st) {
        const uint32_t last = it - 1 - ((it - 1 - st) % S);
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&full[st]), (last / S) & 1) && globaltimer() - t0 < kTimeoutNs) {
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------- MMA issuer --------------------------------
    if (lane == 0) {
      const uint32_t idesc = idesc_f8_n16();
      uint32_t it = 0, kc = 0;
      bool ok = true;
      // one stage of nkb K blocks against the B sub-tiles at b0, b0 + kSubX, ...
      auto consume = [&](int nkb, uint32_t b0) -> bool {
        const int st = it % S;
        if (!mbar_wait(smem_u32(&full[st]), (it / S) & 1, &s_abort)) return false;
        const uint32_t sw = smem_u32(ring + (size_t)st * stage_bytes);
        for (int h = 0; h < nkb; ++h, ++kc) {
          const uint32_t acc = kc % kAcc;
          if (!mbar_wait(smem_u32(&tempty[acc]), ((kc / kAcc) & 1) ^ 1, &s_abort)) return false;
          fence_after();
          const uint32_t d = tmem_base + acc * kN;
          const uint32_t wa = sw + h * kSubW, xb = b0 + h * kSubX;
#pragma unroll
          for (int j = 0; j < kBK / 32; ++j)
            mma_f8(d, smem_desc_sw128(wa + 32 * j), smem_desc_sw128(xb + 32 * j), idesc, j > 0 ? 1u : 0u);
          mma_commit(smem_u32(&tfull[acc]));
        }
        mma_commit(smem_u32(&empty[st]));
        ++it;
        return true;
      };
      // the same walk as the producer's: gate/up stages (B = the stage's token tile), then
      // down stages (B = the expert's staged intermediate rows)
      int64_t u = sc.u_lo;
      int d = sc.d_lo, sub = 0, g = -1, prev_s = -1;
      while (ok && !s_abort) {
        uint32_t b0;
        int nkb;
        bool release_b = false;
        if (u < sc.u_hi) {
          b0 = smem_u32(ring + (size_t)(it % S) * stage_bytes + p.kbs_g * kSubW);
          nkb = p.kbs_g;
          if (++sub == p.ckb / p.kbs_g) sub = 0, ++u;
        } else if (d < sc.d_hi) {
          const int s = d / HB;
          if (s != prev_s) {  // a new expert: its B rows are staged in buffer (g + 1) & 1
            ++g;
            prev_s = s;
            if (!mbar_wait(smem_u32(&bfull[g & 1]), (g >> 1) & 1, &s_abort)) break;
            fence_after();
          }
          b0 = smem_u32(bbuf + (size_t)(g & 1) * bbuf_bytes) + (uint32_t)(sub * p.kbs_d * kSubX);
          nkb = p.kbs_d;
          if (++sub == p.KB2 / p.kbs_d) {
            sub = 0;
            ++d;
            release_b = d >= sc.d_hi || d / HB != s;  // the expert's last block: B may be refilled
          }
        } else {
          break;
        }
        ok = consume(nkb, b0);
        if (ok && release_b) mma_commit(smem_u32(&bempty[g & 1]));
      }
      // MMAs still running write TMEM and read B: wait (bounded) for each accumulator's last
      // commit before the CTA may free TMEM
      for (uint32_t b = 0; b < (uint32_t)kAcc && b < kc; ++b) {
        const uint32_t last = kc - 1 - ((kc - 1 - b) % kAcc);
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&tfull[b]), (last / kAcc) & 1) && globaltimer() - t0 < kTimeoutNs) {
        }
      }
    }
  } else if (warp == 2) {
    // ------------------------ B loader (down blocks) -------------------------------
    // The expert's intermediate rows (one per token, written by the pair finalizers of any
    // CTA) become the MMA's B operand: 16 rows of I bytes in the 128-byte-swizzled K-major
    // layout, one 2 KiB sub-tile per K block, rows beyond the expert's tokens zero.
    int g = -1, prev_s = -1;
    pdl_wait();
    for (int d = sc.d_lo; d < sc.d_hi && !s_abort; ++d) {
      const int s = d / HB;
      if (s == prev_s) continue;
      ++g;
      prev_s = s;
      if (g >= 2 && !__all_sync(0xffffffffu, mbar_wait(smem_u32(&bempty[g & 1]), ((g >> 1) - 1) & 1, &s_abort)))
        break;
      // all of the expert's (gate, up) pairs are re-quantized (bounded wait)
      bool ready = lane == 0 ? wait_count(cnt_exp + s, (uint32_t)NJ, &s_abort) : true;
      ready = __shfl_sync(0xffffffffu, ready ? 1 : 0, 0) != 0;
      if (!ready) break;
      (void)ld_acquire_u32(cnt_exp + s);  // every lane acquires before it reads the rows
      uint8_t* bb = bbuf + (size_t)(g & 1) * bbuf_bytes;
      const int m = tb.m[s];
      const int per_row = p.KB2 * 8;  // 16-byte chunks of one row
      for (int i = lane; i < kMaxRowsPerExpert * per_row; i += 32) {
        const int q = i / per_row, rem = i - q * per_row;
        const int kb = rem >> 3, c16 = rem & 7;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (q < m) v = __ldcg(reinterpret_cast<const uint4*>(p.act_q_in + (int64_t)tb.rt[s][q] * p.I + kb * kBK + c16 * 16));
        *reinterpret_cast<uint4*>(bb + kb * kSubX + q * kBK + ((c16 ^ (q & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bfull[g & 1]));
    }
  } else if (warp == kScaleWarp) {
    // -------------------- scale products, one item ahead ---------------------------
    // Item it's table goes to buffer it & 1: gate/up segments x_s[token][kb] * w_s[block][kb],
    // down blocks act_s[row q][kb] * w_s[e][hb][kb] (once the expert's intermediate rows
    // are complete). The promoters read it while the next one is being formed.
    pdl_wait();  // x_s comes from the quantizing launch
    int item = 0;
    auto begin = [&](int it) -> bool {
      bool ok = true;
      if (it >= 2) ok = mbar_wait(smem_u32(&pempty[it & 1]), ((it >> 1) - 1) & 1, &s_abort);
      return __all_sync(0xffffffffu, ok) != 0;
    };
    for (int64_t u = sc.u_lo; u < sc.u_hi; ++item) {
      const int b = (int)(u / sc.KCH), c0 = (int)(u % sc.KCH);
      const int64_t seg_end = ((int64_t)b + 1) * sc.KCH < sc.u_hi ? ((int64_t)b + 1) * sc.KCH : sc.u_hi;
      const int c1 = (int)(seg_end - (int64_t)b * sc.KCH);
      u = seg_end;
      if (!begin(item)) break;
      float* pr = prod + (item & 1) * prod_kb * kN;
      const int e = tb.ex[slot_of_block(b)], wrb = wrow_block(b);
      const int kb0 = c0 * p.ckb, nkb = (c1 - c0) * p.ckb;
      for (int i = lane; i < nkb * kN; i += 32) {
        const int kbl = i / kN, c = i - kbl * kN;
        const int kb = kb0 + kbl;
        pr[i] = __ldg(p.x_s + (int64_t)c * p.KB + kb) * __ldg(p.wg_s + ((int64_t)e * p.NB + wrb) * p.KB + kb);
      }
      mbar_arrive(smem_u32(&pfull[item & 1]));
    }
    for (int d = sc.d_lo; d < sc.d_hi && !s_abort; ++d, ++item) {
      if (!begin(item)) break;
      const int s = d / HB, hb = d % HB, e = tb.ex[s], m = tb.m[s];
      bool ready = lane == 0 ? wait_count(cnt_exp + s, (uint32_t)NJ, &s_abort) : true;
      if (__shfl_sync(0xffffffffu, ready ? 1 : 0, 0) == 0) break;
      (void)ld_acquire_u32(cnt_exp + s);  // every lane acquires before it reads the scales
      float* pr = prod + (item & 1) * prod_kb * kN;
      for (int i = lane; i < p.KB2 * kN; i += 32) {
        const int kb = i / kN, q = i - kb * kN;
        pr[i] = q < m ? __ldcg(p.act_s + (int64_t)tb.rt[s][q] * NJ + kb) *
                            __ldg(p.wd_s + ((int64_t)e * HB + hb) * p.KB2 + kb)
                      : 0.0f;
      }
      mbar_arrive(smem_u32(&pfull[item & 1]));
    }
  } else if (warp < kFinWarp0) {
    // ------------------------------- promotion --------------------------------------
    // Warp w reads TMEM lanes 32 (w % 4) .. (one weight row per thread) of each K block's
    // accumulator and adds d * (act_scale x weight_scale) per column; gate/up chunks are
    // stored as partial sums, down blocks as rows of y. Nothing here waits on other CTAs.
    const int et = tid - kEpiWarp0 * 32;  // 0..127 = TMEM lane = weight row in the block
    const int quarter = warp & 3;
    uint32_t kc = 0;
    pdl_wait();
    // promote nkb K blocks: acc[c] += d[c] * pr[i][c]
    auto promote = [&](int nkb, float* acc, const float* pr) -> bool {
      bool ok = true;
      for (int i = 0; i < nkb; ++i, ++kc) {
        const uint32_t ab = kc % kAcc;
        if (ok) {
          const int got = mbar_wait(smem_u32(&tfull[ab]), (kc / kAcc) & 1, &s_abort) ? 1 : 0;
          ok = __all_sync(0xffffffffu, got) != 0;
        }
        if (!ok) continue;
        fence_after();
        float d[kN];
        tmem_ld16(tmem_base + ((uint32_t)(32 * quarter) << 16) + ab * kN, d);
        tmem_ld_wait();
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&tempty[ab]));
        const float4* p4 = reinterpret_cast<const float4*>(pr + i * kN);
#pragma unroll
        for (int c4 = 0; c4 < kN / 4; ++c4) {
          const float4 s4 = p4[c4];
          acc[4 * c4 + 0] = fmaf(d[4 * c4 + 0], s4.x, acc[4 * c4 + 0]);
          acc[4 * c4 + 1] = fmaf(d[4 * c4 + 1], s4.y, acc[4 * c4 + 1]);
          acc[4 * c4 + 2] = fmaf(d[4 * c4 + 2], s4.z, acc[4 * c4 + 2]);
          acc[4 * c4 + 3] = fmaf(d[4 * c4 + 3], s4.w, acc[4 * c4 + 3]);
        }
      }
      return ok;
    };
    // an item's scale table is ready, and its queue slot is free of the item kQueue back
    auto begin = [&](int it) -> bool {
      bool ok = true;
      if (it >= kQueue) ok = mbar_wait(smem_u32(&qfree[it % kQueue]), ((it / kQueue) - 1) & 1, &s_abort);
      ok = ok && mbar_wait(smem_u32(&pfull[it & 1]), (it >> 1) & 1, &s_abort);
      return __all_sync(0xffffffffu, ok) != 0;
    };
    // the table is read and the item's rows are written: hand it to the finishers
    auto finish = [&](int it) {
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&pempty[it & 1]));
        mbar_arrive(smem_u32(&qdone[it % kQueue]));
      }
    };
    // one walk over the CTA's items (gate/up segments, then down blocks) with one promotion
    // call site, so the down phase runs code the gate/up phase already brought into the
    // instruction cache
    int item = 0;
    bool ok = true;
    int64_t u = sc.u_lo;
    int d = sc.d_lo;
    while (ok) {
      bool gu;
      int b = 0, c0 = 0, c1 = 1, s = 0, hb = 0;
      if (u < sc.u_hi) {
        gu = true;
        b = (int)(u / sc.KCH);
        c0 = (int)(u % sc.KCH);
        const int64_t seg_end = ((int64_t)b + 1) * sc.KCH < sc.u_hi ? ((int64_t)b + 1) * sc.KCH : sc.u_hi;
        c1 = (int)(seg_end - (int64_t)b * sc.KCH);
        u = seg_end;
      } else if (d < sc.d_hi) {
        gu = false;
        s = d / HB;
        hb = d % HB;
        ++d;
      } else {
        break;
      }
      if (!begin(item)) break;
      const float* pr = prod + (item & 1) * prod_kb * kN;
      const int nkb = gu ? p.ckb : p.KB2;
      // gate/up: one partial sum per chunk, each from zero (the finishers add a block's chunks
      // in K order, so the result does not depend on how the chunks were spread over the
      // CTAs); down: the expert's rows of y
      for (int ch = c0; ch < c1; ++ch) {
        float acc[kN];
#pragma unroll
        for (int c = 0; c < kN; ++c) acc[c] = 0.0f;
        ok = promote(nkb, acc, pr + (ch - c0) * nkb * kN) && ok;
        if (gu) {
          // [chunk][row][8 token columns]: a row's columns are one 32-byte piece
          float4* pp = reinterpret_cast<float4*>(p.part + (((size_t)b * sc.KCH + ch) * kBM + et) * kPartCols);
          __stcg(pp, make_float4(acc[0], acc[1], acc[2], acc[3]));
          __stcg(pp + 1, make_float4(acc[4], acc[5], acc[6], acc[7]));
        } else {
          const int m = tb.m[s], h = hb * kBM + et;
#pragma unroll
          for (int q = 0; q < kMaxRowsPerExpert; ++q)
            if (q < m) __stcg(p.y + (int64_t)tb.rt[s][q] * p.H + h, acc[q]);
        }
      }
      finish(item);
      ++item;
    }
  } else {
    // --------------------------------- finishers ------------------------------------
    // Per item, after the promoters wrote its rows: a gate/up segment counts its arrival at
    // the (gate block j, up block j) pair; the last arrival adds each block's chunks in K
    // order, forms silu(g) * u for the expert's tokens, re-quantizes each token's 1x128 group
    // (scale amax / 448) and counts the pair done for the expert. A down block counts its
    // tokens per (token, block of H); the last arrival for a token reduces that token's
    // active routes in ascending slot order (fp32, from zero) into the output. Thread ft is
    // weight row ft of the block.
    const int ft = tid - kFinWarp0 * 32;
    const int fw = warp - kFinWarp0;
    pdl_wait();  // the counters are zeroed by the quantizing launch
    auto begin = [&](int it) -> bool {
      const bool ok = mbar_wait(smem_u32(&qdone[it % kQueue]), (it / kQueue) & 1, &s_abort);
      return !named_bar_or(kFinBar, kFinThreads, ok ? 0 : 1);
    };
    auto done = [&](int it) {
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&qfree[it % kQueue]));
    };
    int item = 0;
    for (int64_t u = sc.u_lo; u < sc.u_hi; ++item) {
      const int b = (int)(u / sc.KCH);
      const int64_t seg_end = ((int64_t)b + 1) * sc.KCH < sc.u_hi ? ((int64_t)b + 1) * sc.KCH : sc.u_hi;
      u = seg_end;
      if (!begin(item)) break;
      const int s = slot_of_block(b), j = (b >> 1) % NJ, bg = b & ~1;
      if (ft == 0) {
        // the pair's arrivals: every segment of its gate block and of its up block
        int expected = 0;
        for (int h = 0; h < 2; ++h) {
          const int64_t a0 = ((int64_t)bg + h) * sc.KCH;
          expected += cta_of(a0 + sc.KCH - 1, sc.KU, sc.Gg) - cta_of(a0, sc.KU, sc.Gg) + 1;
        }
        fence_acq_rel_gpu();  // this CTA's partial sums (seen through the queue) before the count
        const uint32_t old = atomicAdd(cnt_pair + (size_t)s * NJ + j, 1u);
        s_last = (int)(old + 1 == (uint32_t)expected);
        fence_acq_rel_gpu();
      }
      named_bar(kFinBar, kFinThreads);
      if (s_last) {
        // the gate and up blocks' chunk sums of this row, added in K order: per group of four
        // token columns the call has, every chunk's loads are in flight before the sum
        float gsum[kPartCols], usum[kPartCols];
        const float4* g4 = reinterpret_cast<const float4*>(p.part + ((size_t)bg * sc.KCH * kBM + ft) * kPartCols);
        const float4* u4 = g4 + (size_t)sc.KCH * kBM * 2;
#pragma unroll
        for (int cg = 0; cg < kPartCols / 4; ++cg) {
          float4 gv[kDecodeMaxKch], uv[kDecodeMaxKch];
          const bool need = cg * 4 < p.T;
#pragma unroll
          for (int ch = 0; ch < kDecodeMaxKch; ++ch) {
            if (need && ch < sc.KCH) {
              gv[ch] = __ldcg(g4 + (size_t)ch * kBM * 2 + cg);
              uv[ch] = __ldcg(u4 + (size_t)ch * kBM * 2 + cg);
            } else {
              gv[ch] = uv[ch] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            }
          }
          float4 ga = gv[0], ua = uv[0];
#pragma unroll
          for (int ch = 1; ch < kDecodeMaxKch; ++ch) {
            if (ch < sc.KCH) {
              ga.x += gv[ch].x, ga.y += gv[ch].y, ga.z += gv[ch].z, ga.w += gv[ch].w;
              ua.x += uv[ch].x, ua.y += uv[ch].y, ua.z += uv[ch].z, ua.w += uv[ch].w;
            }
          }
          gsum[4 * cg + 0] = ga.x, gsum[4 * cg + 1] = ga.y, gsum[4 * cg + 2] = ga.z, gsum[4 * cg + 3] = ga.w;
          usum[4 * cg + 0] = ua.x, usum[4 * cg + 1] = ua.y, usum[4 * cg + 2] = ua.z, usum[4 * cg + 3] = ua.w;
        }
        const int m = tb.m[s];
        // silu(g) * u of the token of the expert's q-th row (its column of the sums); compact
        // loops over the expert's tokens, the value recomputed where it is quantized (the same
        // expression on the same inputs: the same bits)
        auto a_of = [&](int q) {
          const int t = tb.rt[s][q] / p.topk;
          float gt = 0.0f, ut = 0.0f;
#pragma unroll
          for (int c = 0; c < kPartCols; ++c)  // a select, not a dynamic index into registers
            if (c == t) gt = gsum[c], ut = usum[c];
          return silu_mul_1(gt, ut);
        };
#pragma unroll 1
        for (int q = 0; q < m; ++q) {
          const float w = warp_max(fabsf(a_of(q)));
          if (lane == 0) red[fw * kMaxRowsPerExpert + q] = w;
        }
        named_bar(kFinBar, kFinThreads);
#pragma unroll 1
        for (int q = 0; q < m; ++q) {
          const float amax = fmaxf(fmaxf(red[q], red[kMaxRowsPerExpert + q]),
                                   fmaxf(red[2 * kMaxRowsPerExpert + q], red[3 * kMaxRowsPerExpert + q]));
          const float scl = div_rn(amax, kE4M3Max);
          const uint8_t code = amax > 0.0f ? (uint8_t)(f2_to_e4m3x2(div_rn(a_of(q), scl), 0.0f) & 0xFF) : (uint8_t)0;
          const int r = tb.rt[s][q];
          p.act_q[(int64_t)r * p.I + j * kBK + ft] = code;
          if (ft == 0) p.act_s[(int64_t)r * NJ + j] = scl;
        }
        named_bar(kFinBar, kFinThreads);  // every row written (and red read) before the count
        if (ft == 0) {
          fence_acq_rel_gpu();
          atomicAdd(cnt_exp + s, 1u);
        }
      }
      done(item);
    }
    for (int d = sc.d_lo; d < sc.d_hi; ++d, ++item) {
      if (!begin(item)) break;
      const int s = d / HB, hb = d % HB, m = tb.m[s];
      if (ft < m) {  // one thread per token of the expert, the counts in parallel
        const int t = tb.rt[s][ft] / p.topk;
        fence_acq_rel_gpu();  // this CTA's rows of y (seen through the queue) before the count
        const uint32_t old = atomicAdd(cnt_tok + (size_t)t * HB + hb, 1u);
        s_mark[ft] = (int)(old + 1 == (uint32_t)tb.nact[t]);
        fence_acq_rel_gpu();
      }
      named_bar(kFinBar, kFinThreads);
      const int h = hb * kBM + ft;
      for (int q = 0; q < m; ++q) {
        if (!s_mark[q]) continue;
        const int t = tb.rt[s][q] / p.topk;
        float v = 0.0f;
        // the token's routes eight at a time: loads first, then the sum in slot order
        for (int j0 = 0; j0 < p.topk; j0 += 8) {
          float wv[8], yv[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int r = t * p.topk + j0 + u;
            const bool act = j0 + u < p.topk && tb.ids[r] >= 0;  // inactive: nothing of it is read
            wv[u] = act ? __ldg(p.rw + r) : 0.0f;
            yv[u] = act ? __ldcg(p.y + (int64_t)tb.canon[r] * p.H + h) : 0.0f;
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int r = t * p.topk + j0 + u;
            if (j0 + u < p.topk && tb.ids[r] >= 0) v = fmaf(wv[u], yv[u], v);
          }
        }
        if (p.out_dtype == FTMOE_OUT_FP32) {
          reinterpret_cast<float*>(p.out)[(int64_t)t * p.ld_out + h] = v;
        } else if (p.out_dtype == FTMOE_OUT_FP16) {
          reinterpret_cast<uint16_t*>(p.out)[(int64_t)t * p.ld_out + h] = __half_as_ushort(__float2half_rn(v));
        } else {
          reinterpret_cast<uint16_t*>(p.out)[(int64_t)t * p.ld_out + h] =
              __bfloat16_as_ushort(__float2bfloat16_rn(v));
        }
      }
      named_bar(kFinBar, kFinThreads);  // s_mark is rewritten by the next block
      done(item);
    }
  }

  fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "n"(kTmemCols));
  }
}

// ---- prep: the token rows quantized per 1x128 into 16 rows (rows >= T zero), the
// counters zeroed, and the output rows of tokens without an active route written as zeros ----
template <bool kVec>
__global__ void __launch_bounds__(512) decode_prep_kernel(const uint16_t* __restrict__ x, int T, int64_t H,
                                                          int64_t ld_x, uint8_t* __restrict__ xq,
                                                          float* __restrict__ xs, const int32_t* __restrict__ ids,
                                                          int topk, int E, uint32_t* __restrict__ cnt, int ncnt,
                                                          uint8_t* __restrict__ out, int64_t ld_out_bytes,
                                                          int64_t row_bytes) {
  pdl_wait();  // the predecessor's outputs are complete from here on
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int64_t ng = H / kGroup;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t w = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); w < kN * ng; w += nwarps) {
    const int64_t row = w / ng, g = w - row * ng;
    if (row < T) {
      quantize_fp8_group<kVec>(x, H, ld_x, xq, xs, ng, row, g, lane);
    } else {
      *reinterpret_cast<uint32_t*>(xq + row * H + g * kGroup + lane * 4) = 0u;
      if (lane == 0) xs[row * ng + g] = 0.0f;
    }
  }
  if (blockIdx.x == 0) {
    for (int i = threadIdx.x; i < ncnt; i += blockDim.x) cnt[i] = 0u;
    for (int t = 0; t < T; ++t) {
      int n = 0;
      for (int j = 0; j < topk; ++j) {
        const int id = ids[t * topk + j];
        n += (id >= 0 && id < E) ? 1 : 0;
      }
      if (n == 0)
        for (int64_t b = threadIdx.x; b < row_bytes; b += blockDim.x) out[t * ld_out_bytes + b] = 0;
    }
  }
}

}  // namespace dk

// ---------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------

static int kbs_for_blocks(int kb) { return kb % 4 == 0 ? 4 : (kb % 2 == 0 ? 2 : 1); }

DecodePlan decode_plan(int64_t T, int32_t topk, int32_t E, int64_t H, int64_t I) {
  DecodePlan pl;
  pl.ok = T >= 1 && T <= kDecodeMaxTokens && T * topk <= kDecodeMaxRoutes && E >= 1 && E <= kDecodeMaxExperts &&
          H % 128 == 0 && I % 128 == 0 && H >= 128 && I >= 128 && H <= 8192 && I <= 2048;
  if (!pl.ok) return pl;
  pl.KB = (int)(H / 128);
  pl.KB2 = (int)(I / 128);
  pl.NJ = pl.KB2;
  pl.NB = 2 * pl.NJ;
  pl.HB = pl.KB;
  pl.kbs_g = kbs_for_blocks(pl.KB);
  // a down stage holds at most a gate/up stage's weight bytes (both are powers of two that
  // divide their K-block counts, so the smaller still divides KB2)
  pl.kbs_d = kbs_for_blocks(pl.KB2) < pl.kbs_g ? kbs_for_blocks(pl.KB2) : pl.kbs_g;
  pl.u_max = (int)(T * topk < E ? T * topk : E);
  // Chunks per gate/up block: as many as the partial-sum budget allows (finer chunks spread
  // the weight stream more evenly over the SMs), a divisor of the block's TMA stages. The
  // chunking depends on the shape only, never on which experts are active.
  const int stages_per_block = pl.KB / pl.kbs_g;
  pl.kch = 1;
  // (at most kDecodeMaxKch chunks, 4 beyond four tokens: the finisher keeps one load per
  // chunk and group of four token columns in flight)
  const int kch_cap = T > 4 ? kDecodeMaxKch / 2 : kDecodeMaxKch;
  for (int d = 1; d <= stages_per_block && d <= kch_cap; ++d)
    if (stages_per_block % d == 0 && (int64_t)pl.u_max * pl.NB * d <= kDecodeMaxChunks) pl.kch = d;
  pl.ckb = pl.KB / pl.kch;
  pl.part_bytes = (size_t)pl.u_max * pl.NB * pl.kch * dk::kPartCols * dk::kBM * 4;
  pl.cnt_words = (size_t)pl.u_max * pl.NJ + pl.u_max + (size_t)T * pl.HB;
  return pl;
}

cudaError_t launch_decode_prep(const uint16_t* x, int64_t T, int64_t H, int64_t ld_x, uint8_t* xq, float* xs,
                               const int32_t* ids, int32_t topk, int32_t E, uint32_t* cnt, size_t ncnt, void* out,
                               int64_t ld_out, int32_t out_dtype, cudaStream_t st) {
  const int64_t ng = H / kGroup;
  const int64_t warps = dk::kN * ng;
  int blocks = (int)cdiv(warps, 16);
  if (blocks < 1) blocks = 1;
  const bool vec = quantize_fp8_vec_ok(x, ld_x, xq, H);
  const int64_t eb = out_dtype == FTMOE_OUT_FP32 ? 4 : 2;
  return launch_kernel(vec ? dk::decode_prep_kernel<true> : dk::decode_prep_kernel<false>, dim3(blocks), dim3(512), 0,
                       st, false, x, (int)T, H, ld_x, xq, xs, ids, (int)topk, (int)E, cnt, (int)ncnt,
                       static_cast<uint8_t*>(out), ld_out * eb, H * eb);
}

cudaError_t launch_decode_fused(const DecodeArgs& a, const DecodePlan& pl, cudaStream_t st, int* unsupported) {
  *unsupported = 0;
  EncodeTiledFn enc = encode_fn();
  if (!enc || !pl.ok || (uintptr_t)a.wg_q % 16 || (uintptr_t)a.wd_q % 16 || (uintptr_t)a.x_q % 16) {
    *unsupported = 1;
    return cudaSuccess;
  }
  const int G = sm_count() < kDecodeGrid ? sm_count() : kDecodeGrid;
  int dev = 0;
  cudaGetDevice(&dev);
  static size_t budget[64] = {};
  size_t max_smem = (dev >= 0 && dev < 64) ? budget[dev] : 0;
  if (max_smem == 0) {
    cudaFuncAttributes fattr;
    if (cudaFuncGetAttributes(&fattr, dk::decode_fused_kernel) != cudaSuccess) return cudaErrorInvalidValue;
    int optin = 0;
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    max_smem = (size_t)optin > fattr.sharedSizeBytes ? (size_t)optin - fattr.sharedSizeBytes : 0;
    if (dev >= 0 && dev < 64) budget[dev] = max_smem;
  }
  const size_t stage = (size_t)pl.kbs_g * (dk::kSubW + dk::kSubX);
  const int prod_kb = pl.KB > pl.KB2 ? pl.KB : pl.KB2;
  const size_t fixed = 1024 + 2 * (size_t)pl.KB2 * dk::kSubX + 2 * (size_t)prod_kb * dk::kN * 4 +
                       4 * dk::kMaxRowsPerExpert * 4 + 8 /*bar align*/;
  int stages = dk::kMaxStages;
  auto bytes = [&](int s) {
    return fixed + (size_t)s * stage + (size_t)(2 * s + 2 * dk::kAcc + 8 + 2 * dk::kQueue) * 8;
  };
  while (stages > 2 && bytes(stages) > max_smem) --stages;
  const size_t smem = bytes(stages);
  if (smem > max_smem) {
    *unsupported = 1;
    return cudaSuccess;
  }
  CUtensorMap mg, md, mx;
  {
    const uint64_t d[4] = {128, (uint64_t)(2 * pl.NJ * 128), (uint64_t)pl.KB, (uint64_t)a.E};
    const uint64_t s[3] = {(uint64_t)a.H, 128, (uint64_t)a.H * 2 * a.I};
    const uint32_t b[4] = {128, 128, (uint32_t)pl.kbs_g, 1};
    if (!encode_u8_tmap(&mg, a.wg_q, 4, d, s, b)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t d[4] = {128, (uint64_t)a.H, (uint64_t)pl.KB2, (uint64_t)a.E};
    const uint64_t s[3] = {(uint64_t)a.I, 128, (uint64_t)a.H * a.I};
    const uint32_t b[4] = {128, 128, (uint32_t)pl.kbs_d, 1};
    if (!encode_u8_tmap(&md, a.wd_q, 4, d, s, b)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t d[3] = {128, (uint64_t)dk::kN, (uint64_t)pl.KB};
    const uint64_t s[2] = {(uint64_t)a.H, 128};
    const uint32_t b[3] = {128, (uint32_t)dk::kN, (uint32_t)pl.kbs_g};
    if (!encode_u8_tmap(&mx, a.x_q, 3, d, s, b)) return cudaErrorInvalidValue;
  }
  dk::Params p;
  p.ids = a.ids;
  p.rw = a.rw;
  p.x_s = a.x_s;
  p.act_q_in = a.act_q;
  p.wg_s = a.wg_s;
  p.wd_s = a.wd_s;
  p.act_q = a.act_q;
  p.act_s = a.act_s;
  p.y = a.y;
  p.part = a.part;
  p.cnt = a.cnt;
  p.out = a.out;
  p.ld_out = a.ld_out;
  p.out_dtype = a.out_dtype;
  p.T = (int)a.T;
  p.topk = a.topk;
  p.E = a.E;
  p.H = (int)a.H;
  p.I = (int)a.I;
  p.KB = pl.KB;
  p.KB2 = pl.KB2;
  p.NJ = pl.NJ;
  p.NB = pl.NB;
  p.HB = pl.HB;
  p.kbs_g = pl.kbs_g;
  p.kbs_d = pl.kbs_d;
  p.stages = stages;
  p.kch = pl.kch;
  p.ckb = pl.ckb;
  p.u_max = pl.u_max;
  static size_t granted[64] = {};
  if (dev < 0 || dev >= 64 || smem > granted[dev]) {
    cudaError_t e = cudaFuncSetAttribute(dk::decode_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) granted[dev] = smem;
  }
  return launch_kernel(dk::decode_fused_kernel, dim3(G), dim3(dk::kThreads), smem, st, true, mg, md, mx, p);
}

FTMOE_DEFINE_ERR_READER(read_err_decode)

}  // namespace ftmoe

// Grouped MXFP8 GEMM on the block-scaled tensor-core MMA (tcgen05 kind::mxf8f6f4).
//
// out[row, n] = sum_k (a[row, k] * 2^(sa[row, k/32] - 127)) * (w[e, n, k] * 2^(sw[e, n, k/32] - 127))
// with e4m3 codes a, w and E8M0 scale bytes sa, sw (one per 32 consecutive elements of a row):
// the MXFP8 variant the SGLang gather page names (Modifications: the mxfp8 branch, a ue8m0
// scale per 32 elements). The scales are native to the MMA
// (tcgen05.mma ... kind::mxf8f6f4.block_scale.scale_vec::1X, K = 32 per instruction, one
// scale per row and instruction), so a unit accumulates all of K in TMEM and the epilogue
// stores the accumulator as it is: no per-block promotion on CUDA cores.
//
// Work layout as in the other grouped GEMMs ("swap AB"): MMA M = 128 weight rows (one weight
// block), MMA N = the token tile (16/32/64/128 from route density); CTA c takes units c, c + G,
// ... of the (expert, token tile, weight block) list, so the CTAs sweep it together and a
// token tile is read by several of them at about the same time, from L2.
//
// Two rings in shared memory:
//   * codes: stages of KBS K blocks of 128 elements (weights 128 rows x 128 B, tokens TT rows x
//     128 B per K block, each a canonical 128-byte-swizzled sub-tile), one TMA box per operand;
//   * scales: slots of one chunk of 4 K blocks (512 elements: 16 scale bytes per row, the
//     narrowest box TMA moves), weights 128 x 16 B and tokens TT x 16 B, loaded with the stage
//     that holds the chunk's first K block.
// Scale factors in TMEM, per chunk slot (32 columns: 16 for the weight rows, 16 for the token
// rows): column 4j + c of lane l (in every lane quarter) holds the four scale bytes of K block
// j of the chunk for row l + 32c, byte s for K elements [32 s, 32 s + 32) of that block; the
// MMA of K block j, step s reads column 4j (+ c by row) and byte s (the scale-factor id of the
// instruction descriptor).
//
// Roles: warp 0 TMA producer; warp 1 MMA issuer and TMEM owner; warps 2-5 copy each chunk's
// scales from shared memory into TMEM; warps 6-13 epilogue. Every wait is bounded: on timeout
// the kernel raises FTMOE_ERR_WAIT_TIMEOUT, stops all roles, lets its own copies and MMAs
// drain, frees TMEM and returns.
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace ftmoe {

namespace mxg {

constexpr int kBM = 128;          // weight rows per tile (MMA M)
constexpr int kBK = 128;          // elements (bytes) per K block
constexpr int kChunk = 4;         // K blocks per scale chunk (512 elements, 16 scale bytes per row)
constexpr int kSfRow = 16;        // scale bytes per row and chunk
constexpr int kScaleWarp0 = 2, kScaleWarps = 4;
constexpr int kEpiWarp0 = kScaleWarp0 + kScaleWarps, kEpiWarps = 8;
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);  // 448
constexpr int kMaxExperts = 1024;
constexpr int kAcc = 2;           // accumulators: the next unit's MMAs run during this unit's epilogue
constexpr int kMaxStages = 8;
constexpr int kMaxSfSlots = 8;    // TMEM scale slots (32 columns each, one chunk)
constexpr int kSmemSlots = 4;     // shared-memory scale slots
// K blocks per code stage: four up to token tile 64, two at 128 (the largest stage)
__host__ __device__ constexpr int kbs_for(int tt) { return tt <= 64 ? 4 : 2; }

template <int TT, int KBS>
struct Sz {
  static constexpr int kW = kBM * kBK;        // 16 KiB of weight codes per K block
  static constexpr int kA = TT * kBK;         // token codes per K block
  static constexpr int kOffA = KBS * kW;
  static constexpr int kStage = KBS * (kW + kA);  // multiple of 1024
  static constexpr int kSW = kBM * kSfRow;    // weight scales per chunk
  static constexpr int kSA = TT * kSfRow;     // token scales per chunk
  static constexpr int kSlot = (kSW + kSA + 127) / 128 * 128;
};

// Instruction descriptor of kind::mxf8f6f4 with block scaling: A = B = E4M3, K-major,
// M = 128, N = n, E8M0 scale factors, scale-factor ids sf (byte sf of each 32-bit scale
// column, for A and for B).
__host__ __device__ constexpr uint32_t idesc_mx(int n, uint32_t sf) {
  return (sf << 4)                          // B scale-factor id
         | (0u << 7) | (0u << 10)           // A, B format: E4M3
         | ((uint32_t)(n >> 3) << 17)       // N >> 3
         | (1u << 23)                       // scale format: UE8M0
         | ((uint32_t)(kBM >> 4) << 24)     // M >> 4
         | (sf << 29);                      // A scale-factor id
}

__device__ __forceinline__ void mma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                       uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(acc)
      : "memory");
}

struct Params {
  const int32_t* offsets;
  float* out;
  int64_t ld_out;
  int64_t a_rows;
  int n, E, kb_count, nb_count, stages, sf_slots;
};

template <int TT, int KBS>
__global__ void __launch_bounds__(kThreads, 1)
    mxfp8_gemm_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_a,
                      const __grid_constant__ CUtensorMap map_sw, const __grid_constant__ CUtensorMap map_sa,
                      Params p) {
  using Z = Sz<TT, KBS>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int S = p.stages, SF = p.sf_slots;
  uint8_t* tiles = smem;
  uint8_t* sslots = smem + (size_t)S * Z::kStage;                        // [kSmemSlots][kSlot]
  int* cum = reinterpret_cast<int*>(sslots + (size_t)kSmemSlots * Z::kSlot);  // [E+2] unit prefix
  int* seg_lo = cum + p.E + 2;
  int* seg_hi = seg_lo + p.E;
  uint64_t* bars = reinterpret_cast<uint64_t*>(((reinterpret_cast<uintptr_t>(seg_hi + p.E)) + 7) & ~(uintptr_t)7);
  uint64_t* full = bars;                      // [S] code stage landed
  uint64_t* empty = full + S;                 // [S] MMAs done reading a code stage
  uint64_t* sland = empty + S;                // [kSmemSlots] scale chunk landed in shared memory
  uint64_t* sdrop = sland + kSmemSlots;       // [kSmemSlots] scale chunk copied out (slot reusable)
  uint64_t* sfree = sdrop + kSmemSlots;       // [SF] MMAs done reading a TMEM scale slot
  uint64_t* sfull = sfree + SF;               // [SF] a chunk's scales are in TMEM
  uint64_t* tfull = sfull + SF;
  uint64_t* tempty = tfull + kAcc;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E, NB = p.nb_count, KB = p.kb_count;
  const int NC = KB / kChunk;  // scale chunks per unit (K is a whole number of chunks)
  // TMEM columns: accumulators [0, kAcc*TT), then 32 scale columns per TMEM scale slot
  const uint32_t sf0 = (uint32_t)((kAcc * TT + 31) / 32 * 32);

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < S; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    for (int i = 0; i < kSmemSlots; ++i) {
      mbar_init(smem_u32(&sland[i]), 1);
      mbar_init(smem_u32(&sdrop[i]), kScaleWarps);
    }
    for (int i = 0; i < SF; ++i) {
      mbar_init(smem_u32(&sfree[i]), 1);
      mbar_init(smem_u32(&sfull[i]), kScaleWarps);
    }
    for (int i = 0; i < kAcc; ++i) {
      mbar_init(smem_u32(&tfull[i]), 1);
      mbar_init(smem_u32(&tempty[i]), kEpiWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0) {
    int run = 0;
    for (int base = 0; base < E; base += 32) {
      const int e = base + lane;
      int u = 0;
      if (e < E) {
        // the segment offsets come from a kernel two launches back, complete by now (see
        // pdl_wait); read them from L2
        int lo = __ldcg(p.offsets + e), hi = __ldcg(p.offsets + e + 1);
        if (lo < 0) lo = 0;
        if (hi > p.a_rows) hi = (int)p.a_rows;
        const int m = hi > lo ? hi - lo : 0;
        u = ((m + TT - 1) / TT) * NB;
        seg_lo[e] = lo;
        seg_hi[e] = hi > lo ? hi : lo;
      }
      int inc = u;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, inc, o);
        if (lane >= o) inc += t;
      }
      if (e < E) cum[e] = run + inc - u;
      run += __shfl_sync(0xffffffffu, inc, 31);
    }
    if (lane == 0) cum[E] = run;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&s_tmem)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_before();
  __syncthreads();
  fence_after();
  // everything above overlapped the previous kernel's tail; the token rows and their scales
  // come from the previous kernel (the producer waits after it has sent the first weight tiles)
  if (!(warp == 0 && lane == 0)) {
    pdl_wait();
    pdl_trigger();
  }
  const uint32_t tmem_base = s_tmem;
  const int total_units = cum[E];
  const int u_begin = (int)blockIdx.x, u_step = (int)gridDim.x;

  auto decode = [&](int u, int& e, int& nb, int& row0, int& rows) {
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cum[mid] <= u) lo = mid; else hi = mid - 1;
    }
    e = lo;
    const int s0 = seg_lo[e], s1 = seg_hi[e];
    const int local = u - cum[e];
    const int tt = local / NB;
    nb = local - tt * NB;
    row0 = s0 + tt * TT;
    rows = min(TT, s1 - row0);
  };

  if (warp == 0) {
    // ------------------------------- TMA producer -------------------------------
    if (lane == 0) {
      const uint64_t pol_w = l2_policy_evict_first(), pol_a = l2_policy_evict_last();
      const int SP = KB / KBS;  // stages per unit (KBS divides a chunk, a chunk divides K)
      uint32_t it = 0, ci = 0;  // stages and scale chunks issued
      bool ok = true;
      // The weight codes and scales of the first stages go out before the wait for the
      // previous kernel; their token tiles (codes and scales) are held back until it is
      // complete. They are sent before anything would wait on a barrier that only their
      // arrival (through the MMA or the scale warps) can release: when every stage is in
      // flight, or before a scale slot is reused.
      bool waited = false;
      int pre_st[kMaxStages], pre_kb[kMaxStages], pre_row0[kMaxStages], pre_slot[kMaxStages];
      int npre = 0;
      auto flush_pre = [&]() {
        pdl_wait();
        pdl_trigger();
        waited = true;
        for (int i = 0; i < npre; ++i) {
          tma_load_3d_hint(smem_u32(tiles + (size_t)pre_st[i] * Z::kStage + Z::kOffA), &map_a,
                           smem_u32(&full[pre_st[i]]), 0, pre_row0[i], pre_kb[i], pol_a);
          if (pre_slot[i] >= 0)
            tma_load_3d_hint(smem_u32(sslots + (size_t)pre_slot[i] * Z::kSlot + Z::kSW), &map_sa,
                             smem_u32(&sland[pre_slot[i]]), 0, pre_row0[i], pre_kb[i] / kChunk, pol_a);
        }
        npre = 0;
      };
      for (int u = u_begin; u < total_units && ok && !s_abort; u += u_step) {
        int e, nb, row0, rows;
        decode(u, e, nb, row0, rows);
        for (int sp = 0; sp < SP; ++sp, ++it) {
          const int st = it % S;
          const int kb0 = sp * KBS;
          const bool opens = kb0 % kChunk == 0;  // the stage's first K block opens a scale chunk
          if (!waited && (npre == S || (opens && ci >= (uint32_t)kSmemSlots))) flush_pre();
          if (!mbar_wait(smem_u32(&empty[st]), ((it / S) & 1) ^ 1, &s_abort)) { ok = false; break; }
          int slot = -1;
          if (opens) {
            slot = (int)(ci % kSmemSlots);
            if (!mbar_wait(smem_u32(&sdrop[slot]), ((ci / kSmemSlots) & 1) ^ 1, &s_abort)) { ok = false; break; }
            const uint32_t sb = smem_u32(&sland[slot]);
            uint8_t* sl = sslots + (size_t)slot * Z::kSlot;
            mbar_expect_tx(sb, Z::kSW + Z::kSA);
            tma_load_4d_hint(smem_u32(sl), &map_sw, sb, 0, nb * kBM, kb0 / kChunk, e, pol_w);
            if (waited) tma_load_3d_hint(smem_u32(sl + Z::kSW), &map_sa, sb, 0, row0, kb0 / kChunk, pol_a);
            ++ci;
          }
          uint8_t* t0 = tiles + (size_t)st * Z::kStage;
          const uint32_t fb = smem_u32(&full[st]);
          mbar_expect_tx(fb, Z::kStage);
          tma_load_4d_hint(smem_u32(t0), &map_w, fb, 0, nb * kBM, kb0, e, pol_w);
          if (waited) {
            tma_load_3d_hint(smem_u32(t0 + Z::kOffA), &map_a, fb, 0, row0, kb0, pol_a);
          } else {
            pre_st[npre] = st;
            pre_kb[npre] = kb0;
            pre_row0[npre] = row0;
            pre_slot[npre] = slot;
            ++npre;
          }
        }
      }
      if (!waited) flush_pre();  // (also after an abort: every armed phase gets its bytes)
      // loads still in flight complete on their barriers: wait for the last phase issued on
      // each (bounded; the phase completes once its bytes land)
      for (int st = 0; st < S && (uint32_t)st < it; ++st) {
        const uint32_t last = it - 1 - ((it - 1 - st) % S);
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&full[st]), (last / S) & 1) && globaltimer() - t0 < kTimeoutNs) {
        }
      }
      for (int sl = 0; sl < kSmemSlots && (uint32_t)sl < ci; ++sl) {
        const uint32_t last = ci - 1 - ((ci - 1 - sl) % kSmemSlots);
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&sland[sl]), (last / kSmemSlots) & 1) && globaltimer() - t0 < kTimeoutNs) {
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------- MMA issuer --------------------------------
    if (lane == 0) {
      uint32_t it = 0, uc = 0, kc = 0;  // stages, units, K blocks consumed
      const int SP = KB / KBS;
      bool ok = true;
      for (int u = u_begin; u < total_units && ok && !s_abort; u += u_step, ++uc) {
        const uint32_t acc = uc % kAcc;
        if (!mbar_wait(smem_u32(&tempty[acc]), ((uc / kAcc) & 1) ^ 1, &s_abort)) { ok = false; break; }
        fence_after();
        const uint32_t d = tmem_base + acc * TT;
        for (int sp = 0; sp < SP && ok; ++sp, ++it) {
          const int st = it % S;
          if (!mbar_wait(smem_u32(&full[st]), (it / S) & 1, &s_abort)) { ok = false; break; }
          const uint32_t t0 = smem_u32(tiles + (size_t)st * Z::kStage);
          for (int h = 0; h < KBS; ++h, ++kc) {
            const int kb = sp * KBS + h;
            const uint32_t chunk = kc / kChunk, j = kc % kChunk;  // this CTA's chunk count
            const uint32_t slot = chunk % SF;
            if (j == 0) {
              if (!mbar_wait(smem_u32(&sfull[slot]), (chunk / SF) & 1, &s_abort)) { ok = false; break; }
              fence_after();
            }
            const uint32_t tw = t0 + h * Z::kW, ta = t0 + Z::kOffA + h * Z::kA;
            const uint32_t sfa = tmem_base + sf0 + 32u * slot + 4u * j;
            const uint32_t sfb = sfa + 16u;
#pragma unroll
            for (int s = 0; s < kBK / 32; ++s)
              mma_mx(d, smem_desc_sw128(tw + 32 * s), smem_desc_sw128(ta + 32 * s), idesc_mx(TT, (uint32_t)s), sfa, sfb,
                     (kb | s) != 0 ? 1u : 0u);
            if (j == kChunk - 1) mma_commit(smem_u32(&sfree[slot]));
          }
          if (!ok) break;
          mma_commit(smem_u32(&empty[st]));
        }
        if (!ok) break;
        mma_commit(smem_u32(&tfull[acc]));
      }
      // drain: the last commit of each accumulator and scale slot before the CTA may free TMEM
      for (uint32_t b = 0; b < (uint32_t)kAcc && b < uc; ++b) {
        const uint32_t last = uc - 1 - ((uc - 1 - b) % kAcc);
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&tfull[b]), (last / kAcc) & 1) && globaltimer() - t0 < kTimeoutNs) {
        }
      }
      const uint32_t nch = kc / kChunk;
      for (uint32_t sl = 0; sl < (uint32_t)SF && sl < nch; ++sl) {
        const uint32_t last = nch - 1 - ((nch - 1 - sl) % SF);
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&sfree[sl]), (last / SF) & 1) && globaltimer() - t0 < kTimeoutNs) {
        }
      }
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------- scale factors -> TMEM -------------------------
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    uint32_t ci = 0;
    bool ok = true;
    for (int u = u_begin; u < total_units && ok; u += u_step) {
      for (int c = 0; c < NC; ++c, ++ci) {
        const uint32_t ss = ci % kSmemSlots, ts = ci % SF;
        int got = mbar_wait(smem_u32(&sland[ss]), (ci / kSmemSlots) & 1, &s_abort) ? 1 : 0;
        if (got) got = mbar_wait(smem_u32(&sfree[ts]), ((ci / SF) & 1) ^ 1, &s_abort) ? 1 : 0;
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        fence_after();
        const uint8_t* sw_t = sslots + (size_t)ss * Z::kSlot;
        const uint8_t* sa_t = sw_t + Z::kSW;
        const uint32_t taddr = tmem_base + ((uint32_t)(32 * quarter) << 16) + sf0 + 32u * ts;
        // column 4j + c of lane l (every lane quarter): the four bytes of K block j for row l + 32c
        uint32_t r[16];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          const uint4 v = *reinterpret_cast<const uint4*>(sw_t + (lane + 32 * cc) * kSfRow);
          r[cc] = v.x;
          r[4 + cc] = v.y;
          r[8 + cc] = v.z;
          r[12 + cc] = v.w;
        }
        tmem_st16(taddr, r);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (lane + 32 * cc < TT) v = *reinterpret_cast<const uint4*>(sa_t + (lane + 32 * cc) * kSfRow);
          r[cc] = v.x;
          r[4 + cc] = v.y;
          r[8 + cc] = v.z;
          r[12 + cc] = v.w;
        }
        tmem_st16(taddr + 16u, r);
        tmem_st_wait();
        fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(smem_u32(&sfull[ts]));
          mbar_arrive(smem_u32(&sdrop[ss]));  // the shared-memory slot may be refilled
        }
      }
    }
  } else {
    // --------------------------------- epilogue ---------------------------------
    const int ew = warp - kEpiWarp0;   // 0..7
    const int half = ew >> 2;          // token-column half
    const int quarter = warp & 3;
    constexpr int HC = TT / 2;
    constexpr int CW = HC < 16 ? HC : 16;
    uint32_t uc = 0;
    for (int u = u_begin; u < total_units; u += u_step, ++uc) {
      int e, nb, row0, rows;
      decode(u, e, nb, row0, rows);
      const uint32_t acc = uc % kAcc;
      const int got = mbar_wait(smem_u32(&tfull[acc]), (uc / kAcc) & 1, &s_abort) ? 1 : 0;
      if (!__all_sync(0xffffffffu, got)) break;
      fence_after();
      const int n = nb * kBM + 32 * quarter + lane;
      const uint32_t taddr = tmem_base + ((uint32_t)(32 * quarter) << 16) + acc * TT + half * HC;
#pragma unroll
      for (int c0 = 0; c0 < HC; c0 += CW) {
        float d[16];
        if constexpr (CW == 8) {
          tmem_ld8(taddr + c0, d);
        } else {
          tmem_ld16(taddr + c0, d);
        }
        tmem_ld_wait();
        if (n < p.n) {
#pragma unroll
          for (int c = 0; c < CW; ++c) {
            const int r = half * HC + c0 + c;
            if (r < rows) p.out[(int64_t)(row0 + r) * p.ld_out + n] = d[c];
          }
        }
      }
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&tempty[acc]));
    }
  }

  fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem_base));
  }
}

}  // namespace mxg

template <int TT>
static cudaError_t launch_mx(const MxGemmArgs& a, cudaStream_t st, int* unsupported) {
  constexpr int KBS = mxg::kbs_for(TT);
  using Z = mxg::Sz<TT, KBS>;
  const int KB = (int)(a.k / 128), NB = (int)cdiv(a.n, 128);
  int dev = 0;
  cudaGetDevice(&dev);
  static size_t budget[64] = {};
  size_t max_smem = (dev >= 0 && dev < 64) ? budget[dev] : 0;
  if (max_smem == 0) {
    cudaFuncAttributes fattr;
    if (cudaFuncGetAttributes(&fattr, mxg::mxfp8_gemm_kernel<TT, KBS>) != cudaSuccess) return cudaErrorInvalidValue;
    int optin = 0;
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    max_smem = (size_t)optin > fattr.sharedSizeBytes ? (size_t)optin - fattr.sharedSizeBytes : 0;
    if (dev >= 0 && dev < 64) budget[dev] = max_smem;
  }
  // TMEM: the accumulators, then 32 scale columns per scale slot, within 512 columns
  const int sf_free = (512 - (mxg::kAcc * TT + 31) / 32 * 32) / 32;
  const int sf_slots = sf_free < mxg::kMaxSfSlots ? sf_free : mxg::kMaxSfSlots;
  const size_t fixed = 1024 + (size_t)mxg::kSmemSlots * Z::kSlot + (size_t)(3 * a.E + 2) * 4 + 8 +
                       (size_t)(2 * mxg::kSmemSlots + 2 * sf_slots + 2 * mxg::kAcc) * 8;
  int stages = mxg::kMaxStages;
  while (stages > 2 && fixed + (size_t)stages * Z::kStage + (size_t)(2 * stages) * 8 > max_smem) --stages;
  const size_t smem = fixed + (size_t)stages * Z::kStage + (size_t)(2 * stages) * 8;
  if (smem > max_smem || stages < 2 || sf_slots < 2) {
    *unsupported = 1;
    return cudaSuccess;
  }
  // codes as (128-byte chunk, row, K block[, expert]) with the 128-byte swizzle; scales as
  // (16-byte chunk, row, scale chunk[, expert]) unswizzled
  CUtensorMap mw, ma, msw, msa;
  const uint64_t kk = (uint64_t)a.k, ks = (uint64_t)(a.k / 32);
  {
    const uint64_t d[4] = {128, (uint64_t)a.n, (uint64_t)KB, (uint64_t)a.E};
    const uint64_t sd[3] = {kk, 128, kk * (uint64_t)a.n};
    const uint32_t bx[4] = {128, (uint32_t)mxg::kBM, (uint32_t)KBS, 1};
    if (!encode_u8_tmap(&mw, a.w_q, 4, d, sd, bx)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t d[3] = {128, (uint64_t)a.a_rows, (uint64_t)KB};
    const uint64_t sd[2] = {kk, 128};
    const uint32_t bx[3] = {128, (uint32_t)TT, (uint32_t)KBS};
    if (!encode_u8_tmap(&ma, a.a_q, 3, d, sd, bx)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t d[4] = {16, (uint64_t)a.n, (uint64_t)(KB / mxg::kChunk), (uint64_t)a.E};
    const uint64_t sd[3] = {ks, 16, ks * (uint64_t)a.n};
    const uint32_t bx[4] = {16, (uint32_t)mxg::kBM, 1, 1};
    if (!encode_u8_tmap_plain(&msw, a.w_sf, 4, d, sd, bx)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t d[3] = {16, (uint64_t)a.a_rows, (uint64_t)(KB / mxg::kChunk)};
    const uint64_t sd[2] = {ks, 16};
    const uint32_t bx[3] = {16, (uint32_t)TT, 1};
    if (!encode_u8_tmap_plain(&msa, a.a_sf, 3, d, sd, bx)) return cudaErrorInvalidValue;
  }
  mxg::Params p;
  p.offsets = a.offsets;
  p.out = a.out;
  p.ld_out = a.ld_out;
  p.a_rows = a.a_rows;
  p.n = (int)a.n;
  p.E = a.E;
  p.kb_count = KB;
  p.nb_count = NB;
  p.stages = stages;
  p.sf_slots = sf_slots;
  static size_t granted[64] = {};
  if (dev < 0 || dev >= 64 || smem > granted[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(mxg::mxfp8_gemm_kernel<TT, KBS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) granted[dev] = smem;
  }
  return launch_kernel(mxg::mxfp8_gemm_kernel<TT, KBS>, dim3(sm_count()), dim3(mxg::kThreads), smem, st, true, mw, ma,
                       msw, msa, p);
}

cudaError_t launch_mxfp8_gemm(const MxGemmArgs& a, cudaStream_t st, int* unsupported) {
  *unsupported = 0;
  // K in whole chunks of 512 elements (a scale row of k/32 bytes moves in 16-byte boxes);
  // TMA needs 16-byte aligned bases
  if (a.k % 512 != 0 || a.k <= 0 || (uintptr_t)a.w_q % 16 != 0 || (uintptr_t)a.a_q % 16 != 0 ||
      (uintptr_t)a.w_sf % 16 != 0 || (uintptr_t)a.a_sf % 16 != 0 || a.E > mxg::kMaxExperts || a.n > (1 << 30) ||
      a.a_rows > (1 << 30)) {
    *unsupported = 1;
    return cudaSuccess;
  }
  switch (a.tok_tile) {
    case 16: return launch_mx<16>(a, st, unsupported);
    case 32: return launch_mx<32>(a, st, unsupported);
    case 64: return launch_mx<64>(a, st, unsupported);
    case 128: return launch_mx<128>(a, st, unsupported);
    default: *unsupported = 1; return cudaSuccess;
  }
}

FTMOE_DEFINE_ERR_READER(read_err_tc_mxfp8)

}  // namespace ftmoe

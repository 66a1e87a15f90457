// Grouped NVFP4 GEMM on the block-scaled tensor-core MMA (tcgen05 kind::mxf4nvf4).
//
// out[row, n] = g_a * g_w[e] * sum_k (a[row,k] * sa[row, k/16]) * (w[e,n,k] * sw[e,n,k/16])
// with e2m1 codes a, w (two per byte, even element in the low nibble), e4m3 block scales
// sa, sw (one per 16 elements) and fp32 tensor scales g_a, g_w[e] -- the NVFP4 variant of
// the prefill GEMM. The dsfp4 page names the format only; the two-level recipe used here is
// g = amax_tensor / (448 * 6) per tensor, one e4m3 scale sb = e4m3(amax_16 / (6 g)) per 16
// consecutive elements of a row, and e2m1 codes of x / (sb * g), rounded to nearest even.
// Unlike the FP8 path, the block scales are native to the MMA
// (tcgen05.mma ... kind::mxf4nvf4.block_scale.scale_vec::4X, K = 64 per instruction, one
// ue4m3 scale per 16 elements of each row), so a unit accumulates all of K in TMEM and the
// epilogue only applies g_a * g_w once.
//
// Work layout as in the FP8 kernel: MMA M = 128 weight rows, MMA N = the token tile; one
// persistent CTA per SM; CTA c takes units c, c + G, ... of the (expert, token tile, weight
// block) list.
// Roles: warp 0 TMA producer (code tiles with the 128-byte swizzle, scale tiles plain);
// warp 1 MMA issuer and TMEM owner; warps 2-5 move each stage's scale factors from shared
// memory into TMEM, warps 6-13 epilogue. Every wait is bounded.
//
// Scale factors in TMEM, per operand and MMA step (K = 64, four e4m3 scales per row): four
// 32-bit columns; column c of lane l holds the four scales of row l + 32c, and every lane
// quarter holds the same copy (each sub-partition reads the scales it needs from its own
// quarter). This is the 128x4 block-scale chunk layout (32 rows of 16 bytes) replicated
// into the four quarters.
#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace ftmoe {

namespace nv {

constexpr int kBM = 128;           // weight rows per tile (MMA M)
constexpr int kBKB = 128;          // code bytes per row per stage = 256 elements
constexpr int kSfPerStage = 16;    // scale bytes per row per stage
constexpr int kScaleWarp0 = 2, kScaleWarps = 4;
constexpr int kEpiWarp0 = kScaleWarp0 + kScaleWarps, kEpiWarps = 8;
constexpr int kThreads = 32 * (kEpiWarp0 + kEpiWarps);  // 448
constexpr int kMaxExperts = 1024;
constexpr int kAcc = 2;            // accumulators: the next unit's MMAs run during this unit's epilogue
constexpr int kMaxStages = 8;
constexpr int kMaxSfSlots = 8;     // TMEM scale slots (32 columns each, one K block)
// K blocks (256 elements) per shared-memory stage: one TMA box per operand brings all of them
// (the tensor maps carry the K-block index as a dimension), because each TMA instruction
// costs the SM a fixed time; two at token tile 128, where a stage is largest.
__host__ __device__ constexpr int kbs_for(int tt) { return tt <= 64 ? 4 : 2; }

// One stage: weight codes [KBS][128 rows][128 B] (each K block a canonical 128-byte-swizzled
// sub-tile), token codes [KBS][TT][128 B], weight scales [KBS][128][16 B], token scales
// [KBS][TT][16 B].
template <int TT, int KBS>
struct Sz {
  static constexpr int kW = kBM * kBKB;             // 16 KiB of weight codes per K block
  static constexpr int kA = TT * kBKB;              // token codes per K block
  static constexpr int kSW = kBM * kSfPerStage;     // weight scales per K block
  static constexpr int kSA = TT * kSfPerStage;      // token scales per K block
  static constexpr int kOffA = KBS * kW;
  static constexpr int kOffSW = kOffA + KBS * kA;
  static constexpr int kOffSA = kOffSW + KBS * kSW;
  static constexpr int kBytes = kOffSA + KBS * kSA;
  static constexpr int kStage = (kBytes + 1023) / 1024 * 1024;
};

// Instruction descriptor of kind::mxf4nvf4: A = B = E2M1, ue4m3 scale factors, both
// operands K-major, M = 128, N = n, K = 64, scale-factor ids 0 (all four scales of a
// 32-bit column are used by scale_vec::4X).
__host__ __device__ constexpr uint32_t idesc_nvf4(int n) {
  return (1u << 7)                          // A format: E2M1
         | (1u << 10)                       // B format: E2M1
         | ((uint32_t)(n >> 3) << 17)       // N >> 3
         | (0u << 23)                       // scale format: UE4M3
         | ((uint32_t)(kBM >> 4) << 24);    // M >> 4
}

__device__ __forceinline__ void mma_nvf4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(acc)
      : "memory");
}

struct Params {
  const int32_t* offsets;
  const float* g_a;   // [1]
  const float* g_w;   // [E]
  float* out;
  int64_t ld_out;
  int64_t a_rows;
  int n, E, kb_count, nb_count, stages, sf_slots;
};

template <int TT, int KBS>
__global__ void __launch_bounds__(kThreads, 1)
    nvfp4_gemm_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_a,
                      const __grid_constant__ CUtensorMap map_sw, const __grid_constant__ CUtensorMap map_sa,
                      Params p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int S = p.stages, SF = p.sf_slots;
  uint8_t* tiles = smem;
  int* cum = reinterpret_cast<int*>(smem + (size_t)S * Sz<TT, KBS>::kStage);  // [E+2] unit prefix
  int* seg_lo = cum + p.E + 2;                                            // [E] rows [seg_lo, seg_hi)
  int* seg_hi = seg_lo + p.E;
  uint64_t* bars = reinterpret_cast<uint64_t*>(((reinterpret_cast<uintptr_t>(seg_hi + p.E)) + 7) & ~(uintptr_t)7);
  uint64_t* full = bars;            // TMA landed (codes and scales of the stage's K blocks)
  uint64_t* empty = bars + S;       // MMAs done reading the stage (for the producer)
  uint64_t* sfree = bars + 2 * S;   // [SF] MMAs done reading a TMEM scale slot (for the scale warps)
  uint64_t* sfull = sfree + SF;     // [SF] scale factors of one K block in TMEM
  uint64_t* tfull = sfull + SF;
  uint64_t* tempty = tfull + kAcc;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E, NB = p.nb_count, KB = p.kb_count;
  // TMEM columns: accumulators [0, kAcc*TT), then 32 scale columns per TMEM scale slot
  // (16 for the weight rows, 16 for the token rows)
  const uint32_t sf0 = (uint32_t)((kAcc * TT + 31) / 32 * 32);

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < S; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
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
        seg_lo[e] = lo;  // kept in shared memory: no global load at unit boundaries
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
  // everything above overlapped the previous kernel's tail; the token rows and their
  // scales come from the previous kernel (the producer thread waits after it has sent the
  // first weight tiles, which do not depend on it)
  if (!(warp == 0 && lane == 0)) {
    pdl_wait();
    pdl_trigger();
  }
  const uint32_t tmem_base = s_tmem;
  const int total_units = cum[E];
  // units c, c + G, ...: the CTAs sweep the (expert, token tile, weight block) list together,
  // so a token tile is read by several CTAs at about the same time and stays in L2
  const int u_begin = (int)blockIdx.x, u_end = total_units, u_step = (int)gridDim.x;

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
      // weight tiles are read once; the token tile is read again by every weight block
      const uint64_t pol_w = l2_policy_evict_first(), pol_a = l2_policy_evict_last();
      uint32_t it = 0;
      const int SP = (KB + KBS - 1) / KBS;  // stages per unit
      int u = u_begin, sp = 0, e = 0, nb = 0, row0 = 0, rows = 0;
      if (u < u_end) decode(u, e, nb, row0, rows);
      auto advance = [&]() {
        if (++sp == SP) {
          sp = 0;
          if ((u += u_step) < u_end) decode(u, e, nb, row0, rows);
        }
      };
      // one box per operand and stage: K blocks [sp * KBS, sp * KBS + KBS)
      auto load_w = [&](uint8_t* t0, uint32_t fb) {
        tma_load_4d_hint(smem_u32(t0), &map_w, fb, 0, nb * kBM, sp * KBS, e, pol_w);
        tma_load_4d_hint(smem_u32(t0 + Sz<TT, KBS>::kOffSW), &map_sw, fb, 0, nb * kBM, sp * KBS, e, pol_w);
      };
      auto load_a = [&](uint8_t* t0, uint32_t fb, int s_sp, int s_row0) {
        tma_load_3d_hint(smem_u32(t0 + Sz<TT, KBS>::kOffA), &map_a, fb, 0, s_row0, s_sp * KBS, pol_a);
        tma_load_3d_hint(smem_u32(t0 + Sz<TT, KBS>::kOffSA), &map_sa, fb, 0, s_row0, s_sp * KBS, pol_a);
      };
      // The weight tiles (codes and scales) of the first pass over the ring go out before
      // the wait: they do not depend on the previous kernel. The token tiles follow.
      int pre_sp[kMaxStages], pre_row0[kMaxStages];
      int npre = 0;
      while (npre < S && u < u_end) {
        uint8_t* t0 = tiles + (size_t)npre * Sz<TT, KBS>::kStage;
        const uint32_t fb = smem_u32(&full[npre]);
        mbar_expect_tx(fb, Sz<TT, KBS>::kBytes);
        load_w(t0, fb);
        pre_sp[npre] = sp;
        pre_row0[npre] = row0;
        ++npre;
        ++it;
        advance();
      }
      pdl_wait();
      pdl_trigger();
      for (int i = 0; i < npre; ++i)
        load_a(tiles + (size_t)i * Sz<TT, KBS>::kStage, smem_u32(&full[i]), pre_sp[i], pre_row0[i]);
      while (u < u_end && !s_abort) {
        const int st = it % S;
        if (!mbar_wait(smem_u32(&empty[st]), ((it / S) & 1) ^ 1, &s_abort)) break;
        uint8_t* t0 = tiles + (size_t)st * Sz<TT, KBS>::kStage;
        const uint32_t fb = smem_u32(&full[st]);
        mbar_expect_tx(fb, Sz<TT, KBS>::kBytes);
        load_w(t0, fb);
        load_a(t0, fb, sp, row0);
        ++it;
        advance();
      }
      const uint32_t issued = it;
      for (int st = 0; st < S && (uint32_t)st < issued; ++st) {
        const uint32_t last = issued - 1 - ((issued - 1 - st) % S);
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&full[st]), (last / S) & 1) && globaltimer() - t0 < kTimeoutNs) {
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------- MMA issuer --------------------------------
    if (lane == 0) {
      uint32_t it = 0, uc = 0, kc = 0;
      constexpr uint32_t idesc = idesc_nvf4(TT);
      const int SP = (KB + KBS - 1) / KBS;
      bool ok = true;
      for (int u = u_begin; u < u_end && ok && !s_abort; u += u_step, ++uc) {
        const uint32_t acc = uc % kAcc;
        if (!mbar_wait(smem_u32(&tempty[acc]), ((uc / kAcc) & 1) ^ 1, &s_abort)) { ok = false; break; }
        fence_after();
        const uint32_t d = tmem_base + acc * TT;
        for (int sp = 0; sp < SP && ok; ++sp, ++it) {
          const int st = it % S;
          if (!mbar_wait(smem_u32(&full[st]), (it / S) & 1, &s_abort)) { ok = false; break; }
          const uint32_t t0 = smem_u32(tiles + (size_t)st * Sz<TT, KBS>::kStage);
          for (int h = 0; h < KBS && sp * KBS + h < KB; ++h, ++kc) {
            const uint32_t slot = kc % SF;
            if (!mbar_wait(smem_u32(&sfull[slot]), (kc / SF) & 1, &s_abort)) { ok = false; break; }
            fence_after();
            const uint32_t tw = t0 + h * Sz<TT, KBS>::kW, ta = t0 + Sz<TT, KBS>::kOffA + h * Sz<TT, KBS>::kA;
            const uint32_t sfa = tmem_base + sf0 + 32u * slot;
            const uint32_t sfb = sfa + 16u;
            const int kb = sp * KBS + h;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              mma_nvf4(d, smem_desc_sw128(tw + 32 * j), smem_desc_sw128(ta + 32 * j), idesc, sfa + 4 * j, sfb + 4 * j,
                       (kb | j) != 0 ? 1u : 0u);
            mma_commit(smem_u32(&sfree[slot]));
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
      for (uint32_t sl = 0; sl < (uint32_t)SF && sl < kc; ++sl) {
        const uint32_t last = kc - 1 - ((kc - 1 - sl) % SF);
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&sfree[sl]), (last / SF) & 1) && globaltimer() - t0 < kTimeoutNs) {
        }
      }
    }
  } else if (warp < kEpiWarp0) {
    // ------------------------- scale factors -> TMEM -------------------------
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int SP = (KB + KBS - 1) / KBS;
    uint32_t it = 0, kc = 0;
    for (int u = u_begin; u < u_end; u += u_step) {
      bool ok = true;
      for (int sp = 0; sp < SP && ok; ++sp, ++it) {
        const int st = it % S;
        for (int h = 0; h < KBS && sp * KBS + h < KB; ++h, ++kc) {
        const uint32_t slot = kc % SF;
        int got = mbar_wait(smem_u32(&full[st]), (it / S) & 1, &s_abort) ? 1 : 0;
        if (got) got = mbar_wait(smem_u32(&sfree[slot]), ((kc / SF) & 1) ^ 1, &s_abort) ? 1 : 0;
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        fence_after();
        const uint8_t* t0 = tiles + (size_t)st * Sz<TT, KBS>::kStage;
        const uint8_t* sw_t = t0 + Sz<TT, KBS>::kOffSW + h * Sz<TT, KBS>::kSW;
        const uint8_t* sa_t = t0 + Sz<TT, KBS>::kOffSA + h * Sz<TT, KBS>::kSA;
        const uint32_t taddr = tmem_base + ((uint32_t)(32 * quarter) << 16) + sf0 + 32u * slot;
        // column 4j + c of lane l (in every lane quarter): the four scales of MMA step j
        // for row l + 32c
        uint32_t r[16];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(sw_t + (lane + 32 * c) * kSfPerStage);
          r[c] = v.x;
          r[4 + c] = v.y;
          r[8 + c] = v.z;
          r[12 + c] = v.w;
        }
        tmem_st16(taddr, r);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (lane + 32 * c < TT) v = *reinterpret_cast<const uint4*>(sa_t + (lane + 32 * c) * kSfPerStage);
          r[c] = v.x;
          r[4 + c] = v.y;
          r[8 + c] = v.z;
          r[12 + c] = v.w;
        }
        tmem_st16(taddr + 16u, r);
        tmem_st_wait();
        fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sfull[slot]));
        }
      }
      if (!ok) break;
    }
  } else {
    // --------------------------------- epilogue ---------------------------------
    const int ew = warp - kEpiWarp0;   // 0..7
    const int half = ew >> 2;          // token-column half
    const int quarter = warp & 3;
    constexpr int HC = TT / 2;
    uint32_t uc = 0;
    for (int u = u_begin; u < u_end; u += u_step, ++uc) {
      int e, nb, row0, rows;
      decode(u, e, nb, row0, rows);
      const float f = __ldg(p.g_a) * __ldg(p.g_w + e);
      const uint32_t acc = uc % kAcc;
      const int got = mbar_wait(smem_u32(&tfull[acc]), (uc / kAcc) & 1, &s_abort) ? 1 : 0;
      if (!__all_sync(0xffffffffu, got)) break;
      fence_after();
      const int n = nb * kBM + 32 * quarter + lane;
      const uint32_t taddr = tmem_base + ((uint32_t)(32 * quarter) << 16) + acc * TT + half * HC;
#pragma unroll
      for (int c0 = 0; c0 < HC; c0 += (HC < 16 ? HC : 16)) {
        float d[16];
        if constexpr (HC == 8) {
          tmem_ld8(taddr + c0, d);
        } else {
          tmem_ld16(taddr + c0, d);
        }
        tmem_ld_wait();
        if (n < p.n) {
#pragma unroll
          for (int c = 0; c < (HC < 16 ? HC : 16); ++c) {
            const int r = half * HC + c0 + c;
            if (r < rows) p.out[(int64_t)(row0 + r) * p.ld_out + n] = d[c] * f;
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

}  // namespace nv

template <int TT>
static cudaError_t launch_nv(const NvGemmArgs& a, cudaStream_t st, int* unsupported) {
  constexpr int KBS = nv::kbs_for(TT);
  using Z = nv::Sz<TT, KBS>;
  const int KB = (int)(a.k / 256), NB = (int)cdiv(a.n, 128);
  int dev = 0;
  cudaGetDevice(&dev);
  static size_t budget[64] = {};
  size_t max_smem = (dev >= 0 && dev < 64) ? budget[dev] : 0;
  if (max_smem == 0) {
    cudaFuncAttributes fattr;
    if (cudaFuncGetAttributes(&fattr, nv::nvfp4_gemm_kernel<TT, KBS>) != cudaSuccess) return cudaErrorInvalidValue;
    int optin = 0;
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    max_smem = (size_t)optin > fattr.sharedSizeBytes ? (size_t)optin - fattr.sharedSizeBytes : 0;
    if (dev >= 0 && dev < 64) budget[dev] = max_smem;
  }
  // TMEM: the accumulators, then 32 scale columns per scale slot, within 512 columns
  const int sf_free = (512 - (nv::kAcc * TT + 31) / 32 * 32) / 32;
  const int sf_slots = sf_free < nv::kMaxSfSlots ? sf_free : nv::kMaxSfSlots;
  const size_t fixed = 1024 + (size_t)(3 * a.E + 2) * 4 + 8 + (size_t)(2 * sf_slots + 2 * nv::kAcc) * 8;
  int stages = nv::kMaxStages;
  while (stages > 2 && fixed + (size_t)stages * Z::kStage + (size_t)(2 * stages) * 8 > max_smem) --stages;
  const size_t smem = fixed + (size_t)stages * Z::kStage + (size_t)(2 * stages) * 8;
  if (smem > max_smem || stages < 2 || sf_slots < 2) {
    *unsupported = 1;
    return cudaSuccess;
  }
  // codes as (128-byte chunk, row, K block[, expert]) and scales as (16-byte chunk, row,
  // K block[, expert]): one box per operand holds KBS K blocks of 256 elements
  CUtensorMap mw, ma, msw, msa;
  const uint64_t kc = (uint64_t)(a.k / 2), ks = (uint64_t)(a.k / 16);
  {
    const uint64_t d[4] = {128, (uint64_t)a.n, (uint64_t)KB, (uint64_t)a.E};
    const uint64_t sd[3] = {kc, 128, kc * (uint64_t)a.n};
    const uint32_t bx[4] = {128, (uint32_t)nv::kBM, (uint32_t)KBS, 1};
    if (!encode_u8_tmap(&mw, a.w_q, 4, d, sd, bx)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t d[3] = {128, (uint64_t)a.a_rows, (uint64_t)KB};
    const uint64_t sd[2] = {kc, 128};
    const uint32_t bx[3] = {128, (uint32_t)TT, (uint32_t)KBS};
    if (!encode_u8_tmap(&ma, a.a_q, 3, d, sd, bx)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t d[4] = {16, (uint64_t)a.n, (uint64_t)KB, (uint64_t)a.E};
    const uint64_t sd[3] = {ks, 16, ks * (uint64_t)a.n};
    const uint32_t bx[4] = {16, (uint32_t)nv::kBM, (uint32_t)KBS, 1};
    if (!encode_u8_tmap_plain(&msw, a.w_sf, 4, d, sd, bx)) return cudaErrorInvalidValue;
  }
  {
    const uint64_t d[3] = {16, (uint64_t)a.a_rows, (uint64_t)KB};
    const uint64_t sd[2] = {ks, 16};
    const uint32_t bx[3] = {16, (uint32_t)TT, (uint32_t)KBS};
    if (!encode_u8_tmap_plain(&msa, a.a_sf, 3, d, sd, bx)) return cudaErrorInvalidValue;
  }
  nv::Params p;
  p.offsets = a.offsets;
  p.g_a = a.a_gscale;
  p.g_w = a.w_gscale;
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
        cudaFuncSetAttribute(nv::nvfp4_gemm_kernel<TT, KBS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) granted[dev] = smem;
  }
  return launch_kernel(nv::nvfp4_gemm_kernel<TT, KBS>, dim3(sm_count()), dim3(nv::kThreads), smem, st, true, mw, ma,
                       msw, msa, p);
}

cudaError_t launch_nvfp4_gemm(const NvGemmArgs& a, cudaStream_t st, int* unsupported) {
  *unsupported = 0;
  // TMA: code rows of k/2 bytes and scale rows of k/16 bytes must be 16-byte multiples
  if (a.k % 256 != 0 || (uintptr_t)a.w_q % 16 != 0 || (uintptr_t)a.a_q % 16 != 0 || (uintptr_t)a.w_sf % 16 != 0 ||
      (uintptr_t)a.a_sf % 16 != 0 || a.E > nv::kMaxExperts || a.n > (1 << 30) || a.a_rows > (1 << 30)) {
    *unsupported = 1;
    return cudaSuccess;
  }
  switch (a.tok_tile) {
    case 16: return launch_nv<16>(a, st, unsupported);
    case 32: return launch_nv<32>(a, st, unsupported);
    case 64: return launch_nv<64>(a, st, unsupported);
    case 128: return launch_nv<128>(a, st, unsupported);
    default: *unsupported = 1; return cudaSuccess;
  }
}

FTMOE_DEFINE_ERR_READER(read_err_nvfp4)

}  // namespace ftmoe

// Grouped block-FP8 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// out[row, n] = sum_kb  s_a[row, kb] * s_w[e, n/128, kb] * sum_{k in kb} a[row, k] * w[e, n, k]
// for the rows of each expert's segment (rows sorted by expert, offsets[e]..offsets[e+1]).
// The 128x128 fp32 weight block scales and 1x128 activation scales are arbitrary fp32
// numbers, which the block-scaled MMA kinds (power-of-two or e4m3 scales per 16/32
// elements) cannot express; so, as the FreeToken block-FP8 page and the SGLang CUTLASS
// path do with their block scales, each 128-wide K block is accumulated separately and
// then rescaled on CUDA cores.
//
// Layout of the work ("swap AB"): the MMA's M = 128 rows are 128 weight rows (one
// weight-scale block row), the MMA's N is the token tile (16/32/64/128 rows of one
// expert, picked from rows per expert because padding is not free -- FreeToken
// "perf(dsfp4): pick the grouped-prefill tile from route density on sm_89").
// A unit is (expert, token tile, one or two weight blocks); with two blocks the token tile
// is shared (see Mode), and the gate/up pairing lets the epilogue apply SiLU-and-mul and the
// FP8 re-quantization of the intermediate. Per 128-wide K block and weight block:
// 4 x tcgen05.mma kind::f8f6f4 (K = 32 each) into a fresh TMEM accumulator; the epilogue
// warps tcgen05.ld it and add d * (s_a[column] * s_w) into fp32 registers, the scale
// products formed once per chunk of K blocks. Up to sixteen TMEM accumulators (512 columns
// at most) rotate so the MMA runs ahead of the promotion.
//
// One persistent CTA per SM; CTA c takes units c, c + G, c + 2G, ... (G CTAs) of the list
// ordered (expert, token tile, weight block), weight blocks innermost. At any moment the CTAs
// work on G consecutive units, a few experts' token tiles, which L2 serves to the CTAs that
// read them at about the same time; every weight tile is read once. (Contiguous ranges per
// CTA kept one token tile per CTA live for its whole run: at token tile 128 and K = 7168 that
// is 152 tiles of 0.9 MB, more than L2 holds, and the re-reads went to DRAM.) The
// weight-scale rows of the next unit and the next chunk of activation scales are fetched
// while the current ones are in use. Roles: warp 0 = TMA producer, warp 1 = MMA
// issuer (and TMEM owner), the last 16 warps = epilogue (four groups of four warps, one
// group per quarter of the token columns; warp w reads TMEM lanes 32*(w%4) .. +31). Every
// mbarrier wait is bounded: on timeout the kernel raises FTMOE_ERR_WAIT_TIMEOUT, stops all
// roles, waits for its own TMA loads still in flight, frees its TMEM and returns.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace ftmoe {

namespace tc {

constexpr int kBM = 128;               // weight rows per tile (MMA M)
constexpr int kBK = 128;               // K bytes per K block = one scale block
constexpr int kMaxExperts = 1024;

// What one unit of work covers, besides its token tile:
//   kSingle     one 128-row weight block; fp32 output columns [128 nb, 128 nb + 128)
//   kPair       two adjacent weight blocks 2p, 2p + 1 that share the token tile; fp32 output
//   kGateUpSilu gate block j (rows 128 j ..) and up block j (rows I + 128 j ..) of a gate/up
//               matrix; the epilogue forms silu(g) * u for intermediate columns
//               [128 j, 128 j + 128) -- exactly one 1x128 group -- and re-quantizes it to FP8
//               with its group scale, so no fp32 gate/up row is ever written
//   kCtaPair    weight blocks 2p and 2p + 1 on the two CTAs of a cluster (two SMs): CTA r
//               streams block 2p + r and loads half of the token tile (rows r TT/2 ..); the
//               first CTA issues tcgen05.mma.cta_group::2 with M = 256, which reads the
//               weights and the token halves of both CTAs and leaves each CTA the fp32
//               accumulator of its own block over all TT token columns
//   kCtaPairComb  kCtaPair for the down GEMM of the forward, with the routing-weighted
//               combine inside: four more warps publish each unit's fp32 rows, count the
//               arrivals per (token, weight block) and, for a token whose last route arrived,
//               add its rows in ascending slot order into the output (see "Fused combine")
// Two weight blocks per token tile halve the token bytes each stage carries for every
// weight byte, so more weight bytes fit in flight in the same shared memory. kPair does it
// on one SM (twice the epilogue work per K block); kCtaPair across two, with the epilogue
// work of one block per SM.
enum Mode { kSingle = 0, kPair = 1, kGateUpSilu = 2, kCtaPair = 3, kCtaPairComb = 4 };
__host__ __device__ constexpr int wb_of(int mode) { return mode == kPair || mode == kGateUpSilu ? 2 : 1; }
__host__ __device__ constexpr bool is_cp(int mode) { return mode == kCtaPair || mode == kCtaPairComb; }

// TMEM accumulators in rotation: as many (weight blocks x TT)-column accumulators as 512
// columns hold, at most 16, so the MMA can run that many K blocks ahead of the promotion
__host__ __device__ constexpr int acc_count(int cols) { return 512 / cols > 16 ? 16 : 512 / cols; }

// Instruction descriptor, kind::f8f6f4: D fp32, A = B = e4m3, both K-major, M = m, N = n.
__host__ __device__ constexpr uint32_t idesc_f8(int n, int m = kBM) {
  return (1u << 4)                      // D format f32
         | (0u << 7) | (0u << 10)       // A, B format e4m3
         | ((uint32_t)(n >> 3) << 17)   // N >> 3
         | ((uint32_t)(m >> 4) << 24);  // M >> 4
}

__device__ __forceinline__ void mma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}

// CTA pair: one MMA over both CTAs' operands (M = 256, each CTA 128 weight rows and half of
// the N token rows); each CTA's TMEM receives its own 128 rows of D
__device__ __forceinline__ void mma_f8_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc)
      : "memory");
}

struct Params {
  const int32_t* offsets;
  const float* a_s;   // [a_rows][kb_count]
  const float* w_s;   // [E][nb_count][kb_count]
  float* out;         // kSingle, kPair: [a_rows][ld_out]
  int64_t ld_out;
  uint8_t* q_out;     // kGateUpSilu: FP8 codes [a_rows][n / 2]
  float* s_out;       // kGateUpSilu: group scales [a_rows][n / 256]
  int64_t a_rows;
  int n, k, E, kb_count, nb_count, stages;
  // kCtaPairComb: the combine out_c[t, :] = round(sum_j rw[t*topk + j] * out[route2dst[t*topk + j], :])
  const int32_t* dst2src;    // grouped row -> token
  const int32_t* route2dst;  // route -> grouped row, -1 for a route without one
  const float* rw;           // routing weights [tokens][topk]
  uint32_t* cnt;             // [tokens][nb_count] arrival counters, zero at launch
  void* out_c;               // [tokens][ld_c] elements of out_dtype
  int64_t ld_c;
  int topk, out_dtype;
};

constexpr int kEpiWarps = 16;                    // 4 column groups x 4 TMEM lane quarters
constexpr int kGroups = kEpiWarps / 4;
constexpr int kMaxKB = 128;                      // K <= 16384
constexpr int kMaxStages = 12;
constexpr int kSaChunk = 8;                      // K blocks of activation scales staged at once
constexpr int kYRing = 4;                        // fused combine: units in flight between the roles
constexpr int kCombK = 8;                        // fused combine: slots a token's last arrival stages

// K blocks per pipeline stage (KBS). One TMA box brings all of them: the tensor maps carry
// the K-block index as a dimension of its own, and each K block lands as its own canonical
// 128-byte-swizzled sub-tile (1024-byte aligned), exactly as in a one-block stage. Each TMA
// instruction costs the SM a fixed time, so fewer, larger boxes move more bytes per SM: four
// K blocks per box up to token tile 64, two at 128 (two or three stages still fit); with two
// weight blocks per unit a box already carries twice the weight bytes per K block. A CTA pair
// at token tile 128 carries four (two stages of 96 KiB): measured on GB300 at 24,576 routes,
// gate/up took 1478 us with four, 1556 us with two and 1711 us with one. A K that is not a
// multiple of 128 keeps one K block per stage and the per-row maps, whose x extent is K
// itself, so the partial last block is zero-filled rather than read past the row.
__host__ __device__ constexpr int kbs_for(int tt, int mode) {
  return mode == kSingle ? (tt <= 64 ? 4 : 2) : (is_cp(mode) ? 4 : (tt <= 32 ? 2 : 1));
}

// Warp roles. Warp 0 issues TMA, warp 1 issues MMAs, the last kEpiWarps warps promote.
// Units with two weight blocks from token tile 64 on hold 2 x TT/4 fp32 accumulators (32
// or 64) per epilogue thread. Those kernels add two idle warps, so that warps 0-3 form a
// warpgroup that gives registers back (setmaxnreg.dec to kCtlRegs) to the four epilogue
// warpgroups (setmaxnreg.inc to kEpiRegs). The launch pool is threads x the kernel's
// register count; the host checks the warpgroups' shares (W::kRegsNeeded) against it
// before launching, since an increase the pool cannot cover would never complete.
// The fused-combine kernel (kCtaPairComb) has a second control warpgroup, the four combine
// warps, and splits registers the same way: 768 threads launch with 80 registers each; both
// control warpgroups keep 64, the epilogue takes 88 (its 32 accumulators and 16 TMEM
// columns in flight fit without spilling).
template <int TT, int MODE>
struct Warps {
  static constexpr bool kComb = MODE == kCtaPairComb;
  static constexpr bool kSplitRegs = (TT >= 64 && wb_of(MODE) == 2) || kComb;
  static constexpr int kCtl = kComb ? 8 : 4;  // TMA, MMA, scale-product tables, one idle warp (+ 4 combine)
  static constexpr int kThreads = 32 * (kCtl + kEpiWarps);
  static constexpr int kCtlRegs = 64, kEpiRegs = kComb ? 88 : 104, kCombRegs = 64;
  static constexpr int kRegsNeeded = kCtlRegs * 128 + (kComb ? kCombRegs * 128 : 0) + kEpiRegs * 32 * kEpiWarps;
};

template <int TT, int KBS, int MODE>
struct Smem {
  static constexpr int kWB = wb_of(MODE);
  static constexpr int kSubW = kBM * kBK;     // 16 KiB: one K block of one weight block
  static constexpr int kSubA = (is_cp(MODE) ? TT / 2 : TT) * kBK;  // one K block of this CTA's tokens
  static constexpr int kTileW = kSubW * KBS * kWB;
  static constexpr int kTileA = kSubA * KBS;
  static constexpr int kStage = kTileW + kTileA;
  // Byte offset of weight block b, K block h inside a stage's weight tile. kPair boxes are
  // 256 rows high, so the two blocks of a K block are adjacent; kGateUpSilu boxes carry the
  // gate half, then the up half, each KBS K blocks long.
  static __device__ __forceinline__ uint32_t w_off(int b, int h) {
    return (uint32_t)((MODE == kPair ? h * kWB + b : b * KBS + h) * kSubW);
  }
  // epilogue tables (bytes): the products act_scale x weight_scale
  // [kGroups][2][kSaChunk][kWB][TT / kGroups] (two chunk buffers), SiLU group maxima per lane
  // quarter and group scales [kGroups][5][TT / kGroups]
  static constexpr int kProdBytes = 2 * kSaChunk * kWB * TT * 4;
  static constexpr int kRedBytes = MODE == kGateUpSilu ? 5 * TT * 4 : 0;
  // fused combine: per combine warp and lane, the rows and weights of the token whose last
  // route it counted [4][32][kCombK] each
  static constexpr int kCombBytes = MODE == kCtaPairComb ? 4 * 32 * kCombK * 8 : 0;
};

// Dynamic shared memory: [stages][W tile | A tile] (1024-aligned), then the epilogue tables,
// the unit prefix table, the expert segment bounds and the barriers.
template <int TT, int KBS, int MODE>
__global__ void __launch_bounds__(Warps<TT, MODE>::kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_a, Params p) {
  using SM = Smem<TT, KBS, MODE>;
  using W = Warps<TT, MODE>;
  constexpr int WB = SM::kWB;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  const int S = p.stages;
  uint8_t* tiles = smem;
  float* prod = reinterpret_cast<float*>(smem + (size_t)S * SM::kStage);
  float* red = prod + SM::kProdBytes / 4;
  int* crow = reinterpret_cast<int*>(red + SM::kRedBytes / 4);  // (fused combine) [4][32][kCombK]
  float* cwt = reinterpret_cast<float*>(crow + SM::kCombBytes / 8);  // [4][32][kCombK]
  int* cum = reinterpret_cast<int*>(cwt + SM::kCombBytes / 8);  // [E+2] unit prefix
  int* seg_lo = cum + p.E + 2;                                   // [E] rows of expert e: [seg_lo, seg_hi)
  int* seg_hi = seg_lo + p.E;
  uint64_t* bars = reinterpret_cast<uint64_t*>(((reinterpret_cast<uintptr_t>(seg_hi + p.E)) + 7) & ~(uintptr_t)7);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  constexpr int kAcc = acc_count(WB * TT);
  constexpr int kTmemCols = kAcc * WB * TT < 32 ? 32 : kAcc * WB * TT;
  uint64_t* tfull = bars + 2 * S;
  uint64_t* tempty = bars + 2 * S + kAcc;
  uint64_t* pfull = tempty + kAcc;   // [2] a chunk's scale products are in place
  uint64_t* pempty = pfull + 2;      // [2] every epilogue warp is done with a chunk buffer
  // (kCtaPairComb) a ring of kYRing unit slots: ydone[i] every epilogue warp has stored its
  // rows of a unit; yfree[i] every combine warp has taken them over
  uint64_t* ydone = pempty + 2;
  uint64_t* yfree = ydone + kYRing;
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int E = p.E, NB = p.nb_count, KB = p.kb_count;
  const int NBU = MODE == kSingle ? NB : NB / 2;  // units per token tile
  // CTA pair: rank 0 issues the MMAs and owns the barriers that both CTAs' loads and
  // epilogues report to; rank 1 works on weight block 2p + 1 and token rows TT/2 ..
  constexpr bool kCP = is_cp(MODE);
  constexpr bool kComb = MODE == kCtaPairComb;
  const uint32_t crank = kCP ? cluster_rank() : 0u;

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int i = 0; i < S; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    for (int i = 0; i < kAcc; ++i) {
      mbar_init(smem_u32(&tfull[i]), 1);
      mbar_init(smem_u32(&tempty[i]), kCP ? 2 * kEpiWarps : kEpiWarps);  // one arrival per epilogue warp
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&pfull[i]), 32);         // every lane of the table warp
      mbar_init(smem_u32(&pempty[i]), kEpiWarps);
    }
    if constexpr (kComb) {
      for (int i = 0; i < kYRing; ++i) {
        mbar_init(smem_u32(&ydone[i]), kEpiWarps);  // this CTA's epilogue warps
        mbar_init(smem_u32(&yfree[i]), 4);          // its combine warps
      }
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // unit prefix: cum[e] = number of units of experts < e (units = token tiles x NBU)
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
        u = ((m + TT - 1) / TT) * NBU;
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
    if constexpr (kCP) {
      // one warp of each CTA of the pair allocates, together: the same columns in both
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                   "r"(kTmemCols));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                   "r"(kTmemCols));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
  }
  fence_before();
  if constexpr (kCP)
    cluster_sync();  // both CTAs' barriers are initialised before either reports to the other
  else
    __syncthreads();
  fence_after();
  // everything above overlapped the previous kernel's tail; the token rows and their
  // scales come from the previous kernel (the producer thread waits after it has sent the
  // first weight tiles, which do not depend on it)
  const bool producer = warp == 0 && lane == 0;
  if (!producer) {
    pdl_wait();
    pdl_trigger();
  }
  const uint32_t tmem_base = s_tmem;
  const int total_units = cum[E];
  // units c, c + G, ...: the CTAs sweep the (expert, token tile, weight block) list together,
  // so a token tile is read by several CTAs at about the same time and stays in L2
  // (a CTA pair counts as one: both CTAs run the same units)
  const int u_begin = kCP ? (int)cluster_id_x() : (int)blockIdx.x;
  const int u_end = total_units;
  const int u_step = kCP ? (int)cluster_count_x() : (int)gridDim.x;

  // unit -> (expert, weight block or block pair, token tile, first row, rows in tile).
  // The fused combine orders the list (block pair, expert, token tile), block pairs
  // outermost: the CTAs then finish every route's rows of one block pair within a short
  // span, while those rows are still in L2 for the token's last arrival to add up. (Measured
  // on GB300 for the plain down GEMM at 24,576 routes, either order takes the same time.)
  auto decode = [&](int u, int& e, int& nb, int& tt, int& row0, int& rows) {
    int key = u, nb_outer = 0;
    if constexpr (kComb) {
      const int tiles = total_units / NBU;  // every expert has NBU units per token tile
      nb_outer = u / tiles;
      key = (u - nb_outer * tiles) * NBU;
    }
    int lo = 0, hi = E - 1;
    while (lo < hi) {  // last e with cum[e] <= key
      const int mid = (lo + hi + 1) >> 1;
      if (cum[mid] <= key) lo = mid; else hi = mid - 1;
    }
    e = lo;
    const int s0 = seg_lo[e], s1 = seg_hi[e];
    const int local = key - cum[e];
    tt = local / NBU;
    nb = kComb ? nb_outer : local - tt * NBU;
    row0 = s0 + tt * TT;
    rows = min(TT, s1 - row0);
  };
  // weight block (row block of the n x k matrix) b of unit index nb
  auto wblock = [&](int nb, int b) {
    return MODE == kSingle ? nb : (MODE == kPair ? 2 * nb + b : (kCP ? 2 * nb + (int)crank : b * NBU + nb));
  };

  if (warp < W::kCtl) {
    // control warpgroup (register split: the whole warpgroup lowers its limit here)
    if constexpr (W::kComb) {
      if (warp >= 4)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(W::kCombRegs));
      else
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(W::kCtlRegs));
    } else if constexpr (W::kSplitRegs) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(W::kCtlRegs));
    }
  if (warp == 0) {
    // ------------------------------- TMA producer -------------------------------
    if (lane == 0) {
      // weight blocks are read once; the activation tile is read again by every weight
      // block of the expert
      const uint64_t pol_w = l2_policy_evict_first(), pol_a = l2_policy_evict_last();
      // stage sp of a unit: K blocks [sp * KBS, sp * KBS + KBS)
      auto load_w = [&](uint32_t dst, uint32_t bar, int sp, int nb, int e, uint64_t pol) {
        if constexpr (kCP)
          tma_load_4d_hint_pair(dst, &map_w, bar, 0, (2 * nb + (int)crank) * kBM, sp * KBS, e, pol);
        else if constexpr (MODE == kGateUpSilu)
          tma_load_5d_hint(dst, &map_w, bar, 0, 0, sp * KBS, nb, 2 * e, pol);
        else if constexpr (MODE == kPair)
          tma_load_4d_hint(dst, &map_w, bar, 0, nb * 2 * kBM, sp * KBS, e, pol);
        else if constexpr (KBS == 1)
          tma_load_3d_hint(dst, &map_w, bar, sp * kBK, nb * kBM, e, pol);
        else
          tma_load_4d_hint(dst, &map_w, bar, 0, nb * kBM, sp * KBS, e, pol);
      };
      auto load_a = [&](uint32_t dst, uint32_t bar, int sp, int row0, uint64_t pol) {
        if constexpr (kCP)
          tma_load_3d_hint_pair(dst, &map_a, bar, 0, row0 + (int)crank * (TT / 2), sp * KBS, pol);
        else if constexpr (KBS == 1 && MODE == kSingle)
          tma_load_2d_hint(dst, &map_a, bar, sp * kBK, row0, pol);
        else
          tma_load_3d_hint(dst, &map_a, bar, 0, row0, sp * KBS, pol);
      };
      uint32_t it = 0;
      const int SP = (KB + KBS - 1) / KBS;  // stages per unit
      // CTA pair: both CTAs' bytes are counted on the first CTA's full barrier, which that
      // CTA alone arms, for both (a box may land before it is armed: the phase cannot
      // complete while the arming arrival is still pending)
      auto full_target = [&](int st) {
        return kCP ? mapa_shared(smem_u32(&full[st]), 0) : smem_u32(&full[st]);
      };
      auto arm_full = [&](int st) {
        if (!kCP || crank == 0) mbar_expect_tx(smem_u32(&full[st]), kCP ? 2 * SM::kStage : SM::kStage);
      };
      int u = u_begin, sp = 0, e = 0, nb = 0, tt = 0, row0 = 0, rows = 0;
      if (u < u_end) decode(u, e, nb, tt, row0, rows);
      auto advance = [&]() {
        if (++sp == SP) {
          sp = 0;
          if ((u += u_step) < u_end) decode(u, e, nb, tt, row0, rows);
        }
      };
      // The weight tiles of the first pass over the ring go out before the wait: they do
      // not depend on the previous kernel. Their token tiles follow once it is complete.
      int pre_sp[kMaxStages], pre_row0[kMaxStages];
      int npre = 0;
      while (npre < S && u < u_end) {
        uint8_t* tw = tiles + (size_t)npre * SM::kStage;
        arm_full(npre);
        load_w(smem_u32(tw), full_target(npre), sp, nb, e, pol_w);
        pre_sp[npre] = sp;
        pre_row0[npre] = row0;
        ++npre;
        ++it;
        advance();
      }
      pdl_wait();
      pdl_trigger();
      for (int i = 0; i < npre; ++i)
        load_a(smem_u32(tiles + (size_t)i * SM::kStage + SM::kTileW), full_target(i), pre_sp[i], pre_row0[i], pol_a);
      while (u < u_end && !s_abort) {
        const int st = it % S;
        const uint32_t ph = (it / S) & 1;
        if (!mbar_wait(smem_u32(&empty[st]), ph ^ 1, &s_abort)) break;
        uint8_t* tw = tiles + (size_t)st * SM::kStage;
        uint8_t* ta = tw + SM::kTileW;
        const uint32_t fb = full_target(st);
        arm_full(st);
        load_w(smem_u32(tw), fb, sp, nb, e, pol_w);
        load_a(smem_u32(ta), fb, sp, row0, pol_a);
        ++it;
        advance();
      }
      // loads still in flight complete on their full barrier: wait for the last phase
      // issued on each stage (a bounded wait; the phase completes once its bytes land). In
      // a CTA pair the first CTA waits for both: its phases count the second CTA's bytes,
      // and the second CTA does not leave before the first (the closing cluster barrier).
      const uint32_t issued = (kCP && crank != 0) ? 0u : it;
      for (int st = 0; st < S && (uint32_t)st < issued; ++st) {
        const uint32_t last = issued - 1 - ((issued - 1 - st) % S);
        const uint32_t ph = (last / S) & 1;
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&full[st]), ph) && globaltimer() - t0 < kTimeoutNs) {
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------- MMA issuer --------------------------------
    // (CTA pair: the first CTA issues every MMA of the pair; the second only holds TMEM)
    if (lane == 0 && crank == 0) {
      uint32_t it = 0, kc = 0;
      constexpr uint32_t idesc = idesc_f8(TT, kCP ? 2 * kBM : kBM);
      const int SP = (KB + KBS - 1) / KBS;
      for (int u = u_begin; u < u_end && !s_abort; u += u_step) {
        bool ok = true;
        for (int sp = 0; sp < SP && ok; ++sp, ++it) {
          const int st = it % S;
          if (!mbar_wait(smem_u32(&full[st]), (it / S) & 1, &s_abort)) { ok = false; break; }
          const uint32_t tw = smem_u32(tiles + (size_t)st * SM::kStage);
          const uint32_t ta = tw + SM::kTileW;
          // the stage's K blocks (a last stage of an odd K has one; TMA zero-filled the other)
          for (int h = 0; h < KBS && sp * KBS + h < KB; ++h, ++kc) {
            const uint32_t acc = kc % kAcc;
            if (!mbar_wait(smem_u32(&tempty[acc]), ((kc / kAcc) & 1) ^ 1, &s_abort)) { ok = false; break; }
            fence_after();
            const uint32_t ta_h = ta + h * SM::kSubA;
#pragma unroll
            for (int b = 0; b < WB; ++b) {
              const uint32_t d = tmem_base + acc * (WB * TT) + b * TT;
              const uint32_t tw_h = tw + SM::w_off(b, h);
#pragma unroll
              for (int j = 0; j < kBK / 32; ++j) {
                if constexpr (kCP)
                  mma_f8_pair(d, smem_desc_sw128(tw_h + 32 * j), smem_desc_sw128(ta_h + 32 * j), idesc, j > 0 ? 1u : 0u);
                else
                  mma_f8(d, smem_desc_sw128(tw_h + 32 * j), smem_desc_sw128(ta_h + 32 * j), idesc, j > 0 ? 1u : 0u);
              }
            }
            // (CTA pair: the accumulator of each CTA is full, on each CTA's barrier)
            if constexpr (kCP)
              mma_commit_pair(smem_u32(&tfull[acc]), 0x3);
            else
              mma_commit(smem_u32(&tfull[acc]));
          }
          if (!ok) break;
          if constexpr (kCP)
            mma_commit_pair(smem_u32(&empty[st]), 0x3);  // both CTAs' stage is free
          else
            mma_commit(smem_u32(&empty[st]));
        }
        if (!ok) break;
      }
      // MMAs still running write TMEM: wait (bounded) for the last commit of each
      // accumulator before the CTA may free it
      for (uint32_t b = 0; b < (uint32_t)kAcc && b < kc; ++b) {
        const uint32_t last = kc - 1 - ((kc - 1 - b) % kAcc);
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(smem_u32(&tfull[b]), (last / kAcc) & 1) && globaltimer() - t0 < kTimeoutNs) {
        }
      }
    }
  } else if (warp == 2) {
    // ------------------------ scale-product tables ------------------------
    // For every (unit, chunk of kSaChunk K blocks) of this CTA, in the epilogue's order, the
    // products s_a[row0 + col][kb] * s_w[e, weight block, kb]: the same for all 128 weight
    // rows, so formed once per token column instead of per element. Two buffers alternate;
    // each lane loads all its scales of a chunk before it waits for the buffer, so the loads
    // of the next chunk are in flight while the epilogue still reads the current one.
    constexpr int NJ = (TT + 31) / 32;  // token columns per lane
    const int nchunks = (KB + kSaChunk - 1) / kSaChunk;
    uint32_t gch = 0;
    bool ok = true;
    for (int u = u_begin; u < u_end && ok; u += u_step) {
      int e, nb, tt, row0, rows;
      decode(u, e, nb, tt, row0, rows);
      for (int ch = 0; ch < nchunks; ++ch, ++gch) {
        // (kernels that split registers keep 64 for this warpgroup: there the weight scales
        // are loaded per block inside the store loop and the columns go in batches)
        constexpr bool kLean = W::kSplitRegs;
        constexpr int JB = kLean ? 1 : NJ;
        auto w_scale = [&](int b, int kbl) {
          const int kb = ch * kSaChunk + kbl;
          return kb < KB ? __ldg(p.w_s + ((int64_t)e * NB + wblock(nb, b)) * KB + kb) : 0.0f;
        };
        float sw[kLean ? 1 : WB][kSaChunk];
        if constexpr (!kLean) {
#pragma unroll
          for (int b = 0; b < WB; ++b)
#pragma unroll
            for (int kbl = 0; kbl < kSaChunk; ++kbl) sw[b][kbl] = w_scale(b, kbl);
        }
        const int buf = (int)(gch & 1);
        // (lean: one column batch at a time, not unrolled, to stay within the registers)
#pragma unroll(kLean ? 1 : NJ)
        for (int j0 = 0; j0 < NJ; j0 += JB) {
          float sa[JB][kSaChunk];
#pragma unroll
          for (int jj = 0; jj < JB; ++jj) {
            const int col = lane + 32 * (j0 + jj);
#pragma unroll
            for (int kbl = 0; kbl < kSaChunk; ++kbl) {
              const int kb = ch * kSaChunk + kbl;
              sa[jj][kbl] =
                  (col < TT && col < rows && kb < KB) ? __ldg(p.a_s + (int64_t)(row0 + col) * KB + kb) : 0.0f;
            }
          }
          if (j0 == 0 && !mbar_wait(smem_u32(&pempty[buf]), ((gch >> 1) & 1) ^ 1, &s_abort)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int b = 0; b < WB; ++b) {
            float swb[kSaChunk];
#pragma unroll
            for (int kbl = 0; kbl < kSaChunk; ++kbl) swb[kbl] = kLean ? w_scale(b, kbl) : sw[kLean ? 0 : b][kbl];
#pragma unroll
            for (int jj = 0; jj < JB; ++jj) {
              const int col = lane + 32 * (j0 + jj);
              if (col < TT) {
                const int g = col / (TT / kGroups), c = col - g * (TT / kGroups);
                float* dst = prod + g * 2 * kSaChunk * WB * (TT / kGroups) + buf * kSaChunk * WB * (TT / kGroups);
#pragma unroll
                for (int kbl = 0; kbl < kSaChunk; ++kbl) dst[(kbl * WB + b) * (TT / kGroups) + c] = sa[jj][kbl] * swb[kbl];
              }
            }
          }
        }
        if (!ok) break;
        mbar_arrive(smem_u32(&pfull[buf]));  // each lane releases its own products
      }
    }
  } else if (kComb && warp >= 4) {
    // ------------------------------ fused combine -------------------------------
    // Combine warp q (0..3) takes the token columns 32q .. 32q + 31 of this CTA's units.
    // Once every epilogue warp has stored a unit's rows (the ring barrier, release and
    // acquire at CTA scope), a gpu-scope fence publishes them -- the fence is cumulative over
    // what this warp observed through the barrier -- and a relaxed atomic counts one arrival
    // per (token, weight block). The arrival that completes a token's active routes acquires
    // the other arrivals' rows (a second fence) and adds the token's rows of this weight block
    // in ascending slot order, with the separate combine kernel's expression and rounding;
    // each row segment is read once, so its L2 lines are dropped, not written back.
    if constexpr (kComb) {
      const int q = warp - 4;
      // out_c[t, 128 nblk + 4 lane ..] from the rows of token t's active routes
      auto combine_token = [&](int t, int nblk) {
        const int col = nblk * kBM + 4 * lane;
        const int64_t rbase = (int64_t)t * p.topk;
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        // slots in batches of kB, the batch's loads issued before its additions
        constexpr int kB = 4;
        for (int j0 = 0; j0 < p.topk; j0 += kB) {
          int row[kB];
          float wt[kB];
#pragma unroll
          for (int i = 0; i < kB; ++i) {
            row[i] = -1;
            wt[i] = 0.0f;
            if (j0 + i < p.topk) {
              const int d = __ldg(p.route2dst + rbase + j0 + i);
              if (d >= 0) {  // a route without a row is skipped unread, as in the combine kernel
                row[i] = d;
                wt[i] = __ldg(p.rw + rbase + j0 + i);
              }
            }
          }
          float4 v[kB];
#pragma unroll
          for (int i = 0; i < kB; ++i) {
            v[i] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (row[i] >= 0) v[i] = __ldcg(reinterpret_cast<const float4*>(p.out + (int64_t)row[i] * p.ld_out + col));
          }
#pragma unroll
          for (int i = 0; i < kB; ++i) {
            if (row[i] >= 0) {
              acc[0] = fmaf(wt[i], v[i].x, acc[0]);
              acc[1] = fmaf(wt[i], v[i].y, acc[1]);
              acc[2] = fmaf(wt[i], v[i].z, acc[2]);
              acc[3] = fmaf(wt[i], v[i].w, acc[3]);
              // the line's eight lanes have all read it (one load instruction of the warp)
              if ((lane & 7) == 0) discard_l2_line(p.out + (int64_t)row[i] * p.ld_out + col);
            }
          }
        }
        const int64_t o = (int64_t)t * p.ld_c + col;
        if (p.out_dtype == FTMOE_OUT_FP32) {
          store4(static_cast<float*>(p.out_c) + o, acc);
        } else {
          uint16_t b[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) b[i] = p.out_dtype == FTMOE_OUT_FP16 ? OutF16::cvt(acc[i]) : OutBf16::cvt(acc[i]);
          store4(static_cast<uint16_t*>(p.out_c) + o, b);
        }
      };
      // topk <= kCombK: each lane's slots are loaded together, and a token whose last route
      // this lane counted has its rows and weights staged in shared memory, so that the warp
      // then issues all of that token's row loads at once
      const bool staged = p.topk <= kCombK;
      int* my_rows = crow + q * 32 * kCombK;
      float* my_wts = cwt + q * 32 * kCombK;
      uint32_t j = 0;
      for (int u = u_begin; u < u_end; u += u_step, ++j) {
        int e, nb, tt, row0, rows;
        decode(u, e, nb, tt, row0, rows);
        const uint32_t slot = j % kYRing;
        if (!mbar_wait(smem_u32(&ydone[slot]), (j / kYRing) & 1, &s_abort)) break;
        fence_acq_rel_gpu();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&yfree[slot]));
        const int nblk = 2 * nb + (int)crank;
        const int c = 32 * q + lane;
        int t = -1;
        bool last = false;
        if (c < rows) {
          t = __ldg(p.dst2src + row0 + c);
          const int64_t rbase = (int64_t)t * p.topk;
          int active = 0;
          if (staged) {
            int sr[kCombK];
#pragma unroll
            for (int i = 0; i < kCombK; ++i) sr[i] = i < p.topk ? __ldg(p.route2dst + rbase + i) : -1;
#pragma unroll
            for (int i = 0; i < kCombK; ++i) active += sr[i] >= 0 ? 1 : 0;
            const uint32_t before = atomicAdd(p.cnt + (int64_t)t * NB + nblk, 1u);
            last = (int)before + 1 == active;
            if (last) {
#pragma unroll
              for (int i = 0; i < kCombK; ++i) {
                my_rows[lane * kCombK + i] = sr[i];
                my_wts[lane * kCombK + i] = sr[i] >= 0 ? __ldg(p.rw + rbase + i) : 0.0f;
              }
            }
          } else {
            for (int i = 0; i < p.topk; ++i) active += __ldg(p.route2dst + rbase + i) >= 0 ? 1 : 0;
            const uint32_t before = atomicAdd(p.cnt + (int64_t)t * NB + nblk, 1u);
            last = (int)before + 1 == active;
          }
        }
        uint32_t m = __ballot_sync(0xffffffffu, last);
        __syncwarp();  // (the lanes' staged rows are visible to the whole warp)
        if (m != 0) fence_acq_rel_gpu();
        while (m != 0) {
          const int i = __ffs((int)m) - 1;
          m &= m - 1;
          const int ti = __shfl_sync(0xffffffffu, t, i);
          if (!staged) {
            combine_token(ti, nblk);
            continue;
          }
          // the token's rows of this weight block, all loads in flight together
          const int col = nblk * kBM + 4 * lane;
          const int* rr = my_rows + i * kCombK;
          const float* ww = my_wts + i * kCombK;
          float4 v[kCombK];
#pragma unroll
          for (int k = 0; k < kCombK; ++k) {
            const int r = rr[k];
            v[k] = r >= 0 ? __ldcg(reinterpret_cast<const float4*>(p.out + (int64_t)r * p.ld_out + col))
                          : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
          }
          float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
          for (int k = 0; k < kCombK; ++k) {
            const int r = rr[k];
            if (r >= 0) {  // a route without a row is skipped unread, as in the combine kernel
              const float wk = ww[k];
              acc[0] = fmaf(wk, v[k].x, acc[0]);
              acc[1] = fmaf(wk, v[k].y, acc[1]);
              acc[2] = fmaf(wk, v[k].z, acc[2]);
              acc[3] = fmaf(wk, v[k].w, acc[3]);
              // the line's eight lanes have all read it (one load instruction of the warp)
              if ((lane & 7) == 0) discard_l2_line(p.out + (int64_t)r * p.ld_out + col);
            }
          }
          const int64_t o = (int64_t)ti * p.ld_c + col;
          if (p.out_dtype == FTMOE_OUT_FP32) {
            store4(static_cast<float*>(p.out_c) + o, acc);
          } else {
            uint16_t b16[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) b16[k] = p.out_dtype == FTMOE_OUT_FP16 ? OutF16::cvt(acc[k]) : OutBf16::cvt(acc[k]);
            store4(static_cast<uint16_t*>(p.out_c) + o, b16);
          }
        }
        __syncwarp();  // the staged rows of this unit are read before the next unit overwrites them
      }
    }
  }
  } else {
    // --------------------------------- epilogue ---------------------------------
    if constexpr (W::kSplitRegs) asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(W::kEpiRegs));
    // Every warp of a column group runs the same sequence of group barriers whatever
    // happens: a failed wait only turns off this warp's TMEM reads and stores for the rest
    // of the unit, and the group leaves together at the next unit boundary.
    constexpr int HC = TT / kGroups;          // token columns of this warp's group
    // TMEM columns read per tcgen05.ld round trip and block (keeps the registers in bounds)
    constexpr int CH = kCP ? 16 : (WB * HC <= 16 ? HC : (W::kSplitRegs ? (TT == 128 ? 4 : 8) : 16 / WB));
    const int ew = warp - W::kCtl;            // 0 .. kEpiWarps-1
    const int grp = ew >> 2;                  // column group
    const int quarter = warp & 3;             // TMEM lane quarter this warp may access
    const int tid_g = (ew & 3) * 32 + lane;   // 0..127 within the group
    float* my_prod = prod + grp * 2 * kSaChunk * WB * HC;  // [2][kSaChunk][WB][HC]
    float* my_red = red + grp * 5 * HC;       // [4][HC] maxima, [HC] scales (kGateUpSilu)
    uint32_t kc = 0;
    float acc[WB][HC];
    uint32_t gch = 0;  // chunks begun so far; chunk gch uses product buffer gch & 1
    // (fused combine) the rows stay in L2 until the token's last route has arrived
    const uint64_t pol_y = kComb ? l2_policy_evict_last() : 0ull;
    uint32_t ucount = 0;  // units of this CTA so far
    for (int u = u_begin; u < u_end; u += u_step, ++ucount) {
      int e, nb, tt, row0, rows;
      decode(u, e, nb, tt, row0, rows);
      // all warps of the group leave together on an abort
      if (named_bar_or(1 + grp, 128, s_abort)) break;
#pragma unroll
      for (int b = 0; b < WB; ++b)
#pragma unroll
        for (int c = 0; c < HC; ++c) acc[b][c] = 0.0f;
      bool ok = true;
      // a group whose token columns all lie past the tile's rows has nothing to promote:
      // it hands each accumulator straight back
      const bool live = grp * HC < rows;
      for (int kb = 0; kb < KB; ++kb, ++kc) {
        const int kbl = kb % kSaChunk;
        const int buf = (int)(gch & 1);
        if (kbl == 0 && ok) {
          // the table warp's products of this chunk
          const int got = mbar_wait(smem_u32(&pfull[buf]), (gch >> 1) & 1, &s_abort) ? 1 : 0;
          ok = __all_sync(0xffffffffu, got) != 0;
        }
        const uint32_t ab = kc % kAcc;
        if (ok) {
          const int got = mbar_wait(smem_u32(&tfull[ab]), (kc / kAcc) & 1, &s_abort) ? 1 : 0;
          ok = __all_sync(0xffffffffu, got) != 0;
        }
        if (ok) {
        fence_after();
        if (!live) {
          fence_before();
          __syncwarp();
          if (lane == 0) {
            if constexpr (kCP)
              mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[ab]), 0));
            else
              mbar_arrive(smem_u32(&tempty[ab]));
          }
        } else {
        const uint32_t taddr = tmem_base + ((uint32_t)(32 * quarter) << 16) + ab * (WB * TT) + grp * HC;
        const float* pp = my_prod + (buf * kSaChunk + kbl) * WB * HC;
#pragma unroll
        for (int c0 = 0; c0 < HC; c0 += CH) {
          float d[WB][CH];
#pragma unroll
          for (int b = 0; b < WB; ++b) tmem_ld<CH>(taddr + b * TT + c0, d[b]);
          tmem_ld_wait();
          if (c0 + CH == HC) {
            // every TMEM read of this accumulator is complete: hand it back to the MMA
            fence_before();
            __syncwarp();
            if (lane == 0) {
              if constexpr (kCP)
                mbar_arrive_cluster(mapa_shared(smem_u32(&tempty[ab]), 0));  // the issuing CTA's barrier
              else
                mbar_arrive(smem_u32(&tempty[ab]));
            }
          }
#pragma unroll
          for (int b = 0; b < WB; ++b) {
            const float4* p4 = reinterpret_cast<const float4*>(pp + b * HC + c0);
#pragma unroll
            for (int c4 = 0; c4 < CH / 4; ++c4) {
              const float4 s4 = p4[c4];
              acc[b][c0 + 4 * c4 + 0] = fmaf(d[b][4 * c4 + 0], s4.x, acc[b][c0 + 4 * c4 + 0]);
              acc[b][c0 + 4 * c4 + 1] = fmaf(d[b][4 * c4 + 1], s4.y, acc[b][c0 + 4 * c4 + 1]);
              acc[b][c0 + 4 * c4 + 2] = fmaf(d[b][4 * c4 + 2], s4.z, acc[b][c0 + 4 * c4 + 2]);
              acc[b][c0 + 4 * c4 + 3] = fmaf(d[b][4 * c4 + 3], s4.w, acc[b][c0 + 4 * c4 + 3]);
            }
          }
        }
        }  // live
        }  // ok
        if (kbl == kSaChunk - 1 || kb == KB - 1) {
          // this warp reads nothing more of the chunk's products (on every path: the table
          // warp must not wait on a warp that gave up)
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&pempty[buf]));
          ++gch;
        }
      }
      const int m = 32 * quarter + lane;  // row of this lane inside a 128-row weight block
      if constexpr (MODE == kGateUpSilu) {
        // a = silu(g) * u for intermediate column 128 nb + m; its group is this unit's
        // 128 rows, so the group maximum is a reduction over the four lane quarters
#pragma unroll
        for (int c = 0; c < HC; ++c) acc[0][c] = silu_mul_1(acc[0][c], acc[1][c]);
        {
          // column maxima of |a| over the warp's 32 rows by a butterfly transpose-reduce:
          // each exchange halves the columns a lane keeps, until lane l holds the maximum of
          // column l / (32 / HC) (HC - 1 + 5 - log2(HC) shuffles instead of 5 per column)
          float v[HC];
#pragma unroll
          for (int c = 0; c < HC; ++c) v[c] = fabsf(acc[0][c]);
#pragma unroll
          for (int st = 0; st < 5; ++st) {
            const int o = 16 >> st;
            constexpr int kLog = HC >= 32 ? 5 : HC >= 16 ? 4 : HC >= 8 ? 3 : HC >= 4 ? 2 : HC >= 2 ? 1 : 0;
            if (st < kLog) {
              const int half = HC >> (st + 1);
              const bool upper = (lane & o) != 0;
#pragma unroll
              for (int i = 0; i < half; ++i) {
                const float send = upper ? v[i] : v[i + half];
                const float keep = upper ? v[i + half] : v[i];
                v[i] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, o));
              }
            } else {
              v[0] = fmaxf(v[0], __shfl_xor_sync(0xffffffffu, v[0], o));
            }
          }
          if ((lane & (32 / HC - 1)) == 0) my_red[quarter * HC + lane / (32 / HC)] = v[0];
        }
        named_bar(1 + grp, 128);
        // one thread per column: the group scale amax / 448
        if (tid_g < HC) {
          const int c = tid_g;
          const float amax = fmaxf(fmaxf(my_red[c], my_red[HC + c]), fmaxf(my_red[2 * HC + c], my_red[3 * HC + c]));
          my_red[4 * HC + c] = div_rn(amax, kE4M3Max);
        }
        named_bar(1 + grp, 128);
        const int ld_q = p.n >> 1, ld_s = NBU;
#pragma unroll
        for (int c = 0; c < HC; ++c) {
          const int r = grp * HC + c;
          const float amax = fmaxf(fmaxf(my_red[c], my_red[HC + c]), fmaxf(my_red[2 * HC + c], my_red[3 * HC + c]));
          const float sc = my_red[4 * HC + c];
          const uint8_t code = amax > 0.0f ? (uint8_t)(f2_to_e4m3x2(div_rn(acc[0][c], sc), 0.0f) & 0xFF) : (uint8_t)0;
          if (ok && r < rows) {
            p.q_out[(int64_t)(row0 + r) * ld_q + nb * kBM + m] = code;
            if (quarter == 0 && lane == 0) p.s_out[(int64_t)(row0 + r) * ld_s + nb] = sc;
          }
        }
      } else {
#pragma unroll
        for (int b = 0; b < WB; ++b) {
          const int n = wblock(nb, b) * kBM + m;
          if (ok && n < p.n) {
#pragma unroll
            for (int c = 0; c < HC; ++c) {
              const int r = grp * HC + c;
              if (r < rows) {
                if constexpr (kComb)
                  st_global_hint(p.out + (int64_t)(row0 + r) * p.ld_out + n, acc[b][c], pol_y);
                else
                  p.out[(int64_t)(row0 + r) * p.ld_out + n] = acc[b][c];
              }
            }
          }
        }
        if constexpr (kComb) {
          // hand the unit's rows to the combine warps (the slot's previous unit, kYRing
          // units back, has been taken over by then)
          const uint32_t slot = ucount % kYRing;
          (void)mbar_wait(smem_u32(&yfree[slot]), ((ucount / kYRing) & 1) ^ 1, &s_abort);
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ydone[slot]));
        }
      }
    }
  }

  fence_before();
  if constexpr (kCP) {
    // neither CTA of the pair leaves, or frees TMEM, while the other may still read its
    // shared memory, signal its barriers or (the MMAs of the first) write its TMEM
    cluster_sync();
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    __syncwarp();
    fence_after();
    if constexpr (kCP)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols));
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols));
  }
}

}  // namespace tc

// ---------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------

static bool encode_u8(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                      const uint32_t* box, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t b[5], es[5] = {1, 1, 1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) st[i] = strides[i];
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, (cuuint32_t)rank, const_cast<void*>(base), d, st, b, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_u8_tmap(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                    const uint32_t* box) {
  return encode_u8(map, base, rank, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

bool encode_u8_tmap_plain(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                          const uint64_t* strides, const uint32_t* box) {
  return encode_u8(map, base, rank, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int sm_count() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

template <int TT, int KBS, int MODE>
static cudaError_t launch_tt(const TcGemmArgs& a, cudaStream_t st, int* unsupported) {
  using SM = tc::Smem<TT, KBS, MODE>;
  EncodeTiledFn enc = encode_fn();
  if (!enc) {
    *unsupported = 1;
    return cudaSuccess;
  }
  const int KB = (int)cdiv(a.k, 128), NB = (int)cdiv(a.n, 128);
  if (KB > tc::kMaxKB) {
    *unsupported = 1;
    return cudaSuccess;
  }
  const size_t fixed =
      1024 /*align*/ + SM::kProdBytes + SM::kRedBytes + SM::kCombBytes + (size_t)(3 * a.E + 2) * 4 + 8;
  // dynamic shared memory budget: the device's opt-in maximum per block minus the
  // kernel's static shared memory
  int dev = 0;
  cudaGetDevice(&dev);
  static size_t budget[64] = {};  // per device: opt-in maximum minus static shared memory
  size_t max_smem = (dev >= 0 && dev < 64) ? budget[dev] : 0;
  if (max_smem == 0) {
    cudaFuncAttributes fattr;
    if (cudaFuncGetAttributes(&fattr, tc::tc_gemm_kernel<TT, KBS, MODE>) != cudaSuccess) return cudaErrorInvalidValue;
    int optin = 0;
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    max_smem = (size_t)optin > fattr.sharedSizeBytes ? (size_t)optin - fattr.sharedSizeBytes : 0;
    if (dev >= 0 && dev < 64) budget[dev] = max_smem;
  }
  using W = tc::Warps<TT, MODE>;
  if constexpr (W::kSplitRegs) {
    // the register split must fit the pool the block is launched with
    static int regs[64] = {};
    int nr = (dev >= 0 && dev < 64) ? regs[dev] : 0;
    if (nr == 0) {
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, tc::tc_gemm_kernel<TT, KBS, MODE>) != cudaSuccess) return cudaErrorInvalidValue;
      nr = fa.numRegs;
      if (dev >= 0 && dev < 64) regs[dev] = nr;
    }
    if ((int64_t)nr * W::kThreads < (int64_t)W::kRegsNeeded) {
      *unsupported = 1;
      return cudaSuccess;
    }
  }
  constexpr int kAcc = tc::acc_count(SM::kWB * TT);
  constexpr int kBars = 2 * kAcc + 4 + (MODE == tc::kCtaPairComb ? 2 * tc::kYRing : 0);
  int stages = tc::kMaxStages;
  while (stages > 2 && fixed + (size_t)stages * SM::kStage + (2 * stages + kBars) * 8 > max_smem) --stages;
  const size_t smem = fixed + (size_t)stages * SM::kStage + (2 * stages + kBars) * 8;
  if (smem > max_smem) {
    *unsupported = 1;
    return cudaSuccess;
  }
  // KBS > 1 or two weight blocks: weights as (128-byte K chunk, row, K block, expert) and
  // tokens as (128-byte K chunk, row, K block), one box holding KBS K blocks (kPair boxes
  // are 256 rows high). kGateUpSilu splits the rows into (row in block, block j) and folds
  // (gate/up half, expert) into one dimension of stride I*k, so one box brings gate block j
  // and up block j. KBS = 1 with one block: rows of K bytes.
  CUtensorMap mw, ma;
  if constexpr (MODE == tc::kGateUpSilu) {
    const uint64_t half = (uint64_t)a.n / 2;
    const uint64_t wd[5] = {128, 128, (uint64_t)KB, half / 128, 2 * (uint64_t)a.E};
    const uint64_t ws[4] = {(uint64_t)a.k, 128, 128 * (uint64_t)a.k, half * (uint64_t)a.k};
    const uint32_t wb[5] = {128, 128, (uint32_t)KBS, 1, 2};
    if (!encode_u8_tmap(&mw, a.w_q, 5, wd, ws, wb)) return cudaErrorInvalidValue;
  } else if constexpr (MODE == tc::kPair || tc::is_cp(MODE) || KBS > 1) {
    // (the CTA pair's loads are always 4-D: this map at every KBS)
    const uint64_t wd[4] = {128, (uint64_t)a.n, (uint64_t)KB, (uint64_t)a.E};
    const uint64_t ws[3] = {(uint64_t)a.k, 128, (uint64_t)a.k * (uint64_t)a.n};
    const uint32_t wb[4] = {128, (uint32_t)(128 * SM::kWB), (uint32_t)KBS, 1};
    if (!encode_u8_tmap(&mw, a.w_q, 4, wd, ws, wb)) return cudaErrorInvalidValue;
  } else {
    const uint64_t wd[3] = {(uint64_t)a.k, (uint64_t)a.n, (uint64_t)a.E};
    const uint64_t ws[2] = {(uint64_t)a.k, (uint64_t)a.k * (uint64_t)a.n};
    const uint32_t wb[3] = {128, 128, 1};
    if (!encode_u8_tmap(&mw, a.w_q, 3, wd, ws, wb)) return cudaErrorInvalidValue;
  }
  if constexpr (MODE != tc::kSingle || KBS > 1) {
    // (a CTA pair loads half of the token tile in each CTA)
    const uint64_t ad[3] = {128, (uint64_t)a.a_rows, (uint64_t)KB};
    const uint64_t as[2] = {(uint64_t)a.k, 128};
    const uint32_t ab[3] = {128, (uint32_t)(tc::is_cp(MODE) ? TT / 2 : TT), (uint32_t)KBS};
    if (!encode_u8_tmap(&ma, a.a_q, 3, ad, as, ab)) return cudaErrorInvalidValue;
  } else {
    const uint64_t ad[2] = {(uint64_t)a.k, (uint64_t)a.a_rows};
    const uint64_t as[1] = {(uint64_t)a.k};
    const uint32_t ab[2] = {128, (uint32_t)TT};
    if (!encode_u8_tmap(&ma, a.a_q, 2, ad, as, ab)) return cudaErrorInvalidValue;
  }
  tc::Params p;
  p.offsets = a.offsets;
  p.a_s = a.a_s;
  p.w_s = a.w_s;
  p.out = a.out;
  p.ld_out = a.ld_out;
  p.q_out = a.q_out;
  p.s_out = a.s_out;
  p.a_rows = a.a_rows;
  p.n = (int)a.n;
  p.k = (int)a.k;
  p.E = a.E;
  p.kb_count = KB;
  p.nb_count = NB;
  p.stages = stages;
  p.dst2src = a.dst2src;
  p.route2dst = a.route2dst;
  p.rw = a.rw;
  p.cnt = a.cnt;
  p.out_c = a.out_c;
  p.ld_c = a.ld_c;
  p.topk = a.topk;
  p.out_dtype = a.out_dtype;
  // raise the kernel's dynamic shared memory limit only when a launch needs more than
  // any earlier one on this device (the attribute is per function and device)
  static size_t granted[64] = {};
  if (dev >= 0 && dev < 64 && smem > granted[dev]) {
    cudaError_t e =
        cudaFuncSetAttribute(tc::tc_gemm_kernel<TT, KBS, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    granted[dev] = smem;
  } else if (dev < 0 || dev >= 64) {
    cudaError_t e =
        cudaFuncSetAttribute(tc::tc_gemm_kernel<TT, KBS, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  if constexpr (tc::is_cp(MODE)) {
    // as many CTA pairs as can be resident at once (one CTA per SM; a pair needs two SMs
    // of one cluster-capable group, so this may be a little under half the SMs)
    static int pairs[64] = {};
    int np = (dev >= 0 && dev < 64) ? pairs[dev] : 0;
    if (np == 0) {
      np = max_active_clusters(tc::tc_gemm_kernel<TT, KBS, MODE>, dim3(W::kThreads), smem, 2, 2 * (sm_count() / 2));
      if (np > sm_count() / 2) np = sm_count() / 2;
      if (dev >= 0 && dev < 64) pairs[dev] = np;
    }
    if (np < 1) {
      *unsupported = 1;
      return cudaSuccess;
    }
    return launch_kernel_cluster(tc::tc_gemm_kernel<TT, KBS, MODE>, dim3(2 * np), dim3(W::kThreads), smem, st, true, 2,
                                 mw, ma, p);
  }
  return launch_kernel(tc::tc_gemm_kernel<TT, KBS, MODE>, dim3(sm_count()), dim3(W::kThreads), smem, st, true, mw,
                       ma, p);
}

template <int MODE>
static cudaError_t launch_mode(const TcGemmArgs& a, cudaStream_t st, int* unsupported) {
  switch (a.tok_tile) {
    case 16: return launch_tt<16, tc::kbs_for(16, MODE), MODE>(a, st, unsupported);
    case 32: return launch_tt<32, tc::kbs_for(32, MODE), MODE>(a, st, unsupported);
    case 64: return launch_tt<64, tc::kbs_for(64, MODE), MODE>(a, st, unsupported);
    case 128: return launch_tt<128, tc::kbs_for(128, MODE), MODE>(a, st, unsupported);
    default: *unsupported = 1; return cudaSuccess;
  }
}

bool tc_gemm_pairs_ok(int64_t n, int64_t k) { return n % 256 == 0 && k % 128 == 0; }

bool tc_gemm_comb_ok(int tok_tile, int64_t n, int64_t k, const void* y, int64_t ld_y, const void* out_c,
                     int64_t ld_c) {
  return (tok_tile == 64 || tok_tile == 128) && tc_gemm_pairs_ok(n, k) && (uintptr_t)y % 128 == 0 && ld_y % 32 == 0 &&
         (uintptr_t)out_c % 16 == 0 && ld_c % 4 == 0;
}

cudaError_t launch_tc_gemm(const TcGemmArgs& a, cudaStream_t st, int* unsupported) {
  *unsupported = 0;
  // TMA needs 16-byte aligned bases and row strides; the kernel indexes rows and
  // columns in 32-bit; the unit prefix table holds up to kMaxExperts experts.
  if (a.k % 16 != 0 || (uintptr_t)a.w_q % 16 != 0 || (uintptr_t)a.a_q % 16 != 0 || a.E > tc::kMaxExperts ||
      a.n > (1 << 30) || a.k > (1 << 30) || a.a_rows > (1 << 30) || a.E > 65535) {
    *unsupported = 1;
    return cudaSuccess;
  }
  // a CTA pair: one weight block per CTA, token tile 64 or 128, whole block pairs and K blocks
  if (a.comb) {
    if (a.ctas != 2 || a.silu || a.wblocks == 2 || a.topk <= 0 ||
        !tc_gemm_comb_ok(a.tok_tile, a.n, a.k, a.out, a.ld_out, a.out_c, a.ld_c)) {
      *unsupported = 1;
      return cudaSuccess;
    }
    return a.tok_tile == 64
               ? launch_tt<64, tc::kbs_for(64, tc::kCtaPairComb), tc::kCtaPairComb>(a, st, unsupported)
               : launch_tt<128, tc::kbs_for(128, tc::kCtaPairComb), tc::kCtaPairComb>(a, st, unsupported);
  }
  if (a.ctas == 2) {
    if (a.silu || a.wblocks == 2 || !tc_gemm_pairs_ok(a.n, a.k) || (a.tok_tile != 64 && a.tok_tile != 128)) {
      *unsupported = 1;
      return cudaSuccess;
    }
    return a.tok_tile == 64
               ? launch_tt<64, tc::kbs_for(64, tc::kCtaPair), tc::kCtaPair>(a, st, unsupported)
               : launch_tt<128, tc::kbs_for(128, tc::kCtaPair), tc::kCtaPair>(a, st, unsupported);
  }
  // two weight blocks per unit need whole 256-row block pairs and whole K blocks
  if (a.wblocks == 2 || a.silu) {
    if (!tc_gemm_pairs_ok(a.n, a.k)) {
      *unsupported = 1;
      return cudaSuccess;
    }
    return a.silu ? launch_mode<tc::kGateUpSilu>(a, st, unsupported) : launch_mode<tc::kPair>(a, st, unsupported);
  }
  if (a.k % 128 != 0) {  // a partial last K block: one K block per stage
    switch (a.tok_tile) {
      case 16: return launch_tt<16, 1, tc::kSingle>(a, st, unsupported);
      case 32: return launch_tt<32, 1, tc::kSingle>(a, st, unsupported);
      case 64: return launch_tt<64, 1, tc::kSingle>(a, st, unsupported);
      case 128: return launch_tt<128, 1, tc::kSingle>(a, st, unsupported);
      default: *unsupported = 1; return cudaSuccess;
    }
  }
  return launch_mode<tc::kSingle>(a, st, unsupported);
}

FTMOE_DEFINE_ERR_READER(read_err_tc_gemm)

}  // namespace ftmoe

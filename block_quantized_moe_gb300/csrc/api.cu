// C ABI of libftmoe: argument validation on the host, then kernel launches on the
// caller's stream. Nothing here allocates, frees or synchronises (except
// ftmoe_read_error_flags), so every entry point defined in this file can be captured in a
// CUDA graph.
#include <string.h>

#include "common.cuh"
#include "internal.h"

using namespace ftmoe;

namespace ftmoe {
bool& pdl_enabled() {
  static thread_local bool on = false;
  return on;
}
}  // namespace ftmoe

namespace {

// Lets the forward's kernels after the first start while their predecessor finishes
// (programmatic dependent launch), and turns that off again on every way out.
struct OverlapScope {
  ~OverlapScope() { pdl_enabled() = false; }
  void enable() { pdl_enabled() = true; }
};

inline cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }
inline ftmoe_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FTMOE_OK : FTMOE_CUDA_ERROR; }
inline size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

bool valid_format(int32_t f) { return f == FTMOE_FMT_FP8 || f == FTMOE_FMT_NVFP4 || f == FTMOE_FMT_MXFP8; }
bool valid_out_dtype(int32_t d) { return d == FTMOE_OUT_BF16 || d == FTMOE_OUT_FP16 || d == FTMOE_OUT_FP32; }

// bytes of one quantized row of k elements and of its scale row
size_t code_row_bytes(int32_t fmt, int64_t k) { return fmt == FTMOE_FMT_NVFP4 ? (size_t)(k / 2) : (size_t)k; }
size_t scale_row_bytes(int32_t fmt, int64_t k) {
  if (fmt == FTMOE_FMT_MXFP8) return (size_t)(k / kMxBlock);
  return fmt == FTMOE_FMT_FP8 ? (size_t)cdiv(k, kGroup) * 4 : (size_t)(k / kNvfp4Block);
}

int pick_tile_value(int64_t routes, int32_t E) {
  const int64_t per = cdiv(routes, E);
  const int cand[4] = {16, 32, 64, 128};
  for (int m : cand)
    if (m >= per) return m;
  return 128;
}

// Weight blocks per tensor-core unit when the caller leaves it open. Two adjacent blocks
// sharing each token tile halve the token bytes a stage carries per weight byte, but double
// the epilogue's work per K block. Below token tile 64 the token tile is small beside the
// weights, and one block per unit keeps twice as many units to spread over the SMs. At 128
// the two-block epilogue (64 fp32 accumulators per thread, eight TMEM round trips per K
// block) bounds the GEMM: measured on GB300 at 24,576 routes, gate/up took 1671 us with two
// blocks and 1563 us with one. So two blocks at token tile 64 only.
int pick_wblocks(int tok_tile, int64_t n, int64_t k) { return tok_tile == 64 && tc_gemm_pairs_ok(n, k) ? 2 : 1; }

// SMs per tensor-core unit when the caller leaves it open: a CTA pair at token tile 128. Each
// CTA then carries half of the token tile beside its weight block, so more weight bytes fit
// in flight, and its epilogue promotes one block. Measured on GB300 at 24,576 routes (256
// experts, top-6, 7168/2048): gate/up 1478 us against 1560 us on one SM, forward 2859 us
// against 2928 us.
int pick_ctas(int tok_tile, int64_t n, int64_t k) { return tok_tile == 128 && tc_gemm_pairs_ok(n, k) ? 2 : 1; }

ftmoe_status check_bank(const ftmoe_expert_bank* w) {
  if (!w || !w->q || !w->scales) return FTMOE_INVALID_ARG;
  if (w->num_experts <= 0 || w->n <= 0 || w->k <= 0 || !valid_format(w->format)) return FTMOE_INVALID_ARG;
  if (w->format == FTMOE_FMT_NVFP4 && (!w->global_scale || w->k % 32 != 0)) return FTMOE_INVALID_ARG;
  if (w->format == FTMOE_FMT_MXFP8 && w->k % kMxBlock != 0) return FTMOE_INVALID_ARG;
  return FTMOE_OK;
}

// MXFP8: the grouped layout on the block-scaled tensor-core kernel only. Scale rows of k/32
// bytes are read by TMA in 16-byte boxes, so k % 512 == 0.
ftmoe_status grouped_gemm_mxfp8(const ftmoe_act* a, const ftmoe_routes* routes, const ftmoe_expert_bank* w,
                                float* out, int64_t ld_out, const ftmoe_tile* tile, int variant, void* stream) {
  if (routes->kind == FTMOE_ROUTES_SLOTS) return FTMOE_UNSUPPORTED;
  if (routes->kind != FTMOE_ROUTES_GROUPED || !routes->offsets) return FTMOE_INVALID_ARG;
  if (a->rows == 0) return FTMOE_OK;
  if (variant == 1) return FTMOE_UNSUPPORTED;
  MxGemmArgs g;
  memset(&g, 0, sizeof(g));
  g.a_q = a->q;
  g.a_sf = static_cast<const uint8_t*>(a->scales);
  g.a_rows = a->rows;
  g.w_q = w->q;
  g.w_sf = static_cast<const uint8_t*>(w->scales);
  g.out = out;
  g.ld_out = ld_out;
  g.n = w->n;
  g.k = w->k;
  g.E = w->num_experts;
  g.offsets = routes->offsets;
  g.tok_tile = (tile && tile->tok_tile) ? tile->tok_tile : pick_tile_value(a->rows, w->num_experts);
  int unsupported = 0;
  cudaError_t e = launch_mxfp8_gemm(g, as_stream(stream), &unsupported);
  if (unsupported) return FTMOE_UNSUPPORTED;
  return from_cuda(e);
}

// NVFP4: the grouped layout on the block-scaled tensor-core kernel only (no streaming
// kernel for e2m1 codes). Scale rows of k/16 bytes are read by TMA, so k % 256 == 0.
ftmoe_status grouped_gemm_nvfp4(const ftmoe_act* a, const ftmoe_routes* routes, const ftmoe_expert_bank* w,
                                float* out, int64_t ld_out, const ftmoe_tile* tile, int variant, void* stream) {
  if (routes->kind == FTMOE_ROUTES_SLOTS) return FTMOE_UNSUPPORTED;
  if (routes->kind != FTMOE_ROUTES_GROUPED || !routes->offsets) return FTMOE_INVALID_ARG;
  if (a->rows == 0) return FTMOE_OK;
  if (!a->global_scale) return FTMOE_INVALID_ARG;
  if (variant == 1) return FTMOE_UNSUPPORTED;
  NvGemmArgs g;
  memset(&g, 0, sizeof(g));
  g.a_q = a->q;
  g.a_sf = static_cast<const uint8_t*>(a->scales);
  g.a_gscale = a->global_scale;
  g.a_rows = a->rows;
  g.w_q = w->q;
  g.w_sf = static_cast<const uint8_t*>(w->scales);
  g.w_gscale = w->global_scale;
  g.out = out;
  g.ld_out = ld_out;
  g.n = w->n;
  g.k = w->k;
  g.E = w->num_experts;
  g.offsets = routes->offsets;
  g.tok_tile = (tile && tile->tok_tile) ? tile->tok_tile : pick_tile_value(a->rows, w->num_experts);
  int unsupported = 0;
  cudaError_t e = launch_nvfp4_gemm(g, as_stream(stream), &unsupported);
  if (unsupported) return FTMOE_UNSUPPORTED;
  return from_cuda(e);
}

ftmoe_status grouped_gemm(const ftmoe_act* a, const ftmoe_routes* routes, const ftmoe_expert_bank* w,
                          float* out, int64_t ld_out, const ftmoe_tile* tile, void* stream,
                          bool is_down) {
  if (!a || !routes || !out) return FTMOE_INVALID_ARG;
  ftmoe_status st = check_bank(w);
  if (st != FTMOE_OK) return st;
  if (a->format != w->format || a->k != w->k || a->rows < 0 || ld_out < w->n) return FTMOE_INVALID_ARG;
  if (a->rows > 0 && (!a->q || !a->scales)) return FTMOE_INVALID_ARG;
  if (tile && tile->tok_tile != 0 && tile->tok_tile != 16 && tile->tok_tile != 32 &&
      tile->tok_tile != 64 && tile->tok_tile != 128)
    return FTMOE_INVALID_ARG;
  if (tile && (tile->variant < 0 || tile->variant > 2)) return FTMOE_INVALID_ARG;
  if (tile && (tile->wblocks < 0 || tile->wblocks > 2)) return FTMOE_INVALID_ARG;
  if (tile && (tile->ctas < 0 || tile->ctas > 2 || (tile->ctas == 2 && tile->wblocks == 2))) return FTMOE_INVALID_ARG;
  const int variant = tile ? tile->variant : 0;
  if (w->format == FTMOE_FMT_NVFP4) return grouped_gemm_nvfp4(a, routes, w, out, ld_out, tile, variant, stream);
  if (w->format == FTMOE_FMT_MXFP8) return grouped_gemm_mxfp8(a, routes, w, out, ld_out, tile, variant, stream);
  // both GEMM kernels read K-contiguous rows through TMA: 16-byte aligned rows
  if (w->k % 16 != 0 || (uintptr_t)w->q % 16 != 0 || (a->rows > 0 && (uintptr_t)a->q % 16 != 0))
    return FTMOE_UNSUPPORTED;

  if (routes->kind == FTMOE_ROUTES_SLOTS) {
    if (!routes->slots || routes->tokens < 0 || routes->topk <= 0) return FTMOE_INVALID_ARG;
    const int64_t R = routes->tokens * routes->topk;
    if (R == 0) return FTMOE_OK;
    const int64_t need_rows = is_down ? R : routes->tokens;
    if (a->rows < need_rows) return FTMOE_INVALID_ARG;
    if (variant == 2 || w->k > kStreamMaxK) return FTMOE_UNSUPPORTED;
    StreamGemmArgs g;
    memset(&g, 0, sizeof(g));
    g.a_q = a->q;
    g.a_s = static_cast<const float*>(a->scales);
    g.w_q = w->q;
    g.w_s = static_cast<const float*>(w->scales);
    g.out = out;
    g.ld_out = ld_out;
    g.n = w->n;
    g.k = w->k;
    g.E = w->num_experts;
    g.grouped = 0;
    g.slots = routes->slots;
    g.routes = R;
    g.act_div = is_down ? 1 : routes->topk;
    g.topk = routes->topk;
    g.a_rows = a->rows;
    return from_cuda(launch_stream_gemm(g, as_stream(stream)));
  }
  if (routes->kind != FTMOE_ROUTES_GROUPED || !routes->offsets) return FTMOE_INVALID_ARG;
  if (a->rows == 0) return FTMOE_OK;
  if (variant != 1) {
    TcGemmArgs t;
    memset(&t, 0, sizeof(t));
    t.a_q = a->q;
    t.a_s = static_cast<const float*>(a->scales);
    t.a_rows = a->rows;
    t.w_q = w->q;
    t.w_s = static_cast<const float*>(w->scales);
    t.out = out;
    t.ld_out = ld_out;
    t.n = w->n;
    t.k = w->k;
    t.E = w->num_experts;
    t.offsets = routes->offsets;
    t.tok_tile = (tile && tile->tok_tile) ? tile->tok_tile : pick_tile_value(a->rows, w->num_experts);
    // (an explicit request for two weight blocks per unit on one SM keeps the unit on one SM)
    const bool two_blocks = tile && tile->wblocks == 2;
    t.ctas = (tile && tile->ctas) ? tile->ctas : (two_blocks ? 1 : pick_ctas(t.tok_tile, w->n, w->k));
    t.wblocks = (tile && tile->wblocks) ? tile->wblocks : (t.ctas == 2 ? 1 : pick_wblocks(t.tok_tile, w->n, w->k));
    int unsupported = 0;
    cudaError_t e = launch_tc_gemm(t, as_stream(stream), &unsupported);
    if (!unsupported) return from_cuda(e);
    if (variant == 2) return FTMOE_UNSUPPORTED;
  }
  if (w->k > kStreamMaxK) return FTMOE_UNSUPPORTED;
  StreamGemmArgs g;
  memset(&g, 0, sizeof(g));
  g.a_q = a->q;
  g.a_s = static_cast<const float*>(a->scales);
  g.w_q = w->q;
  g.w_s = static_cast<const float*>(w->scales);
  g.out = out;
  g.ld_out = ld_out;
  g.n = w->n;
  g.k = w->k;
  g.E = w->num_experts;
  g.grouped = 1;
  g.offsets = routes->offsets;
  g.a_rows = a->rows;
  return from_cuda(launch_stream_gemm(g, as_stream(stream)));
}

ftmoe_status gateup_silu(const ftmoe_act* a, const ftmoe_routes* routes, const ftmoe_expert_bank* w,
                         uint8_t* q_out, float* scales_out, const ftmoe_tile* tile, void* stream) {
  if (!a || !routes || !q_out || !scales_out) return FTMOE_INVALID_ARG;
  ftmoe_status st = check_bank(w);
  if (st != FTMOE_OK) return st;
  if (a->format != w->format || a->k != w->k || a->rows < 0) return FTMOE_INVALID_ARG;
  if (a->rows > 0 && (!a->q || !a->scales)) return FTMOE_INVALID_ARG;
  if (tile && tile->tok_tile != 0 && tile->tok_tile != 16 && tile->tok_tile != 32 &&
      tile->tok_tile != 64 && tile->tok_tile != 128)
    return FTMOE_INVALID_ARG;
  if (routes->kind != FTMOE_ROUTES_GROUPED || !routes->offsets) return FTMOE_INVALID_ARG;
  if (w->format != FTMOE_FMT_FP8 || !tc_gemm_pairs_ok(w->n, w->k) || (uintptr_t)w->q % 16 != 0 ||
      (a->rows > 0 && (uintptr_t)a->q % 16 != 0))
    return FTMOE_UNSUPPORTED;
  if (a->rows == 0) return FTMOE_OK;
  TcGemmArgs t;
  memset(&t, 0, sizeof(t));
  t.a_q = a->q;
  t.a_s = static_cast<const float*>(a->scales);
  t.a_rows = a->rows;
  t.w_q = w->q;
  t.w_s = static_cast<const float*>(w->scales);
  t.n = w->n;
  t.k = w->k;
  t.E = w->num_experts;
  t.offsets = routes->offsets;
  t.tok_tile = (tile && tile->tok_tile) ? tile->tok_tile : pick_tile_value(a->rows, w->num_experts);
  t.wblocks = 2;
  t.silu = 1;
  t.q_out = q_out;
  t.s_out = scales_out;
  int unsupported = 0;
  cudaError_t e = launch_tc_gemm(t, as_stream(stream), &unsupported);
  if (unsupported) return FTMOE_UNSUPPORTED;
  return from_cuda(e);
}

// The forward's down GEMM with the combine inside (tok_tile 64 or 128, CTA pairs): y keeps
// the rows only until each token's last route has been added; out receives the combined rows
// of every token with an active route (the prep launch wrote the others and zeroed cnt).
ftmoe_status down_comb(const ftmoe_act* a, const int32_t* offsets, const ftmoe_expert_bank* w, float* y,
                       int32_t tok_tile, const int32_t* dst2src, const int32_t* route2dst, const float* rw,
                       int32_t topk, uint32_t* cnt, void* out, int64_t ld_out, int32_t out_dtype, void* stream) {
  if (a->rows == 0) return FTMOE_OK;
  TcGemmArgs t;
  memset(&t, 0, sizeof(t));
  t.a_q = a->q;
  t.a_s = static_cast<const float*>(a->scales);
  t.a_rows = a->rows;
  t.w_q = w->q;
  t.w_s = static_cast<const float*>(w->scales);
  t.out = y;
  t.ld_out = w->n;
  t.n = w->n;
  t.k = w->k;
  t.E = w->num_experts;
  t.offsets = offsets;
  t.tok_tile = tok_tile;
  t.wblocks = 1;
  t.ctas = 2;
  t.comb = 1;
  t.dst2src = dst2src;
  t.route2dst = route2dst;
  t.rw = rw;
  t.cnt = cnt;
  t.out_c = out;
  t.ld_c = ld_out;
  t.topk = topk;
  t.out_dtype = out_dtype;
  int unsupported = 0;
  cudaError_t e = launch_tc_gemm(t, as_stream(stream), &unsupported);
  if (unsupported) return FTMOE_UNSUPPORTED;
  return from_cuda(e);
}

struct Layout {
  ftmoe_workspace_layout l;
  bool grouped;
  bool fused;   // SiLU-and-mul inside the gate/up GEMM: no fp32 gate/up buffer
  bool comb;    // the combine inside the down GEMM (CTA pairs), when the output rows allow
  bool decode;  // the fused decode path (prep launch + one persistent kernel)
  DecodePlan plan;
};

ftmoe_status check_shape(const ftmoe_moe_shape* s) {
  if (!s) return FTMOE_INVALID_ARG;
  if (s->tokens < 0 || s->hidden <= 0 || s->inter <= 0 || s->topk <= 0 || s->num_experts <= 0)
    return FTMOE_INVALID_ARG;
  if (!valid_format(s->format) || s->path < 0 || s->path > 5 || !valid_out_dtype(s->out_dtype))
    return FTMOE_INVALID_ARG;
  if (s->tok_tile != 0 && s->tok_tile != 16 && s->tok_tile != 32 && s->tok_tile != 64 && s->tok_tile != 128)
    return FTMOE_INVALID_ARG;
  if (s->format != FTMOE_FMT_FP8 && (s->hidden % 32 != 0 || s->inter % 32 != 0)) return FTMOE_INVALID_ARG;
  return FTMOE_OK;
}

// Automatic path beyond the fused decode path's limits: the grouped tensor-core path. Measured
// on GB300 with four K blocks per TMA box, it matches the route-slot streaming kernel at one token
// (49.6 vs 50.4 us for 8 active routes of 4096/1024) and beats it from two tokens on (68 vs
// 86 us); the route-slot path stays available as path 1.
bool use_grouped(const ftmoe_moe_shape* s) { return s->path != 1 && s->path != 4; }

// The fused decode path (path 4): one persistent kernel after the quantizing launch. The
// automatic choice wherever its limits hold (at most 8 tokens). Measured on GB300 against
// the grouped path (us per forward, one CUDA graph, L2 flushed): hidden 4096, intermediate
// 1024, 64 experts, top-8 -- 1 token with 8/2/0 active routes 45.6 / 36.0 / 11.2 against
// 48.3 / 38.1 / 15.9, 8 tokens with 8/2 active 116.8 / 61.1 against 119.5 / 65.2; hidden
// 2048, intermediate 768, 8 experts, 1 token with 2 active 32.3 against 31.1.
bool use_decode(const ftmoe_moe_shape* s) {
  if (s->format != FTMOE_FMT_FP8 || (s->path != 0 && s->path != 4)) return false;
  return decode_plan(s->tokens, s->topk, s->num_experts, s->hidden, s->inter).ok;
}

// When the automatic path fuses SiLU-and-mul into the gate/up GEMM. Measured on GB300:
//  - A fused unit is twice as large as a one-block unit, so with few units per SM the CTAs
//    finish unevenly: eight decode tokens (64 experts x 8 gate/up block pairs) ran 126.9 us
//    fused against 122.9 us separate. Hence a minimum of kFusedMinUnits units, counted for
//    the most distinct experts the routes can reach.
//  - At token tile 128 only two accumulator pairs fit in TMEM, so the MMA waits while the
//    epilogue forms and re-quantizes a unit's SiLU outputs: at 24,576 routes (256 experts)
//    fused ran 3193 us, separate 3136 us. At tiles 16 and 32 (1,536 and 6,144 routes) fused
//    won, 1667 vs 1698 us and 1932 vs 2031 us.
constexpr int64_t kFusedMinUnits = 2048;

bool use_fused(const ftmoe_moe_shape* s) {
  if (s->path == 3) return true;
  if (s->path != 0 || s->format != FTMOE_FMT_FP8) return false;
  if (!tc_gemm_pairs_ok(2 * s->inter, s->hidden) || s->num_experts > kTcGemmMaxExperts) return false;
  const int64_t R = s->tokens * s->topk;
  const int tile = s->tok_tile ? s->tok_tile : pick_tile_value(R, s->num_experts);
  if (tile > 64) return false;
  const int64_t experts = R < s->num_experts ? R : s->num_experts;
  return experts * (s->inter / 128) >= kFusedMinUnits;
}

// When the down GEMM adds up each token's rows itself: path 5 only. Measured on GB300 at
// 24,576 routes (4,096 tokens, 7168/2048, 256 experts), the forward took 6217 us with the
// combine inside against 2615 us with the combine kernel. The combine warps' work per unit is
// a chain of round trips to memory (the arrival counters' atomics, then each completed
// token's rows), and with the weight stream holding HBM near its bandwidth each round trip
// waits microseconds: without the atomics the forward took 3457 us, without the row loads
// 3852 us, and without any combine work (no output) 2564 us -- so at most about 2% was to
// be won. The automatic path keeps the combine kernel.
bool use_comb(const ftmoe_moe_shape* s) {
  if (s->path != 5 || s->format != FTMOE_FMT_FP8 || s->num_experts > kTcGemmMaxExperts) return false;
  // the combine warps stage a token's slots in registers and shared memory: at most 8
  if (s->topk > 8) return false;
  if (!tc_gemm_pairs_ok(s->hidden, s->inter)) return false;
  const int tile = s->tok_tile ? s->tok_tile : pick_tile_value(s->tokens * s->topk, s->num_experts);
  return tile == 64 || tile == 128;
}

Layout make_layout(const ftmoe_moe_shape* s) {
  Layout L;
  memset(&L, 0, sizeof(L));
  const int64_t T = s->tokens, H = s->hidden, I = s->inter, R = T * s->topk, E = s->num_experts;
  const int32_t f = s->format;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align256(bytes);
    return o;
  };
  L.decode = use_decode(s);
  if (L.decode) {
    // token rows padded to the MMA's 16 columns, the re-quantized intermediate and the down
    // rows per route, the gate/up partial sums and the arrival counters
    L.plan = decode_plan(T, s->topk, (int32_t)E, H, I);
    L.l.x_q = take(16 * H);
    L.l.x_scales = take(16 * (H / 128) * 4);
    L.l.act_q_bytes = R * I;
    L.l.act_q = take(L.l.act_q_bytes);
    L.l.act_scales_bytes = R * (I / 128) * 4;
    L.l.act_scales = take(L.l.act_scales_bytes);
    L.l.down_bytes = (size_t)R * H * 4;
    L.l.down = take(L.l.down_bytes);
    L.l.partials_bytes = L.plan.part_bytes;
    L.l.partials = take(L.l.partials_bytes);
    L.l.counters_bytes = L.plan.cnt_words * 4;
    L.l.counters = take(L.l.counters_bytes);
    L.l.total = off;
    return L;
  }
  L.grouped = use_grouped(s);
  L.fused = L.grouped && use_fused(s);
  L.comb = L.grouped && use_comb(s);
  // (MXFP8 quantizes the gathered rows: no quantized token rows)
  L.l.x_q = take(f == FTMOE_FMT_MXFP8 ? 0 : T * code_row_bytes(f, H));
  L.l.x_scales = take(f == FTMOE_FMT_MXFP8 ? 0 : T * scale_row_bytes(f, H));
  L.l.x_gscale = take(16);
  if (L.grouped) {
    L.l.counts = take(E * 4);
    L.l.offsets = take((E + 1) * 4);
    L.l.dst2src = take(R * 4);
    L.l.route2dst = take(R * 4);
    L.l.rows_q = take(R * code_row_bytes(f, H));
    L.l.rows_scales = take(R * scale_row_bytes(f, H));
  }
  if (!L.fused) {
    L.l.gateup_bytes = (size_t)R * 2 * I * 4;
    L.l.gateup = take(L.l.gateup_bytes);
  }
  L.l.act_q_bytes = R * code_row_bytes(f, I);
  L.l.act_q = take(L.l.act_q_bytes);
  L.l.act_scales_bytes = R * scale_row_bytes(f, I);
  L.l.act_scales = take(L.l.act_scales_bytes);
  L.l.act_gscale = take(16);
  L.l.down_bytes = (size_t)R * H * 4;
  L.l.down = take(L.l.down_bytes);
  if (L.comb) {
    // arrival counters of the fused combine, one per (token, 128-column block of H)
    L.l.counters_bytes = (size_t)T * (H / 128) * 4;
    L.l.counters = take(L.l.counters_bytes);
  }
  L.l.total = off;
  return L;
}

}  // namespace

extern "C" {

const char* ftmoe_status_string(int status) {
  switch (status) {
    case FTMOE_OK: return "ok";
    case FTMOE_INVALID_ARG: return "invalid argument";
    case FTMOE_UNSUPPORTED: return "unsupported by this build";
    case FTMOE_CUDA_ERROR: return "CUDA error";
    case FTMOE_WORKSPACE_TOO_SMALL: return "workspace too small";
    case FTMOE_CHECK_FAILED: return "check failed";
    default: return "unknown status";
  }
}

ftmoe_status ftmoe_pick_tile(int64_t routes, int32_t num_experts, ftmoe_tile* out) {
  if (!out || routes < 0 || num_experts <= 0) return FTMOE_INVALID_ARG;
  memset(out, 0, sizeof(*out));
  out->tok_tile = pick_tile_value(routes, num_experts);
  return FTMOE_OK;
}

ftmoe_status ftmoe_quantize_act(const uint16_t* x, int64_t rows, int64_t k, int64_t ld_x,
                                int32_t format, uint8_t* q, void* scales, float* global_scale,
                                void* stream) {
  if (rows < 0 || k <= 0 || ld_x < k || !valid_format(format)) return FTMOE_INVALID_ARG;
  if (rows == 0) return FTMOE_OK;
  if (!x || !q || !scales) return FTMOE_INVALID_ARG;
  if (format == FTMOE_FMT_FP8)
    return from_cuda(launch_quantize_act_fp8(x, rows, k, ld_x, q, static_cast<float*>(scales),
                                             as_stream(stream)));
  if (format == FTMOE_FMT_MXFP8) {
    if (global_scale || k % kMxBlock != 0) return FTMOE_INVALID_ARG;
    return from_cuda(launch_mxfp8_quant_bf16(x, rows, k, ld_x, nullptr, rows, nullptr, q,
                                             static_cast<uint8_t*>(scales), as_stream(stream)));
  }
  if (!global_scale || k % 32 != 0 || (uintptr_t)q % 8 != 0) return FTMOE_INVALID_ARG;
  return from_cuda(launch_quantize_act_nvfp4(x, rows, k, ld_x, q, static_cast<uint8_t*>(scales),
                                             global_scale, as_stream(stream)));
}

ftmoe_status ftmoe_quantize_weights(const float* w, int32_t num_experts, int64_t n, int64_t k,
                                    int32_t format, uint8_t* q, void* scales, float* global_scale,
                                    void* stream) {
  if (num_experts < 0 || n <= 0 || k <= 0 || !valid_format(format)) return FTMOE_INVALID_ARG;
  if (num_experts == 0) return FTMOE_OK;
  if (!w || !q || !scales) return FTMOE_INVALID_ARG;
  if (format == FTMOE_FMT_FP8)
    return from_cuda(launch_quantize_weights_fp8(w, num_experts, n, k, q, static_cast<float*>(scales),
                                                 as_stream(stream)));
  if (format == FTMOE_FMT_MXFP8) {
    if (global_scale || k % kMxBlock != 0) return FTMOE_INVALID_ARG;
    return from_cuda(launch_mxfp8_quant_f32(w, (int64_t)num_experts * n, k, k, q, static_cast<uint8_t*>(scales),
                                            as_stream(stream)));
  }
  if (!global_scale || k % 32 != 0 || (uintptr_t)q % 8 != 0) return FTMOE_INVALID_ARG;
  return from_cuda(launch_quantize_weights_nvfp4(w, num_experts, n, k, q, static_cast<uint8_t*>(scales),
                                                 global_scale, as_stream(stream)));
}

ftmoe_status ftmoe_segment_routes(const int32_t* expert_ids, int64_t tokens, int32_t topk,
                                  int32_t num_experts, int32_t* counts, int32_t* offsets,
                                  int32_t* dst2src, int32_t* route2dst, void* stream) {
  if (tokens < 0 || topk <= 0 || num_experts <= 0) return FTMOE_INVALID_ARG;
  if (!counts || !offsets) return FTMOE_INVALID_ARG;
  if (tokens > 0 && (!expert_ids || !dst2src || !route2dst)) return FTMOE_INVALID_ARG;
  if (tokens * (int64_t)topk > 0x7fffffff) return FTMOE_UNSUPPORTED;
  return from_cuda(launch_segment(expert_ids, tokens * topk, topk, num_experts, counts, offsets,
                                  dst2src, route2dst, as_stream(stream)));
}

ftmoe_status ftmoe_gather_rows_scales(const uint8_t* src, const void* src_scales, int64_t n_src,
                                      int64_t row_bytes, int64_t scale_bytes,
                                      const int32_t* dst2src, int64_t n_dst,
                                      const int32_t* n_dst_dev, uint8_t* dst, void* dst_scales,
                                      void* stream) {
  if (n_dst < 0 || n_src < 0 || row_bytes <= 0 || scale_bytes < 0) return FTMOE_INVALID_ARG;
  if (n_dst == 0) return FTMOE_OK;  // zero-row short circuit: nothing is launched
  if (!src || !dst2src || !dst) return FTMOE_INVALID_ARG;
  if (scale_bytes > 0 && (!src_scales || !dst_scales)) return FTMOE_INVALID_ARG;
  return from_cuda(launch_gather(src, static_cast<const uint8_t*>(src_scales), n_src, row_bytes,
                                 scale_bytes, dst2src, n_dst, n_dst_dev, dst,
                                 static_cast<uint8_t*>(dst_scales), as_stream(stream)));
}

ftmoe_status ftmoe_gather_quantize_act(const uint16_t* x, int64_t n_src, int64_t k, int64_t ld_x,
                                       const int32_t* dst2src, int64_t n_dst, const int32_t* n_dst_dev,
                                       int32_t format, uint8_t* q, void* scales, void* stream) {
  if (n_dst < 0 || n_src < 0 || k <= 0 || ld_x < k || !valid_format(format)) return FTMOE_INVALID_ARG;
  if (format != FTMOE_FMT_MXFP8) return FTMOE_UNSUPPORTED;
  if (k % kMxBlock != 0) return FTMOE_INVALID_ARG;
  if (n_dst == 0) return FTMOE_OK;
  if (!x || !dst2src || !q || !scales) return FTMOE_INVALID_ARG;
  return from_cuda(launch_mxfp8_quant_bf16(x, n_dst, k, ld_x, dst2src, n_src, n_dst_dev, q,
                                           static_cast<uint8_t*>(scales), as_stream(stream)));
}

ftmoe_status ftmoe_grouped_gemm_gateup(const ftmoe_act* a, const ftmoe_routes* routes,
                                       const ftmoe_expert_bank* w, float* out, int64_t ld_out,
                                       const ftmoe_tile* tile, void* stream) {
  return grouped_gemm(a, routes, w, out, ld_out, tile, stream, false);
}

ftmoe_status ftmoe_grouped_gemm_gateup_silu(const ftmoe_act* a, const ftmoe_routes* routes,
                                            const ftmoe_expert_bank* w, uint8_t* q_out, float* scales_out,
                                            const ftmoe_tile* tile, void* stream) {
  return gateup_silu(a, routes, w, q_out, scales_out, tile, stream);
}

ftmoe_status ftmoe_grouped_gemm_down(const ftmoe_act* a, const ftmoe_routes* routes,
                                     const ftmoe_expert_bank* w, float* out, int64_t ld_out,
                                     const ftmoe_tile* tile, void* stream) {
  return grouped_gemm(a, routes, w, out, ld_out, tile, stream, true);
}

ftmoe_status ftmoe_silu_mul(const float* gu, int64_t rows, int64_t inter, int64_t ld_gu,
                            const int32_t* rows_dev, int32_t format, uint8_t* q, void* scales,
                            float* global_scale, void* stream) {
  if (rows < 0 || inter <= 0 || ld_gu < 2 * inter || !valid_format(format)) return FTMOE_INVALID_ARG;
  if (rows == 0) return FTMOE_OK;
  if (!gu || !q || !scales) return FTMOE_INVALID_ARG;
  if (format == FTMOE_FMT_FP8)
    return from_cuda(launch_silu_mul_fp8(gu, rows, inter, ld_gu, rows_dev, q,
                                         static_cast<float*>(scales), as_stream(stream)));
  if (format == FTMOE_FMT_MXFP8) {
    if (global_scale || inter % kMxBlock != 0) return FTMOE_INVALID_ARG;
    return from_cuda(launch_silu_mul_mxfp8(gu, rows, inter, ld_gu, rows_dev, q, static_cast<uint8_t*>(scales),
                                           as_stream(stream)));
  }
  if (!global_scale || inter % 32 != 0 || (uintptr_t)q % 8 != 0) return FTMOE_INVALID_ARG;
  return from_cuda(launch_silu_mul_nvfp4(gu, rows, inter, ld_gu, rows_dev, q,
                                         static_cast<uint8_t*>(scales), global_scale,
                                         as_stream(stream)));
}

ftmoe_status ftmoe_combine(const float* y, int64_t ld_y, const int32_t* route2dst,
                           const int32_t* expert_ids, const float* weights, int64_t tokens,
                           int32_t topk, int64_t hidden, int32_t out_dtype, void* out,
                           int64_t ld_out, void* stream) {
  if (tokens < 0 || topk <= 0 || hidden <= 0 || ld_y < hidden || ld_out < hidden) return FTMOE_INVALID_ARG;
  if (!valid_out_dtype(out_dtype)) return FTMOE_INVALID_ARG;
  if (tokens == 0) return FTMOE_OK;
  if (!y || !expert_ids || !weights || !out) return FTMOE_INVALID_ARG;
  return from_cuda(launch_combine(y, ld_y, route2dst, expert_ids, weights, tokens, topk, hidden, out_dtype, out,
                                  ld_out, as_stream(stream)));
}

size_t ftmoe_forward_workspace_bytes(const ftmoe_moe_shape* shape) {
  if (check_shape(shape) != FTMOE_OK) return 0;
  return make_layout(shape).l.total;
}

ftmoe_status ftmoe_forward_workspace_layout(const ftmoe_moe_shape* shape, ftmoe_workspace_layout* out) {
  if (!out) return FTMOE_INVALID_ARG;
  ftmoe_status st = check_shape(shape);
  if (st != FTMOE_OK) return st;
  *out = make_layout(shape).l;
  return FTMOE_OK;
}

ftmoe_status ftmoe_moe_forward(const ftmoe_moe_args* args, void* workspace, size_t workspace_bytes,
                               void* stream) {
  if (!args) return FTMOE_INVALID_ARG;
  const ftmoe_moe_shape* s = &args->shape;
  ftmoe_status st = check_shape(s);
  if (st != FTMOE_OK) return st;
  st = check_bank(&args->w_gateup);
  if (st != FTMOE_OK) return st;
  st = check_bank(&args->w_down);
  if (st != FTMOE_OK) return st;
  const int64_t T = s->tokens, H = s->hidden, I = s->inter, E = s->num_experts;
  const int32_t f = s->format;
  const ftmoe_expert_bank& wg = args->w_gateup;
  const ftmoe_expert_bank& wd = args->w_down;
  if (wg.format != f || wd.format != f || wg.num_experts != E || wd.num_experts != E ||
      wg.n != 2 * I || wg.k != H || wd.n != H || wd.k != I)
    return FTMOE_INVALID_ARG;
  if (args->ld_x < H || args->ld_out < H) return FTMOE_INVALID_ARG;
  if (T == 0) return FTMOE_OK;
  if (!args->x || !args->expert_ids || !args->route_weights || !args->out) return FTMOE_INVALID_ARG;
  const Layout L = make_layout(s);
  if (!workspace) return FTMOE_INVALID_ARG;
  if (workspace_bytes < L.l.total) return FTMOE_WORKSPACE_TOO_SMALL;
  // no route-slot kernel for e2m1 codes or E8M0-scaled rows; no fused gate/up + SiLU for them
  if (f != FTMOE_FMT_FP8 && (!L.grouped || L.fused)) return FTMOE_UNSUPPORTED;
  if (s->path == 4 && !L.decode) return FTMOE_UNSUPPORTED;           // outside the fused decode limits

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int64_t R = T * s->topk;
  cudaStream_t strm = as_stream(stream);
  uint8_t* xq = ws + L.l.x_q;
  void* xs = ws + L.l.x_scales;
  float* xg = f == FTMOE_FMT_NVFP4 ? reinterpret_cast<float*>(ws + L.l.x_gscale) : nullptr;
  float* gu = reinterpret_cast<float*>(ws + L.l.gateup);
  uint8_t* aq = ws + L.l.act_q;
  void* as = ws + L.l.act_scales;
  float* ag = f == FTMOE_FMT_NVFP4 ? reinterpret_cast<float*>(ws + L.l.act_gscale) : nullptr;
  float* y = reinterpret_cast<float*>(ws + L.l.down);
  ftmoe_tile tile;
  memset(&tile, 0, sizeof(tile));
  tile.tok_tile = s->tok_tile ? s->tok_tile : pick_tile_value(R, (int32_t)E);

  int32_t* counts = reinterpret_cast<int32_t*>(ws + L.l.counts);
  int32_t* offsets = reinterpret_cast<int32_t*>(ws + L.l.offsets);
  int32_t* dst2src = reinterpret_cast<int32_t*>(ws + L.l.dst2src);
  int32_t* route2dst = reinterpret_cast<int32_t*>(ws + L.l.route2dst);
  // FP8 on the grouped path: quantization and the segmenter share the first launch
  const bool prep = L.grouped && f == FTMOE_FMT_FP8;
  if (prep && R > 0x7fffffff) return FTMOE_UNSUPPORTED;
  // the combine inside the down GEMM where the layout has it and the output rows allow
  const bool comb = L.comb && tc_gemm_comb_ok(tile.tok_tile, H, I, y, H, args->out, args->ld_out);
  if (s->path == 5 && !comb) return FTMOE_UNSUPPORTED;
  uint32_t* comb_cnt = comb ? reinterpret_cast<uint32_t*>(ws + L.l.counters) : nullptr;
  PrepCombine pc;
  memset(&pc, 0, sizeof(pc));
  if (comb) {
    pc.zero_words = comb_cnt;
    pc.n_zero_words = T * (H / 128);
    pc.out_rows = args->out;
    pc.ld_out = args->ld_out;
    pc.out_bytes = s->out_dtype == FTMOE_OUT_FP32 ? 4 : 2;
    pc.hidden = H;
  }

  OverlapScope overlap;
  if (L.decode) {
    uint32_t* cnt = reinterpret_cast<uint32_t*>(ws + L.l.counters);
    st = from_cuda(launch_decode_prep(args->x, T, H, args->ld_x, xq, static_cast<float*>(xs), args->expert_ids,
                                      s->topk, (int32_t)E, cnt, L.plan.cnt_words, args->out, args->ld_out,
                                      s->out_dtype, strm));
    if (st != FTMOE_OK) return st;
    overlap.enable();
    DecodeArgs d;
    memset(&d, 0, sizeof(d));
    d.x_q = xq;
    d.x_s = static_cast<const float*>(xs);
    d.ids = args->expert_ids;
    d.rw = args->route_weights;
    d.wg_q = wg.q;
    d.wg_s = static_cast<const float*>(wg.scales);
    d.wd_q = wd.q;
    d.wd_s = static_cast<const float*>(wd.scales);
    d.act_q = aq;
    d.act_s = static_cast<float*>(as);
    d.y = y;
    d.part = reinterpret_cast<float*>(ws + L.l.partials);
    d.cnt = cnt;
    d.out = args->out;
    d.ld_out = args->ld_out;
    d.out_dtype = s->out_dtype;
    d.T = T;
    d.H = H;
    d.I = I;
    d.topk = s->topk;
    d.E = (int32_t)E;
    int unsupported = 0;
    const cudaError_t e = launch_decode_fused(d, L.plan, strm, &unsupported);
    if (unsupported) return FTMOE_UNSUPPORTED;
    return from_cuda(e);
  }
  // MXFP8 gathers the bf16 activation and quantizes the gathered rows (the SGLang gather
  // page's mxfp8 branch): its first launch is the segmenter
  const bool mx = f == FTMOE_FMT_MXFP8;
  if (prep)
    st = from_cuda(launch_prep_fp8(args->x, T, H, args->ld_x, xq, static_cast<float*>(xs), args->expert_ids, R,
                                   s->topk, (int32_t)E, counts, offsets, dst2src, route2dst, pc, strm));
  else if (mx)
    st = ftmoe_segment_routes(args->expert_ids, T, s->topk, (int32_t)E, counts, offsets, dst2src, route2dst,
                              stream);
  else
    st = ftmoe_quantize_act(args->x, T, H, args->ld_x, f, xq, xs, xg, stream);
  if (st != FTMOE_OK) return st;
  overlap.enable();
  if (!L.grouped) {
    ftmoe_routes rt;
    memset(&rt, 0, sizeof(rt));
    rt.kind = FTMOE_ROUTES_SLOTS;
    rt.topk = s->topk;
    rt.tokens = T;
    rt.slots = args->expert_ids;
    ftmoe_act a1 = {f, 0, T, H, xq, xs, xg};
    st = ftmoe_grouped_gemm_gateup(&a1, &rt, &wg, gu, 2 * I, &tile, stream);
    if (st != FTMOE_OK) return st;
    st = ftmoe_silu_mul(gu, R, I, 2 * I, nullptr, f, aq, as, ag, stream);
    if (st != FTMOE_OK) return st;
    ftmoe_act a2 = {f, 0, R, I, aq, as, ag};
    st = ftmoe_grouped_gemm_down(&a2, &rt, &wd, y, H, &tile, stream);
    if (st != FTMOE_OK) return st;
    return ftmoe_combine(y, H, nullptr, args->expert_ids, args->route_weights, T, s->topk, H, s->out_dtype,
                         args->out, args->ld_out, stream);
  }
  uint8_t* rq = ws + L.l.rows_q;
  void* rs = ws + L.l.rows_scales;
  if (!prep && !mx) {
    st = ftmoe_segment_routes(args->expert_ids, T, s->topk, (int32_t)E, counts, offsets, dst2src,
                              route2dst, stream);
    if (st != FTMOE_OK) return st;
  }
  if (mx)
    st = ftmoe_gather_quantize_act(args->x, T, H, args->ld_x, dst2src, R, offsets + E, f, rq, rs, stream);
  else
    st = ftmoe_gather_rows_scales(xq, xs, T, (int64_t)code_row_bytes(f, H), (int64_t)scale_row_bytes(f, H), dst2src,
                                  R, offsets + E, rq, rs, stream);
  if (st != FTMOE_OK) return st;
  ftmoe_routes rt;
  memset(&rt, 0, sizeof(rt));
  rt.kind = FTMOE_ROUTES_GROUPED;
  rt.offsets = offsets;
  ftmoe_act a1 = {f, 0, R, H, rq, rs, xg};
  if (L.fused) {
    st = ftmoe_grouped_gemm_gateup_silu(&a1, &rt, &wg, aq, static_cast<float*>(as), &tile, stream);
  } else {
    st = ftmoe_grouped_gemm_gateup(&a1, &rt, &wg, gu, 2 * I, &tile, stream);
    if (st != FTMOE_OK) return st;
    st = ftmoe_silu_mul(gu, R, I, 2 * I, offsets + E, f, aq, as, ag, stream);
  }
  if (st != FTMOE_OK) return st;
  ftmoe_act a2 = {f, 0, R, I, aq, as, ag};
  if (comb)
    return down_comb(&a2, offsets, &wd, y, tile.tok_tile, dst2src, route2dst, args->route_weights, s->topk, comb_cnt,
                     args->out, args->ld_out, s->out_dtype, stream);
  st = ftmoe_grouped_gemm_down(&a2, &rt, &wd, y, H, &tile, stream);
  if (st != FTMOE_OK) return st;
  return ftmoe_combine(y, H, route2dst, args->expert_ids, args->route_weights, T, s->topk, H, s->out_dtype,
                       args->out, args->ld_out, stream);
}

ftmoe_status ftmoe_read_error_flags(uint32_t* flags) {
  if (!flags) return FTMOE_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return FTMOE_CUDA_ERROR;
  *flags = read_err_quant() | read_err_segment() | read_err_gather() | read_err_stream_gemm() |
           read_err_tc_gemm() | read_err_nvfp4() | read_err_act() | read_err_selftest() | read_err_decode() |
           read_err_slots() | read_err_mxfp8() | read_err_tc_mxfp8();
  return FTMOE_OK;
}

}  // extern "C"

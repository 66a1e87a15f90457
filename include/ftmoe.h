/*
 * libftmoe -- routed-expert block-quantized MoE FFN for NVIDIA GB300 (sm_103a).
 *
 * The path, per token row x of a top-k routed MoE layer:
 *   1. quantize x once per 1x128 group to FP8-e4m3 with an fp32 scale per group
 *      (SGLang "Gather the cutlass MoE activation and its scales in one launch",
 *      Motivation: the activation is quantized once, k//128 fp32 scales beside k fp8);
 *   2. group the active routes by expert (counts, offsets, dst2src);
 *   3. gather the FP8 rows and their scale rows in one walk of dst2src
 *      (same page, Modifications);
 *   4. grouped gate/up GEMM against FP8 expert weights with 128x128 fp32 block scales
 *      (FreeToken "perf(moe): skip inactive block-fp8 decode routes", first section);
 *   5. SiLU-and-mul, re-quantized per 1x128 for the down GEMM;
 *   6. grouped down GEMM;
 *   7. routing-weighted top-k combine into bf16 (a kernel of its own, or inside the down
 *      GEMM on its CTA-pair kernel: ftmoe_moe_forward, path 5).
 * A negative expert slot is an inactive route: its gate/up and down output tiles are
 * written as exact zeros and nothing else of it is read (FreeToken page, first section).
 *
 * Conventions for every entry point:
 *   - Pointers named in the argument lists are DEVICE pointers unless stated; the caller
 *     allocates and owns all memory. No entry point allocates, frees or synchronises
 *     (ftmoe_read_error_flags excepted), so the stream-ordered calls declared before
 *     ftmoe_moe_forward_noalloc may be captured into a CUDA graph.
 *   - All work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream).
 *     Errors of the asynchronous work surface at the caller's next synchronisation.
 *   - Argument checks run on the host before anything is enqueued and touch no device
 *     memory: a NULL pointer that is needed, a negative or inconsistent size or stride
 *     returns FTMOE_INVALID_ARG; a valid request this build cannot run returns
 *     FTMOE_UNSUPPORTED; a failed launch returns FTMOE_CUDA_ERROR.
 *   - A call with zero rows returns FTMOE_OK without launching anything.
 *   - Sizes and strides are in elements unless named *_bytes. Row bases are computed in
 *     64-bit. Index arrays are int32.
 *   - Index values that the kernels read on the device (expert ids, dst2src entries) and
 *     that fall outside their range are skipped and raise a bit in the device error word
 *     (ftmoe_read_error_flags); they never cause an out-of-bounds access.
 */
#ifndef FTMOE_H
#define FTMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ftmoe_status {
  FTMOE_OK = 0,
  FTMOE_INVALID_ARG = 1,
  FTMOE_UNSUPPORTED = 2,
  FTMOE_CUDA_ERROR = 3,
  FTMOE_WORKSPACE_TOO_SMALL = 4,
  FTMOE_CHECK_FAILED = 5
} ftmoe_status;

/* Storage formats of weights and activations. */
typedef enum ftmoe_format {
  /* FP8-e4m3 codes; activations carry one fp32 scale per 1x128 row group, weights one
   * fp32 scale per 128x128 block on the padded (ceil-div) grid. value = code * scale. */
  FTMOE_FMT_FP8 = 0,
  /* NVFP4: e2m1 codes packed two per byte (even column in the low nibble), one e4m3
   * scale per 16 consecutive elements of a row, one fp32 scale per tensor.
   * value = code * block_scale * global_scale. */
  FTMOE_FMT_NVFP4 = 1,
  /* MXFP8 (SGLang gather page, Modifications: the mxfp8 branch, a ue8m0 scale per 32):
   * e4m3 codes, one E8M0 byte b per 32 consecutive elements of a row, value = code * 2^(b -
   * 127). Quantization (OCP Microscaling recipe): shared = floor(log2(amax)) - 8, clamped to
   * [-127, 127] (zero and subnormal amax give -127), b = shared + 127, code =
   * e4m3_rne_satfinite(x * 2^-shared). No tensor scale (global_scale must be NULL). */
  FTMOE_FMT_MXFP8 = 2
} ftmoe_format;

/* Element type of the forward's output rows (FreeToken "perf(moe): skip inactive block-fp8
 * decode routes", Validation: bf16, fp16 and fp32 outputs). The combine accumulates in fp32
 * either way; bf16 and fp16 are rounded to nearest even once at the end, fp32 is stored as
 * accumulated. */
typedef enum ftmoe_out_dtype {
  FTMOE_OUT_BF16 = 0,
  FTMOE_OUT_FP16 = 1,
  FTMOE_OUT_FP32 = 2
} ftmoe_out_dtype;

/* Device error word bits (see ftmoe_read_error_flags). */
#define FTMOE_ERR_EXPERT_ID_RANGE 0x1u  /* an expert id >= num_experts was skipped */
#define FTMOE_ERR_MAP_RANGE 0x2u        /* a dst2src entry outside [0, n_src) was skipped */
#define FTMOE_ERR_WAIT_TIMEOUT 0x4u     /* a bounded pipeline wait gave up */

/* E expert matrices of shape [n, k] (row = output feature, K-major).
 * FP8:   q      uint8 [E][n][k]
 *        scales float [E][ceil(n/128)][ceil(k/128)]
 * NVFP4: q      uint8 [E][n][k/2]
 *        scales uint8 (e4m3) [E][n][k/16]
 *        global_scale float [E]
 * MXFP8: q      uint8 [E][n][k]
 *        scales uint8 (E8M0) [E][n][k/32]; the grouped GEMM needs k % 512 == 0
 * Gate/up banks hold the gate rows [0, I) then the up rows [I, 2I) of each expert. */
typedef struct ftmoe_expert_bank {
  int32_t format;      /* ftmoe_format */
  int32_t num_experts; /* E */
  int64_t n;
  int64_t k;
  const uint8_t* q;
  const void* scales;
  const float* global_scale; /* NVFP4 only; NULL for FP8 and MXFP8 */
} ftmoe_expert_bank;

/* Quantized activation rows [rows, k] in the same formats (FP8: scales float
 * [rows][ceil(k/128)]; NVFP4: q [rows][k/2], scales e4m3 [rows][k/16], global_scale
 * float[1]; MXFP8: q [rows][k], scales E8M0 [rows][k/32]). Rows are dense (row stride k,
 * resp. k/2 bytes). */
typedef struct ftmoe_act {
  int32_t format;
  int32_t reserved;
  int64_t rows;
  int64_t k;
  const uint8_t* q;
  const void* scales;
  const float* global_scale;
} ftmoe_act;

/* How activation rows and output rows relate to experts.
 * FTMOE_ROUTES_GROUPED: rows are sorted by expert; the rows of expert e are
 *   [offsets[e], offsets[e+1]) (device int32 [E+1], e.g. from ftmoe_segment_routes).
 *   Output row i belongs to activation row i. Rows >= offsets[E] are not touched.
 * FTMOE_ROUTES_SLOTS: one output row per route r in [0, tokens*topk); the route's
 *   expert is slots[r] (device int32; < 0 = inactive, the output row is written as
 *   zeros). The activation row of route r is r / topk for the gate/up GEMM (token
 *   rows) and r for the down GEMM (one intermediate row per route). */
enum { FTMOE_ROUTES_GROUPED = 0, FTMOE_ROUTES_SLOTS = 1 };
typedef struct ftmoe_routes {
  int32_t kind;
  int32_t topk;           /* SLOTS */
  int64_t tokens;         /* SLOTS */
  const int32_t* offsets; /* GROUPED */
  const int32_t* slots;   /* SLOTS */
} ftmoe_routes;

/* GEMM kernel choice. variant: 0 = automatic (SLOTS -> the HBM-streaming CUDA-core
 * kernel, GROUPED -> the tcgen05 tensor-core kernel), 1 = the streaming kernel,
 * 2 = the tcgen05 kernel. tok_tile: token columns per tensor-core tile, one of
 * 16/32/64/128; 0 = ftmoe_pick_tile's choice. wblocks: 128-row weight blocks per
 * tensor-core unit on one SM, sharing one token tile: 1, 2 (adjacent blocks; needs
 * n % 256 == 0 and k % 128 == 0, else the request is treated as unsupported by the tcgen05
 * kernel), or 0 = automatic (2 at token tile 64 where allowed, else 1). ctas: SMs per
 * tensor-core unit: 1, 2 (a CTA pair, a cluster of two CTAs on two SMs: each streams one of
 * two adjacent weight blocks and loads half of the token tile, one MMA of M = 256 covers
 * both; needs token tile 64 or 128, n % 256 == 0, k % 128 == 0 and wblocks 0 or 1, else
 * the request is treated as unsupported by the tcgen05 kernel), or 0 = automatic (2 at token
 * tile 128 where allowed and wblocks is not 2, else 1). Results do not depend on wblocks or
 * ctas: every output element is the same sum in the same order. */
typedef struct ftmoe_tile {
  int32_t tok_tile;
  int32_t variant;
  int32_t wblocks;
  int32_t ctas;
} ftmoe_tile;

const char* ftmoe_status_string(int status);

/* Token tile from route density (FreeToken "perf(dsfp4): pick the grouped-prefill tile
 * from route density on sm_89", Measurements: the best M tile tracks rows per expert,
 * 16 -> 32 -> 128 at about 6 -> 24 -> 96 rows): the smallest of 16/32/64/128 that holds
 * ceil(routes / num_experts) rows, else 128. Pure host function; out is a host pointer. */
ftmoe_status ftmoe_pick_tile(int64_t routes, int32_t num_experts, ftmoe_tile* out);

/* Per-token activation quantization of bf16 x [rows, k] (row stride ld_x elements).
 * FP8 (SGLang gather page, Motivation): per 1x128 group amax = max|x|,
 *   s = amax / 448 (IEEE fp32), q = e4m3_rne_satfinite(x / s); amax = 0 gives s = 0 and
 *   all-zero codes. q uint8 [rows][k]; scales float [rows][ceil(k/128)];
 *   global_scale must be NULL.
 * NVFP4 (requires k % 32 == 0): g = amax_tensor / 2688 is written to global_scale[0];
 *   per 16 elements sb = e4m3(amax_block / (6 g)), q = e2m1_rne(x / (sb g)).
 *   q uint8 [rows][k/2]; scales uint8 [rows][k/16].
 * MXFP8 (requires k % 32 == 0; global_scale must be NULL): per 32 elements the E8M0 byte and
 *   codes of FTMOE_FMT_MXFP8. q uint8 [rows][k]; scales uint8 [rows][k/32]. */
ftmoe_status ftmoe_quantize_act(const uint16_t* x, int64_t rows, int64_t k, int64_t ld_x,
                                int32_t format, uint8_t* q, void* scales, float* global_scale,
                                void* stream);

/* Weight-bank quantization of float32 w [E][n][k] (dense) into the layout of
 * ftmoe_expert_bank: FP8 with one scale per 128x128 block (amax / 448, padded grid),
 * NVFP4 with one global scale per expert matrix (requires k % 32 == 0), or MXFP8 with one
 * E8M0 byte per 32 elements of a row (requires k % 32 == 0; global_scale NULL). */
ftmoe_status ftmoe_quantize_weights(const float* w, int32_t num_experts, int64_t n, int64_t k,
                                    int32_t format, uint8_t* q, void* scales, float* global_scale,
                                    void* stream);

/* Expert segmenter: stable grouping of the active routes by expert.
 * expert_ids int32 [tokens*topk] (route r = t*topk + j; < 0 inactive).
 * Outputs: counts int32 [E]; offsets int32 [E+1] (exclusive prefix, offsets[E] = active
 * routes); dst2src int32 [tokens*topk] capacity, entry d < offsets[E] is the token of
 * grouped row d; route2dst int32 [tokens*topk], the grouped row of route r or -1.
 * Within an expert rows keep route order. All outputs are deterministic.
 * Passages: SGLang gather page, Motivation (the quantized activation is replicated once per
 * routed expert through a dst2src map of m * topk entries, one source token per grouped
 * row); FreeToken "perf(dsfp4): pick the grouped-prefill tile from route density on sm_89",
 * Measurements (the grouped GEMM's rows per expert, which counts[e] holds). */
ftmoe_status ftmoe_segment_routes(const int32_t* expert_ids, int64_t tokens, int32_t topk,
                                  int32_t num_experts, int32_t* counts, int32_t* offsets,
                                  int32_t* dst2src, int32_t* route2dst, void* stream);

/* Fused row + scale gather (SGLang gather page, Modifications): one walk of dst2src
 * copies, for every destination row i, the row_bytes bytes of src row dst2src[i] and
 * the scale_bytes bytes of its scale row. Bytes are copied, never decoded, so any
 * 1-byte code format works (FP8: row_bytes = k, scale_bytes = 4*ceil(k/128)).
 * src [n_src][row_bytes], src_scales [n_src][scale_bytes], dst [n_dst][row_bytes],
 * dst_scales [n_dst][scale_bytes], all dense. n_dst_dev: optional device int32 holding
 * the number of valid destination rows (<= n_dst); rows at or beyond it are left
 * untouched (lets a fixed-size launch follow a device-side count). */
ftmoe_status ftmoe_gather_rows_scales(const uint8_t* src, const void* src_scales, int64_t n_src,
                                      int64_t row_bytes, int64_t scale_bytes,
                                      const int32_t* dst2src, int64_t n_dst,
                                      const int32_t* n_dst_dev, uint8_t* dst, void* dst_scales,
                                      void* stream);

/* Gather of a bf16 activation with quantization of the gathered rows (SGLang gather page,
 * Modifications: the mxfp8 branch gathers a bf16 activation through its own kernel): for
 * every destination row d < n_dst (or < *n_dst_dev when given), the bf16 row x[dst2src[d]]
 * (row stride ld_x elements, n_src rows) is quantized into q [n_dst][k] and scales
 * [n_dst][...] in `format`'s layout. Only FTMOE_FMT_MXFP8 (k % 32 == 0); other formats
 * return FTMOE_UNSUPPORTED. Quantization is per row, so the result equals quantizing the
 * source rows and gathering the codes. A map entry outside [0, n_src) is skipped (its row
 * is left untouched) and raises FTMOE_ERR_MAP_RANGE. n_dst == 0 launches nothing. */
ftmoe_status ftmoe_gather_quantize_act(const uint16_t* x, int64_t n_src, int64_t k, int64_t ld_x,
                                       const int32_t* dst2src, int64_t n_dst, const int32_t* n_dst_dev,
                                       int32_t format, uint8_t* q, void* scales, void* stream);

/* Grouped gate/up GEMM: out[row, c] = sum over 128-wide K blocks kb of
 *   act_scale[row, kb] * w_scale[e, c/128, kb] * sum_{k in kb} a[row, k] * w[e, c, k]
 * for c in [0, w->n) (= 2I), with e the expert of the row (see ftmoe_routes). NVFP4 and
 * MXFP8 banks apply their own scales (code * block scale [* tensor scales]) inside the
 * block-scaled MMA; both take FTMOE_ROUTES_GROUPED only (k % 256 == 0, resp. k % 512 == 0).
 * a->k must equal w->k (= hidden). out float32, row stride ld_out >= w->n.
 * FTMOE_ROUTES_SLOTS: an inactive route's row is written as zeros before anything of
 * that route is read (FreeToken page, first section). tile may be NULL. */
ftmoe_status ftmoe_grouped_gemm_gateup(const ftmoe_act* a, const ftmoe_routes* routes,
                                       const ftmoe_expert_bank* w, float* out, int64_t ld_out,
                                       const ftmoe_tile* tile, void* stream);

/* Grouped gate/up GEMM with SiLU-and-mul and FP8 re-quantization in its epilogue: the
 * composition ftmoe_grouped_gemm_gateup -> ftmoe_silu_mul (FP8) without the fp32 gate/up
 * rows in between. Each tensor-core unit multiplies one token tile by gate block j (rows
 * [128 j, 128 j + 128)) and up block j (rows [I + 128 j, ...)) of the expert, so it holds
 * g and u of intermediate columns [128 j, 128 j + 128) -- one whole 1x128 group -- and
 * writes a = silu(g) * u as e4m3 codes with the group scale amax / 448. The arithmetic
 * (fp32 promotion per K block, silu, division, rounding) is that of the two separate calls,
 * so codes and scales are bit-identical to theirs.
 * FP8 only; routes must be FTMOE_ROUTES_GROUPED; w->n = 2I with I % 128 == 0 and
 * w->k % 128 == 0 (else FTMOE_UNSUPPORTED). q_out uint8 [a->rows][I], scales_out float
 * [a->rows][I / 128], dense; rows at or beyond offsets[E] are not touched. tile->variant
 * and tile->wblocks are ignored. */
ftmoe_status ftmoe_grouped_gemm_gateup_silu(const ftmoe_act* a, const ftmoe_routes* routes,
                                            const ftmoe_expert_bank* w, uint8_t* q_out,
                                            float* scales_out, const ftmoe_tile* tile, void* stream);

/* SiLU-and-mul with re-quantization (FreeToken "perf(moe): skip inactive block-fp8 decode
 * routes", first section: the activation reads the whole gate/up buffer, zero tiles of
 * inactive routes included; its Validation names SiLU-and-mul among the activations):
 * for each row, a[i] = silu(g[i]) * u[i] with
 * g = gu[row, 0:inter], u = gu[row, inter:2*inter], silu(g) = g / (1 + exp(-g)) in fp32;
 * then a is quantized like ftmoe_quantize_act (FP8: q [rows][inter], scales float
 * [rows][ceil(inter/128)]; NVFP4: q [rows][inter/2], scales [rows][inter/16],
 * global_scale float[1] taken over all valid rows; MXFP8: q [rows][inter], scales E8M0
 * [rows][inter/32], global_scale NULL). rows_dev: optional device int32
 * count of valid rows (<= rows); rows beyond it are not touched. An all-zero input
 * row gives scale 0 and zero codes. */
ftmoe_status ftmoe_silu_mul(const float* gu, int64_t rows, int64_t inter, int64_t ld_gu,
                            const int32_t* rows_dev, int32_t format, uint8_t* q, void* scales,
                            float* global_scale, void* stream);

/* Grouped down GEMM (FreeToken "perf(moe): skip inactive block-fp8 decode routes", first
 * section: gate/up and down run the same block-FP8 kernel, and an inactive route's down
 * output tile is written as zeros; SGLang gather page, Motivation: the second grouped GEMM
 * of the blockwise-FP8 MoE): the same contraction as ftmoe_grouped_gemm_gateup with
 * w->n = hidden and w->k = a->k = inter. In FTMOE_ROUTES_SLOTS mode activation row r
 * belongs to route r. */
ftmoe_status ftmoe_grouped_gemm_down(const ftmoe_act* a, const ftmoe_routes* routes,
                                     const ftmoe_expert_bank* w, float* out, int64_t ld_out,
                                     const ftmoe_tile* tile, void* stream);

/* Routing-weighted top-k combine (FreeToken "perf(moe): skip inactive block-fp8 decode
 * routes", first section: the reduction that follows the down GEMM; it reads no routing
 * weight of an inactive route):
 *   out[t, h] = round( sum_{j ascending, expert_ids[t*topk+j] >= 0}
 *                      weights[t*topk+j] * y[row(t*topk+j), h] )   (fp32 accumulate)
 * round = out_dtype's conversion (ftmoe_out_dtype: bf16 or fp16 round to nearest even, fp32
 * none). row(r) = route2dst[r] if route2dst != NULL, else r (route-major y). Inactive slots
 * are skipped without reading their weight or y row. y float [*, hidden] with row stride
 * ld_y; out [tokens, hidden] of out_dtype with row stride ld_out (elements). */
ftmoe_status ftmoe_combine(const float* y, int64_t ld_y, const int32_t* route2dst,
                           const int32_t* expert_ids, const float* weights, int64_t tokens,
                           int32_t topk, int64_t hidden, int32_t out_dtype, void* out,
                           int64_t ld_out, void* stream);

/* ------------------------------------------------------------------------------------
 * Fused forward (FreeToken "perf(moe): skip inactive block-fp8 decode routes": first
 * section, the launch shapes stay fixed and the activation still processes the zeroed
 * buffers; Validation, one CUDA graph replayed while the routes switch between all-active,
 * mixed and all-inactive and the inputs change). Launch shapes depend only on the shape
 * below, never on route content, so one captured CUDA graph can be replayed while routes
 * and inputs change in place.
 * path: 0 = automatic, 1 = route-slot streaming path (FP8 only), 2 = grouped path with
 * the separate SiLU-and-mul kernel, 3 = grouped path with SiLU-and-mul fused into the
 * gate/up GEMM (ftmoe_grouped_gemm_gateup_silu; FP8, I % 128 == 0, H % 128 == 0),
 * 4 = fused decode path: after a launch that quantizes the token rows, gate/up, SiLU-and-mul
 * with FP8 re-quantization, down and the combine run in one persistent tensor-core kernel
 * whose weight stream is split evenly over the SMs (FP8; T <= 8, T*topk <= 64, E <= 1024,
 * H and I multiples of 128, H <= 8192, I <= 2048; a token that lists one expert twice
 * computes that expert once and weights it per listing),
 * 5 = grouped path with the combine inside the down GEMM (FP8; token tile 64 or 128,
 * topk <= 8, H % 256 == 0, I % 128 == 0; out 16-byte aligned with ld_out % 4 == 0): the down GEMM runs
 * on CTA pairs, counts the arrivals of each token's routes per 128 columns and, at the last,
 * adds the token's rows in ascending slot order with the combine's expression and rounding
 * (decode page, first section: the reduction after the down GEMM), so no fp32 row has to
 * travel back from HBM. The down buffer's contents are undefined after such a call (its rows
 * are dropped from L2 once added), and the arrival counters live in the workspace's
 * counters region (zeroed by the call itself).
 * Automatic: the fused decode path where its limits hold; else the grouped path, fused where
 * the token tile is at most 64, the bank has at most 1024 experts and the routes can reach at
 * least 2048 (expert, gate/up block pair) units (min(T*topk, E) * I/128 >= 2048), else with
 * the separate kernel, and the combine kernel (path 5 measured slower on GB300: 6.2 ms
 * against 2.6 ms for 24,576 routes of 7168/2048, its per-token round trips to memory waiting
 * behind the weight stream). Paths 2, 3 and 5 give bit-identical outputs; path 4 adds the partial sums of a gate/up
 * element in another order, so it agrees with them within the fp32 rounding of that sum.
 * NVFP4 and MXFP8 take the grouped path with the separate SiLU-and-mul kernel only (paths 0
 * and 2; 1, 3 and 4 return FTMOE_UNSUPPORTED). MXFP8 segments the routes first, then
 * gathers the bf16 token rows and quantizes the gathered rows (ftmoe_gather_quantize_act);
 * its GEMMs need H % 512 == 0 and I % 512 == 0.
 * ------------------------------------------------------------------------------------ */
typedef struct ftmoe_moe_shape {
  int64_t tokens;     /* T */
  int64_t hidden;     /* H */
  int64_t inter;      /* I (per expert) */
  int32_t topk;
  int32_t num_experts;
  int32_t format;     /* ftmoe_format of weights and activations */
  int32_t tok_tile;   /* 0 = ftmoe_pick_tile(T*topk, E) */
  int32_t path;
  int32_t out_dtype;  /* ftmoe_out_dtype of out (0 = bf16) */
} ftmoe_moe_shape;

typedef struct ftmoe_moe_args {
  ftmoe_moe_shape shape;
  const uint16_t* x;          /* bf16 [T][ld_x] */
  int64_t ld_x;
  const int32_t* expert_ids;  /* int32 [T*topk], < 0 inactive */
  const float* route_weights; /* float [T*topk]; entries of inactive routes are never read */
  ftmoe_expert_bank w_gateup; /* n = 2I, k = H */
  ftmoe_expert_bank w_down;   /* n = H, k = I */
  void* out;                  /* [T][ld_out] elements of shape.out_dtype */
  int64_t ld_out;
} ftmoe_moe_args;

/* Byte offsets of the intermediate buffers inside the forward workspace (each 256-byte
 * aligned). Offsets of buffers a path does not use are 0 with size 0. */
typedef struct ftmoe_workspace_layout {
  size_t x_q, x_scales, x_gscale;            /* quantized token rows */
  size_t counts, offsets, dst2src, route2dst; /* segmenter (grouped path) */
  size_t rows_q, rows_scales;                /* gathered rows (grouped path) */
  size_t gateup, gateup_bytes;               /* float gate/up output [R][2I] (not in path 3) */
  size_t act_q, act_q_bytes, act_scales, act_scales_bytes, act_gscale;
  size_t down, down_bytes;                   /* float down output [R][H] */
  size_t partials, partials_bytes;           /* fused decode path: gate/up partial sums */
  size_t counters, counters_bytes;           /* arrival counters: fused decode path, and the
                                                combine inside the down GEMM ([T][H/128]) */
  size_t total;
} ftmoe_workspace_layout;

size_t ftmoe_forward_workspace_bytes(const ftmoe_moe_shape* shape);
ftmoe_status ftmoe_forward_workspace_layout(const ftmoe_moe_shape* shape,
                                            ftmoe_workspace_layout* out);
ftmoe_status ftmoe_moe_forward(const ftmoe_moe_args* args, void* workspace, size_t workspace_bytes,
                               void* stream);

/* Allocation-free variant of ftmoe_moe_forward (no counterpart in the pages; a service of
 * this library). For callers that cannot allocate device memory themselves: a plugin
 * hosted by a runtime that owns all device memory and exposes no allocator, or a latency
 * path that cannot afford an allocation's implicit synchronisation. The intermediates
 * live in a file-scope device array of 16 MiB that every GPU loading the library keeps
 * until the process exits; shapes whose workspace (ftmoe_forward_workspace_bytes)
 * exceeds it return FTMOE_WORKSPACE_TOO_SMALL. Decode-size shapes fit (8 tokens, top-8,
 * hidden 4096, intermediate 1024 need about 9.2 MiB on the fused decode path).
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 * with that device current and caches it; make that first call before any stream capture.
 * The cached address belongs to the device's primary context: after the context is
 * destroyed and recreated (cudaDeviceReset), the array lives at a new address and the
 * library must be reloaded. Every call on a device shares the one array: calls whose GPU
 * work overlaps (other streams, other threads) race on it and must be serialised by the
 * caller. The forward writes every region of the array before reading it, so a previous
 * call's contents are never used. No cudaMalloc, cudaFree or allocating library routine is
 * called. Inputs, outputs and their ownership are as for ftmoe_moe_forward. */
ftmoe_status ftmoe_moe_forward_noalloc(const ftmoe_moe_args* args, void* stream);

/* Device-side expert-slot pool, one decode step per call (FreeToken hybrid expert-cache page,
 * the pull request that speeds up victim selection in its ensure-experts kernel: Summary,
 * Change and Fix). It keeps a pool of num_slots expert slots on the device and turns a step's
 * routes into slot ids for the forward (a slot id in expert_ids, -1 for a route whose expert
 * is not resident and runs elsewhere):
 *   1. every requested expert that is resident marks its slot used: slot_usage = step, which
 *      makes it the most recently used slot of the pool;
 *   2. the distinct requested experts that are not resident, in order of first appearance
 *      among the routes and at most max_fetch of them, each take the least recently used slot
 *      among those not used in this step (slot_usage < step), ties to the lowest slot; the
 *      slot's previous expert is evicted and fetch_plan[i] = {slot, expert} (int32 pairs,
 *      host's copy list) for i < *n_fetch; when every slot was used in this step the
 *      remaining misses stay missing;
 *   3. expert_ids[r] is rewritten in place to the slot of its expert, or -1 -- after every
 *      route has been read.
 * State (device, owned by the caller, updated in place): slot_expert int32 [num_slots] (expert
 * held, -1 empty), slot_usage int64 [num_slots] (step of last use, -1 never; start with -1),
 * expert_slot int32 [num_experts] (slot of expert e, -1 if not resident); the two maps must be
 * inverse to each other (an empty pool: all -1). step must exceed every slot_usage entry.
 * expert_ids int32 [routes] (< 0 inactive; ids >= num_experts are treated as inactive and
 * raise FTMOE_ERR_EXPERT_ID_RANGE). fetch_plan int32 [max_fetch][2]; n_fetch device int32.
 * Limits: routes <= 16384, num_experts <= 16384 (else FTMOE_INVALID_ARG). One CTA; the
 * results are deterministic. */
ftmoe_status ftmoe_expert_slots(int32_t* expert_ids, int64_t routes, int32_t* slot_expert, int64_t* slot_usage,
                                int32_t num_slots, int32_t* expert_slot, int32_t num_experts, int64_t step,
                                int32_t max_fetch, int32_t* fetch_plan, int32_t* n_fetch, void* stream);

/* Self-test of the bounded pipeline waits (failure detection; the pages have no counterpart).
 * Every wait of the TMA/tensor-core pipelines gives up after a time limit (4 s), raises
 * FTMOE_ERR_WAIT_TIMEOUT in the device error word and lets its kernel return normally, so a
 * stalled pipeline never hangs the GPU. This call launches one CTA whose single waiting
 * thread runs that same bounded wait on a shared-memory mbarrier nothing ever arrives on,
 * with the limit timeout_ns (1 us .. 1 s, else FTMOE_INVALID_ARG). The wait runs out, the
 * kernel raises FTMOE_ERR_WAIT_TIMEOUT and returns; ftmoe_read_error_flags reports the bit.
 * elapsed_ns: optional device pointer receiving the nanoseconds the wait took before it
 * gave up (0 if it completed, which cannot happen). */
ftmoe_status ftmoe_selftest_wait_timeout(uint64_t timeout_ns, unsigned long long* elapsed_ns, void* stream);

/* Self-test of the quantizers' division (step 1 of the path: x divided by the group scale
 * s = amax/448, gather page, Motivation). The FP8 activation and SiLU-and-mul quantizers form
 * one reciprocal per group and correct each quotient with one fused multiply-add (Markstein's
 * method), which must give exactly the IEEE quotient. This call compares that division with
 * the IEEE one (__fdiv_rn) on the device, bit for bit: every divisor mantissa at three
 * exponents against 4096 dividends each, and 1024 divisors against every dividend mantissa
 * (111.7 G quotients). counts: device uint64[2], set to {quotients checked, quotients that
 * differ}; read them after the stream's work completes. NULL counts: FTMOE_INVALID_ARG. */
ftmoe_status ftmoe_selftest_shared_division(unsigned long long* counts, void* stream);

/* Reads and clears the device error word of the current device (FTMOE_ERR_* bits) into
 * *flags (host pointer). Synchronises the device; not for use inside graph capture. */
ftmoe_status ftmoe_read_error_flags(uint32_t* flags);

#ifdef __cplusplus
}
#endif
#endif /* FTMOE_H */

// Host-side launchers shared between the libftmoe translation units (not exported).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ftmoe.h"

namespace ftmoe {

inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Whether launches from this host thread may overlap the previous kernel on the stream
// (programmatic dependent launch). Set by the fused forward for its kernels after the
// first; every kernel waits for its predecessor's data (pdl_wait) before touching it.
//
// Ordering invariant the tensor-core GEMMs rely on: they read the segment offsets before
// their own pdl_wait, so the segmenter (or the prep kernel) must have completed by the time
// a GEMM starts. That holds as long as every kernel launched between the segmenter and a
// GEMM either waits before it triggers its dependents (the gather and the GEMMs do), or
// is itself launched only after a kernel that did (the FP8 SiLU-and-mul kernel triggers
// first, but it follows the gate/up GEMM, which has waited for the gather, which waited
// for the segmenter). A new kernel placed between the segmenter and a GEMM must wait
// before it triggers.
bool& pdl_enabled();

template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                                 bool allow_overlap, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  if (allow_overlap && pdl_enabled()) {
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same as launch_kernel, in clusters of cluster_x CTAs along x (grid.x a multiple of it).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                         cudaStream_t st, bool allow_overlap, int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cluster_x;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (allow_overlap && pdl_enabled()) ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Clusters of cluster_x CTAs of this kernel that can be resident at once on the device (0 if
// the query fails).
template <typename... KArgs>
inline int max_active_clusters(void (*kernel)(KArgs...), dim3 block, size_t smem, int cluster_x, int grid_x) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid_x);
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cluster_x;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) return 0;
  return n;
}

// tc_gemm.cu: host helpers shared by the TMA-fed kernels
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn encode_fn();  // cuTensorMapEncodeTiled from the driver, or NULL
int sm_count();
// 128B-swizzled uint8 tensor map of rank 2 or 3 (dims innermost first, byte strides of the
// outer dims); false if the driver entry point is missing or the encoding is rejected
bool encode_u8_tmap(CUtensorMap* map, const void* base, int rank, const uint64_t* dims, const uint64_t* strides,
                    const uint32_t* box);
// the same without swizzle (small tiles such as scale rows)
bool encode_u8_tmap_plain(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                          const uint64_t* strides, const uint32_t* box);

// quant.cu
cudaError_t launch_quantize_act_fp8(const uint16_t* x, int64_t rows, int64_t k, int64_t ld_x,
                                    uint8_t* q, float* scales, cudaStream_t s);
cudaError_t launch_quantize_act_nvfp4(const uint16_t* x, int64_t rows, int64_t k, int64_t ld_x,
                                      uint8_t* q, uint8_t* scales, float* gscale, cudaStream_t s);
cudaError_t launch_quantize_weights_fp8(const float* w, int32_t E, int64_t n, int64_t k,
                                        uint8_t* q, float* scales, cudaStream_t s);
cudaError_t launch_quantize_weights_nvfp4(const float* w, int32_t E, int64_t n, int64_t k,
                                          uint8_t* q, uint8_t* scales, float* gscale,
                                          cudaStream_t s);
uint32_t read_err_quant();

// segment.cu
cudaError_t launch_segment(const int32_t* ids, int64_t routes, int32_t topk, int32_t E,
                           int32_t* counts, int32_t* offsets, int32_t* dst2src,
                           int32_t* route2dst, cudaStream_t s);
// the fused forward's first kernel: FP8 quantization of x and the segmenter in one grid.
// For the down GEMM's fused combine it also
// zeroes the arrival counters (zero_words words, may be NULL) and writes a zero output row
// for every token without an active route (out_rows: [rows][ld_out] elements of out_bytes
// bytes, hidden of them per row; NULL when the combine runs as its own kernel).
struct PrepCombine {
  uint32_t* zero_words;
  int64_t n_zero_words;
  void* out_rows;
  int64_t ld_out;
  int32_t out_bytes;
  int64_t hidden;
};
cudaError_t launch_prep_fp8(const uint16_t* x, int64_t rows, int64_t k, int64_t ld_x, uint8_t* q, float* scales,
                            const int32_t* ids, int64_t routes, int32_t topk, int32_t E, int32_t* counts,
                            int32_t* offsets, int32_t* dst2src, int32_t* route2dst, const PrepCombine& pc,
                            cudaStream_t s);
uint32_t read_err_segment();

// gather.cu
cudaError_t launch_gather(const uint8_t* src, const uint8_t* src_scales, int64_t n_src,
                          int64_t row_bytes, int64_t scale_bytes, const int32_t* dst2src,
                          int64_t n_dst, const int32_t* n_dst_dev, uint8_t* dst,
                          uint8_t* dst_scales, cudaStream_t s);
uint32_t read_err_gather();

// stream_gemm.cu: HBM-streaming CUDA-core GEMM (route slots or grouped rows)
struct StreamGemmArgs {
  const uint8_t* a_q;      // activation codes [rows][k]
  const float* a_s;        // [rows][ceil(k/128)]
  const uint8_t* w_q;      // [E][n][k]
  const float* w_s;        // [E][ceil(n/128)][ceil(k/128)]
  float* out;              // [*][ld_out]
  int64_t ld_out;
  int64_t n, k;
  int32_t E;
  int32_t grouped;         // 1: GROUPED layout via offsets, 0: SLOTS
  const int32_t* offsets;  // GROUPED
  int64_t a_rows;          // GROUPED: rows of the activation and output buffers
  const int32_t* slots;    // SLOTS
  int64_t routes;          // SLOTS: tokens * topk
  int32_t act_div;         // SLOTS: activation row of route r is r / act_div
  int32_t topk;            // SLOTS
};
// largest K the streaming kernel stages (64 K blocks of fp16 activation codes)
constexpr int64_t kStreamMaxK = 8192;
cudaError_t launch_stream_gemm(const StreamGemmArgs& a, cudaStream_t s);
uint32_t read_err_stream_gemm();

// tc_gemm.cu: tcgen05 grouped GEMM
struct TcGemmArgs {
  const uint8_t* a_q;
  const float* a_s;
  int64_t a_rows;          // allocated rows of the activation buffer
  const uint8_t* w_q;
  const float* w_s;
  float* out;
  int64_t ld_out;
  int64_t n, k;
  int32_t E;
  const int32_t* offsets;
  int32_t tok_tile;
  int32_t wblocks;         // 1: one 128-row weight block per unit, 2: two adjacent blocks
  int32_t ctas;            // 1: a unit on one SM; 2: a CTA pair (cluster of two), one block each
  int32_t silu;            // 1: gate block j + up block j per unit, SiLU-and-mul + FP8 requant
  uint8_t* q_out;          // silu: codes [a_rows][n/2]
  float* s_out;            // silu: scales [a_rows][n/256]
  // comb (CTA pair only): the routing-weighted combine of the rows into out_c inside the
  // GEMM; out keeps the rows only until they are combined (their L2 lines are dropped)
  int32_t comb;
  const int32_t* dst2src;    // grouped row -> token
  const int32_t* route2dst;  // route -> grouped row or -1
  const float* rw;           // routing weights [tokens][topk]
  uint32_t* cnt;             // [tokens][ceil(n/128)] zero-initialised arrival counters
  void* out_c;               // [tokens][ld_c] of out_dtype
  int64_t ld_c;
  int32_t topk, out_dtype;
};
// whether an n x k weight matrix can run two weight blocks per unit (n % 256, k % 128)
bool tc_gemm_pairs_ok(int64_t n, int64_t k);
// whether the down GEMM with these buffers can run with the combine inside (CTA pair at
// token tile 64 or 128, whole block pairs, 128-byte aligned rows of y, 16-byte aligned output rows)
bool tc_gemm_comb_ok(int tok_tile, int64_t n, int64_t k, const void* y, int64_t ld_y, const void* out_c,
                     int64_t ld_c);
// largest expert count the tensor-core GEMM's unit table holds (tc::kMaxExperts in
// tc_gemm.cu, which refuses larger banks as unsupported)
constexpr int32_t kTcGemmMaxExperts = 1024;
cudaError_t launch_tc_gemm(const TcGemmArgs& a, cudaStream_t s, int* unsupported);
uint32_t read_err_tc_gemm();

// tc_nvfp4.cu: grouped NVFP4 GEMM on the block-scaled tcgen05 MMA
struct NvGemmArgs {
  const uint8_t* a_q;       // e2m1 codes [a_rows][k/2]
  const uint8_t* a_sf;      // e4m3 block scales [a_rows][k/16]
  const float* a_gscale;    // device float[1]
  int64_t a_rows;
  const uint8_t* w_q;       // [E][n][k/2]
  const uint8_t* w_sf;      // [E][n][k/16]
  const float* w_gscale;    // device float[E]
  float* out;
  int64_t ld_out;
  int64_t n, k;
  int32_t E;
  const int32_t* offsets;
  int32_t tok_tile;
};
cudaError_t launch_nvfp4_gemm(const NvGemmArgs& a, cudaStream_t s, int* unsupported);
uint32_t read_err_nvfp4();

// tc_mxfp8.cu: block-scaled MXFP8 grouped GEMM (kind::mxf8f6f4)
struct MxGemmArgs {
  const uint8_t* a_q;       // e4m3 codes [a_rows][k]
  const uint8_t* a_sf;      // E8M0 scale bytes [a_rows][k/32]
  int64_t a_rows;
  const uint8_t* w_q;       // [E][n][k]
  const uint8_t* w_sf;      // [E][n][k/32]
  float* out;
  int64_t ld_out;
  int64_t n, k;
  int32_t E;
  const int32_t* offsets;
  int32_t tok_tile;
};
cudaError_t launch_mxfp8_gemm(const MxGemmArgs& a, cudaStream_t s, int* unsupported);
uint32_t read_err_tc_mxfp8();

// mxfp8.cu: MXFP8 quantization (E8M0 scale per 32 elements of a row, k % 32 == 0)
// bf16 rows [rows][k] (stride ld_x); with map, destination row d reads source row map[d]
// (entries outside [0, n_src) raise FTMOE_ERR_MAP_RANGE and leave the row untouched);
// n_dev: optional device count of destination rows to write
cudaError_t launch_mxfp8_quant_bf16(const uint16_t* x, int64_t rows, int64_t k, int64_t ld_x, const int32_t* map,
                                    int64_t n_src, const int32_t* n_dev, uint8_t* q, uint8_t* s, cudaStream_t st);
cudaError_t launch_mxfp8_quant_f32(const float* x, int64_t rows, int64_t k, int64_t ld_x, uint8_t* q, uint8_t* s,
                                   cudaStream_t st);
cudaError_t launch_silu_mul_mxfp8(const float* gu, int64_t rows, int64_t inter, int64_t ld_gu, const int32_t* rows_dev,
                                  uint8_t* q, uint8_t* s, cudaStream_t st);
uint32_t read_err_mxfp8();

// act.cu: silu_mul and combine
cudaError_t launch_silu_mul_fp8(const float* gu, int64_t rows, int64_t inter, int64_t ld_gu,
                                const int32_t* rows_dev, uint8_t* q, float* scales,
                                cudaStream_t s);
cudaError_t launch_silu_mul_nvfp4(const float* gu, int64_t rows, int64_t inter, int64_t ld_gu,
                                  const int32_t* rows_dev, uint8_t* q, uint8_t* scales,
                                  float* gscale, cudaStream_t s);
cudaError_t launch_combine(const float* y, int64_t ld_y, const int32_t* route2dst,
                           const int32_t* ids, const float* w, int64_t tokens, int32_t topk,
                           int64_t hidden, int32_t out_dtype, void* out, int64_t ld_out, cudaStream_t s);
uint32_t read_err_act();

// selftest.cu
uint32_t read_err_selftest();

// slot_pool.cu: device-side expert-slot pool (one CTA; routes and experts staged in shared memory)
constexpr int64_t kSlotPoolMaxRoutes = 16384;
constexpr int32_t kSlotPoolMaxExperts = 16384;
uint32_t read_err_slots();

// decode_fused.cu: the fused decode forward (prep launch + one persistent kernel)
constexpr int kDecodeMaxTokens = 8;     // token columns the kernel keeps
constexpr int kDecodeMaxRoutes = 64;    // tokens * topk
constexpr int kDecodeMaxExperts = 1024; // bitmap of active experts
constexpr int kDecodeGrid = 152;        // persistent CTAs (at most; one per SM)
constexpr int kDecodeMaxChunks = 2048;  // gate/up chunks the partial sums are sized for (8 MiB)
constexpr int kDecodeMaxKch = 8;        // chunks per gate/up block
struct DecodePlan {
  bool ok;
  int KB, KB2, NJ, NB, HB;  // H/128, I/128, I/128, 2I/128, H/128
  int kbs_g, kbs_d;         // K blocks per TMA stage (gate/up, down)
  int u_max;                // most distinct experts the routes can reach
  int kch, ckb;             // chunks per gate/up block, K blocks per chunk
  size_t part_bytes;        // partial sums [u_max * NB * kch][8][128] float
  size_t cnt_words;         // counters: pairs, experts, (token, H block)
};
DecodePlan decode_plan(int64_t T, int32_t topk, int32_t E, int64_t H, int64_t I);
struct DecodeArgs {
  const uint8_t* x_q;   // [16][H] (rows >= T zero), from the prep launch
  const float* x_s;     // [16][H/128]
  const int32_t* ids;
  const float* rw;
  const uint8_t* wg_q;
  const float* wg_s;
  const uint8_t* wd_q;
  const float* wd_s;
  uint8_t* act_q;       // [T*topk][I]
  float* act_s;         // [T*topk][I/128]
  float* y;             // [T*topk][H]
  float* part;
  uint32_t* cnt;
  void* out;
  int64_t ld_out;
  int32_t out_dtype;
  int64_t T, H, I;
  int32_t topk, E;
};
cudaError_t launch_decode_prep(const uint16_t* x, int64_t T, int64_t H, int64_t ld_x, uint8_t* xq, float* xs,
                               const int32_t* ids, int32_t topk, int32_t E, uint32_t* cnt, size_t ncnt, void* out,
                               int64_t ld_out, int32_t out_dtype, cudaStream_t s);
cudaError_t launch_decode_fused(const DecodeArgs& a, const DecodePlan& pl, cudaStream_t s, int* unsupported);
uint32_t read_err_decode();

}  // namespace ftmoe

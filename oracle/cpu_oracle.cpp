// Plain CPU oracle of the routed-expert block-quantized MoE FFN, in C++.
//
// TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's CPU-baseline
// leg may load it; the CUDA library never does, and the two share no code. It restates each
// step from its definition, as the numpy oracle beside it does, and the tests hold the two
// to each other (bit for bit where the result is a code, a scale or an index):
//
//   * FP8 E4M3 (OCP "fn"): sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent field 0
//     is subnormal (2^-6 * m/8); 0x7F / 0xFF are NaN; largest finite 448. E2M1: sign, 2
//     exponent bits (bias 1), 1 mantissa bit; magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6.
//     Encoding rounds to the nearest representable magnitude, a tie to the code whose last
//     bit is 0, saturating at the largest finite magnitude; the sign is kept.
//   * Activation quantization per 1x128 group (SGLang "Gather the cutlass MoE activation and
//     its scales in one launch", Motivation) and weight quantization per 128x128 block
//     (FreeToken "perf(moe): skip inactive block-fp8 decode routes"): amax = max|x|,
//     s = fl32(amax / 448), q = e4m3(fl32(x / s)); amax = 0 gives s = 0 and zero codes.
//   * NVFP4 (the format the dsfp4 density page names; two-level recipe): g = fl32(amax / 2688)
//     per tensor, sb = e4m3(fl32(amax_16 / fl32(6 g))) per 16 elements, eff = fl32(sb * g),
//     q = e2m1(fl32(x / eff)), zero codes where eff = 0.
//   * MXFP8 (the SGLang gather page's mxfp8 branch: a ue8m0 scale per 32; OCP Microscaling
//     recipe): per 32 elements of a row, shared = floor(log2(amax)) - 8 clamped to
//     [-127, 127] (amax = 0 gives -127), scale byte = shared + 127, q = e4m3(x / 2^shared);
//     value = e4m3(q) * 2^(byte - 127).
//   * Segmentation: a stable grouping of the active routes by expert (counting sort).
//   * Gather: byte copies of a row and its scale row by the map.
//   * The FFN: dequantize (code x scale, exact in double), gate/up and down products in
//     double, silu(g) * u in double with g the first half of the gate/up row, the
//     intermediate re-quantized from its float32 value, and the routing-weighted sum over the
//     active slots in ascending order in double. Negative expert ids are inactive routes:
//     nothing of them is read.
//
// Threads: the forward splits its routes by expert over `threads` std::threads; every value
// is computed by one thread in one fixed order, so the result does not depend on the count.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

constexpr int kGroup = 128;     // activation group width, weight block edge
constexpr int kNvBlock = 16;    // elements per NVFP4 block scale
constexpr int kMxBlock = 32;    // elements per MXFP8 scale byte
constexpr int kE8M0Bias = 127;
constexpr int kE4M3Emax = 8;    // exponent of E4M3's largest power of two (256)
constexpr float kE4M3Max = 448.0f;
constexpr float kE2M1Max = 6.0f;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------- number formats

double e4m3_value(uint8_t code) {
  const double sign = (code & 0x80) ? -1.0 : 1.0;
  const int exp = (code >> 3) & 0xF, man = code & 0x7;
  if (exp == 0xF && man == 0x7) return std::nan("");
  if (exp == 0) return sign * std::ldexp(man / 8.0, -6);
  return sign * std::ldexp(1.0 + man / 8.0, exp - 7);
}

double e2m1_value(uint8_t code) {
  const double sign = (code & 0x8) ? -1.0 : 1.0;
  const int exp = (code >> 1) & 0x3, man = code & 0x1;
  if (exp == 0) return sign * (man / 2.0);
  return sign * std::ldexp(1.0 + man / 2.0, exp - 1);
}

struct Tables {
  double e4m3[256];
  double e2m1[16];
  std::vector<double> pos4;  // magnitudes of codes 0x00 .. 0x7E, increasing
  std::vector<double> pos2;  // magnitudes of codes 0x0 .. 0x7, increasing
  Tables() {
    for (int c = 0; c < 256; ++c) e4m3[c] = e4m3_value((uint8_t)c);
    for (int c = 0; c < 16; ++c) e2m1[c] = e2m1_value((uint8_t)c);
    for (int c = 0; c <= 0x7E; ++c) pos4.push_back(e4m3[c]);
    for (int c = 0; c <= 0x7; ++c) pos2.push_back(e2m1[c]);
  }
};

const Tables& tables() {
  static const Tables t;
  return t;
}

// Nearest entry of the increasing magnitude table to mag (>= 0, finite): walk up while the
// next entry is closer; on an exact tie take the even index; past the last entry, the last.
int nearest(const std::vector<double>& table, double mag) {
  int i = 0;
  const int last = (int)table.size() - 1;
  while (i < last) {
    const double below = mag - table[i], above = table[i + 1] - mag;
    if (above < below) {
      ++i;
    } else if (above == below) {
      if ((i + 1) % 2 == 0) ++i;
      break;
    } else {
      break;
    }
  }
  return i;
}

uint8_t encode_e4m3(double v) {
  if (std::isnan(v)) return 0x7F;
  const int c = nearest(tables().pos4, std::fabs(v));
  return (uint8_t)(std::signbit(v) ? (c | 0x80) : c);
}

uint8_t encode_e2m1(double v) {
  const int c = nearest(tables().pos2, std::fabs(v));
  return (uint8_t)(std::signbit(v) ? (c | 0x8) : c);
}

// ---------------------------------------------------------------- quantizers

// One group or block of float values -> codes and its scale (decisions in float32).
float quantize_fp8_values(const float* v, int64_t n, int64_t stride_row, int64_t rows, uint8_t* q,
                          int64_t q_stride) {
  float amax = 0.0f;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t i = 0; i < n; ++i) amax = std::fmax(amax, std::fabs(v[r * stride_row + i]));
  if (amax == 0.0f) {
    for (int64_t r = 0; r < rows; ++r)
      for (int64_t i = 0; i < n; ++i) q[r * q_stride + i] = 0;
    return 0.0f;
  }
  const float s = amax / kE4M3Max;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t i = 0; i < n; ++i) {
      const float scaled = v[r * stride_row + i] / s;
      q[r * q_stride + i] = encode_e4m3((double)scaled);
    }
  return s;
}

void quantize_act_fp8(const float* x, int64_t rows, int64_t k, uint8_t* q, float* s) {
  const int64_t ng = ceil_div(k, kGroup);
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t g = 0; g < ng; ++g) {
      const int64_t c0 = g * kGroup, w = std::min<int64_t>(kGroup, k - c0);
      s[r * ng + g] = quantize_fp8_values(x + r * k + c0, w, 0, 1, q + r * k + c0, 0);
    }
}

void quantize_weight_fp8(const float* w, int64_t n, int64_t k, uint8_t* q, float* s) {
  const int64_t nb = ceil_div(n, kGroup), kb = ceil_div(k, kGroup);
  for (int64_t i = 0; i < nb; ++i)
    for (int64_t j = 0; j < kb; ++j) {
      const int64_t r0 = i * kGroup, c0 = j * kGroup;
      const int64_t h = std::min<int64_t>(kGroup, n - r0), wd = std::min<int64_t>(kGroup, k - c0);
      s[i * kb + j] = quantize_fp8_values(w + r0 * k + c0, wd, k, h, q + r0 * k + c0, k);
    }
}

float nvfp4_global(float amax) { return amax / (kE4M3Max * kE2M1Max); }

void quantize_nvfp4(const float* x, int64_t rows, int64_t k, float global_amax, uint8_t* q, uint8_t* sb,
                    float* g_out) {
  const float g = nvfp4_global(global_amax);
  *g_out = g;
  const int64_t nblk = ceil_div(k, kNvBlock);
  if (g == 0.0f) {
    std::memset(q, 0, (size_t)(rows * k));
    std::memset(sb, 0, (size_t)(rows * nblk));
    return;
  }
  const float six_g = kE2M1Max * g;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < nblk; ++b) {
      const int64_t c0 = b * kNvBlock, w = std::min<int64_t>(kNvBlock, k - c0);
      float amax = 0.0f;
      for (int64_t i = 0; i < w; ++i) amax = std::fmax(amax, std::fabs(x[r * k + c0 + i]));
      const float ratio = amax / six_g;
      const uint8_t code = encode_e4m3((double)ratio);
      sb[r * nblk + b] = code;
      const float eff = (float)tables().e4m3[code] * g;
      for (int64_t i = 0; i < w; ++i) {
        if (eff == 0.0f) {
          q[r * k + c0 + i] = 0;
        } else {
          const float scaled = x[r * k + c0 + i] / eff;
          q[r * k + c0 + i] = encode_e2m1((double)scaled);
        }
      }
    }
}

// floor(log2(amax)) - 8 clamped to [-127, 127]; amax = 0 gives -127. frexp writes amax as
// m * 2^e with m in [0.5, 1), so floor(log2(amax)) = e - 1 with no logarithm taken.
int mx_shared_exp(float amax) {
  const double a = (double)amax;
  if (a == 0.0) return -kE8M0Bias;
  int e = 0;
  (void)std::frexp(a, &e);
  return std::min(kE8M0Bias, std::max(-kE8M0Bias, (e - 1) - kE4M3Emax));
}

// Rows of x -> e4m3 codes and one E8M0 byte per 32 elements (a partial last block takes its
// amax over its valid elements). Dividing by 2^shared is exact in double.
void quantize_mxfp8(const float* x, int64_t rows, int64_t k, uint8_t* q, uint8_t* sb) {
  const int64_t nblk = ceil_div(k, kMxBlock);
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < nblk; ++b) {
      const int64_t c0 = b * kMxBlock, w = std::min<int64_t>(kMxBlock, k - c0);
      float amax = 0.0f;
      for (int64_t i = 0; i < w; ++i) amax = std::fmax(amax, std::fabs(x[r * k + c0 + i]));
      const int e = mx_shared_exp(amax);
      sb[r * nblk + b] = (uint8_t)(e + kE8M0Bias);
      for (int64_t i = 0; i < w; ++i) q[r * k + c0 + i] = encode_e4m3((double)x[r * k + c0 + i] * std::ldexp(1.0, -e));
    }
}

// ---------------------------------------------------------------- dequantized views

// Row r of an FP8 activation / weight matrix with 128-wide scale groups, in double.
struct Fp8Rows {
  const uint8_t* q;
  const float* s;
  int64_t k, scale_cols, rows_per_scale;  // rows_per_scale: 1 (activations) or 128 (weights)
  double at(int64_t r, int64_t c) const {
    return tables().e4m3[q[r * k + c]] * (double)s[(r / rows_per_scale) * scale_cols + c / kGroup];
  }
};

struct Nvfp4Rows {
  const uint8_t* q;   // unpacked codes 0..15
  const uint8_t* sb;  // e4m3 codes, one per 16 elements
  float g;
  int64_t k;
  double at(int64_t r, int64_t c) const {
    return tables().e2m1[q[r * k + c] & 0xF] * tables().e4m3[sb[r * ceil_div(k, kNvBlock) + c / kNvBlock]] *
           (double)g;
  }
};

struct MxRows {
  const uint8_t* q;   // e4m3 codes
  const uint8_t* sb;  // E8M0 bytes, one per 32 elements
  int64_t k;
  double at(int64_t r, int64_t c) const {
    return tables().e4m3[q[r * k + c]] * std::ldexp(1.0, (int)sb[r * ceil_div(k, kMxBlock) + c / kMxBlock] - kE8M0Bias);
  }
};

struct Route {
  int64_t t;
  int j;
};

}  // namespace

extern "C" {

double ftor_e4m3_decode(uint8_t c) { return tables().e4m3[c]; }
double ftor_e2m1_decode(uint8_t c) { return tables().e2m1[c & 0xF]; }
uint8_t ftor_e4m3_encode(double v) { return encode_e4m3(v); }
uint8_t ftor_e2m1_encode(double v) { return encode_e2m1(v); }

void ftor_quantize_act_fp8(const float* x, int64_t rows, int64_t k, uint8_t* q, float* s) {
  quantize_act_fp8(x, rows, k, q, s);
}

void ftor_quantize_weight_fp8(const float* w, int64_t n, int64_t k, uint8_t* q, float* s) {
  quantize_weight_fp8(w, n, k, q, s);
}

float ftor_nvfp4_global_scale(float amax) { return nvfp4_global(amax); }

void ftor_quantize_nvfp4(const float* x, int64_t rows, int64_t k, float global_amax, uint8_t* q, uint8_t* sb,
                         float* g) {
  quantize_nvfp4(x, rows, k, global_amax, q, sb, g);
}

int ftor_mx_shared_exp(float amax) { return mx_shared_exp(amax); }

void ftor_quantize_mxfp8(const float* x, int64_t rows, int64_t k, uint8_t* q, uint8_t* sb) {
  quantize_mxfp8(x, rows, k, q, sb);
}

// Stable grouping of the active routes by expert. Returns 0, or -1 if an id >= E.
int ftor_segment(const int32_t* ids, int64_t tokens, int32_t topk, int32_t E, int32_t* counts,
                 int32_t* offsets, int32_t* dst2src, int32_t* route2dst) {
  const int64_t R = tokens * topk;
  for (int64_t r = 0; r < R; ++r)
    if (ids[r] >= E) return -1;
  for (int32_t e = 0; e < E; ++e) counts[e] = 0;
  for (int64_t r = 0; r < R; ++r)
    if (ids[r] >= 0) ++counts[ids[r]];
  offsets[0] = 0;
  for (int32_t e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  std::vector<int32_t> next(offsets, offsets + E);
  for (int64_t r = 0; r < R; ++r) {
    if (ids[r] < 0) {
      route2dst[r] = -1;
      continue;
    }
    const int32_t d = next[ids[r]]++;
    dst2src[d] = (int32_t)(r / topk);
    route2dst[r] = d;
  }
  return 0;
}

void ftor_gather(const uint8_t* src, const uint8_t* src_scales, int64_t row_bytes, int64_t scale_bytes,
                 const int32_t* map, int64_t n_dst, uint8_t* dst, uint8_t* dst_scales) {
  for (int64_t i = 0; i < n_dst; ++i) {
    std::memcpy(dst + i * row_bytes, src + (int64_t)map[i] * row_bytes, (size_t)row_bytes);
    if (scale_bytes > 0)
      std::memcpy(dst_scales + i * scale_bytes, src_scales + (int64_t)map[i] * scale_bytes, (size_t)scale_bytes);
  }
}

// The whole FFN. fmt 0 = FP8, 1 = NVFP4, 2 = MXFP8.
//   x [T][H] float (exact bf16 values); ids [T][topk] (negative = inactive); w [T][topk].
//   FP8 banks: q uint8 [E][n][k], scales float [E][ceil(n/128)][ceil(k/128)], g unused.
//   NVFP4 banks: q unpacked e2m1 codes [E][n][k], scales e4m3 codes [E][n][ceil(k/16)],
//   g float [E]. MXFP8 banks: q uint8 [E][n][k], scales E8M0 bytes [E][n][ceil(k/32)], g unused.
//   Gate/up: n = 2I (gate rows first), k = H; down: n = H, k = I.
//   subset: token indices to evaluate (NULL = all); out [T][H] double (other rows zero).
//   The NVFP4 tensor scales span the whole call (all tokens; all active routes for the
//   intermediate) even when a subset is evaluated.
// Returns 0, or -1 on an expert id >= E.
int ftor_moe_forward(int fmt, const float* x, int64_t T, int64_t H, int64_t I, int32_t E, int32_t topk,
                     const int32_t* ids, const float* w, const uint8_t* gq, const void* gs, const float* gg,
                     const uint8_t* dq, const void* ds, const float* dg, const int64_t* subset, int64_t n_subset,
                     int threads, double* out) {
  for (int64_t r = 0; r < T * topk; ++r)
    if (ids[r] >= E) return -1;
  if (threads < 1) threads = 1;
  const int64_t N2 = 2 * I;
  // 1. the token rows, quantized over the whole call
  std::vector<uint8_t> xq((size_t)(T * H));
  std::vector<float> xs;
  std::vector<uint8_t> xsb;
  float xg = 0.0f;
  if (fmt == 0) {
    xs.resize((size_t)(T * ceil_div(H, kGroup)));
    quantize_act_fp8(x, T, H, xq.data(), xs.data());
  } else if (fmt == 2) {
    xsb.resize((size_t)(T * ceil_div(H, kMxBlock)));
    quantize_mxfp8(x, T, H, xq.data(), xsb.data());
  } else {
    float amax = 0.0f;
    for (int64_t i = 0; i < T * H; ++i) amax = std::fmax(amax, std::fabs(x[i]));
    xsb.resize((size_t)(T * ceil_div(H, kNvBlock)));
    quantize_nvfp4(x, T, H, amax, xq.data(), xsb.data(), &xg);
  }
  auto xval = [&](int64_t t, int64_t c) {
    if (fmt == 0) return Fp8Rows{xq.data(), xs.data(), H, ceil_div(H, kGroup), 1}.at(t, c);
    if (fmt == 2) return MxRows{xq.data(), xsb.data(), H}.at(t, c);
    return Nvfp4Rows{xq.data(), xsb.data(), xg, H}.at(t, c);
  };
  // 2. routes: the evaluated tokens' active routes; NVFP4 needs every active route's
  //    intermediate for its tensor scale
  std::vector<char> wanted((size_t)T, subset ? 0 : 1);
  if (subset)
    for (int64_t i = 0; i < n_subset; ++i) wanted[(size_t)subset[i]] = 1;
  std::vector<std::vector<Route>> by_expert((size_t)E);
  for (int64_t t = 0; t < T; ++t)
    for (int j = 0; j < topk; ++j) {
      const int32_t e = ids[t * topk + j];
      if (e < 0) continue;
      if (wanted[(size_t)t] || fmt == 1) by_expert[(size_t)e].push_back(Route{t, j});
    }
  // 3. gate/up in double, silu(g) * u in double, kept as float32 (the re-quantized operand)
  std::vector<float> a((size_t)(T * topk * I), 0.0f);
  auto run = [&](auto&& body) {
    std::vector<std::thread> pool;
    for (int th = 0; th < threads; ++th)
      pool.emplace_back([&, th] {
        for (int32_t e = th; e < E; e += threads) body(e);
      });
    for (auto& p : pool) p.join();
  };
  run([&](int32_t e) {
    if (by_expert[(size_t)e].empty()) return;
    std::vector<double> gu((size_t)N2), xrow((size_t)H);
    const uint8_t* q = gq + (size_t)e * N2 * H;
    for (const Route& rt : by_expert[(size_t)e]) {
      for (int64_t c = 0; c < H; ++c) xrow[(size_t)c] = xval(rt.t, c);
      for (int64_t n = 0; n < N2; ++n) {
        double acc = 0.0;
        for (int64_t c = 0; c < H; ++c) {
          double wv;
          if (fmt == 0) {
            const float* s = static_cast<const float*>(gs) + (size_t)e * ceil_div(N2, kGroup) * ceil_div(H, kGroup);
            wv = Fp8Rows{q, s, H, ceil_div(H, kGroup), kGroup}.at(n, c);
          } else if (fmt == 2) {
            const uint8_t* sb = static_cast<const uint8_t*>(gs) + (size_t)e * N2 * ceil_div(H, kMxBlock);
            wv = MxRows{q, sb, H}.at(n, c);
          } else {
            const uint8_t* sb = static_cast<const uint8_t*>(gs) + (size_t)e * N2 * ceil_div(H, kNvBlock);
            wv = Nvfp4Rows{q, sb, gg[e], H}.at(n, c);
          }
          acc += wv * xrow[(size_t)c];
        }
        gu[(size_t)n] = acc;
      }
      float* arow = a.data() + (size_t)(rt.t * topk + rt.j) * I;
      for (int64_t i = 0; i < I; ++i) {
        const double g = gu[(size_t)i], u = gu[(size_t)(I + i)];
        arow[i] = (float)(g / (1.0 + std::exp(-g)) * u);
      }
    }
  });
  // 4. re-quantize each active route's intermediate (NVFP4: one tensor scale over all of them)
  std::vector<uint8_t> aq((size_t)(T * topk * I), 0);
  std::vector<float> as;
  std::vector<uint8_t> asb;
  float ag = 0.0f;
  if (fmt == 0) {
    as.assign((size_t)(T * topk * ceil_div(I, kGroup)), 0.0f);
    for (int64_t r = 0; r < T * topk; ++r)
      if (ids[r] >= 0) quantize_act_fp8(a.data() + r * I, 1, I, aq.data() + r * I, as.data() + r * ceil_div(I, kGroup));
  } else if (fmt == 2) {
    asb.assign((size_t)(T * topk * ceil_div(I, kMxBlock)), 0);
    for (int64_t r = 0; r < T * topk; ++r)
      if (ids[r] >= 0) quantize_mxfp8(a.data() + r * I, 1, I, aq.data() + r * I, asb.data() + r * ceil_div(I, kMxBlock));
  } else {
    float amax = 0.0f;
    for (int64_t r = 0; r < T * topk; ++r)
      if (ids[r] >= 0)
        for (int64_t i = 0; i < I; ++i) amax = std::fmax(amax, std::fabs(a[(size_t)(r * I + i)]));
    asb.assign((size_t)(T * topk * ceil_div(I, kNvBlock)), 0);
    for (int64_t r = 0; r < T * topk; ++r)
      if (ids[r] >= 0)
        quantize_nvfp4(a.data() + r * I, 1, I, amax, aq.data() + r * I, asb.data() + r * ceil_div(I, kNvBlock), &ag);
    ag = nvfp4_global(amax);
  }
  // 5. down in double, for the evaluated tokens' routes
  std::vector<double> y((size_t)(T * topk * H), 0.0);
  run([&](int32_t e) {
    std::vector<double> arow((size_t)I);
    const uint8_t* q = dq + (size_t)e * H * I;
    for (const Route& rt : by_expert[(size_t)e]) {
      if (!wanted[(size_t)rt.t]) continue;
      const int64_t r = rt.t * topk + rt.j;
      for (int64_t c = 0; c < I; ++c)
        arow[(size_t)c] = fmt == 0   ? Fp8Rows{aq.data(), as.data(), I, ceil_div(I, kGroup), 1}.at(r, c)
                          : fmt == 2 ? MxRows{aq.data(), asb.data(), I}.at(r, c)
                                     : Nvfp4Rows{aq.data(), asb.data(), ag, I}.at(r, c);
      for (int64_t h = 0; h < H; ++h) {
        double acc = 0.0;
        for (int64_t c = 0; c < I; ++c) {
          double wv;
          if (fmt == 0) {
            const float* s = static_cast<const float*>(ds) + (size_t)e * ceil_div(H, kGroup) * ceil_div(I, kGroup);
            wv = Fp8Rows{q, s, I, ceil_div(I, kGroup), kGroup}.at(h, c);
          } else if (fmt == 2) {
            const uint8_t* sb = static_cast<const uint8_t*>(ds) + (size_t)e * H * ceil_div(I, kMxBlock);
            wv = MxRows{q, sb, I}.at(h, c);
          } else {
            const uint8_t* sb = static_cast<const uint8_t*>(ds) + (size_t)e * H * ceil_div(I, kNvBlock);
            wv = Nvfp4Rows{q, sb, dg[e], I}.at(h, c);
          }
          acc += wv * arow[(size_t)c];
        }
        y[(size_t)(r * H + h)] = acc;
      }
    }
  });
  // 6. routing-weighted sum over the active slots, ascending
  for (int64_t t = 0; t < T; ++t) {
    double* o = out + t * H;
    for (int64_t h = 0; h < H; ++h) o[h] = 0.0;
    if (!wanted[(size_t)t]) continue;
    for (int j = 0; j < topk; ++j) {
      const int64_t r = t * topk + j;
      if (ids[r] < 0) continue;
      const double wt = (double)w[r];
      for (int64_t h = 0; h < H; ++h) o[h] += wt * y[(size_t)(r * H + h)];
    }
  }
  return 0;
}

int ftor_hardware_threads() {
  const unsigned n = std::thread::hardware_concurrency();
  return n == 0 ? 1 : (int)n;
}

}  // extern "C"

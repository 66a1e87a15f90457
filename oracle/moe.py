"""Plain CPU oracle of the routed-expert block-quantized MoE FFN.

TEST INFRASTRUCTURE ONLY: only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import this module. It shares no code with the
CUDA library and never calls it.

Everything here is the slow, direct definition of each step:

* quantize_act_fp8 / quantize_weight_fp8 -- per 1x128 activation group and per
  128x128 weight block: amax = max|x|, s = fl32(amax / 448), q = e4m3_rne_sat(fl32(x / s)).
  The SGLang page "Gather the cutlass MoE activation and its scales in one
  launch" (Motivation) fixes the grid: the activation is quantized once, with one
  fp32 scale per 128 columns ("k // 128 fp32 against k fp8"); the FreeToken
  page "perf(moe): skip inactive block-fp8 decode routes" gives the padded
  128x128 block-scale grid of the weights.
* segment_routes -- stable counting sort of the active routes by expert; the
  per-expert row counts/offsets that the grouped GEMMs consume and the dst2src
  map ("m * topk entries", SGLang page, Motivation) the gather walks.
* gather_rows_scales -- plain indexing of the FP8 row bytes and their scale row
  by the same map (SGLang page, Modifications / Accuracy Tests).
* gemm_rows -- dequantize to float64 and multiply in float64.
* silu_mul -- silu(g) * u in float64, g = first half, u = second half of the
  gate/up row.
* combine -- routing-weighted sum over the top-k slots, float64, inactive slots
  (negative expert id) contribute nothing and their weights are never read
  (FreeToken page, first section).
* NVFP4 -- e2m1 codes, one e4m3 scale per 16 elements, one fp32 scale per
  tensor (the two-level recipe; the pages name the format only).
* MXFP8 -- e4m3 codes with one power-of-two (E8M0) scale per 32 consecutive
  elements of a row. The SGLang gather page (Modifications) names the format
  ("mxfp8") and its branch, which gathers a bf16 activation and leaves the
  quantization to after the gather; the recipe is the OCP Microscaling one:
  shared exponent floor(log2(amax)) - 8 (8 = the largest exponent of an E4M3
  normal), clamped to E8M0's [-127, 127], codes e4m3_rne_sat(x / 2^shared).

Readings where the pages are silent are listed in the repository's design
notes (gate rows first then up rows; fp32 gate/up intermediate re-quantized per
1x128 before the down GEMM; amax = 0 gives scale 0 and all-zero codes; routing
weights not renormalised over active slots).
"""
import numpy as np

from .formats import (E2M1_MAX, E4M3_MAX, decode_e2m1, decode_e4m3,
                      encode_e2m1, encode_e4m3, round_to_bf16)

GROUP = 128        # activation group width; weight block edge
NVFP4_BLOCK = 16   # elements per e4m3 scale in NVFP4
MX_BLOCK = 32      # elements per E8M0 scale in MXFP8
E4M3_EMAX = 8      # exponent of E4M3's largest power of two (448 = 1.75 * 2^8)
E8M0_BIAS = 127


def ceil_div(a, b):
    return -(-a // b)


# --------------------------------------------------------------------------
# quantization (decisions taken in float32, like the kernels)
# --------------------------------------------------------------------------

def _quantize_fp8_block(vals32: np.ndarray):
    """One block/group of float32 values -> (codes uint8, scale float32).

    amax = max|x|; s = fl32(amax / 448); codes = e4m3_rne_sat(fl32(x / s)).
    amax == 0 gives s = 0 and all-zero codes (no 0/0).
    """
    amax = np.float32(np.max(np.abs(vals32))) if vals32.size else np.float32(0)
    if amax == 0:
        return np.zeros(vals32.shape, np.uint8), np.float32(0)
    s = np.float32(amax) / np.float32(E4M3_MAX)
    v = (vals32 / s).astype(np.float32)  # IEEE fp32 division, one rounding
    return encode_e4m3(v), np.float32(s)


def quantize_act_fp8(x):
    """Per-token 1x128 FP8 quantization.

    x: [rows, k] float32 (bf16 inputs are passed as their exact float32 values).
    Returns q uint8 [rows, k], scales float32 [rows, ceil(k/128)]; a partial last
    group takes its amax over its valid columns only.
    """
    x = np.asarray(x, dtype=np.float32)
    rows, k = x.shape
    ng = ceil_div(k, GROUP)
    q = np.zeros((rows, k), np.uint8)
    s = np.zeros((rows, ng), np.float32)
    for r in range(rows):
        for g in range(ng):
            sl = slice(g * GROUP, min(k, (g + 1) * GROUP))
            q[r, sl], s[r, g] = _quantize_fp8_block(x[r, sl])
    return q, s


def quantize_act_fp8_fast(x):
    """Same result as quantize_act_fp8, vectorised over rows (for large inputs)."""
    x = np.asarray(x, dtype=np.float32)
    rows, k = x.shape
    ng = ceil_div(k, GROUP)
    q = np.zeros((rows, k), np.uint8)
    s = np.zeros((rows, ng), np.float32)
    for g in range(ng):
        sl = slice(g * GROUP, min(k, (g + 1) * GROUP))
        blk = x[:, sl]
        amax = np.max(np.abs(blk), axis=1).astype(np.float32)
        sc = (amax / np.float32(E4M3_MAX)).astype(np.float32)
        safe = np.where(amax == 0, np.float32(1), sc).astype(np.float32)
        v = (blk / safe[:, None]).astype(np.float32)
        codes = encode_e4m3(v)
        codes[amax == 0, :] = 0
        q[:, sl] = codes
        s[:, g] = np.where(amax == 0, np.float32(0), sc)
    return q, s


def quantize_weight_fp8(w):
    """128x128 block FP8 quantization of one weight matrix.

    w: [n, k] float32. Returns q uint8 [n, k], scales float32
    [ceil(n/128), ceil(k/128)] (the padded grid: edge blocks take their amax over
    their valid elements).
    """
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    nb, kb = ceil_div(n, GROUP), ceil_div(k, GROUP)
    q = np.zeros((n, k), np.uint8)
    s = np.zeros((nb, kb), np.float32)
    for i in range(nb):
        rs = slice(i * GROUP, min(n, (i + 1) * GROUP))
        for j in range(kb):
            cs = slice(j * GROUP, min(k, (j + 1) * GROUP))
            q[rs, cs], s[i, j] = _quantize_fp8_block(w[rs, cs])
    return q, s


def quantize_weight_fp8_fast(w):
    """Same result as quantize_weight_fp8, vectorised over blocks (for large matrices)."""
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    nb, kb = ceil_div(n, GROUP), ceil_div(k, GROUP)
    pad = np.zeros((nb * GROUP, kb * GROUP), np.float32)
    pad[:n, :k] = w
    blocks = pad.reshape(nb, GROUP, kb, GROUP)
    amax = np.max(np.abs(blocks), axis=(1, 3)).astype(np.float32)  # padding zeros never win
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    safe = np.where(amax == 0, np.float32(1), s).astype(np.float32)
    v = (blocks / safe[:, None, :, None]).astype(np.float32)
    q = encode_e4m3(v)
    q[np.broadcast_to((amax == 0)[:, None, :, None], q.shape)] = 0
    return q.reshape(nb * GROUP, kb * GROUP)[:n, :k].copy(), s


def dequant_act_fp8(q, s):
    """[rows, k] codes + [rows, ceil(k/128)] scales -> float64 [rows, k]."""
    q = np.asarray(q)
    k = q.shape[1]
    scale_cols = np.repeat(np.asarray(s, np.float64), GROUP, axis=1)[:, :k]
    return decode_e4m3(q) * scale_cols


def dequant_weight_fp8(q, s):
    """[n, k] codes + [ceil(n/128), ceil(k/128)] block scales -> float64 [n, k]."""
    q = np.asarray(q)
    n, k = q.shape
    sc = np.repeat(np.repeat(np.asarray(s, np.float64), GROUP, axis=0), GROUP, axis=1)[:n, :k]
    return decode_e4m3(q) * sc


# --------------------------------------------------------------------------
# NVFP4: e2m1 codes, e4m3 scale per 16 elements, fp32 scale per tensor
# --------------------------------------------------------------------------

def nvfp4_global_scale(amax_tensor):
    """g = fl32(amax / (448 * 6)): maps the largest block scale onto e4m3's top."""
    return np.float32(np.float32(amax_tensor) / np.float32(E4M3_MAX * E2M1_MAX))


def quantize_nvfp4(x, global_amax=None):
    """Two-level FP4 quantization of a [rows, k] float32 tensor.

    g   = fl32(amax_tensor / 2688)                       (per tensor, fp32)
    sb  = e4m3_rne_sat(fl32(amax_block / fl32(6 g)))       (per 16 elements)
    eff = fl32(decode(sb) * g)
    q   = e2m1_rne_sat(fl32(x / eff)), or 0 where eff == 0
    Returns (codes uint8 [rows, k] holding 0..15, block scale codes uint8
    [rows, ceil(k/16)], g float32). g = 0 (all-zero tensor) gives all-zero codes.
    """
    x = np.asarray(x, dtype=np.float32)
    rows, k = x.shape
    if global_amax is None:
        global_amax = np.max(np.abs(x)) if x.size else 0.0
    g = nvfp4_global_scale(global_amax)
    nblk = ceil_div(k, NVFP4_BLOCK)
    q = np.zeros((rows, k), np.uint8)
    sb = np.zeros((rows, nblk), np.uint8)
    if g == 0:
        return q, sb, g
    six_g = np.float32(np.float32(E2M1_MAX) * g)
    for b in range(nblk):
        sl = slice(b * NVFP4_BLOCK, min(k, (b + 1) * NVFP4_BLOCK))
        blk = x[:, sl]
        amax_b = np.max(np.abs(blk), axis=1).astype(np.float32)
        codes = encode_e4m3((amax_b / six_g).astype(np.float32))
        sb[:, b] = codes
        eff = (decode_e4m3(codes).astype(np.float32) * g).astype(np.float32)
        safe = np.where(eff == 0, np.float32(1), eff).astype(np.float32)
        v = (blk / safe[:, None]).astype(np.float32)
        c = encode_e2m1(v)
        c[eff == 0, :] = 0
        q[:, sl] = c
    return q, sb, g


def dequant_nvfp4(q, sb, g):
    """codes [rows, k] (0..15) + block scale codes [rows, ceil(k/16)] + g -> float64."""
    q = np.asarray(q)
    k = q.shape[1]
    bs = np.repeat(decode_e4m3(sb), NVFP4_BLOCK, axis=1)[:, :k]
    return decode_e2m1(q) * bs * np.float64(g)


def pack_e2m1(codes):
    """[rows, k] 4-bit codes -> [rows, ceil(k/2)] bytes, even column in the low nibble."""
    codes = np.asarray(codes, np.uint8)
    rows, k = codes.shape
    if k % 2:
        codes = np.concatenate([codes, np.zeros((rows, 1), np.uint8)], axis=1)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def unpack_e2m1(packed, k):
    packed = np.asarray(packed, np.uint8)
    out = np.zeros((packed.shape[0], packed.shape[1] * 2), np.uint8)
    out[:, 0::2] = packed & 0xF
    out[:, 1::2] = packed >> 4
    return out[:, :k]


# --------------------------------------------------------------------------
# MXFP8: e4m3 codes, one E8M0 (power-of-two) scale per 32 elements of a row
# --------------------------------------------------------------------------

def mx_shared_exp(amax):
    """floor(log2(amax)) - 8, clamped to [-127, 127]; amax == 0 gives -127.

    amax is a float32 magnitude. frexp gives amax = m * 2^e with m in [0.5, 1), so
    floor(log2(amax)) = e - 1 exactly (no floating-point logarithm is taken).
    """
    a = float(np.float32(amax))
    if a == 0.0:
        return -E8M0_BIAS
    _, e = np.frexp(a)
    return int(min(E8M0_BIAS, max(-E8M0_BIAS, (int(e) - 1) - E4M3_EMAX)))


def quantize_mxfp8(x):
    """MXFP8 quantization of a [rows, k] float32 tensor along its rows.

    Per 32 consecutive elements of a row (a partial last block takes its amax over its
    valid elements): shared = mx_shared_exp(amax), scale byte = shared + 127, codes
    e4m3_rne_sat(x / 2^shared). Dividing by a power of two is exact here (the quotient's
    magnitude is below 512 and far above E4M3's smallest step), so the codes follow from
    the inputs alone. Returns (codes uint8 [rows, k], scale bytes uint8 [rows, ceil(k/32)]).
    """
    x = np.asarray(x, dtype=np.float32)
    rows, k = x.shape
    nblk = ceil_div(k, MX_BLOCK)
    q = np.zeros((rows, k), np.uint8)
    sb = np.zeros((rows, nblk), np.uint8)
    for b in range(nblk):
        sl = slice(b * MX_BLOCK, min(k, (b + 1) * MX_BLOCK))
        blk = x[:, sl].astype(np.float64)
        amax = np.max(np.abs(blk), axis=1)
        for r in range(rows):
            e = mx_shared_exp(amax[r])
            sb[r, b] = e + E8M0_BIAS
            q[r, sl] = encode_e4m3(blk[r] * np.ldexp(1.0, -e))
    return q, sb


def quantize_mxfp8_fast(x):
    """Same result as quantize_mxfp8, vectorised over rows and blocks (for large inputs)."""
    x = np.asarray(x, dtype=np.float32)
    rows, k = x.shape
    nblk = ceil_div(k, MX_BLOCK)
    pad = np.zeros((rows, nblk * MX_BLOCK), np.float64)
    pad[:, :k] = x
    blk = pad.reshape(rows, nblk, MX_BLOCK)
    amax = np.max(np.abs(blk), axis=2)  # padding zeros never win
    _, e = np.frexp(amax)
    shared = np.clip(e.astype(np.int64) - 1 - E4M3_EMAX, -E8M0_BIAS, E8M0_BIAS)
    shared = np.where(amax == 0, -E8M0_BIAS, shared)
    q = encode_e4m3(blk * np.ldexp(1.0, -shared)[:, :, None])
    return q.reshape(rows, nblk * MX_BLOCK)[:, :k].copy(), (shared + E8M0_BIAS).astype(np.uint8)


def dequant_mxfp8(q, sb):
    """codes [rows, k] + E8M0 scale bytes [rows, ceil(k/32)] -> float64 [rows, k]."""
    q = np.asarray(q)
    k = q.shape[1]
    scale = np.ldexp(1.0, np.asarray(sb, np.int64) - E8M0_BIAS)
    return decode_e4m3(q) * np.repeat(scale, MX_BLOCK, axis=1)[:, :k]


# --------------------------------------------------------------------------
# routing: segmenter, gather, combine
# --------------------------------------------------------------------------

def segment_routes(expert_ids, num_experts):
    """Group the active routes by expert, stable in route order.

    expert_ids: [tokens, topk] int; a negative id is an inactive route.
    Route r = t * topk + j. Returns dict with
      counts    int32 [E]      rows per expert
      offsets   int32 [E + 1]  exclusive prefix of counts
      dst2src   int32 [R_a]    source token of each grouped row
      route2dst int32 [R]      grouped row of each route, -1 if inactive
    """
    ids = np.asarray(expert_ids, dtype=np.int64)
    tokens, topk = ids.shape
    flat = ids.reshape(-1)
    if np.any(flat >= num_experts):
        raise ValueError("expert id out of range")
    active = np.nonzero(flat >= 0)[0]
    order = active[np.argsort(flat[active], kind="stable")]  # stable: route order within an expert
    counts = np.bincount(flat[active], minlength=num_experts).astype(np.int32)
    offsets = np.zeros(num_experts + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    dst2src = (order // topk).astype(np.int32)
    route2dst = np.full(flat.shape[0], -1, np.int32)
    route2dst[order] = np.arange(order.shape[0], dtype=np.int32)
    return dict(counts=counts, offsets=offsets, dst2src=dst2src, route2dst=route2dst)


def gather_rows_scales(src, src_scales, dst2src):
    """dst[i] = src[dst2src[i]] and dst_scales[i] = src_scales[dst2src[i]], as raw bytes."""
    m = np.asarray(dst2src, dtype=np.int64)
    src = np.asarray(src)
    src_scales = np.asarray(src_scales)
    return src[m].copy(), src_scales[m].copy()


def combine(y, route2dst, expert_ids, weights):
    """out[t] = sum over active slots j (ascending) of w[t, j] * y[route2dst[t*topk+j]], float64.

    Inactive slots (expert id < 0) are skipped without reading their weight.
    y: [rows, hidden] values (any float dtype). Returns float64 [tokens, hidden].
    """
    ids = np.asarray(expert_ids)
    tokens, topk = ids.shape
    y = np.asarray(y, np.float64)
    out = np.zeros((tokens, y.shape[1]), np.float64)
    for t in range(tokens):
        for j in range(topk):
            if ids[t, j] < 0:
                continue
            out[t] += np.float64(weights[t, j]) * y[route2dst[t * topk + j]]
    return out


def silu_mul(gu):
    """[rows, 2I] -> [rows, I]: silu(g) * u with g = columns [0, I), u = columns [I, 2I)."""
    gu = np.asarray(gu, np.float64)
    inter = gu.shape[1] // 2
    g, u = gu[:, :inter], gu[:, inter:]
    return g / (1.0 + np.exp(-g)) * u


def pick_tile(routes, num_experts):
    """Token tile of the grouped GEMM from route density.

    The smallest of 16/32/64/128 that holds ceil(routes / experts) rows, else 128
    (dsfp4 page: the best M tile tracks rows per expert, 16 -> 32 -> 128 at
    about 6 -> 24 -> 96 rows; the picker is a pure function of route count and
    expert count).
    """
    per = ceil_div(int(routes), int(num_experts)) if num_experts > 0 else 0
    for m in (16, 32, 64, 128):
        if m >= per:
            return m
    return 128


# --------------------------------------------------------------------------
# GEMM and the whole FFN
# --------------------------------------------------------------------------

def gemm_rows(a_deq, w_deq):
    """Rows of dequantized activations times one dequantized expert matrix, float64.

    a_deq [m, k], w_deq [n, k] -> [m, n] with out[i, n] = sum_k a[i, k] * w[n, k].
    """
    return np.asarray(a_deq, np.float64) @ np.asarray(w_deq, np.float64).T


class Bank:
    """A quantized expert bank held by the oracle: per-expert codes and scales.

    fmt 'fp8': q [E, n, k] uint8, s [E, ceil(n/128), ceil(k/128)] float32.
    fmt 'nvfp4': q [E, n, k] codes 0..15 (unpacked), sb [E, n, ceil(k/16)] e4m3
    codes, g [E] float32.
    fmt 'mxfp8': q [E, n, k] uint8, s [E, n, ceil(k/32)] E8M0 scale bytes.
    """

    def __init__(self, fmt, q, s, g=None):
        self.fmt, self.q, self.s, self.g = fmt, q, s, g
        self.n = q.shape[1]

    def dequant(self, e):
        if self.fmt == "fp8":
            return dequant_weight_fp8(self.q[e], self.s[e])
        if self.fmt == "mxfp8":
            return dequant_mxfp8(self.q[e], self.s[e])
        return dequant_nvfp4(self.q[e], self.s[e], self.g[e])


class LazyBank:
    """A bank whose experts are quantized on first use from raw(e) -> float32 [n, k].

    Large workloads touch one expert at a time; the result per expert is the same as
    quantize_bank's.
    """

    def __init__(self, raw, n, fmt="fp8"):
        self.raw, self.n, self.fmt = raw, n, fmt
        self._cache = {}

    def parts(self, e):
        if e not in self._cache:
            w = np.asarray(self.raw(e), np.float32)
            if self.fmt == "fp8":
                self._cache[e] = quantize_weight_fp8_fast(w)
            elif self.fmt == "mxfp8":
                self._cache[e] = quantize_mxfp8_fast(w)
            else:
                self._cache[e] = quantize_nvfp4(w)
        return self._cache[e]

    def dequant(self, e):
        p = self.parts(e)
        if self.fmt == "fp8":
            return dequant_weight_fp8(*p)
        if self.fmt == "mxfp8":
            return dequant_mxfp8(*p)
        return dequant_nvfp4(*p)


def quantize_bank(weights_fp32, fmt="fp8"):
    """[E, n, k] float32 -> Bank (each expert quantized independently)."""
    w = np.asarray(weights_fp32, np.float32)
    if fmt == "fp8":
        qs = [quantize_weight_fp8(w[e]) for e in range(w.shape[0])]
        return Bank("fp8", np.stack([a for a, _ in qs]), np.stack([b for _, b in qs]))
    if fmt == "mxfp8":
        qs = [quantize_mxfp8(w[e]) for e in range(w.shape[0])]
        return Bank("mxfp8", np.stack([a for a, _ in qs]), np.stack([b for _, b in qs]))
    qs = [quantize_nvfp4(w[e]) for e in range(w.shape[0])]
    return Bank("nvfp4", np.stack([a for a, _, _ in qs]), np.stack([b for _, b, _ in qs]),
                np.array([c for _, _, c in qs], np.float32))


def quantize_acts(x, fmt, global_amax=None):
    """Activation quantization of either format; returns (dequantized float64, raw parts)."""
    if fmt == "fp8":
        q, s = quantize_act_fp8_fast(x)
        return dequant_act_fp8(q, s), (q, s)
    if fmt == "mxfp8":
        q, sb = quantize_mxfp8_fast(x)
        return dequant_mxfp8(q, sb), (q, sb)
    q, sb, g = quantize_nvfp4(x, global_amax)
    return dequant_nvfp4(q, sb, g), (q, sb, g)


def moe_forward(x, expert_ids, weights, bank_gateup, bank_down, fmt="fp8", tokens_subset=None):
    """The whole routed-expert FFN, float64 after each quantization.

    x [T, H] float32 (exact bf16 values); expert_ids [T, topk] (negative = inactive);
    weights [T, topk] float32; banks: gate/up [E, 2I, H] (gate rows first), down [E, H, I].
    Steps: quantize x per 1x128 (or NVFP4, or MXFP8) -> for each active route: gate/up GEMM in
    float64 -> silu(g)*u -> re-quantize that intermediate (the down GEMM's FP8/FP4
    operand) -> down GEMM in float64 -> routing-weighted combine.
    The grouping (segment + gather) only reorders rows and changes no value, so the
    oracle evaluates each route directly from its token's row.
    tokens_subset: optional list of token indices to evaluate (others left zero);
    NVFP4 global amaxes are still taken over the whole tensors.
    Returns dict(out=float64 [T, H], out_bf16=float64 values of the bf16 rounding,
    and per-route intermediates keyed by (token, slot): gu (gate/up output), a (SiLU-and-mul
    output, before its re-quantization) and y (down output); xdeq the dequantized tokens).
    """
    x = np.asarray(x, np.float32)
    ids = np.asarray(expert_ids)
    T, topk = ids.shape
    H = x.shape[1]
    toks = range(T) if tokens_subset is None else list(tokens_subset)
    xdeq, _ = quantize_acts(x, fmt)
    inter = bank_gateup.n // 2
    # all active routes' intermediates (needed for the NVFP4 tensor-wide amax)
    routes = [(t, j) for t in toks for j in range(topk) if ids[t, j] >= 0]
    if fmt == "nvfp4" and tokens_subset is not None:
        routes_all = [(t, j) for t in range(T) for j in range(topk) if ids[t, j] >= 0]
    else:
        routes_all = routes
    by_expert = {}
    for (t, j) in routes_all:
        by_expert.setdefault(int(ids[t, j]), []).append((t, j))
    a_rows, gu_rows = {}, {}
    for e, lst in by_expert.items():
        wg = bank_gateup.dequant(e)
        rows = np.stack([xdeq[t] for (t, _) in lst])
        gu = gemm_rows(rows, wg)
        act = silu_mul(gu)
        for i, (t, j) in enumerate(lst):
            a_rows[(t, j)] = act[i]
            gu_rows[(t, j)] = gu[i]
    keys = sorted(a_rows.keys())
    y_rows = {}
    if keys:
        A = np.stack([a_rows[k] for k in keys]).astype(np.float32)  # the fp32 intermediate
        gamax = np.max(np.abs(A)) if fmt == "nvfp4" else None
        adeq_all, _ = quantize_acts(A, fmt, gamax)
        adeq = {k: adeq_all[i] for i, k in enumerate(keys)}
        wanted = set(routes)
        for e, lst in by_expert.items():
            lst = [r for r in lst if r in wanted]
            if not lst:
                continue
            wd = bank_down.dequant(e)
            y = gemm_rows(np.stack([adeq[r] for r in lst]), wd)
            for i, r in enumerate(lst):
                y_rows[r] = y[i]
    out = np.zeros((T, H), np.float64)
    for t in toks:
        for j in range(topk):
            if ids[t, j] < 0:
                continue
            out[t] += np.float64(weights[t, j]) * y_rows[(t, j)]
    return dict(out=out, out_bf16=round_to_bf16(out), a=a_rows, gu=gu_rows, y=y_rows, xdeq=xdeq)

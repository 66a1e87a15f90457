"""The oracle at the largest prefill sizes, one expert per task in a pool of spawned workers.

Test infrastructure: every value here comes from `oracle/` functions, called on the same
seeded inputs the GPU side uses. The work is only split by expert (each expert's rows are
independent of the others'), with the NVFP4 intermediate's call-wide tensor scale taken in
a first pass over all routes, as `oracle.moe.moe_forward` does. Raw expert weights are
drawn on the CPU by `synth` in each worker, so no weights cross the process boundary.
"""
import os

import numpy as np

_BLAS_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
_CTX = {}


def _init(ctx):
    _CTX.update(ctx)


def _bank_parts(e, which):
    """(dequantized float64 matrix) of expert e, quantized by the oracle from synth's draw."""
    import synth
    from oracle import moe as M
    H, I, seed, fmt = _CTX["H"], _CTX["I"], _CTX["seed"], _CTX["fmt"]
    n, k = (2 * I, H) if which == "gateup" else (H, I)
    w = synth.expert_weight_fp32(n, k, seed, e, which, "cpu").numpy()
    if fmt == "fp8":
        q, s = M.quantize_weight_fp8_fast(w)
        return M.dequant_weight_fp8(q, s)
    q, sb, g = M.quantize_nvfp4(w)
    return M.dequant_nvfp4(q, sb, g)


def _x_rows(tokens):
    """Dequantized token rows (float64) from the codes and scales the main process made."""
    from oracle import moe as M
    if _CTX["fmt"] == "fp8":
        return M.dequant_act_fp8(_CTX["xq"][tokens], _CTX["xs"][tokens])
    return M.dequant_nvfp4(_CTX["xq"][tokens], _CTX["xs"][tokens], _CTX["xg"])


def expert_amax(task):
    """NVFP4 first pass: largest |silu(g)*u| (as float32) over all routes of one expert, and
    the kernels' fp32 error bound at that element."""
    from common import NVFP4_SUM_REL, _silu_mul_error
    from oracle import moe as M
    e, tokens = task
    if not tokens:
        return 0.0, 0.0
    wg = _bank_parts(e, "gateup")
    x = _x_rows(np.asarray(tokens))
    gu = M.gemm_rows(x, wg)
    a = M.silu_mul(gu)
    absum = np.abs(x) @ np.abs(wg).T
    a32 = np.abs(a.astype(np.float32).astype(np.float64))
    r, c = np.unravel_index(np.argmax(a32), a32.shape)
    ea = _silu_mul_error(gu[r], absum[r], NVFP4_SUM_REL)[c] + 2.0 ** -21 * a32[r, c]
    return float(a32[r, c]), float(ea)


def expert_rows(task):
    """Down-GEMM output rows of one expert's checked routes and their re-quantization
    allowance: returns (y [m, H], extra [m, H]) for tokens[i] in route order."""
    from common import FP32_SUM_REL, NVFP4_SUM_REL, _silu_mul_error
    from oracle import formats as F
    from oracle import moe as M
    e, tokens = task
    if not tokens:
        return None
    fmt, I = _CTX["fmt"], _CTX["I"]
    wg, wd = _bank_parts(e, "gateup"), _bank_parts(e, "down")
    x = _x_rows(np.asarray(tokens))
    gu = M.gemm_rows(x, wg)
    a = M.silu_mul(gu)
    a32 = a.astype(np.float32)
    if fmt == "fp8":
        adeq, _ = M.quantize_acts(a32, "fp8")
    else:
        adeq, _ = M.quantize_acts(a32, "nvfp4", _CTX["gamax"])
    y = M.gemm_rows(adeq, wd)
    absum = np.abs(x) @ np.abs(wg).T
    awd = np.abs(wd)
    extra = np.zeros_like(y)
    rel = FP32_SUM_REL if fmt == "fp8" else NVFP4_SUM_REL
    for i in range(len(tokens)):
        ea = _silu_mul_error(gu[i], absum[i], rel) + 2.0 ** -21 * np.abs(a[i])
        extra[i] = _fp8_extra(a[i], ea, awd, F) if fmt == "fp8" else _nvfp4_extra(a[i], ea, awd, F)
    return y, extra


def _fp8_extra(a, ea, awd, F):
    """One route's allowance for E4M3 re-quantization ties (as tests/common.requant_flip_bound)."""
    pos = F.E4M3_VALUES[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2
    a32 = a.astype(np.float32).astype(np.float64)
    out = np.zeros(awd.shape[0])
    for g0 in range(0, a.shape[0], 128):
        sl = slice(g0, min(a.shape[0], g0 + 128))
        blk = a32[sl]
        amax = np.max(np.abs(blk))
        if amax == 0:
            continue
        s = float(np.float32(np.float32(amax) / np.float32(448.0)))
        v = np.abs(blk) / s
        rel_s = ea[sl][np.argmax(np.abs(blk))] / amax + 2.0 ** -21
        ev = ea[sl] / s + v * rel_s
        k = np.clip(np.searchsorted(mids, v), 1, len(mids) - 1)
        d = np.minimum(np.abs(v - mids[k - 1]), np.abs(v - mids[np.minimum(k, len(mids) - 1)]))
        amb = np.nonzero(d <= ev)[0]
        if amb.size == 0:
            continue
        idx = np.arange(sl.start, sl.stop)[amb]
        step = np.abs(np.diff(pos))[np.clip(np.searchsorted(pos, v[amb]) - 1, 0, len(pos) - 2)] * s
        out += awd[:, idx] @ step
    return out


def _nvfp4_extra(a, ea, awd, F):
    """One route's allowance for the NVFP4 intermediate's block-scale and code ties (as
    tests/common.nvfp4_requant_flip_bound; the tensor scale's uncertainty comes from the
    first pass)."""
    e2 = F.E2M1_VALUES[:8]
    mids2 = (e2[:-1] + e2[1:]) / 2
    e4 = F.E4M3_VALUES[:0x7F]
    mids4 = (e4[:-1] + e4[1:]) / 2
    gamax, rel_g0 = _CTX["gamax"], _CTX["gamax_rel"]
    g = float(np.float32(np.float32(gamax) / np.float32(448.0 * 6.0)))
    rel_g = rel_g0 + 2.0 ** -22
    six_g = float(np.float32(np.float32(6.0) * np.float32(g)))
    a32 = a.astype(np.float32).astype(np.float64)
    out = np.zeros(awd.shape[0])
    for b0 in range(0, a.shape[0], 16):
        blk = np.abs(a32[b0:b0 + 16])
        amax_b = np.max(blk)
        if amax_b == 0:
            continue
        xb = amax_b / six_g
        rel_b = ea[b0 + np.argmax(blk)] / amax_b + rel_g + 2.0 ** -21
        kb = np.clip(np.searchsorted(mids4, xb), 1, len(mids4) - 1)
        db = min(abs(xb - mids4[kb - 1]), abs(xb - mids4[kb]))
        code = int(F.encode_e4m3(np.float32(xb)))
        if db <= rel_b * xb:
            c2 = [c for c in (code - 1, code + 1) if 0 <= c < 0x7F]
            effs = F.E4M3_VALUES[code] * g + max(F.E4M3_VALUES[c] for c in c2) * g
            out += effs * awd[:, b0:b0 + 16].sum(axis=1)
            continue
        eff = float(np.float32(np.float32(F.E4M3_VALUES[code]) * np.float32(g)))
        if eff == 0:
            continue
        v = blk / eff
        ev = ea[b0:b0 + 16] / eff + v * (rel_g + 2.0 ** -21)
        k2 = np.clip(np.searchsorted(mids2, v), 1, len(mids2) - 1)
        d = np.minimum(np.abs(v - mids2[k2 - 1]), np.abs(v - mids2[k2]))
        near = np.where(np.abs(v - mids2[k2 - 1]) <= np.abs(v - mids2[k2]), k2 - 1, k2)
        amb = np.nonzero(d <= ev)[0]
        if amb.size == 0:
            continue
        step = (e2[near[amb] + 1] - e2[near[amb]]) * eff
        out += awd[:, b0 + amb] @ step
    return out


def forward_subsample(x32, ids, weights, subsample, H, I, E, seed, fmt, workers):
    """The oracle's FFN output rows (float64) of the tokens in `subsample` and their
    re-quantization allowance, for raw weights synth.expert_weight_fp32(..., seed, e, tag).

    x32 [T, H] float32 (bf16 values), ids [T, k], weights [T, k] (numpy). Token quantization
    covers all T tokens (the NVFP4 tensor scale spans the call)."""
    import multiprocessing as mp

    from oracle import moe as M
    T, topk = ids.shape
    if fmt == "fp8":
        xq, xs = M.quantize_act_fp8_fast(x32)
        ctx = dict(xq=xq, xs=xs)
    else:
        xq, xs, xg = M.quantize_nvfp4(x32)
        ctx = dict(xq=xq, xs=xs, xg=xg)
    ctx.update(H=H, I=I, seed=seed, fmt=fmt)
    sub = set(int(t) for t in subsample)
    by_e_all = {e: [] for e in range(E)}
    by_e_sub = {e: [] for e in range(E)}
    for t in range(T):
        for j in range(topk):
            e = int(ids[t, j])
            if e < 0:
                continue
            by_e_all[e].append(t)
            if t in sub:
                by_e_sub[e].append((t, j))
    pool_ctx = mp.get_context("spawn")
    # one BLAS thread per worker (the pool provides the parallelism): spawned children
    # inherit the environment before they import numpy
    saved = {v: os.environ.get(v) for v in _BLAS_VARS}
    os.environ.update({v: "1" for v in _BLAS_VARS})
    try:
        return _run(pool_ctx, ctx, by_e_all, by_e_sub, sub, weights, T, H, E, topk, fmt, workers)
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old


def _run(pool_ctx, ctx, by_e_all, by_e_sub, sub, weights, T, H, E, topk, fmt, workers):
    if fmt == "nvfp4":
        with pool_ctx.Pool(workers, initializer=_init, initargs=(ctx,)) as pool:
            res = pool.map(expert_amax, [(e, by_e_all[e]) for e in range(E)], chunksize=1)
        best = max(range(E), key=lambda e: res[e][0])
        ctx["gamax"] = res[best][0]
        ctx["gamax_rel"] = res[best][1] / res[best][0] if res[best][0] > 0 else 0.0
    with pool_ctx.Pool(workers, initializer=_init, initargs=(ctx,)) as pool:
        res = pool.map(expert_rows, [(e, [t for t, _ in by_e_sub[e]]) for e in range(E)], chunksize=1)
    out = np.zeros((T, H))
    extra = np.zeros((T, H))
    w = np.asarray(weights, np.float64)
    # combine in ascending slot order per token, as the oracle's combine does
    contrib = {}
    for e in range(E):
        if res[e] is None:
            continue
        y, ex = res[e]
        for i, (t, j) in enumerate(by_e_sub[e]):
            contrib[(t, j)] = (y[i], ex[i])
    for t in sorted(sub):
        for j in range(topk):
            if (t, j) in contrib:
                y, ex = contrib[(t, j)]
                out[t] += w[t, j] * y
                extra[t] += abs(w[t, j]) * ex
    return out, extra

"""The oracle at the largest prefill sizes, one expert per task in a pool of spawned workers.

Test infrastructure: every value here comes from `oracle/` functions, called on the same
seeded inputs the GPU side uses. The work is only split by expert (each expert's rows are
independent of the others'), with the NVFP4 intermediate's call-wide tensor scale taken in
a first pass over all routes of each call, as `oracle.moe.moe_forward` does. Several calls
that share one weight bank are evaluated in the same passes, so each expert's weights are
drawn and quantized once per pass for all of them. Raw expert weights are drawn on the CPU
by `synth` in each worker, so no weights cross the process boundary. FP8 weights are
quantized by the C++ oracle's quantizer when it loads (held bit for bit to the numpy one by
the CPU tests), else by the numpy oracle.
"""
import os

import numpy as np

_BLAS_VARS = ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")
_CTX = {}


def _init(ctx):
    _CTX.update(ctx)


def _quantize_weight(w, fmt):
    from oracle import moe as M
    if fmt == "fp8":
        try:
            from oracle import cpu as C
            return C.quantize_weight_fp8(w)
        except (OSError, RuntimeError):
            return M.quantize_weight_fp8_fast(w)
    if fmt == "mxfp8":
        return M.quantize_mxfp8_fast(w)
    return M.quantize_nvfp4(w)


def _weights(e, which):
    """Dequantized float64 matrix of expert e, quantized by the oracle from synth's draw."""
    import synth
    from oracle import moe as M
    H, I, seed, fmt = _CTX["H"], _CTX["I"], _CTX["seed"], _CTX["fmt"]
    n, k = (2 * I, H) if which == "gateup" else (H, I)
    w = synth.expert_weight_fp32(n, k, seed, e, which, "cpu").numpy()
    parts = _quantize_weight(w, fmt)
    if fmt == "mxfp8":
        return M.dequant_mxfp8(*parts)
    return M.dequant_weight_fp8(*parts) if fmt == "fp8" else M.dequant_nvfp4(*parts)


def _x_rows(c, tokens):
    """Dequantized token rows (float64) of call c from the codes the main process made."""
    from oracle import moe as M
    call = _CTX["calls"][c]
    if _CTX["fmt"] == "fp8":
        return M.dequant_act_fp8(call["xq"][tokens], call["xs"][tokens])
    if _CTX["fmt"] == "mxfp8":
        return M.dequant_mxfp8(call["xq"][tokens], call["xs"][tokens])
    return M.dequant_nvfp4(call["xq"][tokens], call["xs"][tokens], call["xg"])


def _gateup(c, tokens, wg):
    """Gate/up rows of call c's tokens, silu(g)*u, and the kernels' fp32 error bound on it."""
    from common import FP32_SUM_REL, NVFP4_SUM_REL, _silu_mul_error, mxfp8_sum_rel
    from oracle import moe as M
    x = _x_rows(c, np.asarray(tokens))
    gu = M.gemm_rows(x, wg)
    a = M.silu_mul(gu)
    absum = np.abs(x) @ np.abs(wg).T
    rel = {"fp8": FP32_SUM_REL, "nvfp4": NVFP4_SUM_REL, "mxfp8": mxfp8_sum_rel(_CTX["H"])}[_CTX["fmt"]]
    ea = np.stack([_silu_mul_error(gu[i], absum[i], rel) for i in range(len(tokens))]) + 2.0 ** -21 * np.abs(a)
    return a, ea


def expert_fp8(task):
    """FP8 and MXFP8 (row-wise scales only), one pass: for every call, the down-GEMM output
    rows of expert e's checked routes and their re-quantization allowance, (y [m, H],
    extra [m, H]) per call, tokens in the task's order."""
    from oracle import formats as F
    from oracle import moe as M
    e, per_call = task
    if not any(per_call):
        return None
    wg, wd = _weights(e, "gateup"), _weights(e, "down")
    awd = np.abs(wd)
    out = []
    for c, tokens in enumerate(per_call):
        if not tokens:
            out.append(None)
            continue
        a, ea = _gateup(c, tokens, wg)
        adeq, _ = M.quantize_acts(a.astype(np.float32), _CTX["fmt"])
        y = M.gemm_rows(adeq, wd)
        if _CTX["fmt"] == "mxfp8":
            from common import mxfp8_route_move
            extra = np.stack([awd @ mxfp8_route_move(a[i], ea[i]) for i in range(len(tokens))])
        else:
            extra = np.stack([_fp8_extra(a[i], ea[i], awd, F) for i in range(len(tokens))])
        out.append((y, extra))
    return out


def expert_nvfp4_first(task):
    """NVFP4 first pass, expert e: per call, the largest |silu(g)*u| (as float32) over all of
    the expert's routes with the kernels' error bound at that element, and the intermediate
    rows a and their error bounds ea of the checked routes (for the second pass)."""
    e, per_call_all, per_call_checked = task
    if not any(per_call_all):
        return None
    wg = _weights(e, "gateup")
    out = []
    for c, (tokens, checked) in enumerate(zip(per_call_all, per_call_checked)):
        if not tokens:
            out.append(None)
            continue
        a, ea = _gateup(c, tokens, wg)
        a32 = np.abs(a.astype(np.float32).astype(np.float64))
        r, col = np.unravel_index(np.argmax(a32), a32.shape)
        pos = {t: i for i, t in enumerate(tokens)}
        idx = [pos[t] for t in checked]
        out.append((float(a32[r, col]), float(ea[r, col]), a[idx], ea[idx]))
    return out


def expert_nvfp4_second(task):
    """NVFP4 second pass, expert e: the checked routes' intermediate quantized with each call's
    tensor scale, the down GEMM, and the re-quantization allowance."""
    from oracle import formats as F
    from oracle import moe as M
    e, per_call = task  # per call: None or (a [m, I], ea [m, I])
    if not any(p is not None for p in per_call):
        return None
    wd = _weights(e, "down")
    awd = np.abs(wd)
    out = []
    for c, p in enumerate(per_call):
        if p is None:
            out.append(None)
            continue
        a, ea = p
        call = _CTX["calls"][c]
        adeq, _ = M.quantize_acts(a.astype(np.float32), "nvfp4", call["gamax"])
        y = M.gemm_rows(adeq, wd)
        extra = np.stack([_nvfp4_extra(a[i], ea[i], awd, F, call["gamax"], call["gamax_rel"])
                          for i in range(a.shape[0])])
        out.append((y, extra))
    return out


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


def _nvfp4_extra(a, ea, awd, F, gamax, rel_g0):
    """One route's allowance for the NVFP4 intermediate's block-scale and code ties (as
    tests/common.nvfp4_requant_flip_bound; the tensor scale's uncertainty comes from the
    first pass)."""
    e2 = F.E2M1_VALUES[:8]
    mids2 = (e2[:-1] + e2[1:]) / 2
    e4 = F.E4M3_VALUES[:0x7F]
    mids4 = (e4[:-1] + e4[1:]) / 2
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


def forward_calls(calls, H, I, E, seed, fmt, workers):
    """The oracle's FFN output rows (float64) of the checked tokens of several calls that share
    one weight bank, with their re-quantization allowance.

    calls: list of dicts with x32 [T, H] float32 (bf16 values), ids [T, k], weights [T, k]
    (numpy) and checked (the tokens to evaluate). The bank's raw weights are
    synth.expert_weight_fp32(..., seed, e, tag). Token quantization covers all T tokens of a
    call (the NVFP4 tensor scales span the call). Returns a list of (out [T, H], extra [T, H])."""
    import multiprocessing as mp

    from oracle import moe as M
    ctx_calls = []
    for c in calls:
        if fmt == "fp8":
            xq, xs = M.quantize_act_fp8_fast(c["x32"])
            ctx_calls.append(dict(xq=xq, xs=xs))
        elif fmt == "mxfp8":
            xq, xs = M.quantize_mxfp8_fast(c["x32"])
            ctx_calls.append(dict(xq=xq, xs=xs))
        else:
            xq, xs, xg = M.quantize_nvfp4(c["x32"])
            ctx_calls.append(dict(xq=xq, xs=xs, xg=xg))
    ctx = dict(H=H, I=I, seed=seed, fmt=fmt, calls=ctx_calls)
    # per call and expert: the tokens routed to it, all of them and the checked ones, and the
    # checked routes (token, slot) in the same order
    routes_all, routes_chk = [], []
    for c in calls:
        ids = np.asarray(c["ids"])
        T, topk = ids.shape
        chk = set(int(t) for t in c["checked"])
        by_all = {e: [] for e in range(E)}
        by_chk = {e: [] for e in range(E)}
        for t in range(T):
            for j in range(topk):
                e = int(ids[t, j])
                if e < 0:
                    continue
                by_all[e].append(t)
                if t in chk:
                    by_chk[e].append((t, j))
        routes_all.append(by_all)
        routes_chk.append(by_chk)
    pool_ctx = mp.get_context("spawn")
    # one BLAS thread per worker (the pool provides the parallelism): spawned children
    # inherit the environment before they import numpy
    saved = {v: os.environ.get(v) for v in _BLAS_VARS}
    os.environ.update({v: "1" for v in _BLAS_VARS})
    try:
        if fmt in ("fp8", "mxfp8"):
            tasks = [(e, [[t for t, _ in rc[e]] for rc in routes_chk]) for e in range(E)]
            with pool_ctx.Pool(workers, initializer=_init, initargs=(ctx,)) as pool:
                res = pool.map(expert_fp8, tasks, chunksize=1)
        else:
            tasks = [(e, [ra[e] for ra in routes_all], [[t for t, _ in rc[e]] for rc in routes_chk])
                     for e in range(E)]
            with pool_ctx.Pool(workers, initializer=_init, initargs=(ctx,)) as pool:
                first = pool.map(expert_nvfp4_first, tasks, chunksize=1)
            for ci, cc in enumerate(ctx_calls):
                best = (0.0, 0.0)
                for e in range(E):
                    if first[e] is not None and first[e][ci] is not None and first[e][ci][0] > best[0]:
                        best = first[e][ci][:2]
                cc["gamax"] = best[0]
                cc["gamax_rel"] = best[1] / best[0] if best[0] > 0 else 0.0
            tasks2 = []
            for e in range(E):
                per = []
                for ci in range(len(calls)):
                    f = first[e][ci] if first[e] is not None else None
                    per.append(None if f is None or f[2].shape[0] == 0 else (f[2], f[3]))
                tasks2.append((e, per))
            del first
            with pool_ctx.Pool(workers, initializer=_init, initargs=(ctx,)) as pool:
                res = pool.map(expert_nvfp4_second, tasks2, chunksize=1)
    finally:
        for v, old in saved.items():
            if old is None:
                os.environ.pop(v, None)
            else:
                os.environ[v] = old
    results = []
    for ci, c in enumerate(calls):
        ids = np.asarray(c["ids"])
        T, topk = ids.shape
        out = np.zeros((T, H))
        extra = np.zeros((T, H))
        w = np.asarray(c["weights"], np.float64)
        contrib = {}
        for e in range(E):
            if res[e] is None or res[e][ci] is None:
                continue
            y, ex = res[e][ci]
            for i, (t, j) in enumerate(routes_chk[ci][e]):
                contrib[(t, j)] = (y[i], ex[i])
        # combine in ascending slot order per token, as the oracle's combine does
        for t in sorted(set(int(t) for t in c["checked"])):
            for j in range(topk):
                if (t, j) in contrib:
                    y, ex = contrib[(t, j)]
                    out[t] += w[t, j] * y
                    extra[t] += abs(w[t, j]) * ex
        results.append((out, extra))
    return results


def forward_subsample(x32, ids, weights, subsample, H, I, E, seed, fmt, workers):
    """forward_calls for one call: (out [T, H], extra [T, H]) of the tokens in `subsample`."""
    return forward_calls([dict(x32=x32, ids=ids, weights=weights, checked=subsample)], H, I, E, seed, fmt,
                         workers)[0]

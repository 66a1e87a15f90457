"""Shared helpers of the parity tests: seeded problems and the output tolerance.

Inputs come from `synth` (draws only). The CUDA side quantizes the raw weights with
the library's own kernel; the oracle quantizes the same raw values itself, so no
oracle input ever comes from the CUDA path.
"""
import numpy as np
import torch

import synth
from oracle import moe as M

# Output tolerance of the routed-expert FFN (bf16 outputs), per element.
TOL_REL, TOL_ABS_OF_MAX = 2e-2, 1e-3


# The re-quantization allowance (requant_flip_bound, nvfp4_requant_flip_bound) may carry at
# most this share of a call's output elements; every other element meets the stated
# tolerance on its own.
ALLOWANCE_SHARE_LIMIT = 1e-3


def _log():
    """Session-wide record of the output checks, read by the terminal summary in conftest.py
    (kept under one sys.modules key, whichever name this module was imported by)."""
    import sys
    import types
    mod = sys.modules.get("_ftmoe_check_log")
    if mod is None:
        mod = types.ModuleType("_ftmoe_check_log")
        mod.checks, mod.measures = [], []
        sys.modules["_ftmoe_check_log"] = mod
    return mod


def _test_name():
    import os
    return os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]


def record_measure(what, value, bound):
    """A measured quantity held to a stated bound (e.g. a GEMM's largest relative error)."""
    _log().measures.append(dict(test=_test_name(), what=what, value=float(value), bound=float(bound)))


def tolerance_report(got, ref, extra=0.0):
    """Counts of a comparison with the stated tolerance |got - ref| <= 2e-2 |ref| + 1e-3 max|ref|:
    elements; elements outside it; of those, elements inside it plus the allowance `extra`
    (they pass only because of the allowance); elements outside both; the largest
    |got - ref| / tolerance among the allowance-carried elements."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    tol = TOL_REL * np.abs(ref) + TOL_ABS_OF_MAX * (np.max(np.abs(ref)) if ref.size else 0.0)
    err = np.abs(got - ref)
    plain = err > tol
    fail = err > tol + extra
    carried = plain & ~fail
    worst = float(np.max(err[carried] / tol[carried])) if carried.any() else 0.0
    worst_fail = float(np.max(err[fail] - (tol + np.broadcast_to(extra, err.shape))[fail])) if fail.any() else 0.0
    return dict(n=int(err.size), outside_tolerance=int(plain.sum()), carried_by_allowance=int(carried.sum()),
                failing=int(fail.sum()), max_err_over_tol_carried=worst, worst_excess=worst_fail)


def out_tolerance_violations(got, ref):
    """Number of elements with |got - ref| > 2e-2 |ref| + 1e-3 max|ref|, and the worst excess."""
    r = tolerance_report(got, ref)
    return r["failing"], r["worst_excess"]


def assert_within_tolerance(got, ref, what="output", extra=0.0):
    """Every element within the stated tolerance plus `extra` (the re-quantization allowance,
    zero by default), and at most ALLOWANCE_SHARE_LIMIT of the elements needing the
    allowance at all. The counts go to the session's check record."""
    r = tolerance_report(got, ref, extra)
    _log().checks.append(dict(test=_test_name(), what=what, **r))
    assert r["failing"] == 0, f"{what}: {r['failing']} elements outside tolerance (worst excess {r['worst_excess']:.3e})"
    assert r["carried_by_allowance"] <= ALLOWANCE_SHARE_LIMIT * r["n"], (
        f"{what}: {r['carried_by_allowance']} of {r['n']} elements pass only with the re-quantization allowance")


# Relative bound on the kernels' fp32 error in a gate/up output element, as a fraction of
# the sum of the magnitudes of its products. The worst case of K fp32 additions is about
# K * 2**-24 of that sum; rounding errors add up like a random walk, so the observed error
# is orders of magnitude smaller, and 2**-22 of the sum is still ~100x above it.
FP32_SUM_REL = 2.0 ** -22


def requant_flip_bound(res, expert_ids, weights, bank_gu, bank_dn):
    """Extra output tolerance for re-quantization decisions the kernels may take differently.

    The SiLU-and-mul output is re-quantized to E4M3 before the down GEMM. The kernels decide
    each code from an fp32-accumulated gate/up value, the oracle from the exact one; where
    the scaled value lies within the kernels' fp32 error of a rounding midpoint, either
    neighbouring code is a correct result. For each such element i of route (t, j) the
    output of token t may move by |w_tj| * step_i * |W_down[h, i]|, step_i being the gap
    between the two codes times the group scale. Computed from the oracle's values only.
    """
    from oracle import formats as F
    ids = np.asarray(expert_ids)
    w = np.asarray(weights, np.float64)
    T = ids.shape[0]
    H = res["out"].shape[1]
    extra = np.zeros((T, H))
    pos = F.E4M3_VALUES[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2
    for (t, j), a in res["a"].items():
        e = int(ids[t, j])
        gu = res["gu"][(t, j)]
        inter = a.shape[0]
        xabs = np.abs(res["xdeq"][t])
        absum = np.abs(bank_gu.dequant(e)) @ xabs  # sum of |products| of each gate/up output
        eg = FP32_SUM_REL * absum + 2.0 ** -23 * np.abs(gu)
        g, u = gu[:inter], gu[inter:]
        sig = 1.0 / (1.0 + np.exp(-g))
        dsilu = sig * (1.0 + g * (1.0 - sig))
        ea = np.abs(dsilu * u) * eg[:inter] + np.abs(g * sig) * eg[inter:] + 2.0 ** -21 * np.abs(a)
        a32 = a.astype(np.float32).astype(np.float64)
        ng = -(-inter // 128)
        for gi in range(ng):
            sl = slice(gi * 128, min(inter, (gi + 1) * 128))
            blk = a32[sl]
            amax = np.max(np.abs(blk))
            if amax == 0:
                continue
            s = float(np.float32(np.float32(amax) / np.float32(448.0)))
            v = np.abs(blk) / s
            rel_s = (ea[sl][np.argmax(np.abs(blk))] / amax) + 2.0 ** -21
            ev = ea[sl] / s + v * rel_s
            k = np.clip(np.searchsorted(mids, v), 1, len(mids) - 1)
            d = np.minimum(np.abs(v - mids[k - 1]), np.abs(v - mids[np.minimum(k, len(mids) - 1)]))
            amb = np.nonzero(d <= ev)[0]
            if amb.size == 0:
                continue
            idx = np.arange(sl.start, sl.stop)[amb]
            step = np.abs(np.diff(pos))[np.clip(np.searchsorted(pos, v[amb]) - 1, 0, len(pos) - 2)] * s
            wd = np.abs(bank_dn.dequant(e)[:, idx])  # [H, n_amb]
            extra[t] += abs(w[t, j]) * (wd @ step)
    return extra


# The block-scaled tensor-core MMA accumulates e2m1 x e2m1 products with their e4m3 scales;
# its error is bounded here like an fp32 sum, with 4x the FP8 allowance for the unknown
# internal order of the 64-wide K steps.
NVFP4_SUM_REL = 2.0 ** -20


def _silu_mul_error(gu, absum, rel_sum):
    """Bound on the kernels' fp32 error in silu(g)*u from the gate/up outputs' errors."""
    inter = gu.shape[0] // 2
    eg = rel_sum * absum + 2.0 ** -21 * np.abs(gu)
    g, u = gu[:inter], gu[inter:]
    sig = 1.0 / (1.0 + np.exp(-g))
    dsilu = sig * (1.0 + g * (1.0 - sig))
    return np.abs(dsilu * u) * eg[:inter] + np.abs(g * sig) * eg[inter:]


def nvfp4_requant_flip_bound(res, expert_ids, weights, bank_gu, bank_dn):
    """requant_flip_bound for the NVFP4 intermediate: the tensor scale g (from the amax over
    all routes), each 16-block's e4m3 scale and each e2m1 code are decisions the kernels
    take from fp32 values; where one lies within their error of a rounding midpoint either
    neighbour is correct. An ambiguous block scale moves every element of the block by at
    most one quantization error per candidate (<= one effective scale each); an ambiguous
    code moves its element by the gap between the two codes. Oracle values only."""
    from oracle import formats as F
    ids = np.asarray(expert_ids)
    w = np.asarray(weights, np.float64)
    T = ids.shape[0]
    H = res["out"].shape[1]
    extra = np.zeros((T, H))
    e2 = F.E2M1_VALUES[:8]
    mids2 = (e2[:-1] + e2[1:]) / 2
    e4 = F.E4M3_VALUES[:0x7F]
    mids4 = (e4[:-1] + e4[1:]) / 2
    keys = sorted(res["a"].keys())
    if not keys:
        return extra
    eas = {}
    for (t, j) in keys:
        e = int(ids[t, j])
        gu = res["gu"][(t, j)]
        absum = np.abs(bank_gu.dequant(e)) @ np.abs(res["xdeq"][t])
        a = res["a"][(t, j)]
        eas[(t, j)] = _silu_mul_error(gu, absum, NVFP4_SUM_REL) + 2.0 ** -21 * np.abs(a)
    allabs = np.stack([np.abs(res["a"][k].astype(np.float32).astype(np.float64)) for k in keys])
    alle = np.stack([eas[k] for k in keys])
    am = np.unravel_index(np.argmax(allabs), allabs.shape)
    gamax = allabs[am]
    if gamax == 0:
        return extra
    g = float(np.float32(np.float32(gamax) / np.float32(448.0 * 6.0)))
    rel_g = alle[am] / gamax + 2.0 ** -22
    six_g = float(np.float32(np.float32(6.0) * np.float32(g)))
    for (t, j) in res["y"].keys():
        a32 = res["a"][(t, j)].astype(np.float32).astype(np.float64)
        ea = eas[(t, j)]
        e = int(ids[t, j])
        wd = None
        for b0 in range(0, a32.shape[0], 16):
            blk = np.abs(a32[b0:b0 + 16])
            amax_b = np.max(blk)
            if amax_b == 0:
                continue
            if wd is None:
                wd = np.abs(bank_dn.dequant(e))
            xb = amax_b / six_g
            rel_b = ea[b0 + np.argmax(blk)] / amax_b + rel_g + 2.0 ** -21
            kb = np.clip(np.searchsorted(mids4, xb), 1, len(mids4) - 1)
            db = min(abs(xb - mids4[kb - 1]), abs(xb - mids4[kb]))
            code = int(F.encode_e4m3(np.float32(xb)))
            if db <= rel_b * xb:
                c2 = [c for c in (code - 1, code + 1) if 0 <= c < 0x7F]
                effs = F.E4M3_VALUES[code] * g + max(F.E4M3_VALUES[c] for c in c2) * g
                extra[t] += abs(w[t, j]) * effs * wd[:, b0:b0 + 16].sum(axis=1)
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
            extra[t] += abs(w[t, j]) * (wd[:, b0 + amb] @ step)
    return extra


def mxfp8_sum_rel(k):
    """Bound on the MXFP8 block-scaled MMA's error over K as a share of the sum of the product
    magnitudes: one fp32 ulp (2^-23, truncation) of the running sum per K = 32 instruction.
    The accumulation grows with K, unlike the FP8 path's per-128 promotion on CUDA cores; the
    GEMM test measures it at K = 512 .. 7168 against this bound."""
    return (k / 32) * 2.0 ** -23


def mxfp8_route_move(a, ea):
    """Per intermediate element of one route, how far the kernels' MXFP8 re-quantization may
    move its dequantized value from the oracle's: a (float64 silu(g)*u of the route), ea (the
    kernels' fp32 error bound on it). Per 32 elements the shared exponent floor(log2(amax)) - 8
    and each e4m3 code are decisions taken from fp32 values. Where the oracle's block maximum
    lies within their error of a power of two, the block's scale may be a binade finer or
    coarser: under either an element's code is within an E4M3 step (1/8 of its value) or the
    clamp at 448 (under 1/8 of 512) of it, or below the smallest step, so a quarter of |a| plus
    two of the smallest steps covers it. Where a scaled value lies within their error of a code
    midpoint it may move by one code step."""
    from oracle import formats as F
    pos = F.E4M3_VALUES[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2
    inter = a.shape[0]
    a32 = a.astype(np.float32).astype(np.float64)
    move = np.zeros(inter)
    for b in range(-(-inter // 32)):
        sl = slice(b * 32, min(inter, (b + 1) * 32))
        blk = np.abs(a32[sl])
        amax = float(np.max(blk))
        if amax == 0:
            continue
        sh = M.mx_shared_exp(amax)
        X = 2.0 ** sh
        err_max = float(ea[sl][np.argmax(blk)])
        lo, hi = 2.0 ** (sh + 8), 2.0 ** (sh + 9)  # amax's binade when not clamped
        if amax - err_max < lo or amax + err_max >= hi:
            move[sl] = np.maximum(move[sl], 0.25 * blk + 2.0 ** -8 * X)
        v = blk / X
        ev = ea[sl] / X
        k = np.clip(np.searchsorted(mids, v), 1, len(mids) - 1)
        d = np.minimum(np.abs(v - mids[k - 1]), np.abs(v - mids[np.minimum(k, len(mids) - 1)]))
        step = np.abs(np.diff(pos))[np.clip(np.searchsorted(pos, v) - 1, 0, len(pos) - 2)] * X
        move[sl] = np.maximum(move[sl], np.where(d <= ev, step, 0.0))
    return move


def mxfp8_requant_flip_bound(res, expert_ids, weights, bank_gu, bank_dn):
    """requant_flip_bound for the MXFP8 intermediate (see mxfp8_route_move): each element's
    possible move reaches token t's output through |w_tj| |W_down[h, i]|. Computed from the
    oracle's values only."""
    ids = np.asarray(expert_ids)
    w = np.asarray(weights, np.float64)
    T = ids.shape[0]
    H = res["out"].shape[1]
    extra = np.zeros((T, H))
    for (t, j), a in res["a"].items():
        e = int(ids[t, j])
        gu = res["gu"][(t, j)]
        absum = np.abs(bank_gu.dequant(e)) @ np.abs(res["xdeq"][t])
        ea = _silu_mul_error(gu, absum, mxfp8_sum_rel(res["xdeq"].shape[1])) + 2.0 ** -21 * np.abs(a)
        move = mxfp8_route_move(a, ea)
        nz = np.nonzero(move)[0]
        if nz.size:
            extra[t] += abs(w[t, j]) * (np.abs(bank_dn.dequant(e)[:, nz]) @ move[nz])
    return extra


class Problem:
    """A seeded MoE FFN problem: activations, routes, weights, GPU bank, oracle bank."""

    _bank_cache = {}

    def __init__(self, T, H, I, E, topk, seed, device="cuda", active=None, ids=None, fmt="fp8"):
        import block_quantized_moe_gb300 as ft
        self.T, self.H, self.I, self.E, self.topk, self.seed, self.dev = T, H, I, E, topk, seed, device
        self.fmt = fmt
        self.ft_fmt = {"fp8": ft.FMT_FP8, "nvfp4": ft.FMT_NVFP4, "mxfp8": ft.FMT_MXFP8}[fmt]
        self.x = synth.activations_bf16(T, H, seed, device)
        if ids is None:
            ids = synth.routes(T, topk, E, seed, active_per_token=active, device=device)
        self.ids = ids.to(device)
        self.w = synth.routing_weights(T, topk, seed, device)
        key = (H, I, E, seed, device, fmt)
        if key not in Problem._bank_cache and fmt == "nvfp4":
            parts = []
            for n, k, raw in ((2 * I, H, self.raw_gateup), (H, I, self.raw_down)):
                q = torch.empty(E, n, k // 2, dtype=torch.uint8, device=device)
                sf = torch.empty(E, n, k // 16, dtype=torch.uint8, device=device)
                gs = torch.empty(E, dtype=torch.float32, device=device)
                for e in range(E):
                    ft.ftmoe_quantize_weights(raw(e)[None], q[e:e + 1], sf[e:e + 1], gs[e:e + 1],
                                              fmt=ft.FMT_NVFP4)
                parts.append((q, sf, gs))
            obg = M.LazyBank(lambda e: self.raw_gateup(e).cpu().numpy(), 2 * I, "nvfp4")
            obd = M.LazyBank(lambda e: self.raw_down(e).cpu().numpy(), H, "nvfp4")
            Problem._bank_cache[key] = (parts[0], parts[1], obg, obd)
        if key not in Problem._bank_cache and fmt == "mxfp8":
            parts = []
            for n, k, raw in ((2 * I, H, self.raw_gateup), (H, I, self.raw_down)):
                q = torch.empty(E, n, k, dtype=torch.uint8, device=device)
                sf = torch.empty(E, n, k // 32, dtype=torch.uint8, device=device)
                for e in range(E):
                    ft.ftmoe_quantize_weights(raw(e)[None], q[e:e + 1], sf[e:e + 1], fmt=ft.FMT_MXFP8)
                parts.append((q, sf))
            obg = M.LazyBank(lambda e: self.raw_gateup(e).cpu().numpy(), 2 * I, "mxfp8")
            obd = M.LazyBank(lambda e: self.raw_down(e).cpu().numpy(), H, "mxfp8")
            Problem._bank_cache[key] = (parts[0], parts[1], obg, obd)
        if fmt == "mxfp8":
            (gq, gs), (dq, ds), self.obank_gu, self.obank_dn = Problem._bank_cache[key]
            self.bank_gu = ft.make_bank(gq, gs, fmt=ft.FMT_MXFP8)
            self.bank_dn = ft.make_bank(dq, ds, fmt=ft.FMT_MXFP8)
            self._keep = (gq, gs, dq, ds)
            return
        if fmt == "nvfp4":
            (gq, gs, gg), (dq, ds, dg), self.obank_gu, self.obank_dn = Problem._bank_cache[key]
            self.bank_gu = ft.make_bank(gq, gs, gg, fmt=ft.FMT_NVFP4)
            self.bank_dn = ft.make_bank(dq, ds, dg, fmt=ft.FMT_NVFP4)
            self._keep = (gq, gs, gg, dq, ds, dg)
            return
        if key not in Problem._bank_cache:
            gq = torch.empty(E, 2 * I, H, dtype=torch.uint8, device=device)
            gs = torch.empty(E, -(-2 * I // 128), -(-H // 128), dtype=torch.float32, device=device)
            dq = torch.empty(E, H, I, dtype=torch.uint8, device=device)
            ds = torch.empty(E, -(-H // 128), -(-I // 128), dtype=torch.float32, device=device)
            for e in range(E):
                ft.ftmoe_quantize_weights(self.raw_gateup(e)[None], gq[e:e + 1], gs[e:e + 1])
                ft.ftmoe_quantize_weights(self.raw_down(e)[None], dq[e:e + 1], ds[e:e + 1])
            obg = M.LazyBank(lambda e: self.raw_gateup(e).cpu().numpy(), 2 * I)
            obd = M.LazyBank(lambda e: self.raw_down(e).cpu().numpy(), H)
            Problem._bank_cache[key] = (gq, gs, dq, ds, obg, obd)
        self.gq, self.gs, self.dq, self.ds, self.obank_gu, self.obank_dn = Problem._bank_cache[key]
        self.bank_gu = ft.make_bank(self.gq, self.gs)
        self.bank_dn = ft.make_bank(self.dq, self.ds)

    def raw_gateup(self, e):
        return synth.expert_weight_fp32(2 * self.I, self.H, self.seed, e, "gateup", self.dev)

    def raw_down(self, e):
        return synth.expert_weight_fp32(self.H, self.I, self.seed, e, "down", self.dev)

    def oracle(self, ids=None, weights=None, x=None, tokens_subset=None):
        ids = self.ids if ids is None else ids
        weights = self.w if weights is None else weights
        x = self.x if x is None else x
        return M.moe_forward(x.float().cpu().numpy(), ids.cpu().numpy(), weights.cpu().numpy(),
                             self.obank_gu, self.obank_dn, fmt=self.fmt, tokens_subset=tokens_subset)

    def check(self, out, ids=None, weights=None, x=None, tokens_subset=None):
        """Compare a GPU output with the oracle: the stated tolerance plus the bound for
        intermediate re-quantization decisions that sit on a rounding boundary."""
        ids = self.ids if ids is None else ids
        weights = self.w if weights is None else weights
        res = self.oracle(ids=ids, weights=weights, x=x, tokens_subset=tokens_subset)
        ref = res["out"]
        wv = torch.where(ids >= 0, weights, torch.zeros_like(weights)).cpu().numpy()
        bound = {"fp8": requant_flip_bound, "nvfp4": nvfp4_requant_flip_bound,
                 "mxfp8": mxfp8_requant_flip_bound}[self.fmt]
        extra = bound(res, ids.cpu().numpy(), wv, self.obank_gu, self.obank_dn)
        got = out.float().cpu().numpy()
        rows = list(range(self.T)) if tokens_subset is None else list(tokens_subset)
        what = (f"{self.fmt} forward T={self.T} H={self.H} I={self.I} E={self.E} top-{self.topk}"
                + ("" if tokens_subset is None else f" ({len(rows)}-token sample)"))
        assert_within_tolerance(got[rows], ref[rows], what=what, extra=extra[rows])
        return ref

    def forward(self, path=0, tok_tile=0, ids=None, weights=None, x=None, out=None, ws=None,
                out_dtype=torch.bfloat16):
        import block_quantized_moe_gb300 as ft
        ids = self.ids if ids is None else ids
        weights = self.w if weights is None else weights
        x = self.x if x is None else x
        if out is None:
            out = torch.empty(self.T, self.H, dtype=out_dtype, device=self.dev)
        shape = ft.moe_shape(self.T, self.H, self.I, self.topk, self.E, fmt=self.ft_fmt, tok_tile=tok_tile,
                             path=path, out_dtype=ft.out_dtype_code(out))
        if ws is None:
            ws = torch.empty(ft.ftmoe_forward_workspace_bytes(shape), dtype=torch.uint8, device=self.dev)
        ft.ftmoe_moe_forward(shape, x, ids, weights, self.bank_gu, self.bank_dn, out, ws)
        return out, ws, shape

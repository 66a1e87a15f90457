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


def out_tolerance_violations(got, ref):
    """Number of elements with |got - ref| > 2e-2 |ref| + 1e-3 max|ref|, and the worst excess."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    tol = TOL_REL * np.abs(ref) + TOL_ABS_OF_MAX * (np.max(np.abs(ref)) if ref.size else 0.0)
    excess = np.abs(got - ref) - tol
    return int(np.sum(excess > 0)), float(np.max(excess)) if excess.size else 0.0


def out_tolerance_violations_extra(got, ref, extra):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    tol = TOL_REL * np.abs(ref) + TOL_ABS_OF_MAX * (np.max(np.abs(ref)) if ref.size else 0.0) + extra
    excess = np.abs(got - ref) - tol
    return int(np.sum(excess > 0)), float(np.max(excess)) if excess.size else 0.0


def assert_within_tolerance(got, ref, what="output", extra=0.0):
    n, worst = out_tolerance_violations_extra(got, ref, extra)
    assert n == 0, f"{what}: {n} elements outside tolerance (worst excess {worst:.3e})"


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


class Problem:
    """A seeded MoE FFN problem: activations, routes, weights, GPU bank, oracle bank."""

    _bank_cache = {}

    def __init__(self, T, H, I, E, topk, seed, device="cuda", active=None, ids=None):
        import block_quantized_moe_gb300 as ft
        self.T, self.H, self.I, self.E, self.topk, self.seed, self.dev = T, H, I, E, topk, seed, device
        self.x = synth.activations_bf16(T, H, seed, device)
        if ids is None:
            ids = synth.routes(T, topk, E, seed, active_per_token=active, device=device)
        self.ids = ids.to(device)
        self.w = synth.routing_weights(T, topk, seed, device)
        key = (H, I, E, seed, device)
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
                             self.obank_gu, self.obank_dn, tokens_subset=tokens_subset)

    def check(self, out, ids=None, weights=None, x=None, tokens_subset=None):
        """Compare a GPU output with the oracle: the stated tolerance plus the bound for
        intermediate re-quantization decisions that sit on a rounding boundary."""
        ids = self.ids if ids is None else ids
        weights = self.w if weights is None else weights
        res = self.oracle(ids=ids, weights=weights, x=x, tokens_subset=tokens_subset)
        ref = res["out"]
        wv = torch.where(ids >= 0, weights, torch.zeros_like(weights)).cpu().numpy()
        extra = requant_flip_bound(res, ids.cpu().numpy(), wv, self.obank_gu, self.obank_dn)
        got = out.float().cpu().numpy()
        rows = list(range(self.T)) if tokens_subset is None else list(tokens_subset)
        assert_within_tolerance(got[rows], ref[rows], extra=extra[rows])
        return ref

    def forward(self, path=0, tok_tile=0, ids=None, weights=None, x=None, out=None, ws=None):
        import block_quantized_moe_gb300 as ft
        ids = self.ids if ids is None else ids
        weights = self.w if weights is None else weights
        x = self.x if x is None else x
        shape = ft.moe_shape(self.T, self.H, self.I, self.topk, self.E, tok_tile=tok_tile, path=path)
        if ws is None:
            ws = torch.empty(ft.ftmoe_forward_workspace_bytes(shape), dtype=torch.uint8, device=self.dev)
        if out is None:
            out = torch.empty(self.T, self.H, dtype=torch.bfloat16, device=self.dev)
        ft.ftmoe_moe_forward(shape, x, ids, weights, self.bank_gu, self.bank_dn, out, ws)
        return out, ws, shape

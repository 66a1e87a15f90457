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


def assert_within_tolerance(got, ref, what="output"):
    n, worst = out_tolerance_violations(got, ref)
    assert n == 0, f"{what}: {n} elements outside tolerance (worst excess {worst:.3e})"


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

"""The prefill workloads at full size against the oracle: 256 experts, top-6, hidden 7168,
intermediate 2048, FP8 with 128x128 block scales, NVFP4 and MXFP8.

Every token is compared at 1,536 routes (256 tokens) and 6,144 routes (1,024 tokens); the
24,576-route calls (4,096 tokens) are compared on a seeded random 1,024-token subsample.
The GPU runs each whole call. One weight bank per format serves all of its sizes, so the
oracle draws and quantizes each expert's weights once per pass for all of them (see
fullsize_oracle.py: expert by expert in spawned workers, all of it the oracle's own
arithmetic; the NVFP4 tensor scales span each whole call). Expert weights are drawn on the
CPU so that both sides quantize the same raw values.
"""
import concurrent.futures
import os

import numpy as np
import pytest
import torch

import synth
from common import assert_within_tolerance
from fullsize_oracle import forward_calls

pytestmark = pytest.mark.gpu
DEV = "cuda"
H, I, E, TOPK = 7168, 2048, 256, 6
WEIGHT_SEED = 0xF7E00004
# tokens of each call, its input seed and how many of its tokens the oracle checks
SIZES = {1536: (256, 0xF7E00041, None), 6144: (1024, 0xF7E00042, None), 24576: (4096, 0xF7E00043, 1024)}


@pytest.fixture(scope="module")
def ft():
    import block_quantized_moe_gb300 as ft
    ft.lib()
    return ft


def _bank(ft, n, k, tag, fmt):
    """The GPU bank quantized by libftmoe from the CPU draws (drawn on all host threads)."""
    if fmt == "fp8":
        q = torch.empty(E, n, k, dtype=torch.uint8, device=DEV)
        s = torch.empty(E, -(-n // 128), -(-k // 128), dtype=torch.float32, device=DEV)
        g = None
    elif fmt == "mxfp8":
        q = torch.empty(E, n, k, dtype=torch.uint8, device=DEV)
        s = torch.empty(E, n, k // 32, dtype=torch.uint8, device=DEV)
        g = None
    else:
        q = torch.empty(E, n, k // 2, dtype=torch.uint8, device=DEV)
        s = torch.empty(E, n, k // 16, dtype=torch.uint8, device=DEV)
        g = torch.empty(E, dtype=torch.float32, device=DEV)
    f = {"fp8": ft.FMT_FP8, "nvfp4": ft.FMT_NVFP4, "mxfp8": ft.FMT_MXFP8}[fmt]
    draw = lambda e: synth.expert_weight_fp32(n, k, WEIGHT_SEED, e, tag, "cpu")  # noqa: E731
    threads = max(2, min(16, os.cpu_count() or 4))
    with concurrent.futures.ThreadPoolExecutor(max_workers=threads) as ex:
        for e0 in range(0, E, threads):
            for i, w in enumerate(ex.map(draw, range(e0, min(E, e0 + threads)))):
                e = e0 + i
                ft.ftmoe_quantize_weights(w.to(DEV)[None], q[e:e + 1], s[e:e + 1], None if g is None else g[e:e + 1],
                                          fmt=f)
            torch.cuda.synchronize()
    return (q, s, g), ft.make_bank(q, s, g, fmt=f)


def _call(routes):
    T, seed, checked = SIZES[routes]
    x = synth.activations_bf16(T, H, seed, "cpu")
    ids = synth.routes_fast(T, TOPK, E, seed, "cpu")
    w = synth.routing_weights(T, TOPK, seed, "cpu")
    sub = list(range(T)) if checked is None else synth.subsample(T, checked, seed)
    return x, ids, w, sub


def _gpu_forward(ft, banks, x, ids, w, fmt, path=0):
    T = x.shape[0]
    f = {"fp8": ft.FMT_FP8, "nvfp4": ft.FMT_NVFP4, "mxfp8": ft.FMT_MXFP8}[fmt]
    shape = ft.moe_shape(T, H, I, TOPK, E, fmt=f, path=path)
    ws = torch.empty(ft.ftmoe_forward_workspace_bytes(shape), dtype=torch.uint8, device=DEV)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    ft.ftmoe_moe_forward(shape, x.to(DEV), ids.to(DEV), w.to(DEV), banks[0], banks[1], out, ws)
    torch.cuda.synchronize()
    assert ft.ftmoe_read_error_flags() == 0
    return out


@pytest.mark.parametrize("fmt,sizes", [("fp8", (1536, 6144, 24576)), ("nvfp4", (6144, 24576)),
                                       ("mxfp8", (6144, 24576))])
def test_prefill_full_sizes_against_the_oracle(ft, fmt, sizes):
    keep_gu, bank_gu = _bank(ft, 2 * I, H, "gateup", fmt)
    keep_dn, bank_dn = _bank(ft, H, I, "down", fmt)
    calls, outs = [], []
    for r in sizes:
        x, ids, w, sub = _call(r)
        out = _gpu_forward(ft, (bank_gu, bank_dn), x, ids, w, fmt)
        got = out.float().cpu().numpy()
        assert not np.isnan(got).any()
        if fmt == "fp8" and r == 6144:
            # at 6,144 routes (token tile 32) the automatic forward fuses SiLU-and-mul into the
            # gate/up GEMM; the separate-kernel forward gives the same bits
            assert ft.ftmoe_forward_workspace_layout(ft.moe_shape(x.shape[0], H, I, TOPK, E))["gateup_bytes"] == 0
            sep = _gpu_forward(ft, (bank_gu, bank_dn), x, ids, w, fmt, path=2)
            assert torch.equal(out.view(torch.int16), sep.view(torch.int16))
        if fmt == "fp8" and r == 24576:
            # at 24,576 routes (token tile 128, CTA pairs) the forward that adds up each token's
            # rows inside the down GEMM (path 5) gives the automatic forward's bits
            comb = _gpu_forward(ft, (bank_gu, bank_dn), x, ids, w, fmt, path=5)
            assert torch.equal(out.view(torch.int16), comb.view(torch.int16))
        outs.append((got, sub))
        calls.append(dict(x32=x.float().numpy(), ids=ids.numpy(), weights=w.numpy(), checked=sub))
    del keep_gu, keep_dn, bank_gu, bank_dn
    torch.cuda.empty_cache()
    res = forward_calls(calls, H, I, E, WEIGHT_SEED, fmt, workers=max(2, os.cpu_count() or 4))
    for r, (got, sub), (ref, extra) in zip(sizes, outs, res):
        T = got.shape[0]
        what = f"{fmt} forward, {r:,} routes, {len(sub)} of {T} tokens"
        assert_within_tolerance(got[sub], ref[sub], what=what, extra=extra[sub])

"""The largest prefill workloads at full size, checked on a seeded random 1,024-token
subsample: 256 experts, top-6, hidden 7168, intermediate 2048, 24,576 routes (4,096
tokens), FP8 with 128x128 block scales and NVFP4. The GPU runs the whole call; the oracle
evaluates the subsample's routes (expert by expert in spawned workers, all of it the
oracle's own arithmetic; the NVFP4 tensor scales still span the whole call). Expert
weights are drawn on the CPU so that both sides quantize the same raw values."""
import os

import numpy as np
import pytest
import torch

import synth
from common import assert_within_tolerance
from fullsize_oracle import forward_subsample

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ft():
    import block_quantized_moe_gb300 as ft
    ft.lib()
    return ft


def _bank(ft, E, n, k, seed, tag, fmt):
    if fmt == "fp8":
        q = torch.empty(E, n, k, dtype=torch.uint8, device=DEV)
        s = torch.empty(E, -(-n // 128), -(-k // 128), dtype=torch.float32, device=DEV)
        g = None
    else:
        q = torch.empty(E, n, k // 2, dtype=torch.uint8, device=DEV)
        s = torch.empty(E, n, k // 16, dtype=torch.uint8, device=DEV)
        g = torch.empty(E, dtype=torch.float32, device=DEV)
    f = ft.FMT_FP8 if fmt == "fp8" else ft.FMT_NVFP4
    for e in range(E):
        w = synth.expert_weight_fp32(n, k, seed, e, tag, "cpu").to(DEV)
        ft.ftmoe_quantize_weights(w[None], q[e:e + 1], s[e:e + 1], None if g is None else g[e:e + 1], fmt=f)
    return (q, s, g), ft.make_bank(q, s, g, fmt=f)


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4"])
def test_prefill_24576_routes_on_1024_token_subsample(ft, fmt):
    T, H, I, E, k, seed = 4096, 7168, 2048, 256, 6, 0xF7E00004
    x = synth.activations_bf16(T, H, seed, "cpu")
    ids = synth.routes_fast(T, k, E, seed, "cpu")
    w = synth.routing_weights(T, k, seed, "cpu")
    keep_gu, bank_gu = _bank(ft, E, 2 * I, H, seed, "gateup", fmt)
    keep_dn, bank_dn = _bank(ft, E, H, I, seed, "down", fmt)
    f = ft.FMT_FP8 if fmt == "fp8" else ft.FMT_NVFP4
    shape = ft.moe_shape(T, H, I, k, E, fmt=f)
    ws = torch.empty(ft.ftmoe_forward_workspace_bytes(shape), dtype=torch.uint8, device=DEV)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    ft.ftmoe_moe_forward(shape, x.to(DEV), ids.to(DEV), w.to(DEV), bank_gu, bank_dn, out, ws)
    torch.cuda.synchronize()
    assert ft.ftmoe_read_error_flags() == 0
    got = out.float().cpu().numpy()
    assert not np.isnan(got).any()
    del keep_gu, keep_dn, ws
    torch.cuda.empty_cache()
    sub = synth.subsample(T, 1024, seed)
    ref, extra = forward_subsample(x.float().numpy(), ids.numpy(), w.numpy(), sub, H, I, E, seed, fmt,
                                   workers=max(2, (os.cpu_count() or 4)))
    assert_within_tolerance(got[sub], ref[sub], what=f"{fmt} forward, 24,576 routes", extra=extra[sub])


def test_prefill_6144_routes_fused_equals_separate_and_oracle_sample(ft):
    # 1,024 tokens x top-6 of 256 experts (24 rows per expert, token tile 32): the automatic
    # forward fuses SiLU-and-mul into the gate/up GEMM here. Its whole output must equal the
    # separate-kernel forward bit for bit, and a seeded 2-token sample must match the oracle.
    from common import Problem
    T, H, I, E, k, seed = 1024, 7168, 2048, 256, 6, 0xF7E00006
    ids = synth.routes_fast(T, k, E, seed, DEV)
    p = Problem(T, H, I, E, k, seed=seed, ids=ids)
    assert ft.ftmoe_forward_workspace_layout(ft.moe_shape(T, H, I, k, E))["gateup_bytes"] == 0  # fused
    out_auto, _, _ = p.forward(path=0)
    out_sep, _, _ = p.forward(path=2)
    torch.cuda.synchronize()
    assert ft.ftmoe_read_error_flags() == 0
    assert torch.equal(out_auto.view(torch.int16), out_sep.view(torch.int16))
    p.check(out_auto, tokens_subset=synth.subsample(T, 2, seed))

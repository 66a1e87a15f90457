"""The allocation-free forward (intermediates in the library's own device array) against
the workspace forward, through the C ABI.

Some callers cannot allocate device memory: a plugin inside a runtime that owns every
byte of device memory and offers no allocator, or a latency path that cannot take an
allocation's implicit synchronisation. ftmoe_moe_forward_noalloc serves them from a fixed
file-scope device array. It runs the same kernels as ftmoe_moe_forward on the same inputs,
so its output must equal the workspace forward's bit for bit, call after call (the shared
array keeps the previous call's contents), and it must refuse shapes larger than its array.

This file is collected last, so that a run stopping at its first failure has already run
every other test; it passes alone in a fresh process as well as after the others.
"""
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _problem(ft, T, H, I, E, k, seed):
    x = synth.activations_bf16(T, H, seed, DEV)
    ids = synth.routes(T, k, E, seed, active_per_token=[k, k // 2, 0, k][:T] if T <= 4 else None, device=DEV)
    w = synth.routing_weights(T, k, seed, DEV)
    gq, gs, _ = ft.quantize_weights(torch.stack([synth.expert_weight_fp32(2 * I, H, seed, e, "gateup", DEV)
                                                 for e in range(E)]))
    dq, ds, _ = ft.quantize_weights(torch.stack([synth.expert_weight_fp32(H, I, seed, e, "down", DEV)
                                                 for e in range(E)]))
    return x, ids, w, (gq, gs, dq, ds)


# path 0: the automatic choice; path 3: SiLU-and-mul fused into the gate/up GEMM; path 4: the
# fused decode kernel (its partial sums and counters live in the shared array too)
@pytest.mark.parametrize("path", [0, 3, 4])
def test_noalloc_forward_equals_workspace_forward_two_calls(path):
    import block_quantized_moe_gb300 as ft
    T, H, I, E, k = 4, 1024, 512, 16, 4
    shape = ft.moe_shape(T, H, I, k, E, path=path)
    ws = torch.empty(ft.ftmoe_forward_workspace_bytes(shape), dtype=torch.uint8, device=DEV)
    for call, seed in enumerate((101 + path, 202 + path)):
        x, ids, w, (gq, gs, dq, ds) = _problem(ft, T, H, I, E, k, seed)
        bg, bd = ft.make_bank(gq, gs), ft.make_bank(dq, ds)
        ref = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
        got = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device=DEV)
        ft.ftmoe_moe_forward(shape, x, ids, w, bg, bd, ref, ws)
        ft.ftmoe_moe_forward_noalloc(shape, x, ids, w, bg, bd, got)
        torch.cuda.synchronize()
        assert ft.ftmoe_read_error_flags() == 0, f"call {call}"
        # same kernels, same inputs: identical bits (a region of the shared array read before
        # it is written would show up here)
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), f"call {call}"


def test_noalloc_forward_refuses_shapes_beyond_its_array():
    import block_quantized_moe_gb300 as ft
    shape = ft.moe_shape(4096, 7168, 2048, 6, 256)  # a prefill workspace of ~1.5 GB
    x = torch.zeros(1, 1, dtype=torch.bfloat16, device=DEV)
    dummy = ft.ExpertBank(0, 256, 4096, 7168, None, None, None)
    with pytest.raises(ft.FtmoeError) as ei:
        ft.ftmoe_moe_forward_noalloc(shape, x, x, x, dummy, dummy, x)
    assert ei.value.status == ft.FTMOE_WORKSPACE_TOO_SMALL

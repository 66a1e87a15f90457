"""The routing-weighted combine inside the down GEMM (FP8, CTA pairs, token tile 64 or 128).

The forward's down GEMM can add up each token's rows itself: four combine warps per CTA count
the arrivals of a token's routes per 128-column block and, at the last one, add the token's
rows in ascending slot order with the separate combine kernel's fp32 expression and output
rounding (the decode page's reduction after the down GEMM; inactive slots unread). So:
  - the forward with the combine inside (path 5) equals the forward with every step
    separate (path 2) and the automatic forward bit for bit, in
    bf16, fp16 and fp32, with inactive routes, tokens without an active route, a token that
    lists one expert twice and ragged expert segments;
  - calls on one workspace are independent: the arrival counters are re-zeroed by each call,
    also in a CUDA graph replayed over poisoned intermediates while the routes change;
  - it matches the oracle.
"""
import numpy as np
import pytest
import torch

import synth
from tests.common import Problem

pytestmark = pytest.mark.gpu
DEV = "cuda"
NAN_BITS = 0x7FC00000


@pytest.fixture(scope="module")
def ft():
    import block_quantized_moe_gb300 as ft
    ft.lib()
    return ft


def _same(a, b):
    if a.dtype == torch.float32:
        return torch.equal(a.view(torch.int32), b.view(torch.int32))
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


def _ids_with_gaps(T, k, E, seed):
    """Routes with inactive slots, a few tokens without any active route and one token that
    lists an expert twice."""
    ids = synth.routes(T, k, E, seed, active_per_token=[k, k - 2, 0, k, 1, k - 1] * (T // 6 + 1), device="cpu")
    ids = ids[:T].clone()
    ids[5, 1] = ids[5, 0]  # token 5: its first expert twice
    return ids.to(DEV)


@pytest.mark.parametrize("tok_tile", [64, 128])
@pytest.mark.parametrize("out_dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_comb_forward_equals_separate_forward(ft, tok_tile, out_dtype):
    # 300 tokens x top-6 over 8 experts: about 190 rows per active expert, so two or three
    # token tiles per expert with ragged tails; H = 768: three block pairs
    T, H, I, E, k = 300, 768, 256, 8, 6
    p = Problem(T, H, I, E, k, seed=0xF7E000C1, ids=_ids_with_gaps(T, k, E, 0xC1))
    w = torch.where(p.ids >= 0, p.w, torch.full_like(p.w, float("nan")))  # never read
    sep, _, _ = p.forward(path=2, tok_tile=tok_tile, weights=w, out_dtype=out_dtype)
    out, ws, shape = p.forward(path=5, tok_tile=tok_tile, weights=w, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert ft.ftmoe_read_error_flags() == 0
    assert ft.ftmoe_forward_workspace_layout(shape)["counters_bytes"] == T * (H // 128) * 4
    assert _same(out, sep)
    assert torch.all(out[2].float() == 0)  # a token without an active route
    # the automatic path (the combine kernel) gives the same bits
    auto, auto_ws, auto_shape = p.forward(path=0, tok_tile=tok_tile, weights=w, out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert ft.ftmoe_forward_workspace_layout(auto_shape)["counters_bytes"] == 0
    assert _same(auto, sep)
    if out_dtype == torch.bfloat16:
        p.check(out, weights=w)


def test_comb_calls_on_one_workspace_are_independent(ft):
    T, H, I, E, k = 200, 512, 256, 6, 4
    p = Problem(T, H, I, E, k, seed=0xF7E000C2, active=4)
    other = synth.routes(T, k, E, 0xC3, active_per_token=[4, 2, 0, 3] * 50, device=DEV)
    first, ws, _ = p.forward(path=5, tok_tile=128)
    first = first.clone()
    again, _, _ = p.forward(path=5, tok_tile=128, ws=ws)
    mid, _, _ = p.forward(path=5, tok_tile=128, ids=other, ws=ws)
    mid = mid.clone()
    last, _, _ = p.forward(path=5, tok_tile=128, ws=ws)
    mid_sep, _, _ = p.forward(path=2, tok_tile=128, ids=other)
    torch.cuda.synchronize()
    assert _same(first, again) and _same(first, last)
    assert _same(mid, mid_sep)


def _poison(ws, lay):
    nan = torch.tensor([NAN_BITS], dtype=torch.int32).view(torch.float32).item()
    for off, nbytes, kind in ((lay["gateup"], lay["gateup_bytes"], "f"), (lay["down"], lay["down_bytes"], "f"),
                              (lay["act_q"], lay["act_q_bytes"], "b"),
                              (lay["act_scales"], lay["act_scales_bytes"], "f"),
                              (lay["counters"], lay["counters_bytes"], "b")):
        region = ws[off:off + nbytes]
        if kind == "f":
            region.view(torch.float32).fill_(nan)
        else:
            region.fill_(0xFF)


def test_comb_graph_replay_with_poisoned_intermediates(ft):
    T, H, I, E, k = 256, 1024, 256, 8, 6
    p = Problem(T, H, I, E, k, seed=0xF7E000C4, active=6)
    shape = ft.moe_shape(T, H, I, k, E, tok_tile=128, path=5)
    lay = ft.ftmoe_forward_workspace_layout(shape)
    assert lay["counters_bytes"] > 0
    ws = torch.empty(lay["total"], dtype=torch.uint8, device=DEV)
    x_in = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    ids_in = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w_in = torch.empty(T, k, dtype=torch.float32, device=DEV)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    x_in.copy_(p.x)
    ids_in.copy_(p.ids)
    w_in.copy_(p.w)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ft.ftmoe_moe_forward(shape, x_in, ids_in, w_in, p.bank_gu, p.bank_dn, out, ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ft.ftmoe_moe_forward(shape, x_in, ids_in, w_in, p.bank_gu, p.bank_dn, out, ws)
    for step, active in enumerate([6, 2, 0, 4, 6]):
        ids = synth.routes(T, k, E, 200 + step, active_per_token=active, device=DEV)
        x = synth.activations_bf16(T, H, 200 + step, DEV)
        w = synth.routing_weights(T, k, 200 + step, DEV)
        w = torch.where(ids >= 0, w, torch.full_like(w, float("nan")))
        ids_in.copy_(ids)
        x_in.copy_(x)
        w_in.copy_(w)
        _poison(ws, lay)
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        sep, _, _ = p.forward(path=2, tok_tile=128, ids=ids, weights=w, x=x)
        torch.cuda.synchronize()
        assert _same(out, sep), f"replay {step} ({active} active routes per token)"
        if active == 0:
            assert torch.all(out.float() == 0)
    assert ft.ftmoe_read_error_flags() == 0


def test_comb_refused_where_it_does_not_apply(ft):
    # path 5 needs FP8, whole 256-column block pairs of H and a token tile of 64 or 128
    T, I, E, k = 64, 256, 4, 2
    for H, tile in ((640, 128), (512, 32)):
        shape = ft.moe_shape(T, H, I, k, E, tok_tile=tile, path=5)
        assert ft.ftmoe_forward_workspace_layout(shape)["counters_bytes"] == 0
    p = Problem(T, 512, I, E, k, seed=0xF7E000C5, active=2)
    with pytest.raises(ft.FtmoeError):
        p.forward(path=5, tok_tile=32)
    # an output row stride that is not a multiple of four elements: path 5 refuses it
    wide = torch.zeros(T, 514, dtype=torch.bfloat16, device=DEV)
    view = wide[:, :512]
    with pytest.raises(ft.FtmoeError):
        p.forward(path=5, tok_tile=128, out=view)
    auto, _, _ = p.forward(path=0, tok_tile=128, out=view)
    sep, _, _ = p.forward(path=2, tok_tile=128)
    torch.cuda.synchronize()
    assert _same(auto.contiguous(), sep)

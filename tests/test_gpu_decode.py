"""Decode MoE FFN (the grouped path and the route-slot streaming path) against the oracle,
through the C ABI.

Workloads of the FreeToken decode page ("perf(moe): skip inactive block-fp8 decode
routes", GPU decode A/B): batch 1 (and 8), top-k 8, FP8 block-scaled expert banks,
bf16 activations, with 8/4/2/0 of the 8 routes active. Its validation protocol is
reproduced: one CUDA graph replayed while routes and inputs change, the gate/up,
activation and down buffers NaN-poisoned before each replay, inactive routes exactly
zero, and the output equal to the old clamped-slot / zero-weight path.
"""
import numpy as np
import pytest
import torch

import synth
from tests.common import Problem

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ft():
    import block_quantized_moe_gb300 as ft
    ft.lib()
    return ft


def _check(prob, out, ids=None, weights=None, x=None):
    return prob.check(out, ids=ids, weights=weights, x=x)


@pytest.mark.parametrize("path", [0, 1, 2, 3, 4])
def test_decode_2048_768_two_of_eight_active(ft, path):
    # hidden 2048, intermediate 768, 8 resident experts, top-k 8, 6 of 8 slots -1
    p = Problem(1, 2048, 768, 8, 8, seed=0xF7E00001, active=2)
    assert int((p.ids >= 0).sum()) == 2
    out, _, _ = p.forward(path=path)
    torch.cuda.synchronize()
    _check(p, out)


@pytest.mark.parametrize("path", [1, 2, 3, 4])
@pytest.mark.parametrize("T", [1, 8])
@pytest.mark.parametrize("active", [8, 4, 2, 0])
def test_decode_4096_1024_sweep(ft, T, active, path):
    # path 1: route-slot streaming kernel; path 2: segment + gather + tcgen05 grouped GEMMs;
    # path 3: the same with SiLU-and-mul fused into the gate/up GEMM; path 4: the fused
    # decode kernel (gate/up, SiLU-and-mul, down and combine in one launch)
    p = Problem(T, 4096, 1024, 64, 8, seed=0xF7E00002, active=active)
    out, ws, shape = p.forward(path=path)
    torch.cuda.synchronize()
    ref = _check(p, out)
    if active == 0:
        assert torch.all(out.float() == 0)
        assert np.all(ref == 0)


def _poison(ws, lay):
    nan = torch.tensor([0x7FC00000], dtype=torch.int32).view(torch.float32).item()
    # the fused decode path's partial sums and arrival counters too (the counters must be
    # zeroed by the forward itself on every call)
    for off, nbytes, kind in ((lay["gateup"], lay["gateup_bytes"], "f"), (lay["down"], lay["down_bytes"], "f"),
                              (lay["act_q"], lay["act_q_bytes"], "b"),
                              (lay["act_scales"], lay["act_scales_bytes"], "f"),
                              (lay["partials"], lay["partials_bytes"], "f"),
                              (lay["counters"], lay["counters_bytes"], "b")):
        region = ws[off:off + nbytes]
        if kind == "f":
            region.view(torch.float32).fill_(nan)
        else:
            region.fill_(0xFF)


@pytest.mark.parametrize("T,path", [(1, 1), (8, 1), (8, 2), (8, 3), (1, 4), (8, 4)])
def test_graph_replay_with_poisoned_intermediates(ft, T, path):
    H, I, E, k = 4096, 1024, 64, 8
    p = Problem(T, H, I, E, k, seed=0xF7E00002, active=8)
    shape = ft.moe_shape(T, H, I, k, E, path=path)
    lay = ft.ftmoe_forward_workspace_layout(shape)
    ws = torch.empty(lay["total"], dtype=torch.uint8, device=DEV)
    x_in = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    ids_in = torch.empty(T, k, dtype=torch.int32, device=DEV)
    w_in = torch.empty(T, k, dtype=torch.float32, device=DEV)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    x_in.copy_(p.x)
    ids_in.copy_(p.ids)
    w_in.copy_(p.w)
    # warm up on a side stream, then capture one forward
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ft.ftmoe_moe_forward(shape, x_in, ids_in, w_in, p.bank_gu, p.bank_dn, out, ws, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ft.ftmoe_moe_forward(shape, x_in, ids_in, w_in, p.bank_gu, p.bank_dn, out, ws)
    for step, active in enumerate([8, 2, 0, 4, 8]):
        ids = synth.routes(T, k, E, 100 + step, active_per_token=active, device=DEV)
        x = synth.activations_bf16(T, H, 100 + step, DEV)
        w = synth.routing_weights(T, k, 100 + step, DEV)
        w = torch.where(ids >= 0, w, torch.full_like(w, float("nan")))  # never read
        ids_in.copy_(ids)
        x_in.copy_(x)
        w_in.copy_(w)
        _poison(ws, lay)
        g.replay()
        torch.cuda.synchronize()
        _check(p, out, ids=ids, weights=w, x=x)
        assert not torch.any(torch.isnan(out.float()))
        if path != 1:
            continue  # grouped paths: inactive routes have no rows at all
        # route-slot path: exact zeros in the gate/up, activation and down rows of inactive routes
        R = T * k
        gu = ws[lay["gateup"]:lay["gateup"] + lay["gateup_bytes"]].view(torch.float32).view(R, 2 * I)
        dn = ws[lay["down"]:lay["down"] + lay["down_bytes"]].view(torch.float32).view(R, H)
        aq = ws[lay["act_q"]:lay["act_q"] + lay["act_q_bytes"]].view(R, I)
        asc = ws[lay["act_scales"]:lay["act_scales"] + lay["act_scales_bytes"]].view(torch.float32).view(R, -1)
        inactive = (ids.view(-1) < 0).nonzero().view(-1)
        if inactive.numel():
            for buf in (gu, dn, asc):
                rows = buf[inactive]
                assert torch.all(rows.view(torch.int32) == 0)  # +0.0 exactly, no NaN left
            assert torch.all(aq[inactive] == 0)
        assert not torch.any(torch.isnan(out.float()))


@pytest.mark.parametrize("path", [1, 2, 3, 4])
def test_negative_slots_equal_clamped_zero_weight_path(ft, path):
    T, H, I, E, k = 8, 4096, 1024, 64, 8
    p = Problem(T, H, I, E, k, seed=0xF7E00002, active=2)
    ids_new = p.ids.clone()
    w_new = torch.where(ids_new >= 0, p.w, torch.full_like(p.w, float("nan")))
    ids_old = torch.where(ids_new >= 0, ids_new, torch.zeros_like(ids_new))  # slot 0 ...
    w_old = torch.where(ids_new >= 0, p.w, torch.zeros_like(p.w))             # ... weight 0
    out_new, _, _ = p.forward(path=path, ids=ids_new, weights=w_new)
    out_old, _, _ = p.forward(path=path, ids=ids_old, weights=w_old)
    torch.cuda.synchronize()
    assert torch.equal(out_new.view(torch.int16), out_old.view(torch.int16))


@pytest.mark.parametrize("path", [1, 2, 3, 4])
def test_all_inactive_and_empty_bank_use(ft, path):
    T, H, I, E, k = 8, 4096, 1024, 64, 8
    p = Problem(T, H, I, E, k, seed=0xF7E00002, active=0)
    w = torch.full_like(p.w, float("nan"))
    out, ws, shape = p.forward(path=path, weights=w)
    torch.cuda.synchronize()
    assert torch.all(out.view(torch.int16) == 0)


@pytest.mark.parametrize("path", [1, 4])
def test_out_of_range_expert_id_is_flagged_not_read(ft, path):
    T, H, I, E, k = 1, 2048, 768, 8, 8
    p = Problem(T, H, I, E, k, seed=0xF7E00001, active=2)
    ft.ftmoe_read_error_flags()
    ids = p.ids.clone()
    ids[0, (ids[0] < 0).nonzero()[0, 0]] = E + 3  # one bad id in place of an inactive slot
    w = p.w.clone()
    out, _, _ = p.forward(path=path, ids=ids, weights=w)
    flags = ft.ftmoe_read_error_flags()
    assert flags & ft.ERR_EXPERT_ID_RANGE
    ref_ids = torch.where(ids >= E, torch.full_like(ids, -1), ids)
    _check(p, out, ids=ref_ids, weights=w)

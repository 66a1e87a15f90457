"""Grouped (prefill) path: the tcgen05 grouped GEMM and the segment -> gather -> GEMM ->
SiLU -> GEMM -> combine forward, against the oracle, through the C ABI.

Shapes cover several tiles and ragged tails (N and K not multiples of 128, experts with
0, 1 and more rows than a token tile), every token tile of the density picker
(FreeToken "perf(dsfp4): pick the grouped-prefill tile from route density on sm_89"),
The pages' prefill geometry (256 experts, top-6, hidden 7168, intermediate 2048) is checked
at full size in test_gpu_fullsize.py.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import moe as M
from tests.common import FP32_SUM_REL, Problem, record_measure

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ft():
    import block_quantized_moe_gb300 as ft
    ft.lib()
    return ft


def _grouped_case(ft, E, N, K, counts, seed):
    """Rows sorted by expert with the given per-expert counts; returns GPU inputs and oracle parts
    (the reference rows and each element's sum of |products|)."""
    R = int(sum(counts))
    offsets = np.zeros(E + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    x = synth.activations_bf16(max(R, 1), K, seed, DEV)[:R]
    w = torch.stack([synth.expert_weight_fp32(N, K, seed, e, "w", DEV) for e in range(E)])
    wq, ws, _ = ft.quantize_weights(w)
    aq, as_, _ = ft.quantize_act(x) if R else (torch.zeros(0, K, dtype=torch.uint8, device=DEV),
                                                torch.zeros(0, -(-K // 128), device=DEV), None)
    off_d = torch.from_numpy(offsets).to(DEV)
    ref = np.zeros((R, N))
    absum = np.zeros((R, N))  # sum of |products| of each output element
    if R:
        rq, rs = M.quantize_act_fp8_fast(x.float().cpu().numpy())
        adeq = M.dequant_act_fp8(rq, rs)
        for e in range(E):
            lo, hi = offsets[e], offsets[e + 1]
            if hi > lo:
                wd = M.dequant_weight_fp8(*M.quantize_weight_fp8_fast(w[e].cpu().numpy()))
                ref[lo:hi] = M.gemm_rows(adeq[lo:hi], wd)
                absum[lo:hi] = np.abs(adeq[lo:hi]) @ np.abs(wd).T
    return aq, as_, wq, ws, off_d, ref, absum


def _gemm_tol_ok(got, ref):
    # fp32 accumulation of fp8 products: far inside 1e-4 relative of the row's scale
    scale = np.max(np.abs(ref)) if ref.size else 0.0
    return np.abs(got - ref) <= 1e-4 * np.abs(ref) + 1e-5 * scale


@pytest.mark.parametrize("tok_tile", [16, 32, 64, 128])
def test_tc_gemm_small_ragged(ft, tok_tile):
    E, N, K = 5, 256, 384
    counts = [0, 1, 17, 40, 3]
    aq, as_, wq, ws, off, ref, absum = _grouped_case(ft, E, N, K, counts, seed=11)
    R = ref.shape[0]
    out = torch.full((R + 3, N), float("nan"), device=DEV)
    ft.ftmoe_grouped_gemm_gateup(ft.make_act(aq, as_), ft.grouped_routes(off), ft.make_bank(wq, ws), out,
                                 tok_tile=tok_tile, variant=2)
    flags = ft.ftmoe_read_error_flags()
    assert flags == 0
    got = out.cpu().numpy()
    assert np.all(_gemm_tol_ok(got[:R], ref))
    assert np.all(np.isnan(got[R:]))  # rows beyond the segments are not touched
    # the fp32 promotion's error against the bound the forward checks assume for a gate/up
    # element (FP32_SUM_REL of the sum of the magnitudes of its products, plus the final
    # rounding to fp32)
    err = np.abs(got[:R] - ref)
    assert np.all(err <= FP32_SUM_REL * absum + 2.0 ** -23 * np.abs(ref))
    nz = absum > 0
    record_measure(f"FP8 tcgen05 GEMM max |err| / sum|products| (token tile {tok_tile})",
                   float(np.max(err[nz] / absum[nz])), FP32_SUM_REL)


@pytest.mark.parametrize("N,K", [(200, 320), (384, 1040), (130, 2048)])
def test_tc_gemm_partial_tiles(ft, N, K):
    E = 3
    counts = [33, 0, 70]
    aq, as_, wq, ws, off, ref, absum = _grouped_case(ft, E, N, K, counts, seed=N + K)
    R = ref.shape[0]
    out = torch.full((R, N), float("nan"), device=DEV)
    ft.ftmoe_grouped_gemm_gateup(ft.make_act(aq, as_), ft.grouped_routes(off), ft.make_bank(wq, ws), out,
                                 tok_tile=32, variant=2)
    torch.cuda.synchronize()
    assert np.all(_gemm_tol_ok(out.cpu().numpy(), ref))


def test_tc_gemm_equals_streaming_kernel(ft):
    # the two GPU GEMMs (tensor-core and CUDA-core) agree with each other on the same inputs
    E, N, K = 8, 512, 1024
    counts = [5, 60, 0, 130, 1, 16, 33, 7]
    aq, as_, wq, ws, off, ref, absum = _grouped_case(ft, E, N, K, counts, seed=21)
    R = ref.shape[0]
    o_tc = torch.empty(R, N, device=DEV)
    o_st = torch.empty(R, N, device=DEV)
    act, rt, bank = ft.make_act(aq, as_), ft.grouped_routes(off), ft.make_bank(wq, ws)
    ft.ftmoe_grouped_gemm_gateup(act, rt, bank, o_tc, tok_tile=64, variant=2)
    ft.ftmoe_grouped_gemm_gateup(act, rt, bank, o_st, variant=1)
    torch.cuda.synchronize()
    a, b = o_tc.cpu().numpy(), o_st.cpu().numpy()
    assert np.all(_gemm_tol_ok(a, ref)) and np.all(_gemm_tol_ok(b, ref))
    assert np.all(np.abs(a - b) <= 2e-4 * np.abs(ref) + 2e-5 * np.max(np.abs(ref)))


def test_prefill_forward_medium(ft):
    T, H, I, E, k = 96, 1024, 512, 16, 6
    p = Problem(T, H, I, E, k, seed=0xF7E00004)
    ids = synth.routes(T, k, E, 3, active_per_token=[6, 5, 4, 6] * 24, device=DEV)
    w = torch.where(ids >= 0, p.w, torch.full_like(p.w, float("nan")))
    for path in (2, 3):
        for tok_tile in (0, 16, 128):
            out, _, _ = p.forward(path=path, tok_tile=tok_tile, ids=ids, weights=w)
            torch.cuda.synchronize()
            p.check(out, ids=ids, weights=w)
    # the route-slot streaming path gives the same answer within tolerance
    out_d, _, _ = p.forward(path=1, ids=ids, weights=w)
    torch.cuda.synchronize()
    p.check(out_d, ids=ids, weights=w)


def test_prefill_forward_all_inactive(ft):
    T, H, I, E, k = 16, 512, 256, 8, 4
    p = Problem(T, H, I, E, k, seed=0xF7E00004)
    ids = torch.full((T, k), -1, dtype=torch.int32, device=DEV)
    out, _, _ = p.forward(path=2, ids=ids, weights=torch.full_like(p.w, float("nan")))
    torch.cuda.synchronize()
    assert torch.all(out.view(torch.int16) == 0)

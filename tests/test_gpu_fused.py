"""Two weight blocks per tensor-core unit, CTA pairs, and SiLU-and-mul fused into the gate/up
GEMM.

The tcgen05 grouped GEMM can give each token tile two 128-row weight blocks (adjacent
blocks of one matrix, or gate block j with up block j), on one SM or on the two CTAs of a
cluster (one M = 256 MMA over both). Its per-K-block promotion is the same fp32 arithmetic
in the same order whichever blocks share a tile, so:
  - the GEMM with two blocks per unit, and with CTA pairs, equals the one-block GEMM bit for
    bit;
  - ftmoe_grouped_gemm_gateup_silu equals ftmoe_grouped_gemm_gateup followed by
    ftmoe_silu_mul bit for bit (codes and scales), and both match the oracle;
  - the forward with the fused gate/up (path 3) equals the forward with the separate
    SiLU-and-mul kernel (path 2) bit for bit, and matches the oracle.
Shapes span several token tiles per expert, experts with 0 and 1 rows, ragged segment
tails, one to three chunks of activation scales (K blocks 3, 9, 17) and every token tile.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import moe as M
from tests.common import Problem, assert_within_tolerance

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ft():
    import block_quantized_moe_gb300 as ft
    ft.lib()
    return ft


def _rows_case(ft, E, N, K, counts, seed):
    R = int(sum(counts))
    offsets = np.zeros(E + 1, np.int32)
    offsets[1:] = np.cumsum(counts)
    x = synth.activations_bf16(R, K, seed, DEV)
    w = torch.stack([synth.expert_weight_fp32(N, K, seed, e, "w", DEV) for e in range(E)])
    wq, ws, _ = ft.quantize_weights(w)
    aq, as_, _ = ft.quantize_act(x)
    return x, w, aq, as_, wq, ws, offsets


@pytest.mark.parametrize("tok_tile", [16, 32, 64, 128])
@pytest.mark.parametrize("K", [384, 1152, 2176])
def test_pair_units_equal_single_units(ft, tok_tile, K):
    E, N = 5, 512
    counts = [0, 1, 17, 140, 3]
    x, w, aq, as_, wq, ws, offsets = _rows_case(ft, E, N, K, counts, seed=K + tok_tile)
    R = int(offsets[-1])
    off = torch.from_numpy(offsets).to(DEV)  # kept alive: the routes struct holds its raw pointer
    act, rt, bank = ft.make_act(aq, as_), ft.grouped_routes(off), ft.make_bank(wq, ws)
    o1 = torch.full((R + 2, N), float("nan"), device=DEV)
    o2 = torch.full((R + 2, N), float("nan"), device=DEV)
    ft.ftmoe_grouped_gemm_down(act, rt, bank, o1, tok_tile=tok_tile, variant=2, wblocks=1)
    ft.ftmoe_grouped_gemm_down(act, rt, bank, o2, tok_tile=tok_tile, variant=2, wblocks=2)
    torch.cuda.synchronize()
    assert ft.ftmoe_read_error_flags() == 0
    assert torch.equal(o1[:R].view(torch.int32), o2[:R].view(torch.int32))
    assert torch.all(torch.isnan(o2[R:]))  # rows past the segments are not touched
    # and the oracle: dequantized fp64 GEMM per expert
    rq, rs = M.quantize_act_fp8_fast(x.float().cpu().numpy())
    adeq = M.dequant_act_fp8(rq, rs)
    got = o2[:R].cpu().numpy()
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            wd = M.dequant_weight_fp8(*M.quantize_weight_fp8_fast(w[e].cpu().numpy()))
            ref = M.gemm_rows(adeq[lo:hi], wd)
            scale = np.max(np.abs(ref))
            assert np.all(np.abs(got[lo:hi] - ref) <= 1e-4 * np.abs(ref) + 1e-5 * scale)


@pytest.mark.parametrize("tok_tile", [64, 128])
@pytest.mark.parametrize("K", [384, 1152, 2176])
@pytest.mark.parametrize("E", [5, 48])
def test_cta_pair_units_equal_single_units(ft, tok_tile, K, E):
    # CTA pairs (clusters of two, M = 256): few units (most pairs idle) and more units than
    # pairs (each pair runs several), experts with 0 and 1 rows, ragged tails, one to three
    # chunks of activation scales
    N = 512
    if E == 5:
        counts = [0, 1, 17, 140, 3]
    else:
        rng = np.random.default_rng(K + tok_tile)
        counts = [int(c) for c in rng.integers(0, 300, E)]
        counts[3] = 0
        counts[7] = 1
    x, w, aq, as_, wq, ws, offsets = _rows_case(ft, E, N, K, counts, seed=K + tok_tile + E)
    R = int(offsets[-1])
    off = torch.from_numpy(offsets).to(DEV)  # kept alive: the routes struct holds its raw pointer
    act, rt, bank = ft.make_act(aq, as_), ft.grouped_routes(off), ft.make_bank(wq, ws)
    o1 = torch.full((R + 2, N), float("nan"), device=DEV)
    o2 = torch.full((R + 2, N), float("nan"), device=DEV)
    ft.ftmoe_grouped_gemm_down(act, rt, bank, o1, tok_tile=tok_tile, variant=2, wblocks=1, ctas=1)
    ft.ftmoe_grouped_gemm_down(act, rt, bank, o2, tok_tile=tok_tile, variant=2, ctas=2)
    torch.cuda.synchronize()
    assert ft.ftmoe_read_error_flags() == 0
    assert torch.equal(o1[:R].view(torch.int32), o2[:R].view(torch.int32))
    assert torch.all(torch.isnan(o2[R:]))  # rows past the segments are not touched
    rq, rs = M.quantize_act_fp8_fast(x.float().cpu().numpy())
    adeq = M.dequant_act_fp8(rq, rs)
    got = o2[:R].cpu().numpy()
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            wd = M.dequant_weight_fp8(*M.quantize_weight_fp8_fast(w[e].cpu().numpy()))
            ref = M.gemm_rows(adeq[lo:hi], wd)
            scale = np.max(np.abs(ref))
            assert np.all(np.abs(got[lo:hi] - ref) <= 1e-4 * np.abs(ref) + 1e-5 * scale)


def test_cta_pair_refused_where_it_does_not_apply(ft):
    # token tiles 16 and 32, and matrices that are not whole 256-row block pairs, are
    # unsupported for CTA pairs (the tensor-core variant is forced, so nothing falls back)
    E, N, K = 2, 384, 256
    counts = [20, 5]
    x, w, aq, as_, wq, ws, offsets = _rows_case(ft, E, N, K, counts, seed=3)
    off = torch.from_numpy(offsets).to(DEV)
    act, rt, bank = ft.make_act(aq, as_), ft.grouped_routes(off), ft.make_bank(wq, ws)
    o = torch.empty(25, N, device=DEV)
    for tile in (16, 32, 128):  # N = 384: three blocks, no whole pairs
        with pytest.raises(ft.FtmoeError) as ei:
            ft.ftmoe_grouped_gemm_down(act, rt, bank, o, tok_tile=tile, variant=2, ctas=2)
        assert ei.value.status == ft.FTMOE_UNSUPPORTED


@pytest.mark.parametrize("tok_tile", [16, 32, 64, 128])
@pytest.mark.parametrize("I,K", [(384, 384), (256, 1152), (128, 2176)])
def test_gateup_silu_equals_gateup_then_silu(ft, tok_tile, I, K):
    E = 4
    counts = [9, 0, 130, 1]
    x, w, aq, as_, wq, ws, offsets = _rows_case(ft, E, 2 * I, K, counts, seed=I + K + tok_tile)
    R = int(offsets[-1])
    off = torch.from_numpy(offsets).to(DEV)
    act, rt, bank = ft.make_act(aq, as_), ft.grouped_routes(off), ft.make_bank(wq, ws)
    # separate: fp32 gate/up rows, then SiLU-and-mul with FP8 re-quantization
    gu = torch.empty(R, 2 * I, device=DEV)
    ft.ftmoe_grouped_gemm_gateup(act, rt, bank, gu, tok_tile=tok_tile, variant=2, wblocks=1)
    q1 = torch.empty(R, I, dtype=torch.uint8, device=DEV)
    s1 = torch.empty(R, I // 128, device=DEV)
    ft.ftmoe_silu_mul(gu, q1, s1)
    # fused, into buffers with two poisoned rows past the segments
    q2 = torch.full((R + 2, I), 0xFF, dtype=torch.uint8, device=DEV)
    s2 = torch.full((R + 2, I // 128), float("nan"), device=DEV)
    ft.ftmoe_grouped_gemm_gateup_silu(act, rt, bank, q2, s2, tok_tile=tok_tile)
    torch.cuda.synchronize()
    assert ft.ftmoe_read_error_flags() == 0
    assert torch.equal(q1, q2[:R])
    assert torch.equal(s1.view(torch.int32), s2[:R].view(torch.int32))
    assert torch.all(q2[R:] == 0xFF) and torch.all(torch.isnan(s2[R:]))
    # oracle: a = silu(g) * u from the exact gate/up values; compare dequantized activations
    # (a code may sit next to the oracle's where the value is on a rounding midpoint, so
    # compare values within one code step of the group scale)
    rq, rs = M.quantize_act_fp8_fast(x.float().cpu().numpy())
    adeq = M.dequant_act_fp8(rq, rs)
    got = M.dequant_act_fp8(q2[:R].cpu().numpy(), s2[:R].cpu().numpy())
    for e in range(E):
        lo, hi = offsets[e], offsets[e + 1]
        if hi > lo:
            wd = M.dequant_weight_fp8(*M.quantize_weight_fp8_fast(w[e].cpu().numpy()))
            g = M.gemm_rows(adeq[lo:hi], wd)
            a = g[:, :I] / (1.0 + np.exp(-g[:, :I])) * g[:, I:]
            sc = np.repeat(s2[lo:hi].cpu().numpy().astype(np.float64), 128, axis=1)
            # E4M3 spacing is at most 2**-3 of the value (32 of 448 at the top): half a step
            # plus one step for a midpoint decision
            assert np.all(np.abs(got[lo:hi] - a) <= 0.1875 * np.abs(a) + 2.0 ** -9 * sc + 1e-6)


def test_gateup_silu_rejects_what_it_cannot_pair(ft):
    E, I, K = 2, 192, 256  # 2I = 384 is not a whole number of 256-row pairs
    x, w, aq, as_, wq, ws, offsets = _rows_case(ft, E, 2 * I, K, [3, 4], seed=5)
    R = int(offsets[-1])
    q = torch.empty(R, I, dtype=torch.uint8, device=DEV)
    s = torch.empty(R, 2, device=DEV)
    off = torch.from_numpy(offsets).to(DEV)
    with pytest.raises(ft.FtmoeError):
        ft.ftmoe_grouped_gemm_gateup_silu(ft.make_act(aq, as_), ft.grouped_routes(off), ft.make_bank(wq, ws), q, s)


@pytest.mark.parametrize("T,H,I,E,k,active", [(8, 4096, 1024, 64, 8, 8), (8, 4096, 1024, 64, 8, 2),
                                               (96, 1024, 512, 16, 6, 6), (1, 2048, 768, 8, 8, 2)])
def test_fused_forward_equals_separate_forward(ft, T, H, I, E, k, active):
    p = Problem(T, H, I, E, k, seed=0xF7E00005, active=active)
    out2, _, _ = p.forward(path=2)
    out3, ws3, shape3 = p.forward(path=3)
    torch.cuda.synchronize()
    assert ft.ftmoe_forward_workspace_layout(shape3)["gateup_bytes"] == 0
    assert torch.equal(out2.view(torch.int16), out3.view(torch.int16))
    p.check(out3)


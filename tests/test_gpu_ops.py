"""GPU parity of the single ops against the oracle, through the C ABI.

Bit-exact: quantized codes and scales (compared as integer views), segment outputs,
gathered rows and scales (raw bytes, as the SGLang gather page's tests compare them).
Floating-point outputs: the stated tolerance, or tighter where the arithmetic allows.
"""
import numpy as np
import pytest
import torch

import synth
from oracle import formats as F
from oracle import moe as M

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ft():
    import block_quantized_moe_gb300 as ft
    ft.lib()
    return ft


def _bits(t):
    return t.cpu().numpy().view(np.uint32) if t.dtype == torch.float32 else t.cpu().numpy()


# -- quantization ------------------------------------------------------------------

@pytest.mark.parametrize("rows,k,ld_pad", [(1, 2048, 0), (8, 4096, 0), (37, 896, 0), (5, 200, 8),
                                           (3, 7168, 0), (64, 130, 2), (0, 256, 0), (3, 384, 0), (7, 1000, 0)])
def test_quantize_act_fp8_bitexact(ft, rows, k, ld_pad):
    xf = synth.activations_bf16(rows, k + ld_pad, 1000 + k, DEV)
    if rows:
        xf[0, :min(k, 128)] = 0  # an all-zero group
    x = xf[:, :k]
    ng = -(-k // 128)
    q = torch.full((rows, k), 0xAA, dtype=torch.uint8, device=DEV)
    s = torch.full((rows, ng), float("nan"), dtype=torch.float32, device=DEV)
    ft.ftmoe_quantize_act(x, q, s)
    torch.cuda.synchronize()
    rq, rs = M.quantize_act_fp8_fast(x.float().cpu().numpy())
    assert np.array_equal(q.cpu().numpy(), rq)
    assert np.array_equal(_bits(s), rs.view(np.uint32))


def test_quantize_act_fp8_many_binades_bitexact(ft):
    # 3.7 M elements whose magnitudes span 2^-30 .. 2^30 within a group, so that the quotients
    # x / s cover every binade the e4m3 codes use and many far below: the kernels' division by
    # the group scale must round exactly as IEEE division (the oracle's float32 x / s)
    g = torch.Generator().manual_seed(0xD1)
    rows, k = 512, 7168
    mant = torch.rand(rows, k, generator=g) + 1.0
    expo = torch.randint(-30, 31, (rows, k), generator=g).float()
    sign = torch.where(torch.rand(rows, k, generator=g) < 0.5, -1.0, 1.0)
    x = (sign * mant * torch.pow(2.0, expo)).to(torch.bfloat16).to(DEV)
    q = torch.empty(rows, k, dtype=torch.uint8, device=DEV)
    s = torch.empty(rows, k // 128, dtype=torch.float32, device=DEV)
    ft.ftmoe_quantize_act(x, q, s)
    torch.cuda.synchronize()
    rq, rs = M.quantize_act_fp8_fast(x.float().cpu().numpy())
    assert np.array_equal(_bits(s), rs.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), rq)


def test_quantizer_division_equals_ieee_division(ft):
    # the quantizers divide by the group scale through one reciprocal per group and a
    # Markstein correction; on the device, against __fdiv_rn: every divisor mantissa at three
    # exponents x 4098 dividends, and 1024 divisors x every dividend mantissa
    counts = torch.zeros(2, dtype=torch.int64, device=DEV)
    ft.ftmoe_selftest_shared_division(counts)
    torch.cuda.synchronize()
    checked, differ = counts.tolist()
    assert checked == (1 << 23) * (3 * 4098 + 1024)
    assert differ == 0


def test_quantize_act_fp8_special_values(ft):
    x = torch.zeros(2, 256, dtype=torch.float32)
    x[0, 0], x[0, 1], x[0, 2], x[0, 3] = 448.0, -1e-6, -0.0, 1e-30
    x[1, 128] = -3.0
    x[1, 200] = 2.0 ** -20
    xb = x.to(torch.bfloat16).to(DEV)
    q, s, _ = ft.quantize_act(xb)
    rq, rs = M.quantize_act_fp8(xb.float().cpu().numpy())
    assert np.array_equal(q.cpu().numpy(), rq) and np.array_equal(_bits(s), rs.view(np.uint32))


@pytest.mark.parametrize("E,n,k", [(3, 300, 260), (2, 1536, 2048), (1, 128, 128)])
def test_quantize_weights_fp8_bitexact(ft, E, n, k):
    w = torch.stack([synth.expert_weight_fp32(n, k, 77, e, "wq", DEV) for e in range(E)])
    w[0, :128, :128] = 0
    q, s, _ = ft.quantize_weights(w)
    torch.cuda.synchronize()
    for e in range(E):
        rq, rs = M.quantize_weight_fp8(w[e].cpu().numpy())
        assert np.array_equal(q[e].cpu().numpy(), rq)
        assert np.array_equal(_bits(s[e]), rs.view(np.uint32))


# -- segmenter -----------------------------------------------------------------------

@pytest.mark.parametrize("T,k,E,inactive", [(1, 8, 8, 6), (8, 8, 64, 4), (256, 6, 256, 0),
                                            (4096, 6, 256, 0), (33, 4, 5, 1), (16, 8, 64, 8),
                                            (1000, 7, 9, 2), (8192, 8, 12, 0)])
def test_segment_bitexact(ft, T, k, E, inactive):
    if T * k > 2048:
        ids = synth.routes_fast(T, k, E, 5 + T, DEV)
    else:
        ids = synth.routes(T, k, E, 5 + T, active_per_token=k - inactive, device=DEV)
    counts = torch.full((E,), -7, dtype=torch.int32, device=DEV)
    offsets = torch.full((E + 1,), -7, dtype=torch.int32, device=DEV)
    d2s = torch.full((T * k,), -7, dtype=torch.int32, device=DEV)
    r2d = torch.full((T * k,), -7, dtype=torch.int32, device=DEV)
    ft.ftmoe_segment_routes(ids, E, counts, offsets, d2s, r2d)
    torch.cuda.synchronize()
    ref = M.segment_routes(ids.cpu().numpy(), E)
    n_act = int(ref["offsets"][-1])
    assert np.array_equal(counts.cpu().numpy(), ref["counts"])
    assert np.array_equal(offsets.cpu().numpy(), ref["offsets"])
    assert np.array_equal(d2s.cpu().numpy()[:n_act], ref["dst2src"])
    assert np.array_equal(r2d.cpu().numpy(), ref["route2dst"])


# -- gather (the SGLang page's workload: random FP8 bytes, U(1e-3,1) scales, randint maps)

@pytest.mark.parametrize("k", [2048, 7168, 896])
@pytest.mark.parametrize("tokens", [1, 8, 64, 1024])
def test_gather_bitexact(ft, k, tokens):
    seed = k * 7 + tokens
    src = synth.random_bytes(tokens, k, seed, device=DEV)
    sc = synth.uniform_f32(tokens, -(-k // 128), 1e-3, 1.0, seed, device=DEV)
    m = synth.randint_map(8 * tokens, tokens, seed, device=DEV)
    dst = torch.full((8 * tokens, k), 0x5A, dtype=torch.uint8, device=DEV)
    dsc = torch.full((8 * tokens, -(-k // 128)), float("nan"), dtype=torch.float32, device=DEV)
    ft.ftmoe_gather_rows_scales(src, sc, m, dst, dsc)
    torch.cuda.synchronize()
    rd, rs = M.gather_rows_scales(src.cpu().numpy(), sc.cpu().numpy().view(np.uint32), m.cpu().numpy())
    assert np.array_equal(dst.cpu().numpy(), rd)
    assert np.array_equal(_bits(dsc), rs)


def test_gather_zero_rows_and_device_count(ft):
    src = synth.random_bytes(4, 896, 3, device=DEV)
    sc = synth.uniform_f32(4, 7, 1e-3, 1.0, 3, device=DEV)
    m = torch.tensor([3, 3, 0, 1, 2, 2], dtype=torch.int32, device=DEV)
    dst = torch.zeros(6, 896, dtype=torch.uint8, device=DEV)
    dsc = torch.zeros(6, 7, dtype=torch.float32, device=DEV)
    ft.ftmoe_gather_rows_scales(src, sc, m[:0], dst[:0], dsc[:0])  # zero rows: no launch
    cnt = torch.tensor([4], dtype=torch.int32, device=DEV)
    ft.ftmoe_gather_rows_scales(src, sc, m, dst, dsc, n_dst_dev=cnt)
    torch.cuda.synchronize()
    rd, rs = M.gather_rows_scales(src.cpu().numpy(), sc.cpu().numpy().view(np.uint32), m.cpu().numpy())
    assert np.array_equal(dst.cpu().numpy()[:4], rd[:4]) and np.all(dst.cpu().numpy()[4:] == 0)
    assert np.array_equal(_bits(dsc)[:4], rs[:4])
    # identity map is a no-op copy
    ident = torch.arange(4, dtype=torch.int32, device=DEV)
    d2 = torch.zeros_like(src)
    s2 = torch.zeros_like(sc)
    ft.ftmoe_gather_rows_scales(src, sc, ident, d2, s2)
    torch.cuda.synchronize()
    assert torch.equal(d2, src) and torch.equal(s2.view(torch.int32), sc.view(torch.int32))


def test_gather_out_of_range_map_is_skipped_and_flagged(ft):
    ft.ftmoe_read_error_flags()
    src = synth.random_bytes(4, 256, 4, device=DEV)
    sc = synth.uniform_f32(4, 2, 1e-3, 1.0, 4, device=DEV)
    m = torch.tensor([1, 9, 2], dtype=torch.int32, device=DEV)
    dst = torch.zeros(3, 256, dtype=torch.uint8, device=DEV)
    dsc = torch.zeros(3, 2, dtype=torch.float32, device=DEV)
    ft.ftmoe_gather_rows_scales(src, sc, m, dst, dsc)
    flags = ft.ftmoe_read_error_flags()
    assert flags & ft.ERR_MAP_RANGE
    assert torch.equal(dst[0], src[1]) and torch.equal(dst[2], src[2]) and torch.all(dst[1] == 0)


# -- SiLU-and-mul ----------------------------------------------------------------------

def _e4m3_step(mag):
    e = np.floor(np.log2(np.maximum(mag, 2.0 ** -6)))
    return 2.0 ** (e - 3)


@pytest.mark.parametrize("rows,inter", [(64, 1024), (7, 200), (8, 768), (5, 132), (3, 384)])
def test_silu_mul_fp8(ft, rows, inter):
    g = torch.randn(rows, 2 * inter, generator=torch.Generator().manual_seed(rows + inter)) * 3
    g[0] = 0  # an inactive route's zero row
    gu = g.to(DEV)
    ng = -(-inter // 128)
    q = torch.full((rows, inter), 0xFF, dtype=torch.uint8, device=DEV)
    s = torch.full((rows, ng), float("nan"), dtype=torch.float32, device=DEV)
    ft.ftmoe_silu_mul(gu, q, s)
    torch.cuda.synchronize()
    a = M.silu_mul(g.numpy().astype(np.float64))
    a32 = a.astype(np.float32)
    rq, rs = M.quantize_act_fp8(a32)
    qg, sg = q.cpu().numpy(), s.cpu().numpy()
    assert np.all(qg[0] == 0) and np.all(sg[0] == 0)
    # the kernel's fp32 silu may differ from the fp64 one in the last bits: scales agree to a
    # few ulp, and every code is the nearest E4M3 value of a/s up to that difference
    assert np.allclose(sg, rs, rtol=4 * 2.0 ** -23, atol=0)
    srep = np.repeat(sg.astype(np.float64), 128, axis=1)[:, :inter]
    with np.errstate(invalid="ignore", divide="ignore"):
        v = np.where(srep > 0, a / srep, 0.0)
    err = np.abs(F.decode_e4m3(qg) - v)
    assert np.all(err <= _e4m3_step(np.abs(v)) / 2 + 1e-5 * np.abs(v) + 1e-30)
    assert np.mean(qg == rq) > 0.999


# -- combine ----------------------------------------------------------------------------

def test_combine(ft):
    T, k, H = 16, 8, 4096
    ids = synth.routes(T, k, 64, 9, active_per_token=[8, 4, 2, 0] * 4, device=DEV)
    w = synth.routing_weights(T, k, 9, DEV)
    w[ids < 0] = float("nan")  # never read
    y = torch.randn(T * k, H, device=DEV)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    ft.ftmoe_combine(y, ids, w, out)
    torch.cuda.synchronize()
    ids_n = ids.cpu().numpy()
    ref = M.combine(y.cpu().numpy(), np.arange(T * k), ids_n, w.cpu().numpy())
    got = out.float().cpu().numpy()
    assert not np.any(np.isnan(got))
    assert np.all(got[3::4] == 0)  # tokens with no active slot
    # fp32 accumulation then one bf16 rounding: within one bf16 ulp of the fp64 sum
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-6)


@pytest.mark.parametrize("H,ld_pad", [(4096, 0), (1000, 0), (1002, 0), (520, 3)])
@pytest.mark.parametrize("k", [6, 8, 13])
def test_combine_ragged_hidden_and_slot_counts(ft, H, ld_pad, k):
    # hidden not a multiple of 8 (or of 4), padded row strides, slot counts below, at and past
    # one batch of loads; route-major y, and y rows reached through route2dst
    T = 10
    ids = synth.routes(T, k, 32, 11 + k, active_per_token=[k, 3, 0, 1, k - 1] * 2, device=DEV)
    w = synth.routing_weights(T, k, 11 + k, DEV)
    w[ids < 0] = float("nan")  # never read
    y = torch.randn(T * k, H + ld_pad, device=DEV)
    perm = torch.randperm(T * k, generator=torch.Generator().manual_seed(k)).to(torch.int32).to(DEV)
    y_perm = torch.empty_like(y)
    y_perm[perm.long()] = y
    out = torch.zeros(T, H + ld_pad, dtype=torch.bfloat16, device=DEV)
    out2 = torch.zeros(T, H + ld_pad, dtype=torch.bfloat16, device=DEV)
    ft.ftmoe_combine(y[:, :H], ids, w, out[:, :H])
    ft.ftmoe_combine(y_perm[:, :H], ids, w, out2[:, :H], route2dst=perm)
    torch.cuda.synchronize()
    ref = M.combine(y[:, :H].cpu().numpy(), np.arange(T * k), ids.cpu().numpy(), w.cpu().numpy())
    got = out[:, :H].float().cpu().numpy()
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -8 + 1e-6)
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))  # the padding stays zero too
    assert torch.all(out[:, H:] == 0)


def test_combine_single_route_weight_one_is_the_row(ft):
    T, k, H = 3, 4, 520
    ids = torch.full((T, k), -1, dtype=torch.int32, device=DEV)
    ids[:, 2] = 5
    w = torch.full((T, k), float("nan"), device=DEV)
    w[:, 2] = 1.0
    y = torch.randn(T * k, H, device=DEV)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    ft.ftmoe_combine(y, ids, w, out)
    torch.cuda.synchronize()
    rows = y.view(T, k, H)[:, 2].cpu().numpy()
    assert np.array_equal(out.float().cpu().numpy(), F.round_to_bf16(rows.astype(np.float64)))


# -- the streaming GEMM on its own ------------------------------------------------------

def test_gemm_rejects_unaligned_k(ft):
    # the GEMM kernels read K-contiguous rows through TMA: K must be a multiple of 16
    x = synth.activations_bf16(2, 520, 1, DEV)
    xq, xs, _ = ft.quantize_act(x)
    w = torch.zeros(2, 64, 520, device=DEV)
    wq, wsc, _ = ft.quantize_weights(w)
    ids = torch.zeros(2, 1, dtype=torch.int32, device=DEV)
    out = torch.empty(2, 64, device=DEV)
    with pytest.raises(ft.FtmoeError) as ei:
        ft.ftmoe_grouped_gemm_gateup(ft.make_act(xq, xs), ft.slot_routes(ids), ft.make_bank(wq, wsc), out)
    assert ei.value.status == ft.FTMOE_UNSUPPORTED


@pytest.mark.parametrize("T,H,N,E,k,active", [(1, 2048, 1536, 8, 8, 2), (8, 4096, 2048, 64, 8, 4),
                                              (3, 384, 300, 4, 2, 1), (8, 528, 256, 6, 4, 4),
                                              (8, 1024, 4096, 3, 3, 3)])
def test_stream_gemm_slots_vs_oracle(ft, T, H, N, E, k, active):
    seed = H + N + T
    x = synth.activations_bf16(T, H, seed, DEV)
    ids = synth.routes(T, k, E, seed, active_per_token=active, device=DEV)
    w = torch.stack([synth.expert_weight_fp32(N, H, seed, e, "g", DEV) for e in range(E)])
    wq, wsc, _ = ft.quantize_weights(w)
    xq, xs, _ = ft.quantize_act(x)
    out = torch.full((T * k, N), float("nan"), device=DEV)
    ft.ftmoe_grouped_gemm_gateup(ft.make_act(xq, xs), ft.slot_routes(ids), ft.make_bank(wq, wsc), out)
    torch.cuda.synchronize()
    rq, rs = M.quantize_act_fp8_fast(x.float().cpu().numpy())
    xdeq = M.dequant_act_fp8(rq, rs)
    got = out.cpu().numpy()
    ids_n = ids.cpu().numpy().reshape(-1)
    for r in range(T * k):
        e = ids_n[r]
        if e < 0:
            assert np.all(got[r] == 0) and not np.any(np.signbit(got[r]))
            continue
        wd = M.dequant_weight_fp8(*M.quantize_weight_fp8_fast(w[e].cpu().numpy()))
        ref = wd @ xdeq[r // k]
        # fp32 accumulation of K products: well inside 1e-4 relative of the row scale
        assert np.all(np.abs(got[r] - ref) <= 1e-4 * np.abs(ref) + 1e-5 * np.max(np.abs(ref)))

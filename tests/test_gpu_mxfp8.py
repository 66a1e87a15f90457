"""GPU parity of the MXFP8 variant against the oracle, through the C ABI.

Bit-exact: the MXFP8 quantizers (e4m3 codes and E8M0 scale bytes per 32 elements) of fp32
weights and bf16 activations, and the gather of bf16 rows with quantization of the gathered
rows (the mxfp8 branch of the SGLang gather page). The SiLU-and-mul re-quantization: scale
bytes and codes of the fp32 product, up to one step where the fp32 input sits on a rounding
boundary. The grouped GEMM on the block-scaled tensor-core MMA (kind::mxf8f6f4): the fp64
product of the dequantized operands within an fp32-accumulation bound that grows with K (one
fp32 ulp of the running sum per 32-element MMA step), for every token tile, with ragged
experts, an empty expert and K of one to fourteen 512-element scale chunks. The
forward: the stated output tolerance plus the allowance for re-quantization decisions on a
rounding boundary.
"""
import numpy as np
import pytest
import torch

import synth
from common import Problem, mxfp8_sum_rel, record_measure
from oracle import formats as F
from oracle import moe as M

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ft():
    import block_quantized_moe_gb300 as ft
    ft.lib()
    return ft


# -- quantizers ------------------------------------------------------------------------

@pytest.mark.parametrize("E,n,k", [(3, 256, 512), (2, 130, 96), (1, 512, 7168)])
def test_quantize_weights_mxfp8_bitexact(ft, E, n, k):
    w = torch.stack([synth.expert_weight_fp32(n, k, 91, e, "mx-w", DEV) for e in range(E)])
    w[0, :3, :32] = 0                                 # all-zero blocks
    w[-1, 1, 32:64] *= 2.0 ** -130                    # a block whose amax is subnormal
    w[-1, 2, :] *= 2.0 ** 60                          # large magnitudes
    w[0, 5, 7] = 448.0 * 2.0 ** -3                    # an exact top-of-range value
    q = torch.full((E, n, k), 0xAA, dtype=torch.uint8, device=DEV)
    s = torch.full((E, n, k // 32), 0xAA, dtype=torch.uint8, device=DEV)
    ft.ftmoe_quantize_weights(w, q, s, None, fmt=ft.FMT_MXFP8)
    torch.cuda.synchronize()
    wn = w.cpu().numpy()
    for e in range(E):
        rq, rs = M.quantize_mxfp8(wn[e])
        assert np.array_equal(s[e].cpu().numpy(), rs), e
        assert np.array_equal(q[e].cpu().numpy(), rq), e


@pytest.mark.parametrize("rows,k,ld", [(1, 256, 256), (37, 512, 520), (8, 7168, 7168), (3, 32, 40), (64, 2048, 2048)])
def test_quantize_act_mxfp8_bitexact(ft, rows, k, ld):
    big = synth.activations_bf16(rows, ld, 3000 + k + rows, DEV)
    big[0, :32] = 0
    big[-1, 32:64] *= 1e-30
    x = big[:, :k]
    q = torch.full((rows, k), 0xAA, dtype=torch.uint8, device=DEV)
    s = torch.full((rows, k // 32), 0xAA, dtype=torch.uint8, device=DEV)
    ft.ftmoe_quantize_act(x, q, s, None, fmt=ft.FMT_MXFP8)
    torch.cuda.synchronize()
    rq, rs = M.quantize_mxfp8(x.float().cpu().numpy())
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


@pytest.mark.parametrize("n_src,k,n_dst", [(1, 7168, 8), (64, 2048, 512), (1024, 7168, 8192), (5, 96, 0), (9, 896, 40)])
def test_gather_quantize_mxfp8_bitexact(ft, n_src, k, n_dst):
    x = synth.activations_bf16(n_src, k, 4000 + n_src, DEV)
    dmap = synth.randint_map(n_dst, n_src, 4000 + k, "mx-map", DEV)
    q = torch.full((max(n_dst, 1), k), 0xAA, dtype=torch.uint8, device=DEV)
    s = torch.full((max(n_dst, 1), k // 32), 0xAA, dtype=torch.uint8, device=DEV)
    ft.ftmoe_gather_quantize_act(x, dmap, q, s, n_dst=n_dst)
    torch.cuda.synchronize()
    assert ft.ftmoe_read_error_flags() == 0
    if n_dst == 0:
        assert bool((q == 0xAA).all())  # nothing launched
        return
    rq, rs = M.quantize_mxfp8(x.float().cpu().numpy())
    m = dmap.cpu().numpy()
    assert np.array_equal(q.cpu().numpy(), rq[m])
    assert np.array_equal(s.cpu().numpy(), rs[m])


def test_gather_quantize_mxfp8_device_count_and_bad_entries(ft):
    n_src, k = 6, 512
    x = synth.activations_bf16(n_src, k, 77, DEV)
    dmap = torch.tensor([5, 0, 9, 2, -1, 3, 1, 1], dtype=torch.int32, device=DEV)
    q = torch.full((8, k), 0xAA, dtype=torch.uint8, device=DEV)
    s = torch.full((8, k // 32), 0xAA, dtype=torch.uint8, device=DEV)
    n_dev = torch.tensor([6], dtype=torch.int32, device=DEV)  # rows 6 and 7 are not written
    ft.ftmoe_read_error_flags()
    ft.ftmoe_gather_quantize_act(x, dmap, q, s, n_dst_dev=n_dev)
    torch.cuda.synchronize()
    assert ft.ftmoe_read_error_flags() & ft.ERR_MAP_RANGE
    rq, rs = M.quantize_mxfp8(x.float().cpu().numpy())
    qh, sh = q.cpu().numpy(), s.cpu().numpy()
    for d, src in enumerate(dmap.cpu().tolist()):
        if d >= 6 or not 0 <= src < n_src:
            assert np.all(qh[d] == 0xAA) and np.all(sh[d] == 0xAA), d
        else:
            assert np.array_equal(qh[d], rq[src]) and np.array_equal(sh[d], rs[src]), d


# -- SiLU-and-mul ----------------------------------------------------------------------

@pytest.mark.parametrize("rows,inter,valid", [(9, 256, 9), (40, 2048, 33)])
def test_silu_mul_mxfp8(ft, rows, inter, valid):
    gu_h = torch.randn(rows, 2 * inter, generator=torch.Generator().manual_seed(rows * 5 + inter)) * 3
    gu_h[1] = 0
    gu = gu_h.to(DEV)
    q = torch.full((rows, inter), 0xAA, dtype=torch.uint8, device=DEV)
    s = torch.full((rows, inter // 32), 0xAA, dtype=torch.uint8, device=DEV)
    rows_dev = torch.tensor([valid], dtype=torch.int32, device=DEV)
    ft.ftmoe_silu_mul(gu, q, s, None, fmt=ft.FMT_MXFP8, rows_dev=rows_dev)
    torch.cuda.synchronize()
    a = M.silu_mul(gu_h[:valid].numpy().astype(np.float64))
    rq, rs = M.quantize_mxfp8(a.astype(np.float32))
    qg, sg = q.cpu().numpy()[:valid], s.cpu().numpy()[:valid]
    assert np.all(q.cpu().numpy()[valid:] == 0xAA) and np.all(s.cpu().numpy()[valid:] == 0xAA)
    assert np.all(qg[1] == 0) and np.all(sg[1] == 0)
    # scale bytes: floor(log2) of the fp32 block maximum, one binade off at most where that
    # maximum sits within the kernel's fp32 error of a power of two
    assert np.all(np.abs(sg.astype(np.int32) - rs.astype(np.int32)) <= 1)
    assert np.mean(sg == rs) > 0.999
    # codes: under the kernel's own scale, the nearest e4m3 value of a / 2^shared, up to one
    # step where the exact value sits within fp32 error of a midpoint
    X = np.repeat(np.exp2(sg.astype(np.float64) - 127), 32, axis=1)
    v = a / X
    got = F.decode_e4m3(qg)
    ref = F.decode_e4m3(F.encode_e4m3(v))
    pos = F.E4M3_VALUES[:0x7F]
    idx = np.clip(np.searchsorted(pos, np.abs(v)), 1, len(pos) - 1)
    step = pos[idx] - pos[idx - 1]
    assert np.all(np.abs(got - ref) <= step * 1.0001)
    same = sg == rs
    assert np.mean((qg == rq)[np.repeat(same, 32, axis=1)]) > 0.999


# -- grouped GEMM ----------------------------------------------------------------------

def _random_mx(rows, k, seed, tag):
    """Random e4m3 codes (finite: NaN patterns remapped) and E8M0 scale bytes around 2^0."""
    codes = synth.random_bytes(rows, k, seed, tag + "-q")
    codes[(codes & 0x7F) == 0x7F] ^= 0x01
    sb = synth.random_bytes(rows, k // 32, seed, tag + "-s") % 16 + 119
    return codes, sb


@pytest.mark.parametrize("tile", [16, 32, 64, 128])
@pytest.mark.parametrize("k", [512, 1536, 4096, 7168])
def test_grouped_gemm_mxfp8_vs_oracle(ft, tile, k):
    E, n = 5, 320
    counts = [0, 1, 17, 40, 130]
    R = sum(counts)
    offsets = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32, device=DEV)
    aq, asf = _random_mx(R + 3, k, 21 + k, "act")
    wq, wsf = _random_mx(E * n, k, 22 + k, "w")
    out = torch.full((R + 3, n), float("nan"), device=DEV)
    a_q, a_sf = aq.to(DEV), asf.to(DEV)
    w_q, w_sf = wq.reshape(E, n, k).to(DEV), wsf.reshape(E, n, k // 32).to(DEV)
    act = ft.make_act(a_q, a_sf, fmt=ft.FMT_MXFP8)
    bank = ft.make_bank(w_q, w_sf, fmt=ft.FMT_MXFP8)
    ft.ftmoe_grouped_gemm_gateup(act, ft.grouped_routes(offsets), bank, out, tok_tile=tile, variant=2)
    torch.cuda.synchronize()
    assert ft.ftmoe_read_error_flags() == 0
    got = out.cpu().numpy()
    assert np.all(np.isnan(got[R:])), "rows past offsets[E] must stay untouched"
    adeq = M.dequant_mxfp8(aq.numpy(), asf.numpy())
    wdeq = M.dequant_mxfp8(wq.numpy(), wsf.numpy()).reshape(E, n, k)
    off = offsets.cpu().numpy()
    worst = 0.0
    for e in range(E):
        rows = slice(off[e], off[e + 1])
        if off[e] == off[e + 1]:
            continue
        ref = M.gemm_rows(adeq[rows], wdeq[e])
        absum = np.abs(adeq[rows]) @ np.abs(wdeq[e]).T
        bound = mxfp8_sum_rel(k) * absum + 2.0 ** -21 * np.abs(ref)
        err = np.abs(got[rows] - ref)
        assert np.all(err <= bound + 1e-30), (e, float(np.max(err - bound)))
        nz = absum > 0
        if nz.any():
            worst = max(worst, float(np.max(err[nz] / absum[nz])))
    record_measure(f"MXFP8 block-scaled GEMM max |err| / sum|products| (token tile {tile}, K {k})", worst,
                   mxfp8_sum_rel(k))


def test_grouped_gemm_mxfp8_rejects_slots_and_unaligned_k(ft):
    E, n, k = 2, 128, 256  # K must be a whole number of 512-element scale chunks
    a_q = torch.zeros(4, k, dtype=torch.uint8, device=DEV)
    a_sf = torch.zeros(4, k // 32, dtype=torch.uint8, device=DEV)
    w_q = torch.zeros(E, n, k, dtype=torch.uint8, device=DEV)
    w_sf = torch.zeros(E, n, k // 32, dtype=torch.uint8, device=DEV)
    out = torch.zeros(4, n, device=DEV)
    act = ft.make_act(a_q, a_sf, fmt=ft.FMT_MXFP8)
    bank = ft.make_bank(w_q, w_sf, fmt=ft.FMT_MXFP8)
    offsets = torch.tensor([0, 2, 4], dtype=torch.int32, device=DEV)
    with pytest.raises(ft.FtmoeError) as ei:
        ft.ftmoe_grouped_gemm_gateup(act, ft.grouped_routes(offsets), bank, out)
    assert ei.value.status == ft.FTMOE_UNSUPPORTED
    ids = torch.zeros(4, 1, dtype=torch.int32, device=DEV)
    with pytest.raises(ft.FtmoeError) as ei:
        ft.ftmoe_grouped_gemm_gateup(act, ft.slot_routes(ids), bank, out)
    assert ei.value.status == ft.FTMOE_UNSUPPORTED


# -- forward ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,H,I,E,topk,active,tile", [
    (64, 512, 512, 8, 4, None, 0),
    (24, 1024, 512, 16, 6, [6, 3, 0, 1] * 6, 16),
    (2, 512, 512, 4, 2, None, 0),           # decode sizes run the grouped path too
    (96, 1024, 1024, 16, 6, None, 128),
])
def test_forward_mxfp8_vs_oracle(ft, T, H, I, E, topk, active, tile):
    p = Problem(T, H, I, E, topk, seed=41 + T, active=active, fmt="mxfp8")
    out, _, _ = p.forward(tok_tile=tile)
    torch.cuda.synchronize()
    assert ft.ftmoe_read_error_flags() == 0
    p.check(out)
    # path 2 (grouped, separate SiLU-and-mul) is the automatic path's arithmetic
    out2, _, _ = p.forward(path=2, tok_tile=tile)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))


def test_forward_mxfp8_other_paths_unsupported(ft):
    p = Problem(2, 512, 512, 4, 2, seed=5, fmt="mxfp8")
    for path in (1, 3, 4):
        with pytest.raises(ft.FtmoeError) as ei:
            p.forward(path=path)
        assert ei.value.status == ft.FTMOE_UNSUPPORTED, path

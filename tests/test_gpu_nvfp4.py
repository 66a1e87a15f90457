"""GPU parity of the NVFP4 variant against the oracle, through the C ABI.

Bit-exact: the two-level NVFP4 quantizers (packed e2m1 codes, e4m3 block scales and the
fp32 tensor scale). The SiLU-and-mul re-quantization: every code the nearest e2m1 value
of its fp32 input (which may differ from the fp64 one in the last bits). The grouped
GEMM on the block-scaled tensor-core MMA: the fp64 product of the dequantized operands
within an fp32-accumulation bound, for every token tile, with ragged experts, an empty
expert and an N tail. The forward: the stated output tolerance plus the allowance for
re-quantization decisions on a rounding midpoint.
"""
import numpy as np
import pytest
import torch

import synth
from common import NVFP4_SUM_REL, Problem, record_measure
from oracle import formats as F
from oracle import moe as M

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ft():
    import block_quantized_moe_gb300 as ft
    ft.lib()
    return ft


def _oracle_nvfp4(x32, global_amax=None):
    q, sb, g = M.quantize_nvfp4(x32, global_amax)
    return M.pack_e2m1(q), sb, np.float32(g)


# -- quantizers ------------------------------------------------------------------------

@pytest.mark.parametrize("rows,k", [(1, 256), (37, 512), (8, 7168), (3, 32), (64, 2048)])
def test_quantize_act_nvfp4_bitexact(ft, rows, k):
    x = synth.activations_bf16(rows, k, 2000 + k + rows, DEV)
    x[0, :16] = 0                 # an all-zero 16-block
    x[-1, 16:32] *= 1e-6          # a block far below the tensor's amax (tiny e4m3 scale)
    q = torch.full((rows, k // 2), 0xAA, dtype=torch.uint8, device=DEV)
    s = torch.full((rows, k // 16), 0xAA, dtype=torch.uint8, device=DEV)
    g = torch.full((1,), float("nan"), device=DEV)
    ft.ftmoe_quantize_act(x, q, s, g, fmt=ft.FMT_NVFP4)
    torch.cuda.synchronize()
    rq, rs, rg = _oracle_nvfp4(x.float().cpu().numpy())
    assert g.cpu().numpy().view(np.uint32)[0] == np.float32(rg).view(np.uint32)
    assert np.array_equal(s.cpu().numpy(), rs)
    assert np.array_equal(q.cpu().numpy(), rq)


def test_quantize_act_nvfp4_all_zero(ft):
    x = torch.zeros(4, 256, dtype=torch.bfloat16, device=DEV)
    q = torch.full((4, 128), 0xAA, dtype=torch.uint8, device=DEV)
    s = torch.full((4, 16), 0xAA, dtype=torch.uint8, device=DEV)
    g = torch.full((1,), float("nan"), device=DEV)
    ft.ftmoe_quantize_act(x, q, s, g, fmt=ft.FMT_NVFP4)
    torch.cuda.synchronize()
    assert float(g.item()) == 0.0
    assert not q.any() and not s.any()


@pytest.mark.parametrize("E,n,k", [(3, 256, 512), (2, 130, 96), (1, 512, 7168)])
def test_quantize_weights_nvfp4_bitexact(ft, E, n, k):
    w = torch.stack([synth.expert_weight_fp32(n, k, 77, e, "nvfp4-w", DEV) for e in range(E)])
    w[0, :3, :16] = 0
    q = torch.full((E, n, k // 2), 0xAA, dtype=torch.uint8, device=DEV)
    s = torch.full((E, n, k // 16), 0xAA, dtype=torch.uint8, device=DEV)
    g = torch.full((E,), float("nan"), device=DEV)
    ft.ftmoe_quantize_weights(w, q, s, g, fmt=ft.FMT_NVFP4)
    torch.cuda.synchronize()
    wn = w.cpu().numpy()
    for e in range(E):
        rq, rs, rg = _oracle_nvfp4(wn[e])
        assert g[e].cpu().numpy().view(np.uint32) == np.float32(rg).view(np.uint32), e
        assert np.array_equal(s[e].cpu().numpy(), rs), e
        assert np.array_equal(q[e].cpu().numpy(), rq), e


# -- SiLU-and-mul ----------------------------------------------------------------------

@pytest.mark.parametrize("rows,inter,valid", [(9, 256, 9), (40, 2048, 33)])
def test_silu_mul_nvfp4(ft, rows, inter, valid):
    gu_h = torch.randn(rows, 2 * inter, generator=torch.Generator().manual_seed(rows * 7 + inter)) * 3
    gu_h[1] = 0
    gu = gu_h.to(DEV)
    q = torch.full((rows, inter // 2), 0xAA, dtype=torch.uint8, device=DEV)
    s = torch.full((rows, inter // 16), 0xAA, dtype=torch.uint8, device=DEV)
    g = torch.full((1,), float("nan"), device=DEV)
    rows_dev = torch.tensor([valid], dtype=torch.int32, device=DEV)
    ft.ftmoe_silu_mul(gu, q, s, g, fmt=ft.FMT_NVFP4, rows_dev=rows_dev)
    torch.cuda.synchronize()
    a = M.silu_mul(gu_h[:valid].numpy().astype(np.float64))
    a32 = a.astype(np.float32)
    rq, rs, rg = M.quantize_nvfp4(a32)
    gg = np.float32(g.item())
    # the tensor scale follows the amax of the fp32 intermediate: a few ulp from the oracle's
    assert abs(float(gg) - float(rg)) <= 4 * 2.0 ** -23 * float(rg)
    qg = M.unpack_e2m1(q.cpu().numpy()[:valid], inter)
    sg = s.cpu().numpy()[:valid]
    assert np.all(qg[1] == 0) and np.all(sg[1] == 0)
    assert np.all(q.cpu().numpy()[valid:] == 0xAA) and np.all(s.cpu().numpy()[valid:] == 0xAA)
    # block scales: the e4m3 code of amax_b / (6 g), up to one code where the fp32 input
    # sits on a rounding midpoint
    assert np.all(np.abs(sg.astype(np.int32) - rs.astype(np.int32)) <= 1)
    assert np.mean(sg == rs) > 0.999
    # codes: the nearest e2m1 value of a / (sb g) under the kernel's own block scale
    eff = np.repeat(F.decode_e4m3(sg) * np.float64(gg), 16, axis=1)
    with np.errstate(invalid="ignore", divide="ignore"):
        v = np.where(eff > 0, a / eff, 0.0)
    vq = F.decode_e2m1(qg)
    tab = F.E2M1_VALUES[:8]
    best = np.min(np.abs(np.abs(v)[..., None] - tab), axis=-1)
    assert np.all(np.abs(np.abs(vq) - np.minimum(np.abs(v), 6.0)) <= best + 1e-5 * np.abs(v) + 1e-30)
    assert np.mean(qg == rq) > 0.999


# -- grouped GEMM ----------------------------------------------------------------------

def _random_nvfp4(rows, k, seed, tag):
    """Random packed e2m1 codes and e4m3 block scales (codes 0x28..0x47: 0.25 .. 3.75,
    with a few zero scales)."""
    codes = synth.random_bytes(rows, k // 2, seed, tag + "-q")
    sb = synth.random_bytes(rows, k // 16, seed, tag + "-s") % 32 + 0x28
    sb[synth.random_bytes(rows, k // 16, seed, tag + "-z") < 8] = 0
    return codes, sb


@pytest.mark.parametrize("tile", [16, 32, 64, 128])
def test_grouped_gemm_nvfp4_vs_oracle(ft, tile):
    E, n, k = 5, 320, 512
    counts = [0, 1, 17, 40, 130]
    R = sum(counts)
    offsets = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32, device=DEV)
    aq, asf = _random_nvfp4(R + 3, k, 11, "act")
    wq, wsf = _random_nvfp4(E * n, k, 12, "w")
    ga = torch.tensor([0.37], dtype=torch.float32)
    gw = torch.tensor([0.5, 1.25, 2.0, 0.0625, 3.0], dtype=torch.float32)
    out = torch.full((R + 3, n), float("nan"), device=DEV)
    a_q, a_sf, w_q = aq.to(DEV), asf.to(DEV), wq.reshape(E, n, k // 2).to(DEV)
    w_sf, ga_d, gw_d = wsf.reshape(E, n, k // 16).to(DEV), ga.to(DEV), gw.to(DEV)
    act = ft.make_act(a_q, a_sf, ga_d, fmt=ft.FMT_NVFP4)
    bank = ft.make_bank(w_q, w_sf, gw_d, fmt=ft.FMT_NVFP4)
    ft.ftmoe_grouped_gemm_gateup(act, ft.grouped_routes(offsets), bank, out, tok_tile=tile, variant=2)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.all(np.isnan(got[R:])), "rows past offsets[E] must stay untouched"
    adeq = M.dequant_nvfp4(M.unpack_e2m1(aq.numpy(), k), asf.numpy(), ga.numpy()[0])
    wdeq = M.dequant_nvfp4(M.unpack_e2m1(wq.numpy(), k), wsf.numpy(), 1.0).reshape(E, n, k)
    off = offsets.cpu().numpy()
    worst = 0.0
    for e in range(E):
        rows = slice(off[e], off[e + 1])
        if off[e] == off[e + 1]:
            continue
        ref = M.gemm_rows(adeq[rows], wdeq[e]) * np.float64(gw[e])
        absum = (np.abs(adeq[rows]) @ np.abs(wdeq[e]).T) * float(gw[e])
        bound = NVFP4_SUM_REL * absum + 2.0 ** -21 * np.abs(ref)
        err = np.abs(got[rows] - ref)
        assert np.all(err <= bound + 1e-30), (e, float(np.max(err - bound)))
        nz = absum > 0
        if nz.any():
            worst = max(worst, float(np.max(err[nz] / absum[nz])))
    # the block-scaled MMA's measured error, as a share of the sum of the magnitudes of the
    # products, against the allowance the forward checks take for it
    record_measure(f"NVFP4 block-scaled GEMM max |err| / sum|products| (token tile {tile})", worst, NVFP4_SUM_REL)


def test_grouped_gemm_nvfp4_rejects_slots_and_unaligned_k(ft):
    E, n, k = 2, 128, 96  # k/16 = 6 scale bytes a row: not a 16-byte TMA stride
    a_q = torch.zeros(4, k // 2, dtype=torch.uint8, device=DEV)
    a_sf = torch.zeros(4, k // 16, dtype=torch.uint8, device=DEV)
    g = torch.ones(E, device=DEV)
    w_q = torch.zeros(E, n, k // 2, dtype=torch.uint8, device=DEV)
    w_sf = torch.zeros(E, n, k // 16, dtype=torch.uint8, device=DEV)
    out = torch.zeros(4, n, device=DEV)
    act = ft.make_act(a_q, a_sf, g[:1], fmt=ft.FMT_NVFP4)
    bank = ft.make_bank(w_q, w_sf, g, fmt=ft.FMT_NVFP4)
    offsets = torch.tensor([0, 2, 4], dtype=torch.int32, device=DEV)
    with pytest.raises(ft.FtmoeError) as ei:
        ft.ftmoe_grouped_gemm_gateup(act, ft.grouped_routes(offsets), bank, out)
    assert ei.value.status == 2
    ids = torch.zeros(4, 1, dtype=torch.int32, device=DEV)
    with pytest.raises(ft.FtmoeError) as ei:
        ft.ftmoe_grouped_gemm_gateup(act, ft.slot_routes(ids), bank, out)
    assert ei.value.status == 2


# -- forward ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,H,I,E,topk,active,tile", [
    (64, 512, 256, 8, 4, None, 0),
    (24, 768, 512, 16, 6, [6, 3, 0, 1] * 6, 16),
    (2, 256, 256, 4, 2, None, 0),          # decode sizes run the grouped path too
])
def test_forward_nvfp4_vs_oracle(ft, T, H, I, E, topk, active, tile):
    p = Problem(T, H, I, E, topk, seed=31 + T, active=active, fmt="nvfp4")
    out, _, _ = p.forward(tok_tile=tile)
    torch.cuda.synchronize()
    assert not torch.isnan(out.float()).any()
    p.check(out)
    if active is not None:
        inactive = (p.ids < 0).all(dim=1)
        assert torch.all(out[inactive] == 0)


def test_forward_nvfp4_slot_path_unsupported(ft):
    p = Problem(2, 256, 256, 4, 2, seed=5, fmt="nvfp4")
    with pytest.raises(ft.FtmoeError) as ei:
        p.forward(path=1)
    assert ei.value.status == 2

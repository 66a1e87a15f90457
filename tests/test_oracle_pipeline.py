"""Pins of the oracle's pipeline steps against closed forms, brute force and invariants.

Each test checks the oracle against something other than itself: a closed-form
property of the quantizer, a brute-force double loop for the segmenter, plain
per-element Python loops of the dense FFN (no grouping, no matmul) for the
GEMMs, scipy's logistic function for SiLU, and the inactive-route invariants of
the FreeToken decode page (negative slot = exact zero; equal to the old
clamped-slot / zero-weight path).
"""
import math
import os

import numpy as np
import pytest
from scipy.special import expit

from oracle import formats as F
from oracle import moe as M

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _e4m3_spacing(mag):
    """Distance between adjacent E4M3 values at magnitude `mag` (format definition)."""
    mag = np.asarray(mag, np.float64)
    e = np.floor(np.log2(np.maximum(mag, 2.0 ** -6)))
    return 2.0 ** (e - 3)


# -- FP8 quantizers ------------------------------------------------------------

def test_quantize_act_has_448_code_in_every_nonzero_group():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((7, 300)).astype(np.float32) * rng.uniform(1e-3, 1e3, (7, 1)).astype(np.float32)
    q, s = M.quantize_act_fp8(x)
    assert s.shape == (7, 3)
    for r in range(7):
        for g in range(3):
            blk = q[r, g * 128:(g + 1) * 128]
            assert np.any((blk & 0x7F) == 0x7E)
            assert s[r, g] == np.float32(np.float32(np.max(np.abs(x[r, g * 128:(g + 1) * 128]))) / np.float32(448))


def test_quantize_act_error_bound():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((5, 256)).astype(np.float32)
    q, s = M.quantize_act_fp8(x)
    deq = M.dequant_act_fp8(q, s)
    srep = np.repeat(s.astype(np.float64), 128, axis=1)
    v = x.astype(np.float64) / srep
    err = np.abs(deq / srep - v)
    bound = _e4m3_spacing(np.abs(v)) / 2 + np.abs(v) * 2.0 ** -23
    assert np.all(err <= bound)


def test_quantize_act_power_of_two_amax_round_trips_exactly():
    # amax = 448 * 2**p makes s = 2**p exact; values that are E4M3 values times 2**p survive exactly
    rng = np.random.default_rng(5)
    p = -3
    codes = rng.integers(0, 0x7F, size=(2, 128))
    vals = F.decode_e4m3(codes) * np.where(rng.random((2, 128)) < 0.5, -1, 1) * 2.0 ** p
    vals[:, 17] = 448 * 2.0 ** p
    q, s = M.quantize_act_fp8(vals.astype(np.float32))
    assert np.all(s == np.float32(2.0 ** p))
    assert np.array_equal(M.dequant_act_fp8(q, s), vals)


def test_quantize_act_zero_group_and_partial_group():
    x = np.zeros((2, 200), np.float32)
    x[1, 130] = -3.0  # only element of the 72-wide tail group of row 1
    x[1, 5] = -0.0
    q, s = M.quantize_act_fp8(x)
    assert s.shape == (2, 2)
    assert np.all(s[0] == 0) and np.all(q[0] == 0)
    assert s[1, 0] == 0 and np.all(q[1, :128] == 0)  # amax 0: scale 0, all codes 0x00
    assert s[1, 1] == np.float32(3.0 / 448.0)
    assert q[1, 130] == 0xFE and np.all(np.delete(q[1, 128:], 2) == 0)


def test_quantize_act_negative_value_rounding_to_zero_keeps_sign():
    x = np.zeros((1, 128), np.float32)
    x[0, 0] = 448.0
    x[0, 1] = -1e-6  # x/s = -1e-6 rounds to -0 in E4M3
    q, _ = M.quantize_act_fp8(x)
    assert q[0, 0] == 0x7E and q[0, 1] == 0x80


def test_quantize_act_divides_by_the_scale():
    # amax = 17.5111083984375 (0x418C16C0) gives s = fl32(amax / 448); for x = 0x3D111790,
    # fl32(x / s) is exactly 0.90625, the midpoint of the E4M3 values 0.875 (code 0x36) and
    # 0.9375 (0x37), so dividing rounds to the even code 0x36. Multiplying by
    # fl32(448 / amax) instead rounds x to the other side (0x37).
    amax = np.array([0x418C16C0], np.uint32).view(np.float32)[0]
    xv = np.array([0x3D111790], np.uint32).view(np.float32)[0]
    x = np.zeros((1, 128), np.float32)
    x[0, 0] = amax
    x[0, 1] = xv
    q, s = M.quantize_act_fp8(x)
    assert np.float32(xv / s[0, 0]) == np.float32(0.90625)
    assert q[0, 0] == 0x7E and q[0, 1] == 0x36


def test_quantize_act_fast_equals_plain():
    rng = np.random.default_rng(6)
    x = (rng.standard_normal((33, 900)) * 3).astype(np.float32)
    x[3, :128] = 0
    a = M.quantize_act_fp8(x)
    b = M.quantize_act_fp8_fast(x)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_quantize_weight_blocks_closed_forms():
    rng = np.random.default_rng(7)
    w = (rng.standard_normal((200, 300)) * 0.02).astype(np.float32)
    q, s = M.quantize_weight_fp8(w)
    assert s.shape == (2, 3)
    for i in range(2):
        for j in range(3):
            blk = w[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
            assert s[i, j] == np.float32(np.float32(np.max(np.abs(blk))) / np.float32(448))
            qb = q[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
            assert np.any((qb & 0x7F) == 0x7E)
    deq = M.dequant_weight_fp8(q, s)
    srep = np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)[:200, :300]
    v = w.astype(np.float64) / srep
    assert np.all(np.abs(deq / srep - v) <= _e4m3_spacing(np.abs(v)) / 2 + np.abs(v) * 2.0 ** -23)


def test_quantize_weight_fast_equals_plain():
    rng = np.random.default_rng(16)
    w = (rng.standard_normal((300, 260)) * 0.02).astype(np.float32)
    w[:128, 128:256] = 0  # an all-zero block
    a = M.quantize_weight_fp8(w)
    b = M.quantize_weight_fp8_fast(w)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    lazy = M.LazyBank(lambda e: w, 300)
    assert np.array_equal(lazy.dequant(0), M.dequant_weight_fp8(*a))


# -- NVFP4 ---------------------------------------------------------------------

def test_nvfp4_exact_when_scales_are_exact():
    # global amax 2688 -> g = 1; a block with amax 6 * v (v an E4M3 value) -> sb = code(v), eff = v
    rng = np.random.default_rng(8)
    x = np.zeros((2, 64), np.float64)
    x[0, 0] = 2688.0
    # row 1: four 16-blocks with scales 1, 0.5, 3.25, 2**-6
    for b, sc in enumerate([1.0, 0.5, 3.25, 2.0 ** -6]):
        codes = rng.integers(0, 8, 16)
        vals = F.E2M1_VALUES[codes] * sc * np.where(rng.random(16) < 0.5, -1, 1)
        vals[3] = 6.0 * sc
        x[1, b * 16:(b + 1) * 16] = vals
    q, sb, g = M.quantize_nvfp4(x.astype(np.float32))
    assert g == np.float32(1.0)
    assert sb[0, 0] == 0x7E  # 2688 / 6 = 448
    assert np.array_equal(M.dequant_nvfp4(q, sb, g)[1], x[1])
    assert np.array_equal(M.dequant_nvfp4(q, sb, g)[0], x[0])


def test_nvfp4_zero_tensor_and_zero_block():
    q, sb, g = M.quantize_nvfp4(np.zeros((2, 32), np.float32))
    assert g == 0 and np.all(q == 0) and np.all(sb == 0)
    x = np.zeros((1, 32), np.float32)
    x[0, 20] = 5.0
    q, sb, g = M.quantize_nvfp4(x)
    assert np.all(q[0, :16] == 0) and sb[0, 0] == 0
    assert F.decode_e2m1(q[0, 20]) * F.decode_e4m3(sb[0, 1]) * g == pytest.approx(5.0, rel=0.07)


def test_nvfp4_error_bound_random():
    rng = np.random.default_rng(9)
    x = rng.standard_normal((4, 256)).astype(np.float32)
    q, sb, g = M.quantize_nvfp4(x)
    deq = M.dequant_nvfp4(q, sb, g)
    eff = np.repeat(F.decode_e4m3(sb) * np.float64(g), 16, axis=1)
    # each element is within half an E2M1 step (<= 1.0 * eff at the top) of x/eff, unless saturated at 6
    v = np.abs(x / eff)
    step = np.where(v < 2, 0.5, np.where(v < 4, 1.0, 2.0))
    assert np.all(np.abs(deq / eff - x / eff) <= step / 2 + 1e-6 + np.maximum(v - 6, 0))


def test_pack_unpack_e2m1():
    codes = np.arange(32, dtype=np.uint8).reshape(2, 16) % 16
    packed = M.pack_e2m1(codes)
    assert packed[0, 0] == (0 | (1 << 4))
    assert np.array_equal(M.unpack_e2m1(packed, 16), codes)


# -- segmenter -----------------------------------------------------------------

def _segment_brute(ids, E):
    T, k = ids.shape
    counts = [0] * E
    rows = []
    for e in range(E):
        for t in range(T):
            for j in range(k):
                if ids[t, j] == e:
                    counts[e] += 1
                    rows.append((t * k + j, t))
    route2dst = [-1] * (T * k)
    for d, (r, _) in enumerate(rows):
        route2dst[r] = d
    offsets = [0]
    for c in counts:
        offsets.append(offsets[-1] + c)
    return counts, offsets, [t for _, t in rows], route2dst


@pytest.mark.parametrize("T,k,E,frac_inactive", [(1, 8, 8, 0.75), (8, 8, 64, 0.5), (37, 6, 16, 0.0), (5, 4, 3, 1.0), (64, 8, 256, 0.1)])
def test_segment_matches_brute_force(T, k, E, frac_inactive):
    rng = np.random.default_rng(T * 131 + E)
    ids = np.stack([rng.permutation(E)[:k] if E >= k else rng.integers(0, E, k) for _ in range(T)]).astype(np.int32)
    ids[rng.random(ids.shape) < frac_inactive] = -1
    seg = M.segment_routes(ids, E)
    counts, offsets, dst2src, route2dst = _segment_brute(ids, E)
    assert seg["counts"].tolist() == counts
    assert seg["offsets"].tolist() == offsets
    assert seg["dst2src"].tolist() == dst2src
    assert seg["route2dst"].tolist() == route2dst
    assert seg["offsets"][-1] == int((ids >= 0).sum())


def test_segment_rejects_out_of_range():
    with pytest.raises(ValueError):
        M.segment_routes(np.array([[0, 5]], np.int32), 4)


# -- gather --------------------------------------------------------------------

def test_gather_identity_duplicates_and_empty():
    rng = np.random.default_rng(10)
    src = rng.integers(0, 256, (6, 896), dtype=np.uint8)
    sc = rng.uniform(1e-3, 1, (6, 7)).astype(np.float32)
    d, ds = M.gather_rows_scales(src, sc, np.arange(6))
    assert np.array_equal(d, src) and np.array_equal(ds.view(np.uint32), sc.view(np.uint32))
    m = np.array([2, 2, 5, 0, 2], np.int32)
    d, ds = M.gather_rows_scales(src, sc, m)
    for i, r in enumerate(m):
        assert d[i].tobytes() == src[r].tobytes()
        assert ds[i].tobytes() == sc[r].tobytes()
    d, ds = M.gather_rows_scales(src, sc, np.zeros(0, np.int32))
    assert d.shape == (0, 896) and ds.shape == (0, 7)


# -- SiLU and combine ------------------------------------------------------------

def test_silu_mul_against_library_and_closed_forms():
    rng = np.random.default_rng(11)
    gu = rng.standard_normal((3, 8)) * 4
    ref = gu[:, :4] * expit(gu[:, :4]) * gu[:, 4:]
    assert np.allclose(M.silu_mul(gu), ref, rtol=1e-14, atol=0)
    g = math.log(3.0)  # sigmoid(ln 3) = 3/4
    assert M.silu_mul(np.array([[g, 2.0]]))[0, 0] == pytest.approx(0.75 * g * 2.0, rel=1e-15)
    assert M.silu_mul(np.array([[0.0, 5.0]]))[0, 0] == 0.0


def test_combine_single_route_and_inactive():
    y = np.arange(12, dtype=np.float64).reshape(3, 4) - 5
    ids = np.array([[-1, 2, -1], [-1, -1, -1]], np.int32)
    w = np.array([[np.nan, 1.0, np.nan], [np.nan, np.nan, np.nan]], np.float32)
    route2dst = np.array([-1, 1, -1, -1, -1, -1], np.int32)
    out = M.combine(y, route2dst, ids, w)
    assert np.array_equal(out[0], y[1])
    assert np.all(out[1] == 0) and not np.any(np.isnan(out))


def test_pick_tile_matches_page_table():
    # (routes, experts, best M tile) from the dsfp4 page's sm_89 measurements table
    rows = [ln.split() for ln in open(os.path.join(GOLDEN, "dsfp4_tile_by_density.txt"))
            if ln.strip() and not ln.startswith("#")]
    assert len(rows) == 6
    for routes, experts, _rpe, _shape, bm in rows:
        assert M.pick_tile(int(routes), int(experts)) == int(bm)
    assert M.pick_tile(8, 64) == 16 and M.pick_tile(64 * 200, 64) == 128 and M.pick_tile(2048, 64) == 32


# -- GEMMs and the whole FFN against a per-element brute force -------------------

def _dense_ffn_brute(x, ids, wts, bank_gu, bank_dn):
    """Per token, per active slot: explicit loops over every output and input element."""
    T, H = x.shape
    k = ids.shape[1]
    I2 = bank_gu.q.shape[1]
    I = I2 // 2
    xq, xs = M.quantize_act_fp8(x)
    out = np.zeros((T, H))
    for t in range(T):
        xrow = [F.E4M3_VALUES[xq[t, c]] * float(xs[t, c // 128]) for c in range(H)]
        for j in range(k):
            e = int(ids[t, j])
            if e < 0:
                continue
            gq, gs = bank_gu.q[e], bank_gu.s[e]
            gu = [math.fsum(F.E4M3_VALUES[gq[n, c]] * float(gs[n // 128, c // 128]) * xrow[c] for c in range(H))
                  for n in range(I2)]
            act = [gu[i] / (1.0 + math.exp(-gu[i])) * gu[I + i] for i in range(I)]
            aq, as_ = M.quantize_act_fp8(np.array([act], np.float32))
            arow = [F.E4M3_VALUES[aq[0, c]] * float(as_[0, c // 128]) for c in range(I)]
            dq, ds = bank_dn.q[e], bank_dn.s[e]
            for h in range(H):
                y = math.fsum(F.E4M3_VALUES[dq[h, c]] * float(ds[h // 128, c // 128]) * arow[c] for c in range(I))
                out[t, h] += float(wts[t, j]) * y
    return out


def _tiny_problem(seed, T=3, H=256, I=128, E=4, k=2):
    rng = np.random.default_rng(seed)
    x = F.bf16_bits_to_f32(F.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)))
    wg = (rng.standard_normal((E, 2 * I, H)) * 0.02).astype(np.float32)
    wd = (rng.standard_normal((E, H, I)) * 0.02).astype(np.float32)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    logits = rng.standard_normal((T, k))
    wts = (np.exp(logits) / np.exp(logits).sum(1, keepdims=True)).astype(np.float32)
    return x, ids, wts, M.quantize_bank(wg), M.quantize_bank(wd)


def test_forward_matches_per_element_brute_force():
    x, ids, wts, bg, bd = _tiny_problem(12)
    ids[1, 0] = -1
    ref = _dense_ffn_brute(x, ids, wts, bg, bd)
    got = M.moe_forward(x, ids, wts, bg, bd)["out"]
    scale = np.max(np.abs(ref))
    # both are float64 evaluations of the same quantized operands; only the order of
    # the sums differs (and a requantization tie could flip on a 1-ulp difference)
    assert np.allclose(got, ref, rtol=1e-9, atol=1e-12 * scale)


def _dense_ffn_brute_nvfp4(x, ids, wts, bank_gu, bank_dn):
    """The NVFP4 FFN in per-element loops, in two passes: every active route's SiLU-and-mul
    row first (its tensor scale is taken over all of them), then the down projection."""
    T, H = x.shape
    k = ids.shape[1]
    I2 = bank_gu.q.shape[1]
    I = I2 // 2

    def w_val(bank, e, n, c):
        return F.E2M1_VALUES[bank.q[e][n, c]] * F.E4M3_VALUES[bank.s[e][n, c // 16]] * float(bank.g[e])

    xq, xsb, xg = M.quantize_nvfp4(x)
    acts = {}
    for t in range(T):
        xrow = [F.E2M1_VALUES[xq[t, c]] * F.E4M3_VALUES[xsb[t, c // 16]] * float(xg) for c in range(H)]
        for j in range(k):
            e = int(ids[t, j])
            if e < 0:
                continue
            gu = [math.fsum(w_val(bank_gu, e, n, c) * xrow[c] for c in range(H)) for n in range(I2)]
            acts[(t, j)] = [gu[i] / (1.0 + math.exp(-gu[i])) * gu[I + i] for i in range(I)]
    out = np.zeros((T, H))
    if not acts:
        return out
    amax = max(abs(np.float32(v)) for row in acts.values() for v in row)
    for (t, j), act in acts.items():
        e = int(ids[t, j])
        aq, asb, ag = M.quantize_nvfp4(np.array([act], np.float32), amax)
        arow = [F.E2M1_VALUES[aq[0, c]] * F.E4M3_VALUES[asb[0, c // 16]] * float(ag) for c in range(I)]
        for h in range(H):
            y = math.fsum(w_val(bank_dn, e, h, c) * arow[c] for c in range(I))
            out[t, h] += float(wts[t, j]) * y
    return out


def test_nvfp4_forward_matches_per_element_brute_force():
    x, ids, wts, _, _ = _tiny_problem(21)
    rng = np.random.default_rng(21)
    wg = (rng.standard_normal((4, 256, 256)) * 0.02).astype(np.float32)
    wd = (rng.standard_normal((4, 256, 128)) * 0.02).astype(np.float32)
    bg, bd = M.quantize_bank(wg, "nvfp4"), M.quantize_bank(wd, "nvfp4")
    ids[2, 1] = -1
    ref = _dense_ffn_brute_nvfp4(x, ids, wts, bg, bd)
    got = M.moe_forward(x, ids, wts, bg, bd, fmt="nvfp4")["out"]
    assert np.allclose(got, ref, rtol=1e-9, atol=1e-12 * np.max(np.abs(ref)))


def test_nvfp4_token_subset_keeps_the_call_wide_tensor_scales():
    # a subset evaluates fewer tokens but quantizes with the whole call's amaxes, so its
    # rows are the full call's rows
    x, ids, wts, _, _ = _tiny_problem(22, T=5)
    rng = np.random.default_rng(22)
    bg = M.quantize_bank((rng.standard_normal((4, 256, 256)) * 0.02).astype(np.float32), "nvfp4")
    bd = M.quantize_bank((rng.standard_normal((4, 256, 128)) * 0.02).astype(np.float32), "nvfp4")
    x[4] *= 8.0  # the largest activation and intermediate sit in a token left out below
    full = M.moe_forward(x, ids, wts, bg, bd, fmt="nvfp4")["out"]
    sub = M.moe_forward(x, ids, wts, bg, bd, fmt="nvfp4", tokens_subset=[0, 2])["out"]
    scale = np.max(np.abs(full))
    # BLAS may order the down GEMM's sums differently for fewer stacked rows
    assert np.allclose(sub[[0, 2]], full[[0, 2]], rtol=1e-12, atol=1e-15 * scale)
    assert not np.any(sub[[1, 3, 4]])
    alone = M.moe_forward(x[:1], ids[:1], wts[:1], bg, bd, fmt="nvfp4")["out"]
    # a call of its own has its own tensor scales: a quantization-level difference
    assert np.max(np.abs(alone[0] - full[0])) > 1e-4 * scale


def test_grouped_rows_equal_per_route_rows():
    # segment + gather + per-expert GEMM over grouped rows == per-route GEMM on token rows
    x, ids, wts, bg, bd = _tiny_problem(13, T=9, E=5, k=3)
    ids[2, 1] = -1
    xq, xs = M.quantize_act_fp8(x)
    seg = M.segment_routes(ids, 5)
    aq, as_ = M.gather_rows_scales(xq, xs, seg["dst2src"])
    adeq = M.dequant_act_fp8(aq, as_)
    G = np.zeros((aq.shape[0], bg.q.shape[1]))
    for e in range(5):
        lo, hi = seg["offsets"][e], seg["offsets"][e + 1]
        G[lo:hi] = M.gemm_rows(adeq[lo:hi], bg.dequant(e))
    xdeq = M.dequant_act_fp8(xq, xs)
    for t in range(9):
        for j in range(3):
            r = t * 3 + j
            if ids[t, j] < 0:
                assert seg["route2dst"][r] == -1
                continue
            d = seg["route2dst"][r]
            # BLAS may order the sums differently for a block of rows than for one row
            assert np.allclose(G[d], M.gemm_rows(xdeq[t:t + 1], bg.dequant(ids[t, j]))[0], rtol=1e-12, atol=1e-15)


def test_one_hot_activation_reproduces_weight_column():
    _, _, _, bg, _ = _tiny_problem(14)
    x = np.zeros((1, 256), np.float32)
    x[0, 77] = 448.0 * 2.0 ** -5  # quantizes exactly: s = 2**-5, code 0x7E
    xq, xs = M.quantize_act_fp8(x)
    got = M.gemm_rows(M.dequant_act_fp8(xq, xs), bg.dequant(2))[0]
    col = F.E4M3_VALUES[bg.q[2][:, 77]] * np.repeat(bg.s[2][:, 0].astype(np.float64), 128)
    assert np.array_equal(got, col * 448.0 * 2.0 ** -5)


def test_inactive_invariants():
    x, ids, wts, bg, bd = _tiny_problem(15, T=4, E=4, k=3)
    # all inactive -> exact zero output
    none = np.full_like(ids, -1)
    nanw = np.full_like(wts, np.nan)
    r = M.moe_forward(x, none, nanw, bg, bd)
    assert np.all(r["out"] == 0)
    # -1 slots equal the clamped-slot-0 / zero-weight path, exactly
    ids2 = ids.copy()
    ids2[0, 1] = -1
    ids2[3, :2] = -1
    w_new = wts.copy()
    w_new[ids2 < 0] = np.nan  # never read
    clamped = np.where(ids2 < 0, 0, ids2)  # the old path: slot 0 with routing weight 0
    w_old = np.where(ids2 < 0, np.float32(0), wts).astype(np.float32)
    a = M.moe_forward(x, ids2, w_new, bg, bd)["out"]
    b = M.moe_forward(x, clamped, w_old, bg, bd)["out"]
    # the clamped routes enlarge expert 0's row block, which can change BLAS's summation
    # order in the last float64 bit; the values must otherwise agree
    assert np.allclose(a, b, rtol=1e-12, atol=1e-15)
    assert not np.any(np.isnan(a))

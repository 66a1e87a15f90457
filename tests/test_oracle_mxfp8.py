"""Pins of the oracle's MXFP8 quantizer and forward (oracle/moe.py).

MXFP8 (the mxfp8 branch the SGLang gather page names) is taken with the OCP Microscaling
recipe: per 32 consecutive elements of a row, shared = floor(log2(amax)) - 8 clamped to
[-127, 127] (one E8M0 byte, bias 127), codes e4m3_rne_sat(x / 2^shared). The pins check it
against things other than itself: closed forms, the fp32 bit pattern as a second way to
take floor(log2), torch's float8_e4m3fn cast as a second E4M3 encoder, an error bound, and
per-element brute-force FFN loops.
"""
import math

import numpy as np
import torch

from oracle import formats as F
from oracle import moe as M


def _floor_log2_bits(a32):
    """floor(log2(a)) of positive float32 values from their bit patterns (subnormals too)."""
    bits = np.asarray(a32, np.float32).view(np.uint32).astype(np.int64)
    exp = (bits >> 23) & 0xFF
    man = bits & 0x7FFFFF
    out = exp - 127
    sub = exp == 0
    # a subnormal is man * 2^-149: its leading bit sits at position floor(log2(man))
    out[sub] = np.floor(np.log2(np.maximum(man[sub], 1))).astype(np.int64) - 149
    return out


def test_shared_exponent_closed_forms():
    cases = {1.0: -8, 448.0: 0, 447.5: 0, 256.0: 0, 255.9: -1, 1.75: -8, 2.0: -7, 0.5: -9,
             2.0 ** -126: -127, 2.0 ** -119: -127, 2.0 ** -118: -126, 2.0 ** 127: 119,
             3.0e38: 119, 0.0: -127}
    for a, want in cases.items():
        assert M.mx_shared_exp(np.float32(a)) == want, a
    # a float32 subnormal amax clamps to the smallest E8M0 scale
    assert M.mx_shared_exp(np.float32(2.0 ** -140)) == -127


def test_shared_exponent_matches_the_bit_pattern():
    rng = np.random.default_rng(1)
    a = np.abs(rng.standard_normal(4000) * np.exp2(rng.uniform(-150, 127, 4000))).astype(np.float32)
    a = a[(a > 0) & np.isfinite(a)]
    want = np.clip(_floor_log2_bits(a) - 8, -127, 127)
    got = np.array([M.mx_shared_exp(v) for v in a])
    assert np.array_equal(got, want)


def test_block_of_exact_values_round_trips_with_its_scale():
    # amax = 448 * 2^e: shared = e, every value below is an E4M3 value times 2^e
    e = -5
    vals = np.array([448.0, -448.0, 1.0, -0.5, 0.0, 2.0 ** -9, 240.0, -1.5] * 4, np.float64) * 2.0 ** e
    q, sb = M.quantize_mxfp8(vals.astype(np.float32)[None, :])
    assert sb[0, 0] == e + 127
    assert np.array_equal(M.dequant_mxfp8(q, sb)[0], vals)
    assert q[0, 0] == 0x7E and q[0, 1] == 0xFE and q[0, 2] == 0x38


def test_amax_mantissa_above_1_75_saturates_to_448():
    # amax = 1.875 * 2^k gives shared = k - 8 and amax / 2^shared = 480 > 448: the element
    # encoding clamps to the largest normal (the OCP recipe keeps the scale and clamps)
    k = 3
    blk = np.zeros(32, np.float32)
    blk[0] = 1.875 * 2.0 ** k
    blk[1] = -1.875 * 2.0 ** k
    blk[2] = 1.75 * 2.0 ** k
    q, sb = M.quantize_mxfp8(blk[None, :])
    assert sb[0, 0] == k - 8 + 127
    assert q[0, 0] == 0x7E and q[0, 1] == 0xFE and q[0, 2] == 0x7E
    assert M.dequant_mxfp8(q, sb)[0, 0] == 448.0 * 2.0 ** (k - 8)


def test_zero_block_and_partial_last_block():
    x = np.zeros((2, 70), np.float32)
    x[0, 33] = 3.0          # block 1 only
    x[1, 65:70] = [1, -2, 4, 0, 0.25]  # the partial block of 6 valid elements
    q, sb = M.quantize_mxfp8(x)
    assert sb.shape == (2, 3)
    assert sb[0, 0] == 0 and sb[0, 2] == 0 and sb[0, 1] == 1 - 8 + 127
    assert np.all(q[0, :32] == 0) and np.all(q[0, 64:] == 0)
    assert sb[1, 2] == 2 - 8 + 127
    assert np.array_equal(M.dequant_mxfp8(q, sb)[1, 64:], [0, 1, -2, 4, 0, 0.25])


def test_codes_match_torch_after_the_exact_scaling():
    # a second E4M3 encoder: torch's cast of the (exactly) scaled and clamped values
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((64, 256)) * np.exp2(rng.integers(-40, 40, (64, 1)))).astype(np.float32)
    x[3, 5] = 0.0
    q, sb = M.quantize_mxfp8(x)
    blocks = x.reshape(64, 8, 32)
    amax = np.max(np.abs(blocks), axis=2)
    shared = np.clip(_floor_log2_bits(np.maximum(amax, np.float32(1e-45))) - 8, -127, 127)
    shared[amax == 0] = -127
    assert np.array_equal(sb.astype(np.int64) - 127, shared)
    v = (blocks.astype(np.float64) * np.exp2(-shared)[:, :, None]).astype(np.float32)
    v = np.clip(v, -448.0, 448.0)
    ref = torch.from_numpy(v.reshape(64, 256)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)


def test_error_bound():
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((32, 512)) * np.exp2(rng.uniform(-10, 10, (32, 1)))).astype(np.float32)
    q, sb = M.quantize_mxfp8(x)
    d = M.dequant_mxfp8(q, sb)
    X = np.repeat(np.exp2(sb.astype(np.float64) - 127), 32, axis=1)
    v = np.abs(x.astype(np.float64)) / X
    # half an E4M3 step at v's binade (2^-10 below the normal range), clamped values aside
    step = np.where(v >= 2.0 ** -6, np.exp2(np.floor(np.log2(np.maximum(v, 2.0 ** -6))) - 3), 2.0 ** -9)
    ok = v <= 448.0
    assert np.all(np.abs(d - x)[ok] <= 0.5 * step[ok] * X[ok] * (1 + 1e-12))
    assert np.all(np.abs(d)[~ok] == 448.0 * X[~ok])


def test_fast_equals_plain():
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((9, 200)) * np.exp2(rng.uniform(-30, 30, (9, 1)))).astype(np.float32)
    x[4, :] = 0
    a = M.quantize_mxfp8(x)
    b = M.quantize_mxfp8_fast(x)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def _dense_ffn_brute_mx(x, ids, wts, bank_gu, bank_dn):
    """The MXFP8 FFN in per-element loops: x rows and the SiLU-and-mul rows quantized per
    32 elements, both GEMMs and the combine in math.fsum."""
    T, H = x.shape
    k = ids.shape[1]
    I2 = bank_gu.q.shape[1]
    I = I2 // 2

    def val(q, sb, n, c):
        return F.E4M3_VALUES[q[n, c]] * 2.0 ** (int(sb[n, c // 32]) - 127)

    xq, xs = M.quantize_mxfp8(x)
    out = np.zeros((T, H))
    for t in range(T):
        xrow = [val(xq, xs, t, c) for c in range(H)]
        for j in range(k):
            e = int(ids[t, j])
            if e < 0:
                continue
            gq, gs = bank_gu.q[e], bank_gu.s[e]
            gu = [math.fsum(val(gq, gs, n, c) * xrow[c] for c in range(H)) for n in range(I2)]
            act = [gu[i] / (1.0 + math.exp(-gu[i])) * gu[I + i] for i in range(I)]
            aq, asb = M.quantize_mxfp8(np.array([act], np.float32))
            arow = [val(aq, asb, 0, c) for c in range(I)]
            dq, ds = bank_dn.q[e], bank_dn.s[e]
            for h in range(H):
                y = math.fsum(val(dq, ds, h, c) * arow[c] for c in range(I))
                out[t, h] += float(wts[t, j]) * y
    return out


def test_forward_matches_per_element_brute_force():
    rng = np.random.default_rng(31)
    T, H, I, E, k = 3, 256, 128, 4, 2
    x = F.bf16_bits_to_f32(F.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)))
    wg = (rng.standard_normal((E, 2 * I, H)) * 0.02).astype(np.float32)
    wd = (rng.standard_normal((E, H, I)) * 0.02).astype(np.float32)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[1, 1] = -1
    logits = rng.standard_normal((T, k))
    wts = (np.exp(logits) / np.exp(logits).sum(1, keepdims=True)).astype(np.float32)
    bg, bd = M.quantize_bank(wg, "mxfp8"), M.quantize_bank(wd, "mxfp8")
    assert bg.s.shape == (E, 2 * I, H // 32) and bd.s.shape == (E, H, I // 32)
    ref = _dense_ffn_brute_mx(x, ids, wts, bg, bd)
    got = M.moe_forward(x, ids, wts, bg, bd, fmt="mxfp8")["out"]
    assert np.allclose(got, ref, rtol=1e-9, atol=1e-12 * np.max(np.abs(ref)))
    # a lazily quantized bank gives the same forward
    lg = M.LazyBank(lambda e: wg[e], 2 * I, "mxfp8")
    ld = M.LazyBank(lambda e: wd[e], H, "mxfp8")
    got2 = M.moe_forward(x, ids, wts, lg, ld, fmt="mxfp8")["out"]
    assert np.array_equal(got, got2)

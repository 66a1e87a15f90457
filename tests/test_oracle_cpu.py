"""Pins of the C++ CPU oracle (oracle/cpu_oracle.cpp).

It is a second, independently written oracle of the same definitions. Its pins:
- the numpy oracle, itself pinned in test_oracle_formats.py and test_oracle_pipeline.py:
  codecs, encoders, quantizers, segmenter and gather bit for bit;
- the per-element brute-force dense FFN loops of test_oracle_pipeline.py and
  test_oracle_mxfp8.py (no grouping, no matmul) for the whole forward in all three formats;
- the decode page's inactive-route invariants;
- thread-count independence.
"""
import numpy as np
import pytest

from oracle import cpu as C
from oracle import formats as F
from oracle import moe as M
from test_oracle_mxfp8 import _dense_ffn_brute_mx
from test_oracle_pipeline import _dense_ffn_brute, _dense_ffn_brute_nvfp4, _tiny_problem


def _bits(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def test_codec_tables_match_the_numpy_oracle():
    got = C.e4m3_decode(np.arange(256, dtype=np.uint8))
    ref = F.E4M3_VALUES
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(got[~np.isnan(ref)], ref[~np.isnan(ref)])
    assert np.array_equal(C.e2m1_decode(np.arange(16, dtype=np.uint8)), F.E2M1_VALUES)


def test_e4m3_encoder_on_every_bf16_value_and_every_midpoint():
    bits = np.arange(1 << 16, dtype=np.uint32)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]  # finite bf16 patterns
    vals = F.bf16_bits_to_f32(bits.astype(np.uint16)).astype(np.float64)
    pos = F.E4M3_VALUES[:0x7F]
    mids = (pos[:-1] + pos[1:]) / 2
    near = np.concatenate([mids, np.nextafter(mids.astype(np.float32), np.float32(0)).astype(np.float64),
                           np.nextafter(mids.astype(np.float32), np.float32(1e9)).astype(np.float64)])
    v = np.concatenate([vals, near, -near, [448.0, 464.0, 480.0, 1e30, -1e30, 0.0, -0.0]])
    assert np.array_equal(C.e4m3_encode(v), F.encode_e4m3(v))


def test_e2m1_encoder_on_midpoints_saturation_and_signs():
    pos = F.E2M1_VALUES[:8]
    mids = (pos[:-1] + pos[1:]) / 2
    v = np.concatenate([pos, mids, mids - 1e-6, mids + 1e-6, [6.5, 7.0, 100.0, 0.0, -0.0]])
    v = np.concatenate([v, -v])
    assert np.array_equal(C.e2m1_encode(v), F.encode_e2m1(v))


def test_fp8_quantizers_match_the_numpy_oracle():
    rng = np.random.default_rng(31)
    x = rng.standard_normal((7, 300)).astype(np.float32) * rng.uniform(1e-3, 1e3, (7, 1)).astype(np.float32)
    x[2] = 0.0                      # amax = 0: scale 0, zero codes
    x[3, :5] = -1e-30               # negative values that round to zero keep their sign
    q, s = C.quantize_act_fp8(x)
    qr, sr = M.quantize_act_fp8(x)
    assert np.array_equal(q, qr) and np.array_equal(_bits(s), _bits(sr))
    w = (rng.standard_normal((300, 260)) * 0.02).astype(np.float32)
    w[128:256, 128:256] = 0.0       # an all-zero block
    q, s = C.quantize_weight_fp8(w)
    qr, sr = M.quantize_weight_fp8(w)
    assert np.array_equal(q, qr) and np.array_equal(_bits(s), _bits(sr))


def test_nvfp4_quantizer_matches_the_numpy_oracle():
    rng = np.random.default_rng(32)
    x = rng.standard_normal((5, 70)).astype(np.float32)
    x[1, 16:32] = 0.0               # a zero block
    for amax in (None, 9.5):        # the tensor's own amax, and a wider call-wide one
        q, sb, g = C.quantize_nvfp4(x, amax)
        qr, sbr, gr = M.quantize_nvfp4(x, amax)
        assert np.array_equal(q, qr) and np.array_equal(sb, sbr) and _bits(g) == _bits(gr)
    q, sb, g = C.quantize_nvfp4(np.zeros((2, 32), np.float32))
    assert g == 0 and not q.any() and not sb.any()


@pytest.mark.parametrize("T,k,E,frac", [(1, 8, 8, 0.75), (37, 6, 16, 0.0), (64, 8, 256, 0.1), (5, 3, 3, 1.0)])
def test_segment_and_gather_match_the_numpy_oracle(T, k, E, frac):
    rng = np.random.default_rng(T * 31 + E)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[rng.random((T, k)) < frac] = -1
    got, ref = C.segment_routes(ids, E), M.segment_routes(ids, E)
    for key in ("counts", "offsets", "dst2src", "route2dst"):
        assert np.array_equal(got[key], ref[key]), key
    src = rng.integers(0, 256, (T, 896), dtype=np.uint8)
    sc = rng.uniform(1e-3, 1, (T, 7)).astype(np.float32)
    d, ds = C.gather_rows_scales(src, sc, ref["dst2src"])
    dr, dsr = M.gather_rows_scales(src, sc, ref["dst2src"])
    assert np.array_equal(d, dr) and np.array_equal(_bits(ds), _bits(dsr))
    with pytest.raises(ValueError):
        C.segment_routes(np.array([[0, E]], np.int32), E)


def _bank(b, fmt):
    return (b.q, b.s) if fmt in ("fp8", "mxfp8") else (b.q, b.s, b.g)


def test_mxfp8_quantizer_matches_the_numpy_oracle():
    rng = np.random.default_rng(34)
    x = rng.standard_normal((6, 200)).astype(np.float32) * rng.uniform(1e-3, 1e3, (6, 1)).astype(np.float32)
    x[1, 32:64] = 0.0                # a zero block: byte 0 (shared -127), zero codes
    x[2, :7] = -1e-30                # negatives that round to zero keep their sign
    x[3, 64] = 3.0e38                # the clamp at +127
    x[4, 96:128] = 1.875 * 2.0 ** 5  # a block maximum that saturates to 448 under 2^(5-8)
    x[5, 160:192] = 0.0
    x[5, 160] = 1e-40                # a block whose maximum is subnormal: the clamp at -127
    q, sb = C.quantize_mxfp8(x)
    qr, sbr = M.quantize_mxfp8(x)
    assert np.array_equal(q, qr) and np.array_equal(sb, sbr)
    for a in (0.0, 1e-40, 1.0, 448.0, 255.9, 256.0, 3.0e38, 2.0 ** -126):
        assert C.mx_shared_exp(a) == M.mx_shared_exp(a), a


def test_mxfp8_forward_matches_per_element_brute_force():
    rng = np.random.default_rng(35)
    T, H, I, E, k = 3, 256, 128, 4, 2
    x = F.bf16_bits_to_f32(F.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)))
    bg = M.quantize_bank((rng.standard_normal((E, 2 * I, H)) * 0.02).astype(np.float32), "mxfp8")
    bd = M.quantize_bank((rng.standard_normal((E, H, I)) * 0.02).astype(np.float32), "mxfp8")
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    ids[2, 0] = -1
    logits = rng.standard_normal((T, k))
    wts = (np.exp(logits) / np.exp(logits).sum(1, keepdims=True)).astype(np.float32)
    ref = _dense_ffn_brute_mx(x, ids, wts, bg, bd)
    got = C.moe_forward(x, ids, wts, _bank(bg, "mxfp8"), _bank(bd, "mxfp8"), fmt="mxfp8")
    assert np.allclose(got, ref, rtol=1e-9, atol=1e-12 * np.max(np.abs(ref)))


def test_fp8_forward_matches_per_element_brute_force():
    x, ids, wts, bg, bd = _tiny_problem(12)
    ids[1, 0] = -1
    ref = _dense_ffn_brute(x, ids, wts, bg, bd)
    got = C.moe_forward(x, ids, wts, _bank(bg, "fp8"), _bank(bd, "fp8"))
    assert np.allclose(got, ref, rtol=1e-9, atol=1e-12 * np.max(np.abs(ref)))


def test_nvfp4_forward_matches_per_element_brute_force():
    x, ids, wts, _, _ = _tiny_problem(21)
    rng = np.random.default_rng(21)
    bg = M.quantize_bank((rng.standard_normal((4, 256, 256)) * 0.02).astype(np.float32), "nvfp4")
    bd = M.quantize_bank((rng.standard_normal((4, 256, 128)) * 0.02).astype(np.float32), "nvfp4")
    ids[2, 1] = -1
    ref = _dense_ffn_brute_nvfp4(x, ids, wts, bg, bd)
    got = C.moe_forward(x, ids, wts, _bank(bg, "nvfp4"), _bank(bd, "nvfp4"), fmt="nvfp4")
    assert np.allclose(got, ref, rtol=1e-9, atol=1e-12 * np.max(np.abs(ref)))


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4", "mxfp8"])
def test_forward_matches_the_numpy_oracle_and_does_not_depend_on_threads(fmt):
    x, ids, wts, _, _ = _tiny_problem(33, T=12, H=256, I=128, E=6, k=3)
    rng = np.random.default_rng(33)
    ids[rng.random(ids.shape) < 0.2] = -1
    bg = M.quantize_bank((rng.standard_normal((6, 256, 256)) * 0.02).astype(np.float32), fmt)
    bd = M.quantize_bank((rng.standard_normal((6, 256, 128)) * 0.02).astype(np.float32), fmt)
    ref = M.moe_forward(x, ids, wts, bg, bd, fmt=fmt)["out"]
    outs = [C.moe_forward(x, ids, wts, _bank(bg, fmt), _bank(bd, fmt), fmt=fmt, threads=n) for n in (1, 3, 8)]
    assert all(np.array_equal(outs[0], o) for o in outs[1:])
    scale = np.max(np.abs(ref))
    assert np.allclose(outs[0], ref, rtol=1e-12, atol=1e-14 * scale)
    # a token subset returns the full call's rows (NVFP4: the tensor scales still span the call)
    sub = C.moe_forward(x, ids, wts, _bank(bg, fmt), _bank(bd, fmt), fmt=fmt, tokens_subset=[1, 4, 11], threads=2)
    assert np.array_equal(sub[[1, 4, 11]], outs[0][[1, 4, 11]])
    assert not np.any(np.delete(sub, [1, 4, 11], axis=0))


def test_forward_inactive_invariants():
    x, ids, wts, bg, bd = _tiny_problem(15, T=4, E=4, k=3)
    none = np.full_like(ids, -1)
    assert not np.any(C.moe_forward(x, none, np.full_like(wts, np.nan), _bank(bg, "fp8"), _bank(bd, "fp8")))
    ids2 = ids.copy()
    ids2[0, 1] = -1
    ids2[3, :2] = -1
    w_new = wts.copy()
    w_new[ids2 < 0] = np.nan  # never read
    clamped = np.where(ids2 < 0, 0, ids2)  # the old path: slot 0 with routing weight 0
    w_old = np.where(ids2 < 0, np.float32(0), wts).astype(np.float32)
    a = C.moe_forward(x, ids2, w_new, _bank(bg, "fp8"), _bank(bd, "fp8"))
    b = C.moe_forward(x, clamped, w_old, _bank(bg, "fp8"), _bank(bd, "fp8"))
    assert np.array_equal(a, b) and not np.any(np.isnan(a))


def test_forward_at_the_decode_2048_768_workload_matches_the_numpy_oracle():
    # one token, hidden 2048, intermediate 768, 8 experts, top-8 with 2 of 8 slots active
    import synth
    T, H, I, E, k, seed = 1, 2048, 768, 8, 8, 0xF7E00001
    x = synth.activations_bf16(T, H, seed, "cpu").float().numpy()
    ids = synth.routes(T, k, E, seed, active_per_token=2, device="cpu").numpy()
    w = synth.routing_weights(T, k, seed, "cpu").numpy()
    used = sorted(int(e) for e in ids.reshape(-1) if e >= 0)
    raw_g = {e: synth.expert_weight_fp32(2 * I, H, seed, e, "gateup", "cpu").numpy() for e in used}
    raw_d = {e: synth.expert_weight_fp32(H, I, seed, e, "down", "cpu").numpy() for e in used}
    bg = M.LazyBank(lambda e: raw_g[e], 2 * I)
    bd = M.LazyBank(lambda e: raw_d[e], H)
    ref = M.moe_forward(x, ids, w, bg, bd)["out"]
    # the C++ oracle quantizes the same raw weights itself
    gq = np.zeros((E, 2 * I, H), np.uint8)
    gs = np.zeros((E, 2 * I // 128, H // 128), np.float32)
    dq = np.zeros((E, H, I), np.uint8)
    ds = np.zeros((E, H // 128, I // 128), np.float32)
    for e in used:
        gq[e], gs[e] = C.quantize_weight_fp8(raw_g[e])
        dq[e], ds[e] = C.quantize_weight_fp8(raw_d[e])
        assert np.array_equal(gq[e], bg.parts(e)[0]) and np.array_equal(_bits(gs[e]), _bits(bg.parts(e)[1]))
    got = C.moe_forward(x, ids, w, (gq, gs), (dq, ds), threads=4)
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-14 * np.max(np.abs(ref)))

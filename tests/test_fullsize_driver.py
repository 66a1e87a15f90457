"""The full-size oracle driver (tests/fullsize_oracle.py) against the oracle itself.

The driver splits the FFN by expert across spawned workers; on a small problem its rows
must equal `oracle.moe.moe_forward` evaluated directly (only the order of float64 sums
differs), and its re-quantization allowance must equal the single-process bound's."""
import numpy as np
import pytest

import synth
from common import mxfp8_requant_flip_bound, nvfp4_requant_flip_bound, requant_flip_bound
from fullsize_oracle import forward_calls, forward_subsample
from oracle import moe as M


@pytest.mark.parametrize("fmt", ["fp8", "nvfp4", "mxfp8"])
def test_driver_equals_the_oracle_forward(fmt):
    T, H, I, E, k, seed = 12, 256, 128, 6, 3, 77
    x = synth.activations_bf16(T, H, seed, "cpu").float().numpy()
    ids = synth.routes(T, k, E, seed, active_per_token=[3, 2, 0, 3] * 3, device="cpu").numpy()
    w = synth.routing_weights(T, k, seed, "cpu").numpy()
    sub = [0, 3, 4, 7, 11]
    got, extra = forward_subsample(x, ids, w, sub, H, I, E, seed, fmt, workers=2)
    bg = M.LazyBank(lambda e: synth.expert_weight_fp32(2 * I, H, seed, e, "gateup", "cpu").numpy(), 2 * I, fmt)
    bd = M.LazyBank(lambda e: synth.expert_weight_fp32(H, I, seed, e, "down", "cpu").numpy(), H, fmt)
    res = M.moe_forward(x, ids, w, bg, bd, fmt=fmt, tokens_subset=sub)
    ref = res["out"]
    scale = np.max(np.abs(ref))
    assert np.allclose(got[sub], ref[sub], rtol=1e-12, atol=1e-15 * scale)
    assert not np.any(got[[t for t in range(T) if t not in sub]])
    wv = np.where(ids >= 0, w, 0.0)
    bound = {"fp8": requant_flip_bound, "nvfp4": nvfp4_requant_flip_bound, "mxfp8": mxfp8_requant_flip_bound}[fmt]
    ref_extra = bound(res, ids, wv, bg, bd)
    assert np.allclose(extra[sub], ref_extra[sub], rtol=1e-6, atol=1e-12 * scale)


def test_driver_calls_sharing_one_bank_equal_separate_runs():
    # two calls on one bank in the same passes give each call's own rows (NVFP4: each call's
    # tensor scales are its own)
    H, I, E, k, seed = 256, 128, 5, 2, 91
    calls = []
    for T, s in ((7, 1), (10, 2)):
        x = synth.activations_bf16(T, H, seed + s, "cpu").float().numpy()
        ids = synth.routes(T, k, E, seed + s, device="cpu").numpy()
        w = synth.routing_weights(T, k, seed + s, "cpu").numpy()
        calls.append(dict(x32=x, ids=ids, weights=w, checked=list(range(0, T, 2))))
    for fmt in ("fp8", "nvfp4", "mxfp8"):
        both = forward_calls(calls, H, I, E, seed, fmt, workers=2)
        for c, (out, extra) in zip(calls, both):
            one, one_extra = forward_subsample(c["x32"], c["ids"], c["weights"], c["checked"], H, I, E, seed, fmt,
                                               workers=2)
            assert np.array_equal(out, one) and np.array_equal(extra, one_extra)

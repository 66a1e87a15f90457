"""Pins of the oracle's number-format codecs against the format definitions and torch.

The codecs are pinned against things other than themselves: values printed in the
OCP 8-bit / MX format definitions, torch's float8_e4m3fn and bfloat16 casts
(independent implementations), and exhaustive tie/midpoint checks.
"""
import numpy as np
import pytest
import torch

from oracle import formats as F


# -- E4M3 ------------------------------------------------------------------

def test_e4m3_decode_spec_points():
    # values given by the OCP FP8 definition for E4M3
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6,
             0x38: 1.0, 0x3C: 1.5, 0x40: 2.0, 0x7E: 448.0, 0x77: 240.0, 0xFE: -448.0,
             0xB8: -1.0}
    for c, v in cases.items():
        assert F.decode_e4m3(c) == v, hex(c)
    assert np.isnan(F.decode_e4m3(0x7F)) and np.isnan(F.decode_e4m3(0xFF))
    assert np.signbit(F.decode_e4m3(0x80)) and F.decode_e4m3(0x80) == 0.0


def test_e4m3_decode_matches_torch_exhaustive():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = F.decode_e4m3(np.arange(256))
    assert np.array_equal(np.isnan(ref), np.isnan(ours))
    ok = ~np.isnan(ref)
    assert np.array_equal(ref[ok], ours[ok])
    assert np.array_equal(np.signbit(ref[ok]), np.signbit(ours[ok]))


def _torch_e4m3(v32):
    return torch.from_numpy(v32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_e4m3_encode_matches_torch_all_bf16_in_range():
    # every bfloat16 bit pattern whose value is finite and within [-448, 448]
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = F.bf16_bits_to_f32(bits)
    keep = np.isfinite(v) & (np.abs(v) <= 448.0)
    v = v[keep]
    assert np.array_equal(F.encode_e4m3(v), _torch_e4m3(v))


def test_e4m3_encode_midpoints_and_neighbours():
    pos = F.E4M3_VALUES[:0x7F]
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)  # exact in fp32
    assert np.array_equal(mids.astype(np.float64), (pos[:-1] + pos[1:]) / 2)
    up = np.nextafter(mids, np.float32(np.inf))
    dn = np.nextafter(mids, np.float32(-np.inf))
    v = np.concatenate([mids, up, dn, -mids, -up, -dn]).astype(np.float32)
    assert np.array_equal(F.encode_e4m3(v), _torch_e4m3(v))
    # a tie goes to the even code
    codes = F.encode_e4m3(mids)
    assert np.all(codes % 2 == 0)


def test_e4m3_encode_saturates_and_keeps_sign():
    assert F.encode_e4m3(np.float32(1e6)) == 0x7E
    assert F.encode_e4m3(np.float32(-1e6)) == 0xFE
    assert F.encode_e4m3(np.float32(470.0)) == 0x7E
    assert F.encode_e4m3(np.float32(-0.0)) == 0x80
    assert F.encode_e4m3(np.float32(-1e-9)) == 0x80  # rounds to -0
    assert F.encode_e4m3(np.float32(np.nan)) == 0x7F
    # smallest subnormal and half of it (a tie to the even code 0)
    assert F.encode_e4m3(np.float32(2.0 ** -9)) == 0x01
    assert F.encode_e4m3(np.float32(2.0 ** -10)) == 0x00
    assert F.encode_e4m3(np.float32(3 * 2.0 ** -10)) == 0x02


def test_e4m3_random_values_match_torch():
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(200_000) * 100).astype(np.float32)
    v = v[np.abs(v) <= 448]
    assert np.array_equal(F.encode_e4m3(v), _torch_e4m3(v))


# -- E2M1 ------------------------------------------------------------------

def test_e2m1_table_is_the_ocp_one():
    # magnitudes of FP4 E2M1 as printed by the OCP MX specification
    assert list(F.E2M1_VALUES[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert list(F.E2M1_VALUES[8:]) == [-0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0]


@pytest.mark.parametrize("v,code", [
    (0.25, 0x0), (0.75, 0x2), (1.25, 0x2), (1.75, 0x4), (2.5, 0x4), (3.5, 0x6), (5.0, 0x6),
    (0.2499, 0x0), (0.2501, 0x1), (5.0001, 0x7), (6.0, 0x7), (7.0, 0x7), (1e9, 0x7),
    (-0.75, 0xA), (-6.5, 0xF), (0.0, 0x0), (-0.0, 0x8),
])
def test_e2m1_encode_ties_even_and_saturation(v, code):
    assert F.encode_e2m1(np.float32(v)) == code


def test_e2m1_encode_is_nearest():
    vals = F.E2M1_VALUES[:8]
    x = np.linspace(0, 7, 7001)
    codes = F.encode_e2m1(x)
    got = F.decode_e2m1(codes)
    best = np.min(np.abs(vals[None, :] - np.minimum(x, 6.0)[:, None]), axis=1)
    assert np.allclose(np.abs(got - np.minimum(x, 6.0)), best)


# -- bfloat16 ---------------------------------------------------------------

def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(2)
    v = np.concatenate([
        (rng.standard_normal(100_000) * 10).astype(np.float32),
        (rng.standard_normal(1000) * 1e-38).astype(np.float32),  # subnormal range
        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 65504.0], np.float32),
    ])
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(F.round_to_bf16(v.astype(np.float64)), ref)
    ref_bits = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(F.f32_to_bf16_bits(v), ref_bits)


def test_bf16_bits_roundtrip():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = F.bf16_bits_to_f32(bits)
    fin = np.isfinite(v)
    assert np.array_equal(F.f32_to_bf16_bits(v[fin]), bits[fin])

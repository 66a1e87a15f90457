"""Number formats of the block-quantized MoE path, written from their definitions.

TEST INFRASTRUCTURE ONLY. This module belongs to the CPU oracle; only the test
suite, the smoke check and the benchmark's CPU-baseline leg may use it. The
product path never imports it.

Formats:

* FP8 E4M3 (OCP 8-bit floating point, "fn" variant): 1 sign bit, 4 exponent
  bits with bias 7, 3 mantissa bits; exponent field 0 is subnormal
  (value 2**-6 * m/8); 0x7F / 0xFF are NaN; no infinities; largest finite
  magnitude 448 (0x7E). This is the "FP8-e4m3" the FreeToken block-FP8 decode
  page ("perf(moe): skip inactive block-fp8 decode routes") and the SGLang
  gather page ("Gather the cutlass MoE activation and its scales in one
  launch", Motivation) store their activations and weights in.
* FP4 E2M1 (OCP MX 4-bit float): 1 sign, 2 exponent bits with bias 1,
  1 mantissa bit; magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; no NaN or infinity.
  Used by the NVFP4 variant the dsfp4 page ("pick the grouped-prefill tile
  from route density on sm_89") names.
* bfloat16: the upper 16 bits of an IEEE binary32.

Rounding is round-to-nearest, ties to the even code, with saturation to the
largest finite magnitude ("satfinite"). The encoders find the nearest code by
brute force over the sorted table of representable magnitudes, which is the
definition of round-to-nearest; a tie goes to the code whose least significant
bit is 0, which is the definition of ties-to-even.
"""
import numpy as np

E4M3_MAX = 448.0
E2M1_MAX = 6.0


def _e4m3_decode_one(code: int) -> float:
    sign = -1.0 if code & 0x80 else 1.0
    exp = (code >> 3) & 0xF
    man = code & 0x7
    if exp == 0xF and man == 0x7:
        return float("nan")
    if exp == 0:
        return sign * (2.0 ** -6) * (man / 8.0)
    return sign * (2.0 ** (exp - 7)) * (1.0 + man / 8.0)


def _e2m1_decode_one(code: int) -> float:
    sign = -1.0 if code & 0x8 else 1.0
    exp = (code >> 1) & 0x3
    man = code & 0x1
    if exp == 0:
        return sign * 1.0 * (man / 2.0)  # subnormal: 2**(1-1) * m/2
    return sign * (2.0 ** (exp - 1)) * (1.0 + man / 2.0)


#: value of every E4M3 code, float64, indexed by the code byte (NaN at 0x7F, 0xFF)
E4M3_VALUES = np.array([_e4m3_decode_one(c) for c in range(256)], dtype=np.float64)
#: value of every E2M1 code, float64, indexed by the 4-bit code
E2M1_VALUES = np.array([_e2m1_decode_one(c) for c in range(16)], dtype=np.float64)

# Non-negative finite magnitudes in code order. For both formats the positive
# codes are monotone in value, so position i in this table is code i.
_E4M3_POS = E4M3_VALUES[:0x7F].copy()  # codes 0x00 .. 0x7E
_E2M1_POS = E2M1_VALUES[:8].copy()      # codes 0x0 .. 0x7
assert np.all(np.diff(_E4M3_POS) > 0) and np.all(np.diff(_E2M1_POS) > 0)


def _nearest_code(mag: np.ndarray, table: np.ndarray) -> np.ndarray:
    """Index of the nearest entry of `table` to each magnitude, ties to the even index.

    The decision boundaries of round-to-nearest are the midpoints between adjacent
    entries: a magnitude above the midpoint of entries i and i+1 rounds to i+1, one
    below it to i, and one exactly on it to whichever of i, i+1 is even. Counting the
    midpoints strictly below `mag` gives the index for all non-tie inputs; a tie adds
    one when i+1 is even. Magnitudes beyond the last entry saturate to it (no midpoint
    lies above the last entry). `mag` must be >= 0 and finite; midpoints of these
    formats are exact in float32 and float64.
    """
    mids = (table[:-1] + table[1:]) / 2
    below = np.searchsorted(mids, mag, side="left")  # midpoints strictly below mag
    at = np.minimum(below, len(mids) - 1)
    tie_up = (mids[at] == mag) & ((at + 1) % 2 == 0)
    return below + tie_up


def encode_e4m3(v) -> np.ndarray:
    """float32/float64 array -> E4M3 code bytes, round-to-nearest-even, satfinite.

    The sign of the input is kept (a negative value that rounds to zero gives
    0x80). NaN input gives 0x7F. Inputs are rounded from their exact value.
    """
    v = np.asarray(v, dtype=np.float64)
    neg = np.signbit(v)
    mag = np.abs(v)
    nan = np.isnan(mag)
    mag = np.where(nan, 0.0, mag)
    code = _nearest_code(mag, _E4M3_POS).astype(np.uint8)
    code = np.where(neg, code | 0x80, code).astype(np.uint8)
    return np.where(nan, np.uint8(0x7F), code).astype(np.uint8)


def decode_e4m3(code) -> np.ndarray:
    return E4M3_VALUES[np.asarray(code, dtype=np.uint8)]


def encode_e2m1(v) -> np.ndarray:
    """float array -> 4-bit E2M1 codes (uint8 holding 0..15), RNE, saturating at 6."""
    v = np.asarray(v, dtype=np.float64)
    neg = np.signbit(v)
    mag = np.abs(v)
    code = _nearest_code(mag, _E2M1_POS).astype(np.uint8)
    return np.where(neg, code | 0x8, code).astype(np.uint8)


def decode_e2m1(code) -> np.ndarray:
    return E2M1_VALUES[np.asarray(code, dtype=np.uint8) & 0xF]


def bf16_bits_to_f32(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float32 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


def round_to_bf16(v) -> np.ndarray:
    """Exact value -> nearest bfloat16 value (as float64), ties to even, no saturation.

    bfloat16 keeps 8 significant bits, so for |v| in [2**e, 2**(e+1)) the spacing is
    2**(e-7); below the normal range (e < -126) the spacing stays 2**-133.
    """
    v = np.asarray(v, dtype=np.float64)
    out = v.copy()  # zeros (with their sign) and non-finite values pass through
    nz = (v != 0) & np.isfinite(v)
    e = np.floor(np.log2(np.abs(v[nz])))
    # guard floor(log2) at exact powers of two computed inexactly
    e = np.where(np.abs(v[nz]) < 2.0 ** e, e - 1, e)
    e = np.where(np.abs(v[nz]) >= 2.0 ** (e + 1), e + 1, e)
    q = 2.0 ** (np.maximum(e, -126.0) - 7.0)
    out[nz] = np.rint(v[nz] / q) * q
    return out


def f32_to_bf16_bits(v) -> np.ndarray:
    """Value -> bfloat16 bit pattern (uint16) of its RNE rounding."""
    r = round_to_bf16(v).astype(np.float32)  # exact: a bf16 value is an fp32 value
    return (r.view(np.uint32) >> 16).astype(np.uint16)

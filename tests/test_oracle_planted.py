"""Planted mistakes: each plausible error, planted in a copy of an oracle, must fail a pin.

C++ oracle: the source is copied, one mistake is written into the copy, the copy is built
into a library of its own and bound in place of the real one, and the pins' comparisons run
against it (against the numpy oracle bit for bit, and against the per-element brute-force
FFN loops). The unmodified copy passes every comparison; every mutant fails at least one.
numpy oracle (MXFP8): a constant of the recipe is replaced in the module, and the MXFP8 pins
of test_oracle_mxfp8.py are run against it.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle import build_cpu_oracle
from oracle import cpu as C
from oracle import formats as F
from oracle import moe as M
from test_oracle_mxfp8 import _dense_ffn_brute_mx
from test_oracle_pipeline import _dense_ffn_brute, _tiny_problem

pytestmark = pytest.mark.skipif(shutil.which("g++") is None and shutil.which("c++") is None,
                                reason="no C++ compiler")

# (name, text in cpu_oracle.cpp, replacement)
CPP_MUTANTS = [
    ("gate and up swapped", "const double g = gu[(size_t)i], u = gu[(size_t)(I + i)];",
     "const double u = gu[(size_t)i], g = gu[(size_t)(I + i)];"),
    ("multiply by 448 / amax instead of dividing by s", "const float scaled = v[r * stride_row + i] / s;",
     "const float scaled = v[r * stride_row + i] * (kE4M3Max / amax);"),
    ("ties to the odd code", "if ((i + 1) % 2 == 0) ++i;", "if ((i + 1) % 2 == 1) ++i;"),
    ("routing weight dropped", "for (int64_t h = 0; h < H; ++h) o[h] += wt * y[(size_t)(r * H + h)];",
     "for (int64_t h = 0; h < H; ++h) o[h] += y[(size_t)(r * H + h)];"),
    ("unstable segment order", "    const int32_t d = next[ids[r]]++;",
     "    const int32_t d = offsets[ids[r] + 1] - 1 - (next[ids[r]]++ - offsets[ids[r]]);"),
    ("route index in place of the token index", "dst2src[d] = (int32_t)(r / topk);", "dst2src[d] = (int32_t)r;"),
    ("MXFP8: ceil for floor in the shared exponent", "(e - 1) - kE4M3Emax", "e - kE4M3Emax"),
    ("MXFP8: scale byte bias 126", "sb[r * nblk + b] = (uint8_t)(e + kE8M0Bias);",
     "sb[r * nblk + b] = (uint8_t)(e + 126);"),
    ("MXFP8: no clamp", "return std::min(kE8M0Bias, std::max(-kE8M0Bias, (e - 1) - kE4M3Emax));",
     "return (e - 1) - kE4M3Emax;"),
    ("MXFP8: multiply by 2^shared", "std::ldexp(1.0, -e));", "std::ldexp(1.0, e));"),
]
# (blocks of 16 instead of 32 changes the scale rows' size the binding allocates, so it is
# planted in the numpy recipe below, not here)


def _build_copy(tmp_path, name, text, repl):
    src = open(build_cpu_oracle.SRC).read()
    if text is not None:
        assert src.count(text) == 1, name
        src = src.replace(text, repl)
    path = os.path.join(str(tmp_path), "mutant.cpp")
    with open(path, "w") as f:
        f.write(src)
    lib = os.path.join(str(tmp_path), "mutant.so")
    cxx = shutil.which("g++") or shutil.which("c++")
    subprocess.run([cxx, "-O1", "-std=c++17", "-ffp-contract=off", "-fPIC", "-shared", "-pthread", "-o", lib, path],
                   check=True, capture_output=True)
    return C.bind(ctypes.CDLL(lib))


def _checks():
    """The pins' comparisons, each True when the C++ oracle (as bound now) agrees."""
    out = {}
    rng = np.random.default_rng(41)
    x = rng.standard_normal((5, 300)).astype(np.float32) * rng.uniform(1e-3, 1e3, (5, 1)).astype(np.float32)
    x[2] = 0.0
    x[3, :5] = -1e-30
    # a quotient on a tie that dividing by s and multiplying by 448/amax round apart
    x[4, :128] = 0.0
    x[4, 0] = np.array([0x418C16C0], np.uint32).view(np.float32)[0]
    x[4, 1] = np.array([0x3D111790], np.uint32).view(np.float32)[0]
    q, s = C.quantize_act_fp8(x)
    qr, sr = M.quantize_act_fp8(x)
    out["fp8 quantizer"] = np.array_equal(q, qr) and np.array_equal(s.view(np.uint32), sr.view(np.uint32))
    # a value half-way between two e4m3 codes (ties to the even code)
    v = np.array([1.0625, 1.1875, 17.0, -3.25], np.float64)
    out["e4m3 encoder"] = np.array_equal(C.e4m3_encode(v), F.encode_e4m3(v))
    xm = x.copy()
    xm[1, 32:64] = 0.0
    xm[4, 96:128] = 1.875 * 2.0 ** 5
    xm[0, 160:192] = 0.0
    xm[0, 160] = 1e-40
    q, sb = C.quantize_mxfp8(xm)
    qr, sbr = M.quantize_mxfp8(xm)
    out["mxfp8 quantizer"] = (np.array_equal(q, qr) and np.array_equal(sb, sbr) and
                              all(C.mx_shared_exp(a) == M.mx_shared_exp(a) for a in (0.0, 1e-40, 1.0, 448.0, 3e38)))
    ids = np.array([[2, 0, 1], [1, 2, -1], [0, 1, 2], [2, 1, 0]], np.int32)
    got, ref = C.segment_routes(ids, 3), M.segment_routes(ids, 3)
    out["segmenter"] = all(np.array_equal(got[key], ref[key]) for key in ("counts", "offsets", "dst2src", "route2dst"))
    xt, idt, wt, bg, bd = _tiny_problem(12)
    ref = _dense_ffn_brute(xt, idt, wt, bg, bd)
    got = C.moe_forward(xt, idt, wt, (bg.q, bg.s), (bd.q, bd.s))
    out["fp8 forward"] = bool(np.allclose(got, ref, rtol=1e-9, atol=1e-12 * np.max(np.abs(ref))))
    rng = np.random.default_rng(42)
    T, H, I, E, k = 3, 256, 128, 4, 2
    xx = F.bf16_bits_to_f32(F.f32_to_bf16_bits(rng.standard_normal((T, H)).astype(np.float32)))
    mg = M.quantize_bank((rng.standard_normal((E, 2 * I, H)) * 0.02).astype(np.float32), "mxfp8")
    md = M.quantize_bank((rng.standard_normal((E, H, I)) * 0.02).astype(np.float32), "mxfp8")
    mid = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    mw = rng.uniform(0.1, 1.0, (T, k)).astype(np.float32)
    ref = _dense_ffn_brute_mx(xx, mid, mw, mg, md)
    got = C.moe_forward(xx, mid, mw, (mg.q, mg.s), (md.q, md.s), fmt="mxfp8")
    out["mxfp8 forward"] = bool(np.allclose(got, ref, rtol=1e-9, atol=1e-12 * np.max(np.abs(ref))))
    return out


def test_unmodified_copy_passes_every_check(tmp_path, monkeypatch):
    monkeypatch.setattr(C, "_lib", _build_copy(tmp_path, "none", None, None))
    failed = [name for name, ok in _checks().items() if not ok]
    assert not failed, failed


@pytest.mark.parametrize("name,text,repl", CPP_MUTANTS, ids=[m[0] for m in CPP_MUTANTS])
def test_planted_mistake_in_the_cpp_oracle_fails_a_pin(tmp_path, monkeypatch, name, text, repl):
    monkeypatch.setattr(C, "_lib", _build_copy(tmp_path, name, text, repl))
    res = _checks()
    assert not all(res.values()), f"'{name}' passed every check"


@pytest.mark.parametrize("const,value", [("E4M3_EMAX", 7), ("E8M0_BIAS", 126), ("MX_BLOCK", 16)])
def test_planted_constant_in_the_numpy_mxfp8_recipe_fails_a_pin(monkeypatch, const, value):
    import test_oracle_mxfp8 as P
    pins = [P.test_shared_exponent_closed_forms, P.test_shared_exponent_matches_the_bit_pattern,
            P.test_block_of_exact_values_round_trips_with_its_scale, P.test_amax_mantissa_above_1_75_saturates_to_448,
            P.test_zero_block_and_partial_last_block, P.test_codes_match_torch_after_the_exact_scaling,
            P.test_error_bound, P.test_forward_matches_per_element_brute_force]
    monkeypatch.setattr(M, const, value)
    failures = 0
    for pin in pins:
        try:
            pin()
        except Exception:  # noqa: BLE001 - a failed assertion or a shape the pin cannot use
            failures += 1
    assert failures > 0, f"{const} = {value} passed every MXFP8 pin"


# numpy oracle (oracle/moe.py): each mistake is written into a copy of the module's source,
# the copy is executed as a module of its own, and the pins of test_oracle_pipeline.py run
# with it in place of the real module.
NUMPY_MUTANTS = [
    ("gate and up swapped", "g, u = gu[:, :inter], gu[:, inter:]", "u, g = gu[:, :inter], gu[:, inter:]"),
    ("weight block scales transposed", "sc = np.repeat(np.repeat(np.asarray(s, np.float64), GROUP, axis=0)",
     "sc = np.repeat(np.repeat(np.asarray(s, np.float64).T, GROUP, axis=0)"),
    ("routing weight dropped", "out[t] += np.float64(weights[t, j]) * y_rows[(t, j)]", "out[t] += y_rows[(t, j)]"),
    ("unstable segment order", 'order = active[np.argsort(flat[active], kind="stable")]',
     'order = active[::-1][np.argsort(flat[active][::-1], kind="stable")]'),
    ("route index in place of the token index", "dst2src = (order // topk).astype(np.int32)",
     "dst2src = order.astype(np.int32)"),
    ("multiply by 448 / amax instead of dividing by s", "v = (vals32 / s).astype(np.float32)",
     "v = (vals32 * (np.float32(E4M3_MAX) / amax)).astype(np.float32)"),
    ("intermediate not re-quantized", "adeq_all, _ = quantize_acts(A, fmt, gamax)",
     "adeq_all = A.astype(np.float64)"),
]


def _numpy_mutant(text, repl):
    import types
    path = os.path.join(os.path.dirname(M.__file__), "moe.py")
    src = open(path).read()
    if text is not None:
        assert src.count(text) == 1, text
        src = src.replace(text, repl)
    mod = types.ModuleType("oracle.moe_planted")
    mod.__package__ = "oracle"
    mod.__file__ = path
    exec(compile(src, path, "exec"), mod.__dict__)
    return mod


def _pipeline_pins_failing(monkeypatch, mod):
    import inspect

    import test_oracle_pipeline as P
    monkeypatch.setattr(P, "M", mod)
    failing = []
    for name, fn in sorted(vars(P).items()):
        if not name.startswith("test_") or not callable(fn):
            continue
        params = inspect.signature(fn).parameters
        calls = [()] if not params else [(8, 8, 64, 0.5), (37, 6, 16, 0.0)]
        for args in calls:
            try:
                fn(*args)
            except Exception:  # noqa: BLE001 - a failed assertion or an operand the pin cannot use
                failing.append(name)
                break
    return failing


def test_unmodified_numpy_copy_passes_the_pipeline_pins(monkeypatch):
    assert _pipeline_pins_failing(monkeypatch, _numpy_mutant(None, None)) == []


@pytest.mark.parametrize("name,text,repl", NUMPY_MUTANTS, ids=[m[0] for m in NUMPY_MUTANTS])
def test_planted_mistake_in_the_numpy_oracle_fails_a_pin(monkeypatch, name, text, repl):
    assert _pipeline_pins_failing(monkeypatch, _numpy_mutant(text, repl)), f"'{name}' passed every pin"

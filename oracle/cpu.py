"""ctypes binding of the C++ CPU oracle (cpu_oracle.cpp), with numpy arrays in and out.

TEST INFRASTRUCTURE ONLY, like the rest of `oracle/`: the tests, the smoke check and the
benchmark's CPU-baseline legs may use it. It is a second, independently written oracle of
the same definitions as `oracle.moe` and `oracle.formats`; the tests hold the two to each
other. Argument marshalling only: every step runs in the C++ code.
"""
import ctypes
import os

import numpy as np

from . import build_cpu_oracle

_lib = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32


def lib():
    """The loaded C++ oracle, built on first use if needed."""
    global _lib
    if _lib is None:
        _lib = bind(ctypes.CDLL(build_cpu_oracle.build()))
    return _lib


def bind(h):
    """Sets the C signatures on a loaded oracle library (also used for copies of it that the
    tests build with planted mistakes); returns it."""
    h.ftor_e4m3_decode.restype = ctypes.c_double
    h.ftor_e4m3_decode.argtypes = [ctypes.c_uint8]
    h.ftor_e2m1_decode.restype = ctypes.c_double
    h.ftor_e2m1_decode.argtypes = [ctypes.c_uint8]
    h.ftor_e4m3_encode.restype = ctypes.c_uint8
    h.ftor_e4m3_encode.argtypes = [ctypes.c_double]
    h.ftor_e2m1_encode.restype = ctypes.c_uint8
    h.ftor_e2m1_encode.argtypes = [ctypes.c_double]
    h.ftor_quantize_act_fp8.argtypes = [_P, _I64, _I64, _P, _P]
    h.ftor_quantize_weight_fp8.argtypes = [_P, _I64, _I64, _P, _P]
    h.ftor_nvfp4_global_scale.restype = ctypes.c_float
    h.ftor_nvfp4_global_scale.argtypes = [ctypes.c_float]
    h.ftor_quantize_nvfp4.argtypes = [_P, _I64, _I64, ctypes.c_float, _P, _P, _P]
    h.ftor_mx_shared_exp.restype = ctypes.c_int
    h.ftor_mx_shared_exp.argtypes = [ctypes.c_float]
    h.ftor_quantize_mxfp8.argtypes = [_P, _I64, _I64, _P, _P]
    h.ftor_segment.restype = ctypes.c_int
    h.ftor_segment.argtypes = [_P, _I64, _I32, _I32, _P, _P, _P, _P]
    h.ftor_gather.argtypes = [_P, _P, _I64, _I64, _P, _I64, _P, _P]
    h.ftor_moe_forward.restype = ctypes.c_int
    h.ftor_moe_forward.argtypes = [ctypes.c_int, _P, _I64, _I64, _I64, _I32, _I32, _P, _P, _P, _P, _P, _P,
                                   _P, _P, _P, _I64, ctypes.c_int, _P]
    h.ftor_hardware_threads.restype = ctypes.c_int
    return h


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def hardware_threads():
    return int(lib().ftor_hardware_threads())


def e4m3_decode(codes):
    f = lib().ftor_e4m3_decode
    return np.array([f(int(c)) for c in np.asarray(codes, np.uint8).reshape(-1)]).reshape(np.shape(codes))


def e4m3_encode(values):
    f = lib().ftor_e4m3_encode
    v = np.asarray(values, np.float64)
    return np.array([f(float(x)) for x in v.reshape(-1)], np.uint8).reshape(v.shape)


def e2m1_decode(codes):
    f = lib().ftor_e2m1_decode
    return np.array([f(int(c)) for c in np.asarray(codes, np.uint8).reshape(-1)]).reshape(np.shape(codes))


def e2m1_encode(values):
    f = lib().ftor_e2m1_encode
    v = np.asarray(values, np.float64)
    return np.array([f(float(x)) for x in v.reshape(-1)], np.uint8).reshape(v.shape)


def quantize_act_fp8(x):
    x = _c(x, np.float32)
    rows, k = x.shape
    q = np.zeros((rows, k), np.uint8)
    s = np.zeros((rows, -(-k // 128)), np.float32)
    lib().ftor_quantize_act_fp8(_ptr(x), rows, k, _ptr(q), _ptr(s))
    return q, s


def quantize_weight_fp8(w):
    w = _c(w, np.float32)
    n, k = w.shape
    q = np.zeros((n, k), np.uint8)
    s = np.zeros((-(-n // 128), -(-k // 128)), np.float32)
    lib().ftor_quantize_weight_fp8(_ptr(w), n, k, _ptr(q), _ptr(s))
    return q, s


def quantize_nvfp4(x, global_amax=None):
    x = _c(x, np.float32)
    rows, k = x.shape
    if global_amax is None:
        global_amax = float(np.max(np.abs(x))) if x.size else 0.0
    q = np.zeros((rows, k), np.uint8)
    sb = np.zeros((rows, -(-k // 16)), np.uint8)
    g = np.zeros(1, np.float32)
    lib().ftor_quantize_nvfp4(_ptr(x), rows, k, ctypes.c_float(global_amax), _ptr(q), _ptr(sb), _ptr(g))
    return q, sb, np.float32(g[0])


def mx_shared_exp(amax):
    return int(lib().ftor_mx_shared_exp(ctypes.c_float(float(amax))))


def quantize_mxfp8(x):
    x = _c(x, np.float32)
    rows, k = x.shape
    q = np.zeros((rows, k), np.uint8)
    sb = np.zeros((rows, -(-k // 32)), np.uint8)
    lib().ftor_quantize_mxfp8(_ptr(x), rows, k, _ptr(q), _ptr(sb))
    return q, sb


def segment_routes(expert_ids, num_experts):
    ids = _c(expert_ids, np.int32)
    tokens, topk = ids.shape
    R = tokens * topk
    counts = np.zeros(num_experts, np.int32)
    offsets = np.zeros(num_experts + 1, np.int32)
    dst2src = np.zeros(R, np.int32)
    route2dst = np.zeros(R, np.int32)
    if lib().ftor_segment(_ptr(ids), tokens, topk, num_experts, _ptr(counts), _ptr(offsets), _ptr(dst2src),
                          _ptr(route2dst)) != 0:
        raise ValueError("expert id out of range")
    return dict(counts=counts, offsets=offsets, dst2src=dst2src[:offsets[-1]], route2dst=route2dst)


def gather_rows_scales(src, src_scales, dst2src):
    src = _c(src, np.uint8)
    sc = np.ascontiguousarray(src_scales)
    scb = sc.view(np.uint8).reshape(sc.shape[0], -1)
    m = _c(dst2src, np.int32)
    dst = np.zeros((m.shape[0], src.shape[1]), np.uint8)
    dsc = np.zeros((m.shape[0], scb.shape[1]), np.uint8)
    lib().ftor_gather(_ptr(src), _ptr(scb), src.shape[1], scb.shape[1], _ptr(m), m.shape[0], _ptr(dst), _ptr(dsc))
    return dst, dsc.view(sc.dtype).reshape((m.shape[0],) + sc.shape[1:])


def moe_forward(x, expert_ids, weights, bank_gateup, bank_down, fmt="fp8", tokens_subset=None, threads=1):
    """The whole FFN (see cpu_oracle.cpp). Banks: fp8 (q [E, n, k] uint8, s [E, nb, kb] float32);
    nvfp4 (q [E, n, k] unpacked codes, sb [E, n, ceil(k/16)] uint8, g [E] float32); mxfp8
    (q [E, n, k] uint8, sb [E, n, ceil(k/32)] E8M0 bytes).
    Returns float64 [T, H] (rows outside tokens_subset are zero)."""
    x = _c(x, np.float32)
    ids = _c(expert_ids, np.int32)
    w = _c(weights, np.float32)
    T, H = x.shape
    topk = ids.shape[1]
    gq = _c(bank_gateup[0], np.uint8)
    dq = _c(bank_down[0], np.uint8)
    E = gq.shape[0]
    I = gq.shape[1] // 2
    if fmt == "fp8":
        gs, ds = _c(bank_gateup[1], np.float32), _c(bank_down[1], np.float32)
        gg = dg = None
    elif fmt == "mxfp8":
        gs, ds = _c(bank_gateup[1], np.uint8), _c(bank_down[1], np.uint8)
        gg = dg = None
    else:
        gs, ds = _c(bank_gateup[1], np.uint8), _c(bank_down[1], np.uint8)
        gg, dg = _c(bank_gateup[2], np.float32), _c(bank_down[2], np.float32)
    sub = None if tokens_subset is None else _c(list(tokens_subset), np.int64)
    out = np.zeros((T, H), np.float64)
    rc = lib().ftor_moe_forward({"fp8": 0, "nvfp4": 1, "mxfp8": 2}[fmt], _ptr(x), T, H, I, E, topk, _ptr(ids), _ptr(w), _ptr(gq),
                                _ptr(gs), _ptr(gg), _ptr(dq), _ptr(ds), _ptr(dg), _ptr(sub),
                                0 if sub is None else sub.shape[0], int(threads), _ptr(out))
    if rc != 0:
        raise ValueError("expert id out of range")
    return out

"""Python binding of libftmoe, the GB300 (sm_103a) block-quantized MoE FFN library.

Argument marshalling only: every function here forwards torch tensors' device
pointers, sizes and the current CUDA stream to the C entry point of the same name
declared in include/ftmoe.h. All arithmetic runs in the library's CUDA kernels;
there is no host or PyTorch fallback. If libftmoe.so is missing or cannot be
loaded, every call raises.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libftmoe.so")

FTMOE_OK, FTMOE_INVALID_ARG, FTMOE_UNSUPPORTED, FTMOE_CUDA_ERROR, FTMOE_WORKSPACE_TOO_SMALL, FTMOE_CHECK_FAILED = range(6)
FMT_FP8, FMT_NVFP4, FMT_MXFP8 = 0, 1, 2
ROUTES_GROUPED, ROUTES_SLOTS = 0, 1
ERR_EXPERT_ID_RANGE, ERR_MAP_RANGE, ERR_WAIT_TIMEOUT = 0x1, 0x2, 0x4
OUT_BF16, OUT_FP16, OUT_FP32 = 0, 1, 2
_OUT_DTYPES = {torch.bfloat16: OUT_BF16, torch.float16: OUT_FP16, torch.float32: OUT_FP32}

c_i32, c_i64, c_ptr, c_size = ctypes.c_int32, ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t


class FtmoeError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {status} ({_status_string(status)})")


class ExpertBank(ctypes.Structure):
    _fields_ = [("format", c_i32), ("num_experts", c_i32), ("n", c_i64), ("k", c_i64),
                ("q", c_ptr), ("scales", c_ptr), ("global_scale", c_ptr)]


class Act(ctypes.Structure):
    _fields_ = [("format", c_i32), ("reserved", c_i32), ("rows", c_i64), ("k", c_i64),
                ("q", c_ptr), ("scales", c_ptr), ("global_scale", c_ptr)]


class Routes(ctypes.Structure):
    _fields_ = [("kind", c_i32), ("topk", c_i32), ("tokens", c_i64), ("offsets", c_ptr), ("slots", c_ptr)]


class Tile(ctypes.Structure):
    _fields_ = [("tok_tile", c_i32), ("variant", c_i32), ("wblocks", c_i32), ("ctas", c_i32)]


class MoeShape(ctypes.Structure):
    _fields_ = [("tokens", c_i64), ("hidden", c_i64), ("inter", c_i64), ("topk", c_i32),
                ("num_experts", c_i32), ("format", c_i32), ("tok_tile", c_i32), ("path", c_i32),
                ("out_dtype", c_i32)]


class MoeArgs(ctypes.Structure):
    _fields_ = [("shape", MoeShape), ("x", c_ptr), ("ld_x", c_i64), ("expert_ids", c_ptr),
                ("route_weights", c_ptr), ("w_gateup", ExpertBank), ("w_down", ExpertBank),
                ("out", c_ptr), ("ld_out", c_i64)]


_LAYOUT_FIELDS = ["x_q", "x_scales", "x_gscale", "counts", "offsets", "dst2src", "route2dst",
                  "rows_q", "rows_scales", "gateup", "gateup_bytes", "act_q", "act_q_bytes",
                  "act_scales", "act_scales_bytes", "act_gscale", "down", "down_bytes", "partials",
                  "partials_bytes", "counters", "counters_bytes", "total"]


class WorkspaceLayout(ctypes.Structure):
    _fields_ = [(n, c_size) for n in _LAYOUT_FIELDS]


# (name, restype, argtypes) of every exported entry point
_SIGNATURES = [
    ("ftmoe_status_string", ctypes.c_char_p, [c_i32]),
    ("ftmoe_pick_tile", c_i32, [c_i64, c_i32, ctypes.POINTER(Tile)]),
    ("ftmoe_quantize_act", c_i32, [c_ptr, c_i64, c_i64, c_i64, c_i32, c_ptr, c_ptr, c_ptr, c_ptr]),
    ("ftmoe_quantize_weights", c_i32, [c_ptr, c_i32, c_i64, c_i64, c_i32, c_ptr, c_ptr, c_ptr, c_ptr]),
    ("ftmoe_segment_routes", c_i32, [c_ptr, c_i64, c_i32, c_i32, c_ptr, c_ptr, c_ptr, c_ptr, c_ptr]),
    ("ftmoe_gather_rows_scales", c_i32, [c_ptr, c_ptr, c_i64, c_i64, c_i64, c_ptr, c_i64, c_ptr,
                                         c_ptr, c_ptr, c_ptr]),
    ("ftmoe_gather_quantize_act", c_i32, [c_ptr, c_i64, c_i64, c_i64, c_ptr, c_i64, c_ptr, c_i32, c_ptr, c_ptr,
                                          c_ptr]),
    ("ftmoe_grouped_gemm_gateup", c_i32, [ctypes.POINTER(Act), ctypes.POINTER(Routes),
                                          ctypes.POINTER(ExpertBank), c_ptr, c_i64,
                                          ctypes.POINTER(Tile), c_ptr]),
    ("ftmoe_grouped_gemm_gateup_silu", c_i32, [ctypes.POINTER(Act), ctypes.POINTER(Routes),
                                               ctypes.POINTER(ExpertBank), c_ptr, c_ptr,
                                               ctypes.POINTER(Tile), c_ptr]),
    ("ftmoe_silu_mul", c_i32, [c_ptr, c_i64, c_i64, c_i64, c_ptr, c_i32, c_ptr, c_ptr, c_ptr, c_ptr]),
    ("ftmoe_grouped_gemm_down", c_i32, [ctypes.POINTER(Act), ctypes.POINTER(Routes),
                                        ctypes.POINTER(ExpertBank), c_ptr, c_i64,
                                        ctypes.POINTER(Tile), c_ptr]),
    ("ftmoe_combine", c_i32, [c_ptr, c_i64, c_ptr, c_ptr, c_ptr, c_i64, c_i32, c_i64, c_i32, c_ptr, c_i64,
                              c_ptr]),
    ("ftmoe_forward_workspace_bytes", c_size, [ctypes.POINTER(MoeShape)]),
    ("ftmoe_forward_workspace_layout", c_i32, [ctypes.POINTER(MoeShape), ctypes.POINTER(WorkspaceLayout)]),
    ("ftmoe_moe_forward", c_i32, [ctypes.POINTER(MoeArgs), c_ptr, c_size, c_ptr]),
    ("ftmoe_moe_forward_noalloc", c_i32, [ctypes.POINTER(MoeArgs), c_ptr]),
    ("ftmoe_selftest_wait_timeout", c_i32, [ctypes.c_uint64, c_ptr, c_ptr]),
    ("ftmoe_selftest_shared_division", c_i32, [c_ptr, c_ptr]),
    ("ftmoe_expert_slots", c_i32, [c_ptr, c_i64, c_ptr, c_ptr, c_i32, c_ptr, c_i32, c_i64, c_i32, c_ptr, c_ptr,
                                   c_ptr]),
    ("ftmoe_read_error_flags", c_i32, [ctypes.POINTER(ctypes.c_uint32)]),
]

_lib_handle = None


def lib():
    """The loaded libftmoe (ctypes.CDLL). Raises if it was not built."""
    global _lib_handle
    if _lib_handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libftmoe.so not found at {LIB_PATH}; build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        h = ctypes.CDLL(LIB_PATH)
        for name, res, args in _SIGNATURES:
            fn = getattr(h, name)
            fn.restype, fn.argtypes = res, args
        _lib_handle = h
    return _lib_handle


def _status_string(s):
    try:
        return lib().ftmoe_status_string(s).decode()
    except Exception:  # noqa: BLE001 - message only
        return "?"


def _check(fn, status):
    if status != FTMOE_OK:
        raise FtmoeError(fn, status)


def _p(t):
    """Device (or host) pointer of a tensor, None for None."""
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


# ---------------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ---------------------------------------------------------------------------------

def ftmoe_pick_tile(routes, num_experts):
    t = Tile()
    _check("ftmoe_pick_tile", lib().ftmoe_pick_tile(int(routes), int(num_experts), ctypes.byref(t)))
    return t.tok_tile


def ftmoe_quantize_act(x, q, scales, global_scale=None, fmt=FMT_FP8, rows=None, k=None, stream=None):
    rows = x.shape[0] if rows is None else rows
    k = x.shape[1] if k is None else k
    ld = x.stride(0) if x.dim() == 2 else k
    _check("ftmoe_quantize_act", lib().ftmoe_quantize_act(
        _p(x), rows, k, ld, fmt, _p(q), _p(scales), _p(global_scale), _stream(stream)))


def ftmoe_quantize_weights(w, q, scales, global_scale=None, fmt=FMT_FP8, stream=None):
    E, n, k = w.shape
    _check("ftmoe_quantize_weights", lib().ftmoe_quantize_weights(
        _p(w), E, n, k, fmt, _p(q), _p(scales), _p(global_scale), _stream(stream)))


def ftmoe_segment_routes(expert_ids, num_experts, counts, offsets, dst2src, route2dst, stream=None):
    T, topk = expert_ids.shape
    _check("ftmoe_segment_routes", lib().ftmoe_segment_routes(
        _p(expert_ids), T, topk, num_experts, _p(counts), _p(offsets), _p(dst2src), _p(route2dst),
        _stream(stream)))


def ftmoe_gather_rows_scales(src, src_scales, dst2src, dst, dst_scales, n_dst=None, n_dst_dev=None,
                             stream=None):
    n_src = src.shape[0]
    row_bytes = src.shape[1] * src.element_size()
    scale_bytes = src_scales.shape[1] * src_scales.element_size() if src_scales is not None else 0
    n_dst = dst2src.shape[0] if n_dst is None else n_dst
    _check("ftmoe_gather_rows_scales", lib().ftmoe_gather_rows_scales(
        _p(src), _p(src_scales), n_src, row_bytes, scale_bytes, _p(dst2src), n_dst, _p(n_dst_dev),
        _p(dst), _p(dst_scales), _stream(stream)))


def ftmoe_gather_quantize_act(x, dst2src, q, scales, fmt=FMT_MXFP8, n_dst=None, n_dst_dev=None, stream=None):
    """bf16 rows x[dst2src[d]] quantized into q [n_dst, k] and scales (MXFP8: [n_dst, k/32])."""
    n_src, k = x.shape
    n_dst = dst2src.shape[0] if n_dst is None else n_dst
    _check("ftmoe_gather_quantize_act", lib().ftmoe_gather_quantize_act(
        _p(x), n_src, k, x.stride(0), _p(dst2src), n_dst, _p(n_dst_dev), fmt, _p(q), _p(scales), _stream(stream)))


def make_bank(q, scales, global_scale=None, fmt=FMT_FP8):
    """ExpertBank view of tensors q [E, n, k(/2)], scales, global_scale."""
    E, n, kk = q.shape
    k = 2 * kk if fmt == FMT_NVFP4 else kk
    return ExpertBank(fmt, E, n, k, _p(q), _p(scales), _p(global_scale))


def make_act(q, scales, global_scale=None, fmt=FMT_FP8):
    rows, kk = q.shape
    k = 2 * kk if fmt == FMT_NVFP4 else kk
    return Act(fmt, 0, rows, k, _p(q), _p(scales), _p(global_scale))


def grouped_routes(offsets):
    return Routes(ROUTES_GROUPED, 0, 0, _p(offsets), None)


def slot_routes(expert_ids):
    T, topk = expert_ids.shape
    return Routes(ROUTES_SLOTS, topk, T, None, _p(expert_ids))


def _tile(tok_tile=0, variant=0, wblocks=0, ctas=0):
    return Tile(tok_tile, variant, wblocks, ctas)


def ftmoe_grouped_gemm_gateup(act, routes, bank, out, tok_tile=0, variant=0, wblocks=0, ctas=0, stream=None):
    t = _tile(tok_tile, variant, wblocks, ctas)
    _check("ftmoe_grouped_gemm_gateup", lib().ftmoe_grouped_gemm_gateup(
        ctypes.byref(act), ctypes.byref(routes), ctypes.byref(bank), _p(out), out.stride(0),
        ctypes.byref(t), _stream(stream)))


def ftmoe_grouped_gemm_gateup_silu(act, routes, bank, q, scales, tok_tile=0, stream=None):
    t = _tile(tok_tile)
    _check("ftmoe_grouped_gemm_gateup_silu", lib().ftmoe_grouped_gemm_gateup_silu(
        ctypes.byref(act), ctypes.byref(routes), ctypes.byref(bank), _p(q), _p(scales),
        ctypes.byref(t), _stream(stream)))


def ftmoe_grouped_gemm_down(act, routes, bank, out, tok_tile=0, variant=0, wblocks=0, ctas=0, stream=None):
    t = _tile(tok_tile, variant, wblocks, ctas)
    _check("ftmoe_grouped_gemm_down", lib().ftmoe_grouped_gemm_down(
        ctypes.byref(act), ctypes.byref(routes), ctypes.byref(bank), _p(out), out.stride(0),
        ctypes.byref(t), _stream(stream)))


def ftmoe_silu_mul(gu, q, scales, global_scale=None, fmt=FMT_FP8, rows=None, rows_dev=None, stream=None):
    rows = gu.shape[0] if rows is None else rows
    inter = gu.shape[1] // 2
    _check("ftmoe_silu_mul", lib().ftmoe_silu_mul(
        _p(gu), rows, inter, gu.stride(0), _p(rows_dev), fmt, _p(q), _p(scales), _p(global_scale),
        _stream(stream)))


def out_dtype_code(out):
    """ftmoe_out_dtype of an output tensor (bf16, fp16 or fp32)."""
    if out.dtype not in _OUT_DTYPES:
        raise ValueError(f"output dtype {out.dtype} is not one of bf16, fp16, fp32")
    return _OUT_DTYPES[out.dtype]


def ftmoe_combine(y, expert_ids, weights, out, route2dst=None, stream=None):
    T, topk = expert_ids.shape
    H = out.shape[1]
    _check("ftmoe_combine", lib().ftmoe_combine(
        _p(y), y.stride(0), _p(route2dst), _p(expert_ids), _p(weights), T, topk, H, out_dtype_code(out),
        _p(out), out.stride(0), _stream(stream)))


def moe_shape(tokens, hidden, inter, topk, num_experts, fmt=FMT_FP8, tok_tile=0, path=0, out_dtype=OUT_BF16):
    return MoeShape(tokens, hidden, inter, topk, num_experts, fmt, tok_tile, path, out_dtype)


def _check_out(shape, out):
    if out_dtype_code(out) != shape.out_dtype:
        raise ValueError(f"output tensor is {out.dtype}, the shape says out_dtype {shape.out_dtype}")


def ftmoe_forward_workspace_bytes(shape):
    return int(lib().ftmoe_forward_workspace_bytes(ctypes.byref(shape)))


def ftmoe_forward_workspace_layout(shape):
    lay = WorkspaceLayout()
    _check("ftmoe_forward_workspace_layout",
           lib().ftmoe_forward_workspace_layout(ctypes.byref(shape), ctypes.byref(lay)))
    return {n: int(getattr(lay, n)) for n in _LAYOUT_FIELDS}


def ftmoe_moe_forward(shape, x, expert_ids, route_weights, bank_gateup, bank_down, out, workspace,
                      stream=None):
    _check_out(shape, out)
    args = MoeArgs(shape, _p(x), x.stride(0), _p(expert_ids), _p(route_weights), bank_gateup,
                   bank_down, _p(out), out.stride(0))
    _check("ftmoe_moe_forward", lib().ftmoe_moe_forward(
        ctypes.byref(args), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def ftmoe_moe_forward_noalloc(shape, x, expert_ids, route_weights, bank_gateup, bank_down, out, stream=None):
    """The fused forward with its intermediates in the library's own device array (no workspace)."""
    _check_out(shape, out)
    args = MoeArgs(shape, _p(x), x.stride(0), _p(expert_ids), _p(route_weights), bank_gateup,
                   bank_down, _p(out), out.stride(0))
    _check("ftmoe_moe_forward_noalloc", lib().ftmoe_moe_forward_noalloc(ctypes.byref(args), _stream(stream)))


def ftmoe_expert_slots(expert_ids, slot_expert, slot_usage, expert_slot, step, max_fetch, fetch_plan, n_fetch,
                       stream=None):
    """One step of the device-side expert-slot pool: expert_ids (int32, any shape) become slot
    ids in place; the pool state tensors are updated in place."""
    _check("ftmoe_expert_slots", lib().ftmoe_expert_slots(
        _p(expert_ids), expert_ids.numel(), _p(slot_expert), _p(slot_usage), slot_expert.numel(),
        _p(expert_slot), expert_slot.numel(), int(step), int(max_fetch), _p(fetch_plan), _p(n_fetch),
        _stream(stream)))


def ftmoe_selftest_wait_timeout(timeout_ns, elapsed_ns=None, stream=None):
    """One bounded pipeline wait that nothing completes, given up after timeout_ns."""
    _check("ftmoe_selftest_wait_timeout", lib().ftmoe_selftest_wait_timeout(
        int(timeout_ns), _p(elapsed_ns), _stream(stream)))


def ftmoe_selftest_shared_division(counts, stream=None):
    """The quantizers' division by a shared group scale against IEEE division on the device;
    counts (int64 tensor [2]) receives {quotients checked, quotients that differ}."""
    _check("ftmoe_selftest_shared_division", lib().ftmoe_selftest_shared_division(_p(counts), _stream(stream)))


def ftmoe_read_error_flags():
    v = ctypes.c_uint32(0)
    _check("ftmoe_read_error_flags", lib().ftmoe_read_error_flags(ctypes.byref(v)))
    return int(v.value)


# ---------------------------------------------------------------------------------
# allocation helpers (torch allocates; the library computes)
# ---------------------------------------------------------------------------------

def cdiv(a, b):
    return -(-a // b)


def quantize_act(x, fmt=FMT_FP8, stream=None):
    """bf16 [rows, k] -> (q, scales, global_scale) allocated with torch on x's device."""
    rows, k = x.shape
    dev = x.device
    if fmt == FMT_FP8:
        q = torch.empty(rows, k, dtype=torch.uint8, device=dev)
        s = torch.empty(rows, cdiv(k, 128), dtype=torch.float32, device=dev)
        ftmoe_quantize_act(x, q, s, None, fmt, stream=stream)
        return q, s, None
    if fmt == FMT_MXFP8:
        q = torch.empty(rows, k, dtype=torch.uint8, device=dev)
        s = torch.empty(rows, k // 32, dtype=torch.uint8, device=dev)
        ftmoe_quantize_act(x, q, s, None, fmt, stream=stream)
        return q, s, None
    q = torch.empty(rows, k // 2, dtype=torch.uint8, device=dev)
    s = torch.empty(rows, k // 16, dtype=torch.uint8, device=dev)
    g = torch.empty(1, dtype=torch.float32, device=dev)
    ftmoe_quantize_act(x, q, s, g, fmt, stream=stream)
    return q, s, g


def quantize_weights(w, fmt=FMT_FP8, stream=None):
    """float32 [E, n, k] -> (q, scales, global_scale) in the ExpertBank layout."""
    E, n, k = w.shape
    dev = w.device
    if fmt == FMT_FP8:
        q = torch.empty(E, n, k, dtype=torch.uint8, device=dev)
        s = torch.empty(E, cdiv(n, 128), cdiv(k, 128), dtype=torch.float32, device=dev)
        ftmoe_quantize_weights(w, q, s, None, fmt, stream=stream)
        return q, s, None
    if fmt == FMT_MXFP8:
        q = torch.empty(E, n, k, dtype=torch.uint8, device=dev)
        s = torch.empty(E, n, k // 32, dtype=torch.uint8, device=dev)
        ftmoe_quantize_weights(w, q, s, None, fmt, stream=stream)
        return q, s, None
    q = torch.empty(E, n, k // 2, dtype=torch.uint8, device=dev)
    s = torch.empty(E, n, k // 16, dtype=torch.uint8, device=dev)
    g = torch.empty(E, dtype=torch.float32, device=dev)
    ftmoe_quantize_weights(w, q, s, g, fmt, stream=stream)
    return q, s, g

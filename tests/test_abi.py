"""The C ABI library builds, loads and exports every symbol include/ftmoe.h declares;
host-side argument checks answer without touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ftmoe.h")


@pytest.fixture(scope="module")
def ft():
    from block_quantized_moe_gb300 import build_lib
    build_lib.build()
    import block_quantized_moe_gb300 as ft
    ft.lib()
    return ft


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ftmoe_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for want in ["ftmoe_quantize_act", "ftmoe_gather_rows_scales", "ftmoe_grouped_gemm_gateup",
                 "ftmoe_silu_mul", "ftmoe_grouped_gemm_down", "ftmoe_combine", "ftmoe_moe_forward",
                 "ftmoe_segment_routes", "ftmoe_pick_tile"]:
        assert want in names


def test_library_exports_every_declared_symbol(ft):
    lib = ctypes.CDLL(ft.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    bound = {n for n, _, _ in ft._SIGNATURES}
    assert set(declared_functions()) <= bound


def test_pick_tile_host_function(ft):
    assert ft.ftmoe_pick_tile(1536, 256) == 16
    assert ft.ftmoe_pick_tile(6144, 256) == 32
    assert ft.ftmoe_pick_tile(24576, 256) == 128
    assert ft.ftmoe_pick_tile(64, 64) == 16
    with pytest.raises(ft.FtmoeError):
        ft.ftmoe_pick_tile(10, 0)


def test_status_strings(ft):
    assert ft.lib().ftmoe_status_string(0) == b"ok"
    assert ft.lib().ftmoe_status_string(1) == b"invalid argument"


def test_invalid_arguments_rejected_on_host(ft):
    L = ft.lib()
    # NULL input with rows > 0
    assert L.ftmoe_quantize_act(None, 4, 128, 128, 0, None, None, None, None) == ft.FTMOE_INVALID_ARG
    # ld < k
    assert L.ftmoe_quantize_act(ctypes.c_void_p(16), 4, 128, 64, 0, ctypes.c_void_p(16),
                                ctypes.c_void_p(16), None, None) == ft.FTMOE_INVALID_ARG
    # unknown format
    assert L.ftmoe_quantize_act(ctypes.c_void_p(16), 4, 128, 128, 7, ctypes.c_void_p(16),
                                ctypes.c_void_p(16), None, None) == ft.FTMOE_INVALID_ARG
    # NVFP4 needs k % 32 == 0 and a global scale
    assert L.ftmoe_quantize_act(ctypes.c_void_p(16), 4, 48, 48, 1, ctypes.c_void_p(16),
                                ctypes.c_void_p(16), ctypes.c_void_p(16), None) == ft.FTMOE_INVALID_ARG
    # zero rows: OK without any launch
    assert L.ftmoe_quantize_act(None, 0, 128, 128, 0, None, None, None, None) == ft.FTMOE_OK
    assert L.ftmoe_gather_rows_scales(None, None, 5, 896, 28, None, 0, None, None, None, None) == ft.FTMOE_OK
    assert L.ftmoe_gather_rows_scales(None, None, 5, 896, 28, None, 3, None, None, None, None) == ft.FTMOE_INVALID_ARG
    assert L.ftmoe_segment_routes(None, 4, 2, 0, None, None, None, None, None) == ft.FTMOE_INVALID_ARG
    assert L.ftmoe_combine(None, 16, None, None, None, 0, 2, 16, 0, None, 16, None) == ft.FTMOE_OK
    assert L.ftmoe_combine(None, 8, None, None, None, 2, 2, 16, 0, None, 16, None) == ft.FTMOE_INVALID_ARG
    # output element types: bf16, fp16, fp32; anything else is refused
    for d in (ft.OUT_BF16, ft.OUT_FP16, ft.OUT_FP32):
        assert L.ftmoe_combine(None, 16, None, None, None, 0, 2, 16, d, None, 16, None) == ft.FTMOE_OK
    assert L.ftmoe_combine(None, 16, None, None, None, 0, 2, 16, 3, None, 16, None) == ft.FTMOE_INVALID_ARG
    # the expert-slot pool: sizes and the pointers it needs are checked on the host
    fake = ctypes.c_void_p(256)
    assert L.ftmoe_expert_slots(fake, 4, fake, fake, 0, fake, 8, 0, 1, fake, fake, None) == ft.FTMOE_INVALID_ARG
    assert L.ftmoe_expert_slots(fake, 4, fake, fake, 4, fake, 20000, 0, 1, fake, fake, None) == ft.FTMOE_INVALID_ARG
    assert L.ftmoe_expert_slots(fake, 20000, fake, fake, 4, fake, 8, 0, 1, fake, fake, None) == ft.FTMOE_INVALID_ARG
    assert L.ftmoe_expert_slots(fake, 4, fake, fake, 4, fake, 8, 0, 2, None, fake, None) == ft.FTMOE_INVALID_ARG
    # the wait self-test takes a limit of 1 us .. 1 s
    assert L.ftmoe_selftest_wait_timeout(999, None, None) == ft.FTMOE_INVALID_ARG
    assert L.ftmoe_selftest_wait_timeout(2 * 10 ** 9, None, None) == ft.FTMOE_INVALID_ARG
    assert L.ftmoe_selftest_shared_division(None, None) == ft.FTMOE_INVALID_ARG


def test_forward_workspace_layout(ft):
    s = ft.moe_shape(8, 4096, 1024, 8, 64, path=2)
    n = ft.ftmoe_forward_workspace_bytes(s)
    lay = ft.ftmoe_forward_workspace_layout(s)
    assert lay["total"] == n
    R = 64
    assert lay["gateup_bytes"] == R * 2 * 1024 * 4 and lay["down_bytes"] == R * 4096 * 4
    assert lay["act_q_bytes"] == R * 1024 and lay["act_scales_bytes"] == R * 8 * 4
    fused = ft.ftmoe_forward_workspace_layout(ft.moe_shape(8, 4096, 1024, 8, 64, path=3))
    assert fused["gateup"] == 0 and fused["gateup_bytes"] == 0  # no fp32 gate/up rows
    assert fused["total"] == n - R * 2 * 1024 * 4
    for key in ("x_q", "x_scales", "gateup", "act_q", "act_scales", "down"):
        assert lay[key] % 256 == 0
    assert lay["rows_q"] > 0  # eight tokens take the grouped path: gather buffers
    auto2 = ft.ftmoe_forward_workspace_layout(ft.moe_shape(2, 4096, 1024, 8, 64))
    assert auto2["rows_q"] == 0 and auto2["partials_bytes"] > 0  # automatic at 2 tokens: fused decode
    auto16 = ft.ftmoe_forward_workspace_layout(ft.moe_shape(16, 4096, 1024, 8, 64))
    assert auto16["rows_q"] > 0  # beyond 8 tokens: the grouped path
    slot = ft.ftmoe_forward_workspace_layout(ft.moe_shape(2, 4096, 1024, 8, 64, path=1))
    assert slot["rows_q"] == 0 and slot["dst2src"] == 0  # route-slot path: no gather buffers
    g = ft.ftmoe_forward_workspace_layout(ft.moe_shape(256, 7168, 2048, 6, 256))
    assert g["rows_q"] > 0 and g["dst2src"] > 0
    bad = ft.moe_shape(8, 4096, 1024, 8, 64, tok_tile=48)
    assert ft.ftmoe_forward_workspace_bytes(bad) == 0
    assert ft.ftmoe_forward_workspace_bytes(ft.moe_shape(8, 4096, 1024, 8, 64, out_dtype=3)) == 0
    # the output element type does not change the workspace
    sizes = {ft.ftmoe_forward_workspace_bytes(ft.moe_shape(8, 4096, 1024, 8, 64, out_dtype=d))
             for d in (ft.OUT_BF16, ft.OUT_FP16, ft.OUT_FP32)}
    assert len(sizes) == 1 and sizes.pop() > 0


def test_binding_checks_the_output_tensor_against_the_shape(ft):
    import torch
    shape = ft.moe_shape(2, 256, 128, 2, 4, out_dtype=ft.OUT_FP16)
    with pytest.raises(ValueError):
        ft._check_out(shape, torch.empty(2, 256, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        ft.out_dtype_code(torch.empty(2, 256, dtype=torch.float64))
    ft._check_out(shape, torch.empty(2, 256, dtype=torch.float16))


def test_forward_rejects_inconsistent_banks(ft):
    # Every call here must be refused by the host checks: the pointers are fake, so a call
    # that got as far as a launch would fault on a GPU.
    s = ft.moe_shape(2, 256, 128, 2, 4)
    bank_gu = ft.ExpertBank(0, 4, 300, 256, ctypes.c_void_p(256), ctypes.c_void_p(256), None)  # n != 2I
    bank_dn = ft.ExpertBank(0, 4, 256, 128, ctypes.c_void_p(256), ctypes.c_void_p(256), None)
    args = ft.MoeArgs(s, ctypes.c_void_p(256), 256, ctypes.c_void_p(256), ctypes.c_void_p(256),
                      bank_gu, bank_dn, ctypes.c_void_p(256), 256)
    assert ft.lib().ftmoe_moe_forward(ctypes.byref(args), ctypes.c_void_p(256), 1 << 30, None) == ft.FTMOE_INVALID_ARG
    args.w_gateup.n = 2 * 128
    args.w_down.num_experts = 5  # bank E != shape E
    assert ft.lib().ftmoe_moe_forward(ctypes.byref(args), ctypes.c_void_p(256), 1 << 30, None) == ft.FTMOE_INVALID_ARG
    args.w_down.num_experts = 4
    assert ft.lib().ftmoe_moe_forward(ctypes.byref(args), ctypes.c_void_p(256), 16, None) == ft.FTMOE_WORKSPACE_TOO_SMALL


def test_automatic_forward_path_choice(ft):
    # the fused decode path up to 8 tokens (FP8); beyond, SiLU-and-mul fused into the gate/up
    # GEMM (no fp32 gate/up buffer) where the token tile is at most 64 and
    # min(T * topk, E) * I / 128 >= 2048; the separate kernel otherwise and for NVFP4
    lay = ft.ftmoe_forward_workspace_layout
    assert lay(ft.moe_shape(8, 4096, 1024, 8, 64))["partials_bytes"] > 0         # fused decode path
    assert lay(ft.moe_shape(16, 4096, 1024, 8, 64))["gateup_bytes"] > 0
    assert lay(ft.moe_shape(4096, 7168, 2048, 6, 256))["gateup_bytes"] > 0       # tile 128
    assert lay(ft.moe_shape(4096, 7168, 2048, 6, 256, tok_tile=32))["gateup_bytes"] == 0
    assert lay(ft.moe_shape(1024, 7168, 2048, 6, 256))["gateup_bytes"] == 0
    assert lay(ft.moe_shape(256, 7168, 2048, 6, 256))["gateup_bytes"] == 0
    assert lay(ft.moe_shape(8, 4096, 1024, 8, 64, path=3))["gateup_bytes"] == 0
    assert lay(ft.moe_shape(1, 4096, 1024, 8, 64))["partials_bytes"] > 0
    assert lay(ft.moe_shape(1, 2048, 768, 8, 8))["partials_bytes"] > 0
    assert lay(ft.moe_shape(1, 4096, 1024, 8, 64, path=2))["gateup_bytes"] > 0
    assert lay(ft.moe_shape(8, 4096, 1024, 8, 64, fmt=ft.FMT_NVFP4))["gateup_bytes"] > 0
    assert lay(ft.moe_shape(8, 4096, 1024, 8, 64, path=2))["gateup_bytes"] > 0
    assert lay(ft.moe_shape(2048, 7168, 2048, 6, 2048))["gateup_bytes"] > 0  # beyond the GEMM's 1024 experts
    assert lay(ft.moe_shape(1, 2048, 768, 8, 8, path=3))["gateup_bytes"] == 0
    # the combine inside the down GEMM (arrival counters, one word per token and 128 columns):
    # path 5 only (FP8, token tile 64 or 128); the automatic path keeps the combine kernel
    assert lay(ft.moe_shape(4096, 7168, 2048, 6, 256))["counters_bytes"] == 0
    assert lay(ft.moe_shape(4096, 7168, 2048, 6, 256, path=5))["counters_bytes"] == 4096 * 56 * 4
    assert lay(ft.moe_shape(4096, 7168, 2048, 6, 256, path=3))["counters_bytes"] == 0
    assert lay(ft.moe_shape(1024, 7168, 2048, 6, 256, path=5))["counters_bytes"] == 0         # tile 32
    assert lay(ft.moe_shape(1024, 7168, 2048, 6, 256, tok_tile=64, path=5))["counters_bytes"] == 1024 * 56 * 4
    assert lay(ft.moe_shape(4096, 7168, 2048, 6, 256, fmt=ft.FMT_NVFP4, path=5))["counters_bytes"] == 0
    assert lay(ft.moe_shape(4096, 7168, 2048, 6, 256, fmt=ft.FMT_MXFP8, path=5))["counters_bytes"] == 0
    assert lay(ft.moe_shape(8, 4096, 1024, 8, 64, path=5))["counters_bytes"] == 0             # tile 16
    assert lay(ft.moe_shape(4096, 7168, 2048, 9, 256, path=5))["counters_bytes"] == 0         # topk > 8
    with pytest.raises(ft.FtmoeError):
        lay(ft.moe_shape(8, 4096, 1024, 8, 64, path=6))


def test_fused_decode_workspace(ft):
    # path 4: token rows padded to 16, the intermediate and the down rows per route, the
    # gate/up partial sums and the arrival counters; no gather or fp32 gate/up rows
    lay = ft.ftmoe_forward_workspace_layout
    d = lay(ft.moe_shape(8, 4096, 1024, 8, 64, path=4))
    R = 64
    assert d["gateup_bytes"] == 0 and d["rows_q"] == 0 and d["dst2src"] == 0
    assert d["act_q_bytes"] == R * 1024 and d["act_scales_bytes"] == R * 8 * 4 and d["down_bytes"] == R * 4096 * 4
    assert d["partials_bytes"] > 0 and d["counters_bytes"] == 4 * (64 * 8 + 64 + 8 * 32)
    for key in ("x_q", "x_scales", "act_q", "act_scales", "down", "partials", "counters"):
        assert d[key] % 256 == 0
    assert d["total"] <= 16 << 20  # the decode shapes still fit the allocation-free forward's array
    # outside its limits (more than 8 tokens, NVFP4, I > 2048) the path is unsupported: the
    # layout falls back to another path's and the forward refuses path 4
    assert lay(ft.moe_shape(9, 4096, 1024, 8, 64, path=4))["partials_bytes"] == 0
    assert lay(ft.moe_shape(8, 4096, 1024, 8, 64, path=4, fmt=ft.FMT_NVFP4))["partials_bytes"] == 0
    assert lay(ft.moe_shape(8, 4096, 4096, 8, 64, path=4))["partials_bytes"] == 0


def test_two_block_and_fused_gemm_host_checks(ft):
    # Every call here must be refused (or finish without a launch) on the host: the
    # pointers are fake, so a call that reached a kernel would fault on a GPU.
    L = ft.lib()
    fake = ctypes.c_void_p(256)
    bank = ft.ExpertBank(ft.FMT_FP8, 4, 384, 256, fake, fake, None)      # 2I = 384: not whole 256-row pairs
    act = ft.Act(ft.FMT_FP8, 0, 8, 256, fake, fake, None)
    rt = ft.Routes(ft.ROUTES_GROUPED, 0, 0, fake, None)
    t = ft.Tile(16, 0, 0, 0)
    silu = L.ftmoe_grouped_gemm_gateup_silu
    assert silu(ctypes.byref(act), ctypes.byref(rt), ctypes.byref(bank), fake, fake, ctypes.byref(t),
                None) == ft.FTMOE_UNSUPPORTED
    bank.n = 512
    bank.k = 200  # K not a whole number of 128-wide blocks
    act.k = 200
    assert silu(ctypes.byref(act), ctypes.byref(rt), ctypes.byref(bank), fake, fake, ctypes.byref(t),
                None) == ft.FTMOE_UNSUPPORTED
    bank.k = act.k = 256
    assert silu(ctypes.byref(act), ctypes.byref(rt), ctypes.byref(bank), None, fake, ctypes.byref(t),
                None) == ft.FTMOE_INVALID_ARG
    slots = ft.Routes(ft.ROUTES_SLOTS, 8, 1, None, fake)  # the fused GEMM takes grouped rows only
    assert silu(ctypes.byref(act), ctypes.byref(slots), ctypes.byref(bank), fake, fake, ctypes.byref(t),
                None) == ft.FTMOE_INVALID_ARG
    nv = ft.ExpertBank(ft.FMT_NVFP4, 4, 512, 256, fake, fake, fake)
    act_nv = ft.Act(ft.FMT_NVFP4, 0, 8, 256, fake, fake, fake)
    assert silu(ctypes.byref(act_nv), ctypes.byref(rt), ctypes.byref(nv), fake, fake, ctypes.byref(t),
                None) == ft.FTMOE_UNSUPPORTED
    act.rows = 0  # zero rows: OK without a launch
    assert silu(ctypes.byref(act), ctypes.byref(rt), ctypes.byref(bank), fake, fake, ctypes.byref(t),
                None) == ft.FTMOE_OK
    # ftmoe_tile.wblocks outside {0, 1, 2}, ctas outside {0, 1, 2}, and a CTA pair asked for
    # two weight blocks per CTA are refused by the GEMM entry points
    act.rows = 8
    for bad in (ft.Tile(16, 2, 3, 0), ft.Tile(128, 2, 0, 3), ft.Tile(128, 2, 0, -1), ft.Tile(128, 2, 2, 2)):
        for fn in (L.ftmoe_grouped_gemm_gateup, L.ftmoe_grouped_gemm_down):
            assert fn(ctypes.byref(act), ctypes.byref(rt), ctypes.byref(bank), fake, 512, ctypes.byref(bad),
                      None) == ft.FTMOE_INVALID_ARG

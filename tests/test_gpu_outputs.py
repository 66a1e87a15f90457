"""Output element types of the forward and the combine (bf16, fp16, fp32), and the bounded
pipeline wait made to run out, through the C ABI.

The FreeToken decode page's validation covers bf16, fp16 and fp32 outputs. The combine
accumulates in fp32 whatever the output type, so the three outputs of one forward are the
same fp32 sums: fp32 stores them as they are, bf16 and fp16 round them to nearest even once.
That gives exact relations between the three, beside the oracle comparison of each.
"""
import numpy as np
import pytest
import torch

import synth
from common import Problem

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ft():
    import block_quantized_moe_gb300 as ft
    ft.lib()
    return ft


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16, torch.float32])
def test_combine_single_route_of_weight_one_is_the_rounded_row(ft, dtype):
    # one active slot of weight 1 per token: the output is that route's row in the output type
    T, k, H = 5, 4, 384
    y = (torch.randn(T * k, H, generator=torch.Generator().manual_seed(3)) * 7).to(DEV)
    ids = torch.full((T, k), -1, dtype=torch.int32, device=DEV)
    slot = torch.tensor([0, 3, 1, 2, 3], device=DEV)
    ids[torch.arange(T, device=DEV), slot] = 1
    w = torch.full((T, k), float("nan"), device=DEV)  # inactive weights are never read
    w[torch.arange(T, device=DEV), slot] = 1.0
    out = torch.full((T, H + 8), -1.0, device=DEV).to(dtype)[:, :H]  # row stride H + 8
    ft.ftmoe_combine(y, ids, w, out)
    torch.cuda.synchronize()
    rows = y.view(T, k, H)[torch.arange(T, device=DEV), slot]
    assert torch.equal(out, rows.to(dtype))


@pytest.mark.parametrize("path", [0, 1, 3, 4])
def test_forward_output_types_agree_and_match_the_oracle(ft, path):
    T, H, I, E, k = 8, 1024, 512, 16, 4
    p = Problem(T, H, I, E, k, seed=0xF7E0_0F16, active=[4, 3, 0, 4, 2, 4, 1, 4])
    o32, _, _ = p.forward(path=path, out_dtype=torch.float32)
    o16, _, _ = p.forward(path=path, out_dtype=torch.float16)
    obf, _, _ = p.forward(path=path, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert ft.ftmoe_read_error_flags() == 0
    # the same fp32 sums, rounded to nearest even once for the 16-bit types
    assert torch.equal(o16, o32.to(torch.float16))
    assert torch.equal(obf, o32.to(torch.bfloat16))
    for out in (o32, o16, obf):
        p.check(out)
    inactive = (p.ids < 0).all(dim=1)
    assert torch.all(o32[inactive] == 0)


def test_forward_refuses_an_unknown_output_type(ft):
    p = Problem(2, 256, 128, 4, 2, seed=5)
    shape = ft.moe_shape(2, 256, 128, 2, 4, out_dtype=3)
    out = torch.empty(2, 256, dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=DEV)
    args = ft.MoeArgs(shape, ft._p(p.x), p.x.stride(0), ft._p(p.ids), ft._p(p.w), p.bank_gu, p.bank_dn,
                      ft._p(out), out.stride(0))
    import ctypes
    assert ft.lib().ftmoe_moe_forward(ctypes.byref(args), ft._p(ws), ws.numel(), None) == ft.FTMOE_INVALID_ARG


def test_bounded_wait_runs_out_and_the_context_stays_usable(ft):
    # a pipeline wait that nothing completes gives up after its limit (1 ms here), raises
    # FTMOE_ERR_WAIT_TIMEOUT in the device error word and lets the kernel return: no trap,
    # no hang, and the next calls on the same context run normally
    assert ft.ftmoe_read_error_flags() == 0
    elapsed = torch.zeros(1, dtype=torch.int64, device=DEV)
    ft.ftmoe_selftest_wait_timeout(1_000_000, elapsed)
    torch.cuda.synchronize()
    assert ft.ftmoe_read_error_flags() == ft.ERR_WAIT_TIMEOUT
    ns = int(elapsed.item())
    assert 1_000_000 <= ns < 100_000_000, ns
    assert ft.ftmoe_read_error_flags() == 0  # reading clears the word
    p = Problem(2, 256, 128, 4, 2, seed=11)
    out, _, _ = p.forward()
    torch.cuda.synchronize()
    assert ft.ftmoe_read_error_flags() == 0
    p.check(out)

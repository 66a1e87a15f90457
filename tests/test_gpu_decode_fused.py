"""The fused decode path (path 4: one persistent kernel for gate/up, SiLU-and-mul with FP8
re-quantization, down and the combine, after a launch that quantizes the token rows) against
the oracle, through the C ABI.

Beyond the decode workloads of test_gpu_decode.py (which run path 4 beside the other paths):
random route sets with mixed active counts, K-block counts that are not multiples of the TMA
stage (one- and two-K-block stages), a token that lists one expert twice, repeated calls
giving identical bits, and batch invariance -- a token's output does not depend on which
experts the other tokens of the call activate, because the gate/up chunking and the order of
its sums are fixed by the shape.
"""
import pytest
import torch

import synth
from tests.common import Problem

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ft():
    import block_quantized_moe_gb300 as ft
    ft.lib()
    return ft


def test_random_route_sets_against_the_oracle(ft):
    T, H, I, E, k = 8, 2048, 768, 32, 8
    p = Problem(T, H, I, E, k, seed=0xDEC0DE)
    for i in range(6):
        active = [(i * 3 + t * 5) % (k + 1) for t in range(T)]
        ids = synth.routes(T, k, E, 700 + i, active_per_token=active, device=DEV)
        x = synth.activations_bf16(T, H, 700 + i, DEV)
        w = synth.routing_weights(T, k, 700 + i, DEV)
        w = torch.where(ids >= 0, w, torch.full_like(w, float("nan")))  # never read
        out, _, _ = p.forward(path=4, ids=ids, weights=w, x=x)
        torch.cuda.synchronize()
        assert ft.ftmoe_read_error_flags() == 0
        p.check(out, ids=ids, weights=w, x=x)
        assert torch.all(out[(ids < 0).all(dim=1)] == 0)


@pytest.mark.parametrize("T,H,I,E,k", [
    (3, 384, 256, 5, 3),     # three K blocks: one-K-block stages, two-K-block down
    (5, 640, 384, 9, 4),     # five and three K blocks
    (2, 256, 128, 4, 2),     # one intermediate block
    (8, 1024, 2048, 16, 4),  # the largest intermediate the path takes
])
def test_odd_shapes_against_the_oracle(ft, T, H, I, E, k):
    p = Problem(T, H, I, E, k, seed=T * 131 + H)
    out, _, _ = p.forward(path=4)
    torch.cuda.synchronize()
    assert ft.ftmoe_read_error_flags() == 0
    p.check(out)


def test_a_token_listing_one_expert_twice(ft):
    # each listing is a route of its own (the oracle evaluates every route independently)
    T, H, I, E, k = 2, 512, 256, 6, 4
    p = Problem(T, H, I, E, k, seed=17)
    ids = torch.tensor([[3, 3, 1, -1], [3, 5, -1, 0]], dtype=torch.int32, device=DEV)
    out, _, _ = p.forward(path=4, ids=ids)
    torch.cuda.synchronize()
    assert ft.ftmoe_read_error_flags() == 0
    p.check(out, ids=ids)


def test_repeated_calls_give_identical_bits(ft):
    T, H, I, E, k = 8, 4096, 1024, 64, 8
    p = Problem(T, H, I, E, k, seed=0xF7E00002, active=[8, 5, 0, 2, 8, 1, 7, 3])
    a, ws, _ = p.forward(path=4)
    b, _, _ = p.forward(path=4, ws=ws)
    c, _, _ = p.forward(path=4)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_batch_invariance(ft):
    # token 0 keeps its routes and input while the other tokens switch to other experts:
    # its output row stays the same bits
    T, H, I, E, k = 8, 2048, 768, 32, 8
    p = Problem(T, H, I, E, k, seed=0xBA7C)
    rows = []
    for i in range(3):
        ids = synth.routes(T, k, E, 900 + i, device=DEV)
        ids[0] = p.ids[0]
        x = synth.activations_bf16(T, H, 900 + i, DEV)
        x[0] = p.x[0]
        w = synth.routing_weights(T, k, 900 + i, DEV)
        w[0] = p.w[0]
        out, _, _ = p.forward(path=4, ids=ids, weights=w, x=x)
        torch.cuda.synchronize()
        rows.append(out[0].clone())
    for r in rows[1:]:
        assert torch.equal(r.view(torch.int16), rows[0].view(torch.int16))


def test_outside_the_limits_path_4_is_refused(ft):
    p = Problem(9, 256, 128, 4, 2, seed=3)  # nine tokens
    with pytest.raises(ft.FtmoeError) as ei:
        p.forward(path=4)
    assert ei.value.status == ft.FTMOE_UNSUPPORTED

"""The device-side expert-slot pool (ftmoe_expert_slots) in lockstep with the oracle's model of
the contract, call by call, through the C ABI -- the test design the FreeToken cache page
describes (Test: the kernel against a model of the LRU contract, from an empty to a full pool,
for pools that fit one tile and pools that do not). Every output is compared bit for bit: the
rewritten route ids, the copy plan and its length, and the whole pool state."""
import random

import numpy as np
import pytest
import torch

from oracle import slots as P

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def ft():
    import block_quantized_moe_gb300 as ft
    ft.lib()
    return ft


@pytest.mark.parametrize("S,E,R,steps", [(8, 64, 16, 60), (3000, 4096, 256, 12), (256, 256, 6144, 6),
                                         (1, 5, 4, 20)])
def test_lockstep_with_the_oracle(ft, S, E, R, steps):
    rng = random.Random(S * 7 + R)
    se, su, es = P.pool_state(S, E)
    d_se = torch.full((S,), -1, dtype=torch.int32, device=DEV)
    d_su = torch.full((S,), -1, dtype=torch.int64, device=DEV)
    d_es = torch.full((E,), -1, dtype=torch.int32, device=DEV)
    plan = torch.full((S + 4, 2), -7, dtype=torch.int32, device=DEV)
    nf = torch.zeros(1, dtype=torch.int32, device=DEV)
    for st in range(steps):
        # a working set that drifts, so that the pool fills, hits and evicts
        hot = rng.randrange(0, E)
        routes = [(hot + rng.randrange(-2, 3 * S // 2 + 3)) % E if rng.random() > 0.1 else -1 for _ in range(R)]
        max_fetch = rng.randrange(0, min(S, 40) + 2)
        ids = torch.tensor(routes, dtype=torch.int32, device=DEV)
        ft.ftmoe_expert_slots(ids, d_se, d_su, d_es, st, max_fetch, plan, nf)
        torch.cuda.synchronize()
        want_ids, want_plan, _ = P.step(routes, se, su, es, st, max_fetch)
        n = int(nf.item())
        assert n == len(want_plan), st
        assert ids.cpu().tolist() == want_ids, st
        assert [tuple(p) for p in plan[:n].cpu().tolist()] == want_plan, st
        assert d_se.cpu().tolist() == se and d_su.cpu().tolist() == su and d_es.cpu().tolist() == es, st
    assert ft.ftmoe_read_error_flags() == 0


def test_out_of_range_ids_are_inactive_and_flagged(ft):
    S, E = 4, 6
    d_se = torch.full((S,), -1, dtype=torch.int32, device=DEV)
    d_su = torch.full((S,), -1, dtype=torch.int64, device=DEV)
    d_es = torch.full((E,), -1, dtype=torch.int32, device=DEV)
    plan = torch.zeros(S, 2, dtype=torch.int32, device=DEV)
    nf = torch.zeros(1, dtype=torch.int32, device=DEV)
    ft.ftmoe_read_error_flags()
    ids = torch.tensor([2, 9, -3, 2, 5], dtype=torch.int32, device=DEV)
    ft.ftmoe_expert_slots(ids, d_se, d_su, d_es, 0, 4, plan, nf)
    flags = ft.ftmoe_read_error_flags()
    assert flags & ft.ERR_EXPERT_ID_RANGE
    assert ids.cpu().tolist() == [0, -1, -1, 0, 1] and int(nf.item()) == 2


def test_the_slot_ids_feed_the_forward(ft):
    # the pool's output is the forward's expert_ids over a bank laid out by slot: routes whose
    # expert was not fetched are -1 (inactive here), the rest read the expert's weights from
    # its slot. The output equals the forward over expert ids with the unfetched routes set
    # to -1 and the bank indexed by expert.
    from tests.common import Problem
    T, H, I, E, k, S = 4, 512, 256, 12, 4, 6
    p = Problem(T, H, I, E, k, seed=3)
    d_se = torch.full((S,), -1, dtype=torch.int32, device=DEV)
    d_su = torch.full((S,), -1, dtype=torch.int64, device=DEV)
    d_es = torch.full((E,), -1, dtype=torch.int32, device=DEV)
    plan = torch.zeros(S, 2, dtype=torch.int32, device=DEV)
    nf = torch.zeros(1, dtype=torch.int32, device=DEV)
    slots = p.ids.clone()
    ft.ftmoe_expert_slots(slots, d_se, d_su, d_es, 0, 5, plan, nf)
    torch.cuda.synchronize()
    held = d_se.cpu().numpy()
    # the slot bank: slot s holds the weights of expert held[s] (what the caller's copy plan moves)
    order = torch.tensor([e if e >= 0 else 0 for e in held], dtype=torch.long, device=DEV)
    # the bank structs hold raw pointers: keep the slot-ordered tensors alive
    keep = [t[order].contiguous() for t in (p.gq, p.gs, p.dq, p.ds)]
    bank_gu = ft.make_bank(keep[0], keep[1])
    bank_dn = ft.make_bank(keep[2], keep[3])
    shape = ft.moe_shape(T, H, I, k, S, path=2)
    ws = torch.empty(ft.ftmoe_forward_workspace_bytes(shape), dtype=torch.uint8, device=DEV)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=DEV)
    ft.ftmoe_moe_forward(shape, p.x, slots, p.w, bank_gu, bank_dn, out, ws)
    ids_expert = torch.where(slots >= 0, p.ids, torch.full_like(p.ids, -1))
    ref, _, _ = p.forward(path=2, ids=ids_expert)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert np.all(held[slots[slots >= 0].cpu().numpy()] == p.ids[slots >= 0].cpu().numpy())

"""Pins of the expert-slot pool oracle (oracle/slots.py): a worked example checked by hand,
closed-form cases, and invariants checked on random step sequences against an independent
formulation of the victim choice (the minimum of (usage, slot) pairs), so that a plausible
mistake -- ties to the highest slot, evicting a slot used this step, fetching a repeated
expert twice, rewriting routes before the fetches -- fails one of them."""
import random

from oracle import slots as P


def test_worked_example():
    # slots 0..3 hold experts 10..13, last used at steps 5, 2, 2, 7; step 8 asks for 11
    # (resident in slot 1), then 20 and 21 (missing), and may fetch both
    slot_expert, usage, expert_slot = P.pool_state(4, 32)
    for s, (e, u) in enumerate(zip((10, 11, 12, 13), (5, 2, 2, 7))):
        slot_expert[s], usage[s], expert_slot[e] = e, u, s
    ids, plan, bad = P.step([11, 20, -1, 21, 20], slot_expert, usage, expert_slot, 8, 2)
    # 11 hits slot 1 (now used at step 8). 20 takes the least recently used slot not used in
    # step 8: slot 2 (usage 2; slot 1 also had 2 but is now 8). 21 then takes slot 0 (5 < 7).
    assert plan == [(2, 20), (0, 21)]
    assert ids == [1, 2, -1, 0, 2]
    assert slot_expert == [21, 11, 20, 13] and usage == [8, 8, 8, 7]
    assert expert_slot[10] == -1 and expert_slot[12] == -1 and bad == []


def test_empty_pool_fills_the_lowest_slots_first():
    slot_expert, usage, expert_slot = P.pool_state(5, 9)
    ids, plan, _ = P.step([4, 7, 4, 2], slot_expert, usage, expert_slot, 0, 8)
    assert plan == [(0, 4), (1, 7), (2, 2)] and ids == [0, 1, 0, 2]
    # the next step's miss evicts nothing while empty slots (usage -1) remain
    ids, plan, _ = P.step([8], slot_expert, usage, expert_slot, 1, 1)
    assert plan == [(3, 8)] and ids == [3]


def test_no_fetch_budget_leaves_misses_unserved():
    slot_expert, usage, expert_slot = P.pool_state(2, 4)
    P.step([0, 1], slot_expert, usage, expert_slot, 0, 2)
    ids, plan, _ = P.step([2, 0, 3], slot_expert, usage, expert_slot, 1, 0)
    assert plan == [] and ids == [-1, 0, -1] and slot_expert == [0, 1]


def test_slots_used_in_the_step_are_never_victims():
    # two slots, both hit in this step: a third expert cannot be placed
    slot_expert, usage, expert_slot = P.pool_state(2, 4)
    P.step([0, 1], slot_expert, usage, expert_slot, 0, 2)
    ids, plan, _ = P.step([1, 2, 0], slot_expert, usage, expert_slot, 1, 4)
    assert plan == [] and ids == [1, -1, 0]
    # one slot hit: the other is the only candidate
    ids, plan, _ = P.step([3, 1], slot_expert, usage, expert_slot, 2, 4)
    assert plan == [(0, 3)] and ids == [0, 1]


def test_out_of_range_ids_are_inactive_and_reported():
    slot_expert, usage, expert_slot = P.pool_state(3, 4)
    ids, plan, bad = P.step([1, 9, -5, 1], slot_expert, usage, expert_slot, 0, 3)
    assert ids == [0, -1, -1, 0] and plan == [(0, 1)] and bad == [9]


def test_random_sequences_keep_the_invariants():
    rng = random.Random(7)
    for S, E, R in ((8, 20, 16), (3, 6, 8), (16, 64, 48), (1, 3, 4)):
        slot_expert, usage, expert_slot = P.pool_state(S, E)
        for st in range(40):
            routes = [rng.randrange(-2, E) for _ in range(R)]
            max_fetch = rng.randrange(0, S + 2)
            before_usage = list(usage)
            before_slot = list(expert_slot)
            ids, plan, _ = P.step(routes, slot_expert, usage, expert_slot, st, max_fetch)
            req = [e for e in routes if e >= 0]
            hits = {e for e in req if before_slot[e] >= 0}
            # the victims, recomputed as the minimum (usage, slot) pair among the slots not
            # used in this step, one fetch after another
            u = list(before_usage)
            for e in hits:
                u[before_slot[e]] = st
            for s, e in plan:
                cand = [(u[x], x) for x in range(S) if u[x] < st]
                assert (u[s], s) == min(cand)
                u[s] = st
            assert len(plan) <= max_fetch
            fetched = [e for _, e in plan]
            misses = []
            for e in req:
                if before_slot[e] < 0 and e not in misses:
                    misses.append(e)
            assert fetched == misses[:len(fetched)]  # first-appearance order, each at most once
            assert all(before_slot[e] == expert_slot[e] for e in hits)  # hits are never evicted
            # the slot map is a bijection between resident experts and occupied slots
            for s, e in enumerate(slot_expert):
                assert e < 0 or expert_slot[e] == s
            for e, s in enumerate(expert_slot):
                assert s < 0 or slot_expert[s] == e
            # every route maps to a slot holding its expert, or to -1 if it is not resident
            for e, new in zip(routes, ids):
                if e < 0:
                    assert new == -1
                else:
                    assert new == expert_slot[e] and (new < 0 or usage[new] == st)

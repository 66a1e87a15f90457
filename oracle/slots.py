"""Expert-slot pool with least-recently-used victims, one decode step at a time: the contract of
the hybrid expert cache's victim selection on the FreeToken cache page (the pull request that
speeds up victim selection in its ensure-experts kernel: Summary, Change and Fix), written as
plain per-step Python.

TEST INFRASTRUCTURE, like the rest of `oracle/`: only the tests may call it.

State of a pool of S slots over E experts:
  slot_expert[S]  the expert a slot holds, -1 if empty;
  slot_usage[S]   the step the slot was last used at (int64), -1 if never;
  expert_slot[E]  the slot holding expert e, -1 if e is not resident.

One step takes the routes' expert ids (negative = inactive; ids >= E are treated as inactive
and reported), the step number (larger than every usage in the pool) and how many missing
experts the step may fetch:
  1. every requested expert that is resident marks its slot used: usage = step (the page's
     Phase 1, which makes those slots the most recently used of the pool);
  2. the distinct requested experts that are not resident, in the order they first appear
     among the routes, up to max_fetch of them, each take the least recently used slot among
     those not used in this step (usage < step), ties to the lowest slot (Change, second
     point); the slot's previous expert is evicted, its usage becomes step, and the copy
     plan records (slot, expert); when no slot is left the remaining misses stay missing;
  3. each route's id is rewritten to its expert's slot, or -1 when the expert is not
     resident (the route runs elsewhere) -- after every route's expert has been read (Fix).
"""


def pool_state(S, E):
    """An empty pool: no slot holds an expert, no slot was ever used."""
    return [-1] * S, [-1] * S, [-1] * E


def step(expert_ids, slot_expert, slot_usage, expert_slot, step_no, max_fetch):
    """One step; returns (new route ids, copy plan [(slot, expert)], ids that were out of
    range) and updates the three state lists in place."""
    E = len(expert_slot)
    S = len(slot_expert)
    experts = []
    bad = []
    for e in expert_ids:
        e = int(e)
        if e >= E:
            bad.append(e)
            e = -1
        experts.append(e if e >= 0 else -1)
    # 1. hits
    for e in experts:
        if e >= 0 and expert_slot[e] >= 0:
            slot_usage[expert_slot[e]] = step_no
    # 2. misses in order of first appearance
    misses = []
    for e in experts:
        if e >= 0 and expert_slot[e] < 0 and e not in misses:
            misses.append(e)
    plan = []
    for e in misses[:max_fetch]:
        victim = -1
        for s in range(S):
            if slot_usage[s] < step_no and (victim < 0 or slot_usage[s] < slot_usage[victim]):
                victim = s
        if victim < 0:
            break
        old = slot_expert[victim]
        if old >= 0:
            expert_slot[old] = -1
        slot_expert[victim] = e
        expert_slot[e] = victim
        slot_usage[victim] = step_no
        plan.append((victim, e))
    # 3. routes to slots
    new_ids = [expert_slot[e] if e >= 0 else -1 for e in experts]
    return new_ids, plan, bad

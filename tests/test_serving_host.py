"""Host logic of the continuous-batching simulator (CPU): admission under the
concurrency cap and the memory budget, slot recycling, and block
bookkeeping, driven the way ``serving.simulate`` drives it."""

import pytest

from linear_attention_diffusion_feature_b300 import capacity
from linear_attention_diffusion_feature_b300.serving import Scheduler, ServeConfig


def _run(cfg, hybrid):
    sched = Scheduler(cfg, hybrid)
    commits = {}          # rid -> step indices of its commits
    seen_steps = {}       # rid -> steps it was active in
    steps = 0
    while not sched.done():
        plan = sched.plan()
        assert plan.active, "stalled: nothing active"
        assert len(plan.active) <= cfg.max_concurrency
        assert sched.used <= cfg.memory_budget
        slots = [r.slot for r in plan.active]
        assert len(set(slots)) == len(slots), "two active requests share a slot"
        assert all(0 <= s < cfg.max_concurrency for s in slots)
        for r, c in zip(plan.active, plan.commit):
            seen_steps.setdefault(r.rid, []).append(steps)
            if c:
                commits.setdefault(r.rid, []).append(steps)
        sched.finish(plan)
        steps += 1
        assert steps < 100000
    return sched, commits, seen_steps


@pytest.mark.parametrize("hybrid", [True, False])
def test_every_request_generates_its_blocks(hybrid):
    cfg = ServeConfig(n_requests=40, max_concurrency=8, gen_tokens=128, steps_per_block=3,
                      memory_budget=1 << 40)
    sched, commits, seen = _run(cfg, hybrid)
    assert len(sched.finished) == 40
    assert sched.tokens_done == 40 * 128
    assert sched.used == 0 and sorted(sched.free_slots) == list(range(8))
    for rid, steps in seen.items():
        # active for gen_blocks * steps_per_block consecutive steps, committing
        # on every steps_per_block-th of them
        assert steps == list(range(steps[0], steps[0] + 4 * 3))
        assert commits[rid] == [steps[0] + 3 * j + 2 for j in range(4)]
    assert sched.peak_active == 8


def test_slots_are_recycled():
    cfg = ServeConfig(n_requests=10, max_concurrency=2, gen_tokens=64, steps_per_block=1,
                      memory_budget=1 << 40)
    sched, _, _ = _run(cfg, True)
    assert {r.slot for r in sched.finished} == {0, 1}


def test_budget_caps_concurrency_and_hybrid_admits_more():
    cfg = ServeConfig(n_requests=200, max_concurrency=128, gen_tokens=2048,
                      steps_per_block=1, memory_budget=40 << 30)
    hyb = Scheduler(cfg, True)
    soft = Scheduler(cfg, False)
    # the budget in requests of the longest prompt, from the capacity model
    per_soft = capacity.request_bytes(512 + 2048, 20, 0)
    per_hyb = capacity.request_bytes(512 + 2048, 14, 6)
    assert soft.capacity_limit() == (40 << 30) // per_soft == 102
    assert hyb.capacity_limit() == (40 << 30) // per_hyb == 143
    ph, ps = hyb.plan(), soft.plan()
    # the first step admits up to the cap (hybrid) or the budget (softmax)
    assert len(ph.active) == 128
    assert 102 <= len(ps.active) < 128
    assert soft.used <= cfg.memory_budget < soft.used + soft.request_bytes(soft.waiting[0])


def test_request_larger_than_budget_is_never_admitted():
    cfg = ServeConfig(n_requests=3, max_concurrency=4, gen_tokens=64, memory_budget=1000)
    sched = Scheduler(cfg, False)
    plan = sched.plan()
    assert plan.active == [] and len(sched.waiting) == 3

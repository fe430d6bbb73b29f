"""Host-side slot planner of the partially resident pool (CPU only)."""
import pytest

from w4a16_routed_expert_gb300 import build as B
from w4a16_routed_expert_gb300 import capi


@pytest.fixture(scope="module", autouse=True)
def _lib():
    B.build()
    capi.lib()


def _check_plan(p, res, C):
    # every demanded expert is computed exactly once, waves hold <= C experts
    # in distinct slots
    assert len(res["wave"]) == len(res["experts"])
    for w in range(res["n_waves"]):
        slots = [s for s, ww in zip(res["slot"], res["wave"]) if ww == w]
        assert 0 < len(slots) <= C and len(set(slots)) == len(slots)
        assert all(0 <= s < C for s in slots)


def test_fixed_order_lru_gets_no_hits_on_a_cyclic_working_set():
    # moe-stream, "Findings": experts visited in a fixed order with LRU and a
    # cache smaller than the working set -> the needed expert is always the
    # one just evicted: zero hits.
    W, C = 128, 32
    p = capi.SlotPlanner(W, C)
    for call in range(4):
        res = p.plan(range(W), capi.MOE_PLAN_FIXED_ORDER_LRU)
        assert sum(res["hit"]) == 0
        _check_plan(p, res, C)


def test_hits_first_keeps_the_resident_set():
    W, C = 128, 32
    p = capi.SlotPlanner(W, C)
    res = p.plan(range(W))
    assert sum(res["hit"]) == 0 and res["n_waves"] == 4
    _check_plan(p, res, C)
    for call in range(3):
        res = p.plan(range(W))
        assert sum(res["hit"]) == C  # the last wave's experts stay resident
        assert res["n_waves"] == 4
        # hits are computed in wave 0
        assert all(w == 0 for w, h in zip(res["wave"], res["hit"]) if h)
        _check_plan(p, res, C)


def test_subset_demand_and_victim_order():
    p = capi.SlotPlanner(16, 4)
    r1 = p.plan([1, 2])
    assert r1["n_waves"] == 1 and r1["hit"] == [0, 0]
    r2 = p.plan([2, 3, 4, 5])  # 2 is a hit; 3,4,5 take the 2 empty slots then the LRU one (expert 1)
    assert r2["hit"] == [1, 0, 0, 0] and r2["n_waves"] == 1
    assert p.slot_of(1) == -1 and p.slot_of(2) == r1["slot"][1]
    r3 = p.plan([2])
    assert r3["hit"] == [1]


def test_invalidate_and_bad_requests():
    p = capi.SlotPlanner(8, 2)
    p.plan([0, 1])
    s = p.slot_of(0)
    p.invalidate(s)
    assert p.slot_of(0) == -1
    assert p.plan([0])["hit"] == [0]
    with pytest.raises(ValueError):
        p.plan([0, 0])
    with pytest.raises(ValueError):
        p.plan([8])
    with pytest.raises(ValueError):
        capi.SlotPlanner(0, 1)

"""Pins of the residency-tier oracle (oracle/tier.py) against facts it does not compute itself.

The facts are:
- LRU residency by stack distance, from the access history;
- the inclusion property of a stack algorithm;
- the closed form of a cyclic access pattern;
- heat from a brute-force count;
- the pinned sets from full sorts (usage heat at start-up, decayed session heat live);
- the halving closed form of the session-heat decay;
- conservation of prefetched loads;
- the per-call guarantees the readings state.

CPU only.
"""
import numpy as np
import pytest

from gen.trace import routing_trace
from oracle.tier import LRU_HIT, MISS, PIN_HIT, TierOracle


def test_lru_hits_equal_stack_distance():
    """one expert per call: a lookup hits iff fewer than n_lru distinct other experts were
    used since its last use, and the evicted expert is the least recently used resident"""
    rng = np.random.default_rng(1)
    seq = [int(e) for e in rng.zipf(1.3, 3000) % 40]
    for cap in (1, 3, 8, 17):
        t = TierOracle(1, 40, 0, cap)
        last = {}
        for i, e in enumerate(seq):
            resident_before = t.resident(0)
            classes, fetched, evicted = t.lookup(0, [e])
            if e in last:
                distinct_since = len(set(seq[last[e] + 1:i]) - {e})
                expect = LRU_HIT if distinct_since < cap else MISS
            else:
                expect = MISS
            assert classes == [expect]
            if evicted:
                assert len(resident_before) == cap
                oldest = min(resident_before, key=lambda x: last[x])
                assert evicted == [oldest]
            last[e] = i


def test_lru_inclusion_property():
    actual, _ = routing_trace(2, 200, 1, 64, 8)
    caps = (8, 9, 12, 20, 40)
    tiers = [TierOracle(1, 64, 0, c) for c in caps]
    for step in actual:
        for t in tiers:
            t.lookup(0, step[0])
        res = [t.resident(0) for t in tiers]
        for a, b in zip(res, res[1:]):
            assert a <= b
    misses = [t.stats["misses"] for t in tiers]
    assert misses == sorted(misses, reverse=True)


@pytest.mark.parametrize("cap", [1, 4, 16])
def test_cyclic_pattern_closed_form(cap):
    t = TierOracle(1, 64, 0, cap)
    for i in range(10 * (cap + 1)):
        t.lookup(0, [i % (cap + 1)])
    assert t.stats["misses"] == 10 * (cap + 1) and t.stats["lru_hits"] == 0
    t = TierOracle(1, 64, 0, cap)
    for i in range(10 * cap):
        t.lookup(0, [i % cap])
    assert t.stats["misses"] == cap and t.stats["lru_hits"] == 9 * cap


def test_calls_keep_their_own_experts_and_heat_is_a_count():
    actual, predicted = routing_trace(3, 120, 3, 48, 6)
    t = TierOracle(3, 48, 4, 6)
    count = np.zeros((3, 48), dtype=np.int64)
    for s, step in enumerate(actual):
        for l in range(3):
            t.prefetch(l, predicted[s][l])  # counts no heat
            _, _, evicted = t.lookup(l, step[l])
            count[l, step[l]] += 1
            assert not set(evicted) & set(step[l].tolist())
            assert set(step[l].tolist()) <= t.resident(l)
            assert len(t.lru[l]) <= 6 and not (t.pinned[l] & set(t.lru[l]))
            assert len(set(t.lru[l])) == len(t.lru[l])
        if s % 30 == 29:
            for l in range(3):
                t.repin(l)
    assert np.array_equal(np.array(t.heat), count)
    assert np.array_equal(np.array(t.session), count)  # no decay yet: the same count


def test_autopin_equals_full_sort():
    rng = np.random.default_rng(4)
    E, n_pin = 50, 7
    for trial in range(20):
        t = TierOracle(1, E, n_pin, 10)
        heat = rng.integers(0, 4, E)  # many ties, some zeros
        if trial == 0:
            heat[:] = 0
        t.set_heat(0, heat.tolist())
        for e in rng.choice(E, 10, replace=False):  # some experts sit in the LRU list
            t.lookup(0, [int(e)])
        t.set_heat(0, heat.tolist())
        lru_before, old = list(t.lru[0]), set(t.pinned[0])
        fetched, dropped = t.autopin(0)
        order = sorted(range(E), key=lambda e: (-int(heat[e]), e))  # full stable sort
        expect = {e for e in order[:n_pin] if heat[e] > 0}
        assert t.pinned[0] == expect
        assert fetched == sorted(expect - old - set(lru_before))
        assert dropped == sorted(old - expect)
        assert t.lru[0] == [e for e in lru_before if e not in expect]


def test_live_repin_equals_full_sort_with_incumbents_first():
    """live repin ranks pinned experts and every expert with session heat > 0 by heat, then
    incumbents first, then id: an expert displaces a pinned one only if strictly hotter"""
    rng = np.random.default_rng(8)
    E, n_pin = 40, 6
    for trial in range(25):
        t = TierOracle(1, E, n_pin, E)
        t.set_heat(0, rng.integers(0, 3, E).tolist())
        t.autopin(0)  # some incumbents
        for _ in range(int(rng.integers(0, 30))):
            t.lookup(0, sorted(rng.choice(E, int(rng.integers(1, 5)), replace=False).tolist()))
        for _ in range(int(rng.integers(0, 3))):
            t.decay()
        old, sess = set(t.pinned[0]), list(t.session[0])
        t.repin(0)
        cand = [e for e in range(E) if sess[e] > 0 or e in old]
        order = sorted(cand, key=lambda e: (-sess[e], e not in old, e))  # full sort
        assert t.pinned[0] == set(order[:n_pin])
    # a session map of zeros changes nothing
    t = TierOracle(1, E, n_pin, E)
    t.set_heat(0, list(range(E)))
    t.autopin(0)
    before = set(t.pinned[0])
    assert t.repin(0) == ([], []) and t.pinned[0] == before


def test_decay_halves_session_heat():
    """u uses followed by m decays leave floor(u / 2^m) of session heat; usage heat keeps u"""
    t = TierOracle(2, 16, 0, 16)
    uses = {3: 1, 5: 7, 9: 13, 15: 64}
    for e, u in uses.items():
        for _ in range(u):
            t.lookup(1, [e])
    for m in range(8):
        for e, u in uses.items():
            assert t.session[1][e] == u >> m and t.heat[1][e] == u
        t.decay()


def test_pinned_experts_hit_and_leave_the_lru_alone():
    t = TierOracle(1, 32, 3, 4)
    t.set_heat(0, [5 if e in (2, 9, 30) else 0 for e in range(32)])
    t.autopin(0)
    t.lookup(0, [1, 4])
    before = list(t.lru[0])
    classes, fetched, evicted = t.lookup(0, [2, 9, 30])
    assert classes == [PIN_HIT] * 3 and fetched == [] and evicted == []
    assert t.lru[0] == before
    # a call of n_lru unpinned experts plus pinned ones is accepted, one more is rejected
    t.lookup(0, [2, 3, 5, 6, 7, 9])
    with pytest.raises(ValueError):
        t.lookup(0, [3, 5, 6, 7, 8])


def test_perfect_prefetch_leaves_no_misses_and_loads_are_conserved():
    actual, _ = routing_trace(5, 150, 2, 64, 8)
    t = TierOracle(2, 64, 0, 12)
    for step in actual:
        for l in range(2):
            t.prefetch(l, step[l])
            classes, fetched, _ = t.lookup(l, step[l])
            assert MISS not in classes and fetched == []
    st = t.stats
    assert st["misses"] == 0 and st["prefetch_wasted"] == 0
    assert st["prefetch_used"] == st["prefetch_fetches"]
    # with a 71.6%-accurate prediction every prefetched load is used, wasted, or still marked
    actual, predicted = routing_trace(6, 150, 2, 64, 8)
    t = TierOracle(2, 64, 2, 12)
    for s, step in enumerate(actual):
        for l in range(2):
            t.prefetch(l, predicted[s][l])
            t.lookup(l, step[l])
        if s == 75:
            t.repin(0)
            t.repin(1)
    st = t.stats
    marked = sum(len(m) for m in t.marked)
    assert st["prefetch_fetches"] == st["prefetch_used"] + st["prefetch_wasted"] + marked
    assert st["prefetch_used"] > 0 and st["prefetch_wasted"] > 0


@pytest.mark.parametrize("ids", [[3, 3], [5, 2], [-1], [64]])
def test_rejected_calls_change_nothing(ids):
    t = TierOracle(1, 64, 0, 4)
    t.lookup(0, [1, 2])
    snap = (list(t.lru[0]), list(t.heat[0]), dict(t.stats))
    with pytest.raises(ValueError):
        t.lookup(0, ids)
    with pytest.raises(ValueError):
        t.prefetch(0, ids)
    assert (list(t.lru[0]), list(t.heat[0]), dict(t.stats)) == snap


TIER_MUTANTS = {
    1: ("evicts the most recently used expert", ["test_lru_hits_equal_stack_distance"]),
    2: ("repin ties go to the higher id", ["test_autopin_equals_full_sort"]),
    3: ("prefetch counts heat", ["test_calls_keep_their_own_experts_and_heat_is_a_count"]),
    4: ("LRU hits are not promoted", ["test_lru_hits_equal_stack_distance"]),
    5: ("repin pins experts never used", ["test_autopin_equals_full_sort"]),
    6: ("a used prefetch stays marked", ["test_perfect_prefetch_leaves_no_misses_and_loads_are_conserved"]),
    7: ("decay leaves the session heat as it is", ["test_decay_halves_session_heat"]),
    8: ("incumbents lose ties at a repin", ["test_live_repin_equals_full_sort_with_incumbents_first"]),
}


@pytest.mark.parametrize("n", sorted(TIER_MUTANTS))
def test_tier_pin_catches_planted_mistake(n, monkeypatch):
    import oracle.tier as tier
    monkeypatch.setattr(tier, "MUTANT", n)
    for name in TIER_MUTANTS[n][1]:
        with pytest.raises(AssertionError):
            globals()[name]()

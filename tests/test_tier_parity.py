"""The library's tier manager (coli_tier_*) against the residency-tier oracle, op by op.

Seeded random sequences of lookups, prefetches, repins and heat restores run on both sides.
After every op these must be identical:
- the hit classes, the loads, and the evictions and drops, in order;
- the pinned sets and the LRU order;
- the heat and the counters.

Slots are the library's own choice, so they are checked for validity instead:
- each resident expert holds one distinct slot in range;
- a slot stays with its expert until that expert is evicted or dropped;
- a load goes to a slot that was free, or that the same call freed.

Host code only: no GPU is used.
"""
import os
import struct

import numpy as np
import pytest

from gen.trace import routing_trace
from int4_routed_expert_quantize_gb300 import _build, coli
from oracle.tier import TierOracle


@pytest.fixture(scope="module")
def lib():
    if os.environ.get("COLI_TIER_HOST_SO"):  # a host-only (sanitized) build is under test
        return coli.use_host_library(os.environ["COLI_TIER_HOST_SO"])
    if _build.is_stale():
        _build.build()
    coli._lib = None
    return coli.lib()


def snapshot(t, o):
    """compare the full state of library tier t and oracle o; return slot_of per layer"""
    slots = []
    n_slots = o.n_pin + o.n_lru
    for l in range(o.n_layers):
        pinned, lru, slot_of = t.state(l)
        assert pinned.tolist() == sorted(o.pinned[l])
        assert lru.tolist() == o.lru[l]
        assert t.heat(l).tolist() == o.heat[l]
        assert t.session_heat(l).tolist() == o.session[l]
        res = np.flatnonzero(slot_of >= 0)
        assert set(res.tolist()) == o.resident(l)
        used = slot_of[res]
        assert used.min(initial=0) >= 0 and used.max(initial=0) < n_slots
        assert len(set(used.tolist())) == used.size
        slots.append(slot_of.copy())
    assert t.stats() == o.stats
    return slots


def check_moves(before, after, fetch_ids, fetch_slots, freed_ids, freed_slots):
    """slot bookkeeping of one op on one layer"""
    assert before[freed_ids].tolist() == freed_slots.tolist()
    assert np.all(after[freed_ids[~np.isin(freed_ids, fetch_ids)]] == -1)
    assert after[fetch_ids].tolist() == fetch_slots.tolist()
    busy_before = set(before[before >= 0].tolist()) - set(freed_slots.tolist())
    assert not busy_before & set(fetch_slots.tolist())
    kept = (before >= 0) & (after >= 0)
    kept[fetch_ids] = False
    assert np.array_equal(before[kept], after[kept])


CONFIGS = [  # n_layers, n_experts, n_pin, n_lru, per_call
    (3, 64, 4, 8, 8),
    (2, 32, 0, 8, 8),       # no pinned store
    (2, 40, 40, 6, 6),      # pinned store as large as the layer
    (1, 16, 2, 1, 1),       # one LRU place, one expert per call
    (4, 256, 16, 24, 8),    # GLM-like: 256 experts, top-8
    (2, 48, 5, 48, 12),     # LRU as large as the layer
]


@pytest.mark.parametrize("cfg", CONFIGS, ids=[f"L{c[0]}E{c[1]}p{c[2]}r{c[3]}k{c[4]}" for c in CONFIGS])
@pytest.mark.parametrize("seed", [0, 1])
def test_tier_matches_oracle(lib, cfg, seed):
    n_layers, E, n_pin, n_lru, k = cfg
    actual, predicted = routing_trace(100 + seed, 60, n_layers, E, k)
    t, o = coli.Tier(n_layers, E, n_pin, n_lru), TierOracle(n_layers, E, n_pin, n_lru)
    rng = np.random.default_rng(seed)
    slots = snapshot(t, o)
    for s in range(len(actual)):
        for l in range(n_layers):
            op = rng.random()
            if op < 0.5:
                r = t.prefetch(l, predicted[s][l])
                f, ev = o.prefetch(l, predicted[s][l])
                assert r["fetch_ids"].tolist() == f and r["evict_ids"].tolist() == ev
                new = snapshot(t, o)
                check_moves(slots[l], new[l], r["fetch_ids"], r["fetch_slots"], r["evict_ids"],
                            r["evict_slots"])
                slots = new
            ids = actual[s][l]
            try:
                o_res = o.lookup(l, ids)
            except ValueError:  # more unpinned experts than LRU places: both reject
                with pytest.raises(coli.ColiError):
                    t.lookup(l, ids)
                assert all(np.array_equal(a, b) for a, b in zip(snapshot(t, o), slots))
                continue
            r = t.lookup(l, ids)
            cls, f, ev = o_res
            assert r["cls"].tolist() == cls
            assert r["fetch_ids"].tolist() == f and r["evict_ids"].tolist() == ev
            new = snapshot(t, o)
            assert r["slot"].tolist() == new[l][ids].tolist()
            check_moves(slots[l], new[l], r["fetch_ids"], r["fetch_slots"], r["evict_ids"],
                        r["evict_slots"])
            slots = new
        if rng.random() < 0.1:
            t.decay()
            o.decay()
        if rng.random() < 0.15:
            l = int(rng.integers(n_layers))
            if rng.random() < 0.3:  # restore a saved usage map and pin from it
                heat = rng.integers(0, 5, E)
                t.set_heat(l, heat)
                o.set_heat(l, heat.tolist())
                r = t.autopin(l)
                f, dropped = o.autopin(l)
            else:  # live repin by the session heat
                r = t.repin(l)
                f, dropped = o.repin(l)
            assert r["fetch_ids"].tolist() == f and r["drop_ids"].tolist() == dropped
            new = snapshot(t, o)
            check_moves(slots[l], new[l], r["fetch_ids"], r["fetch_slots"], r["drop_ids"],
                        r["drop_slots"])
            slots = new
    st = t.stats()
    assert st["misses"] + st["lru_hits"] + st["pin_hits"] > 0


def test_rejected_calls_change_nothing(lib):
    t, o = coli.Tier(1, 32, 2, 4), TierOracle(1, 32, 2, 4)
    t.lookup(0, [1, 2, 3])
    o.lookup(0, [1, 2, 3])
    before = snapshot(t, o)
    for ids in ([3, 3], [5, 2], [-1], [32], [4, 5, 6, 7, 8]):
        with pytest.raises(coli.ColiError) as e:
            t.lookup(0, ids)
        assert e.value.status == -1
        assert snapshot(t, o)[0].tolist() == before[0].tolist()
    with pytest.raises(coli.ColiError):
        t.prefetch(0, [1, 2, 3, 4, 5])  # more than n_lru predictions
    for bad_layer in (-1, 1):
        with pytest.raises(coli.ColiError):
            t.lookup(bad_layer, [1])
        with pytest.raises(coli.ColiError):
            t.repin(bad_layer)
    with pytest.raises(coli.ColiError):
        t.set_heat(0, np.full(32, -1))
    snapshot(t, o)


@pytest.mark.parametrize("cfg", [(0, 8, 0, 1), (1, 0, 0, 1), (1, 8, 9, 1), (1, 8, 0, 0),
                                 (1, 8, 0, 9), (1, 8, -1, 1), (4097, 8, 0, 1), (1, 65537, 0, 1),
                                 (257, 65536, 0, 1)])  # the last: more than 2^24 entries
def test_create_rejects_bad_config(lib, cfg):
    with pytest.raises(coli.ColiError) as e:
        coli.Tier(*cfg)
    assert e.value.status == -1


def test_empty_call_is_a_no_op(lib):
    t = coli.Tier(1, 8, 1, 2)
    r = t.lookup(0, [])
    assert r["cls"].size == 0 and r["fetch_ids"].size == 0
    assert t.stats() == dict.fromkeys(coli.TIER_STATS, 0)


def test_usage_file_layout_and_round_trip(lib, tmp_path):
    t = coli.Tier(2, 3, 1, 2)
    t.set_heat(0, [5, 0, 2 ** 40])
    t.set_heat(1, [1, 2, 3])
    path = tmp_path / "usage.bin"
    t.save_usage(path)
    data = path.read_bytes()
    # written out by hand: magic, int32 n_layers = 2, int32 n_experts = 3, six int64 counts
    expect = (b"COLIUSE1" + b"\x02\x00\x00\x00" + b"\x03\x00\x00\x00"
              + b"\x05" + b"\x00" * 7 + b"\x00" * 8 + b"\x00" * 5 + b"\x01" + b"\x00" * 2
              + b"\x01" + b"\x00" * 7 + b"\x02" + b"\x00" * 7 + b"\x03" + b"\x00" * 7)
    assert data == expect
    u = coli.Tier(2, 3, 1, 2)
    u.load_usage(path)
    assert u.heat(0).tolist() == [5, 0, 2 ** 40] and u.heat(1).tolist() == [1, 2, 3]
    # start-up autopin: the hottest expert of each layer is pinned from the learned usage
    assert u.autopin(0)["fetch_ids"].tolist() == [2] and u.autopin(1)["fetch_ids"].tolist() == [2]
    # the session heat starts empty in the new process: a live repin changes nothing
    assert u.repin(0)["fetch_ids"].size == 0 and u.repin(0)["drop_ids"].size == 0


def test_usage_file_rejections_leave_heat_alone(lib, tmp_path):
    t = coli.Tier(2, 3, 1, 2)
    t.set_heat(0, [7, 8, 9])
    good = tmp_path / "good.bin"
    t.save_usage(good)
    data = good.read_bytes()
    u = coli.Tier(2, 3, 1, 2)
    u.set_heat(1, [4, 4, 4])
    cases = {
        "magic.bin": (b"COLIUSE2" + data[8:], -1),
        "shape.bin": (data[:8] + struct.pack("<ii", 2, 4) + data[16:], -1),
        "short.bin": (data[:-3], -7),
        "long.bin": (data + b"\x00", -1),
        "negative.bin": (data[:16] + struct.pack("<q", -1) + data[24:], -1),
    }
    for name, (blob, status) in cases.items():
        p = tmp_path / name
        p.write_bytes(blob)
        with pytest.raises(coli.ColiError) as e:
            u.load_usage(p)
        assert e.value.status == status, name
        assert u.heat(0).tolist() == [0, 0, 0] and u.heat(1).tolist() == [4, 4, 4]
    with pytest.raises(coli.ColiError) as e:
        u.load_usage(tmp_path / "missing.bin")
    assert e.value.status == -7
    with pytest.raises(coli.ColiError) as e:
        t.save_usage(tmp_path)  # a directory cannot be opened for writing
    assert e.value.status == -7


def test_glm_sized_trace_hit_rates(lib):
    """a GLM-sized layer set (8 layers x 256 experts, top-8 per call) behaves as the oracle
    does over a longer trace, with lookahead prefetch and a repin every 64 steps"""
    n_layers, E, n_pin, n_lru, k = 8, 256, 32, 64, 8
    actual, predicted = routing_trace(7, 256, n_layers, E, k)
    t, o = coli.Tier(n_layers, E, n_pin, n_lru), TierOracle(n_layers, E, n_pin, n_lru)
    for s in range(len(actual)):
        for l in range(n_layers):
            if l + 1 < n_layers:
                t.prefetch(l + 1, predicted[s][l + 1])
                o.prefetch(l + 1, predicted[s][l + 1])
            r = t.lookup(l, actual[s][l])
            assert r["cls"].tolist() == o.lookup(l, actual[s][l])[0]
        if s % 32 == 31:
            t.decay()
            o.decay()
        if s % 64 == 63:
            for l in range(n_layers):
                assert t.repin(l)["fetch_ids"].tolist() == o.repin(l)[0]
    assert t.stats() == o.stats
    st = o.stats
    assert st["pin_hits"] > 0 and st["lru_hits"] > 0 and st["prefetch_used"] > 0


def _same(t, o, layers):
    for l in layers:
        pinned, lru, slot_of = t.state(l)
        assert pinned.tolist() == sorted(o.pinned[l]) and lru.tolist() == o.lru[l]
        assert set(np.flatnonzero(slot_of >= 0).tolist()) == o.resident(l)
    assert t.stats() == o.stats


def test_largest_configurations(lib):
    # 65536 experts with as many pinned and LRU slots: ids at both ends of the range
    E = 65536
    t, o = coli.Tier(1, E, E, E), TierOracle(1, E, E, E)
    for ids in ([0, 1, E - 2, E - 1], [5, 40000, E - 1], list(range(E - 64, E))):
        r = t.lookup(0, ids)
        assert r["cls"].tolist() == o.lookup(0, ids)[0]
    heat = np.zeros(E, np.int64)
    heat[[3, E - 1, 777]] = [9, 9, 2]
    t.set_heat(0, heat)
    o.set_heat(0, heat.tolist())
    assert t.autopin(0)["fetch_ids"].tolist() == o.autopin(0)[0]
    assert t.repin(0)["drop_ids"].tolist() == o.repin(0)[1]
    _same(t, o, [0])
    # 4096 layers
    t, o = coli.Tier(4096, 8, 1, 2), TierOracle(4096, 8, 1, 2)
    for l in (0, 1, 4094, 4095):
        assert t.lookup(l, [1, 7])["cls"].tolist() == o.lookup(l, [1, 7])[0]
        t.repin(l)
        o.repin(l)
    _same(t, o, [0, 4095])


def test_degenerate_cases(lib):
    E = 16
    # equal heat everywhere: the lowest ids are pinned
    t, o = coli.Tier(1, E, 4, 4), TierOracle(1, E, 4, 4)
    t.set_heat(0, np.full(E, 3))
    o.set_heat(0, [3] * E)
    assert t.autopin(0)["fetch_ids"].tolist() == o.autopin(0)[0] == [0, 1, 2, 3]
    # predicted experts that are pinned load nothing and keep their pinned place
    r = t.prefetch(0, [0, 1, 2, 3])
    assert r["fetch_ids"].size == 0 and o.prefetch(0, [0, 1, 2, 3]) == ([], [])
    _same(t, o, [0])
    # no pinned slots: a repin pins nothing and drops nothing
    t, o = coli.Tier(1, E, 0, 3), TierOracle(1, E, 0, 3)
    t.lookup(0, [2, 4])
    o.lookup(0, [2, 4])
    r = t.repin(0)
    assert r["fetch_ids"].size == 0 and r["drop_ids"].size == 0 and o.repin(0) == ([], [])
    _same(t, o, [0])
    # a cleared map keeps the pinned experts; an expert displaces one only if strictly hotter
    t, o = coli.Tier(1, E, 2, 2), TierOracle(1, E, 2, 2)
    for tier in (t, o):
        tier.set_heat(0, [1] * E if tier is o else np.ones(E))
        tier.autopin(0)  # pins 0 and 1
        tier.set_heat(0, [0] * E if tier is o else np.zeros(E))
    r = t.autopin(0)
    assert r["drop_ids"].size == 0 and o.autopin(0) == ([], [])
    hot = [0] * E
    hot[7], hot[9], hot[0] = 2, 1, 1  # 7 is hotter than both; 9 ties with pinned 0
    t.set_heat(0, np.array(hot))
    o.set_heat(0, hot)
    r = t.autopin(0)
    f, dropped = o.autopin(0)
    assert r["fetch_ids"].tolist() == f == [7] and r["drop_ids"].tolist() == dropped == [1]
    _same(t, o, [0])


def test_null_arguments(lib, tmp_path):
    """the C ABI's NULL rules: a NULL handle or input is EINVAL; every output may be NULL"""
    import ctypes
    L = coli.lib()
    EINVAL = -1
    h = ctypes.c_void_p()
    cfg = coli.TierConfig(1, 8, 1, 2)
    assert L.coli_tier_create(None, ctypes.byref(h)) == EINVAL
    assert L.coli_tier_create(ctypes.byref(cfg), None) == EINVAL
    assert L.coli_tier_create(ctypes.byref(cfg), ctypes.byref(h)) == 0
    ids = np.array([1, 5], np.int32)
    p = ids.ctypes.data
    assert L.coli_tier_lookup(None, 0, p, 2, *[None] * 8) == EINVAL
    assert L.coli_tier_lookup(h, 0, None, 2, *[None] * 8) == EINVAL
    assert L.coli_tier_lookup(h, 0, None, 0, *[None] * 8) == 0  # an empty call needs no ids
    assert L.coli_tier_lookup(h, 0, p, 2, *[None] * 8) == 0    # outputs are optional
    assert L.coli_tier_prefetch(None, 0, p, 2, *[None] * 6) == EINVAL
    assert L.coli_tier_prefetch(h, 0, p, 2, *[None] * 6) == 0
    assert L.coli_tier_repin(None, 0, *[None] * 6) == EINVAL
    assert L.coli_tier_repin(h, 0, *[None] * 6) == 0
    assert L.coli_tier_autopin(None, 0, *[None] * 6) == EINVAL
    assert L.coli_tier_decay(None) == EINVAL
    assert L.coli_tier_session_heat(h, 0, None) == EINVAL
    assert L.coli_tier_session_heat(None, 0, p) == EINVAL
    assert L.coli_tier_state(None, 0, *[None] * 5) == EINVAL
    assert L.coli_tier_state(h, 0, *[None] * 5) == 0
    assert L.coli_tier_heat(h, 0, None) == EINVAL and L.coli_tier_heat(None, 0, p) == EINVAL
    assert L.coli_tier_set_heat(h, 0, None) == EINVAL
    assert L.coli_tier_stats(h, None) == EINVAL and L.coli_tier_stats(None, p) == EINVAL
    path = str(tmp_path / "u.bin").encode()
    assert L.coli_tier_save_usage(h, None) == EINVAL and L.coli_tier_save_usage(None, path) == EINVAL
    assert L.coli_tier_load_usage(h, None) == EINVAL and L.coli_tier_load_usage(None, path) == EINVAL
    # the calls with NULL outputs still did their work: 1 and 5 were used once each, and the
    # repin pinned the lower of the two
    heat = np.empty(8, np.int64)
    assert L.coli_tier_heat(h, 0, heat.ctypes.data) == 0
    assert heat.tolist() == [0, 1, 0, 0, 0, 1, 0, 0]
    pinned, n_pinned = np.empty(1, np.int32), ctypes.c_int()
    assert L.coli_tier_state(h, 0, pinned.ctypes.data, ctypes.byref(n_pinned), None, None, None) == 0
    assert n_pinned.value == 1 and pinned[0] == 1
    L.coli_tier_destroy(h)
    L.coli_tier_destroy(None)  # a no-op

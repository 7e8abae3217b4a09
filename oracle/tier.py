"""CPU oracle of the expert residency tiers.  TEST INFRASTRUCTURE ONLY.

Where each step comes from:
- "colibrì 架构概述" §4, the expert cache and scheduling layer. Each layer keeps an LRU cache
  (ecache) and a pinned hot store (pin). tier.h repins by heat. pilot_prefetch is a
  router-lookahead read-ahead.
- §5, the life of a token. The moe step looks up pin, then ecache, and loads the expert on a
  miss (expert_load); LRU promotion follows the expert computation. The continuous
  optimisations are pilot_prefetch (layer L+1's router predicts the next layer's experts)
  and repin_pass (at safe turn boundaries, the heat map swaps cold pinned experts for hot
  ones). At start-up the hottest experts learned in the usage file are pinned (autopin).
- README "統一記憶體階層": a learning cache records where the workload routes and pins the
  hottest experts.
- README "絕不為同一次硬碟讀取等待兩遍": the router lookahead preloads the next layer's
  experts.
- ai4coding.ru "colibrì: движок GLM-5.2", "Обучающийся кэш": the usage file records which
  experts the workload reaches, and start-up pins the hottest. The optional live repin
  (--repin N) swaps cold pinned experts for hotter ones by a decaying session heat map.

Readings (the pages name the steps, not their details):
- One tier object covers every MoE layer. Each layer has a pinned set of at most n_pin
  experts and an LRU list of at most n_lru experts, most recently used first. The shared
  expert is always resident and is not tracked.
- lookup(layer, ids) takes the distinct routed experts of one call (the batch union), in
  ascending order. It classifies each as PIN_HIT, LRU_HIT or MISS, and adds 1 to each
  one's usage heat and session heat.
- The misses are loaded. Then every unpinned expert of the call moves to the front of the
  LRU list (hits and misses alike, in ascending order, so the largest id ends in front), and
  the list is cut back to n_lru entries from its tail; the cut entries are evicted, least
  recently used first.
- So a call never evicts an expert it uses itself, and the recency order does not depend on
  the capacity (LRU stays a stack algorithm). That needs at most n_lru unpinned ids per
  call; a call with more is rejected and changes nothing.
- prefetch(layer, ids) treats the predicted experts as a call would, but counts no heat
  and no hits. It loads the predicted experts that are not resident, moves every unpinned
  predicted expert to the front in the same way, and cuts the list back. So a prefetch
  never evicts an expert it predicts. Each expert it loads is marked as prefetched.
- A later lookup that hits a marked expert counts the prefetch as used, and so does a repin
  that pins it (its load is kept). An eviction of a marked expert counts it as wasted. At
  most n_lru ids per call.
- Two heats per (layer, expert). Usage heat is a cumulative use count; set_heat restores a
  saved usage map. Session heat counts uses too, but decay() halves it for every layer
  (integer halving, rounding down). The pages give no decay rate: the caller's interval
  between decays sets the half-life.
- autopin(layer) pins by usage heat (start-up); repin(layer) pins by session heat (live).
- Both rank the candidates by heat, higher first. The candidates are the pinned experts and
  every expert with heat > 0. On equal heat a pinned expert goes first, then the lower id.
  The top n_pin form the new pinned set. So an expert replaces a pinned one only if it is
  strictly hotter, and a map of zeros changes nothing.
- A repin or autopin drops the experts that leave the pinned set. An entering expert that
  sits in the LRU list moves out of the list (no load); any other entering expert is
  loaded.

Pure Python over lists and sets, so the steps can be checked by eye.  Nothing here is
shared with the library's own tier manager.
"""

PIN_HIT, LRU_HIT, MISS = 0, 1, 2

# MUTANT plants one known mistake (tests/test_tier_oracle.py checks that a pin catches each);
# the oracle the tests trust has MUTANT == 0.
MUTANT = 0

STAT_KEYS = ("pin_hits", "lru_hits", "misses", "evictions", "prefetch_fetches",
             "prefetch_used", "prefetch_wasted", "repin_fetches")


class TierOracle:
    def __init__(self, n_layers, n_experts, n_pin, n_lru):
        if n_layers < 1 or n_experts < 1 or n_pin < 0 or n_lru < 1 or n_pin > n_experts:
            raise ValueError("bad tier configuration")
        self.n_layers, self.n_experts, self.n_pin, self.n_lru = n_layers, n_experts, n_pin, n_lru
        self.pinned = [set() for _ in range(n_layers)]
        self.lru = [[] for _ in range(n_layers)]  # most recently used first
        self.heat = [[0] * n_experts for _ in range(n_layers)]  # usage heat
        self.session = [[0] * n_experts for _ in range(n_layers)]  # decayed session heat
        self.marked = [set() for _ in range(n_layers)]  # prefetched, not used yet
        self.stats = dict.fromkeys(STAT_KEYS, 0)

    def _check_ids(self, layer, ids):
        if not 0 <= layer < self.n_layers:
            raise ValueError("layer out of range")
        ids = [int(e) for e in ids]
        for i, e in enumerate(ids):
            if not 0 <= e < self.n_experts or (i and ids[i - 1] >= e):
                raise ValueError("ids must be distinct, ascending and in range")
        return ids

    def _evict_tail(self, layer):
        victim = self.lru[layer].pop(0 if MUTANT == 1 else -1)
        self.stats["evictions"] += 1
        if victim in self.marked[layer]:
            self.marked[layer].discard(victim)
            self.stats["prefetch_wasted"] += 1
        return victim

    def _to_front(self, layer, ids):
        lru = self.lru[layer]
        for e in ids:
            if e in lru:
                lru.remove(e)
            lru.insert(0, e)

    def _cut_back(self, layer):
        evicted = []
        while len(self.lru[layer]) > self.n_lru:
            evicted.append(self._evict_tail(layer))
        return evicted

    def lookup(self, layer, ids):
        """One call's experts ("colibrì 架构概述" §5, moe step: pin, then ecache, else
        expert_load; LRU promotion after the experts ran).
        -> (classes, fetched ids, evicted ids), all in the order they happened"""
        ids = self._check_ids(layer, ids)
        pinned, lru = self.pinned[layer], self.lru[layer]
        if sum(1 for e in ids if e not in pinned) > self.n_lru:
            raise ValueError("more unpinned experts in one call than LRU places")
        # check the pinned store, then the LRU cache; the rest are misses
        classes = [PIN_HIT if e in pinned else LRU_HIT if e in lru else MISS for e in ids]
        for e, c in zip(ids, classes):
            self.heat[layer][e] += 1
            self.session[layer][e] += 1
            self.stats[("pin_hits", "lru_hits", "misses")[c]] += 1
            if c == LRU_HIT and e in self.marked[layer]:
                if MUTANT != 6:
                    self.marked[layer].discard(e)
                self.stats["prefetch_used"] += 1
        # misses are loaded; the call's unpinned experts become the most recently used
        fetched = [e for e, c in zip(ids, classes) if c == MISS]
        moved = [e for e, c in zip(ids, classes) if c == MISS or (c == LRU_HIT and MUTANT != 4)]
        self._to_front(layer, moved)
        return classes, fetched, self._cut_back(layer)

    def prefetch(self, layer, ids):
        """Predicted experts of a layer ("colibrì 架构概述" §5 pilot_prefetch; README
        "絕不為同一次硬碟讀取等待兩遍", router lookahead). -> (fetched ids, evicted ids)"""
        ids = self._check_ids(layer, ids)
        if len(ids) > self.n_lru:
            raise ValueError("more predicted experts than LRU places")
        pinned, lru = self.pinned[layer], self.lru[layer]
        fetched = [e for e in ids if e not in pinned and e not in lru]
        for e in fetched:
            self.marked[layer].add(e)
            self.stats["prefetch_fetches"] += 1
            if MUTANT == 3:
                self.heat[layer][e] += 1
        self._to_front(layer, [e for e in ids if e not in pinned])
        return fetched, self._cut_back(layer)

    def _pin_by(self, layer, h):
        if not 0 <= layer < self.n_layers:
            raise ValueError("layer out of range")
        old = self.pinned[layer]
        tie = -1 if MUTANT == 2 else 1
        incumbent_first = MUTANT != 8
        candidates = [e for e in range(self.n_experts) if h[e] > 0 or e in old or MUTANT == 5]
        ranked = sorted(candidates,
                        key=lambda e: (-h[e], 0 if (e in old and incumbent_first) else 1, tie * e))
        new = set(ranked[:self.n_pin])
        fetched = []
        for e in sorted(new - old):
            if e in self.lru[layer]:
                self.lru[layer].remove(e)
                if e in self.marked[layer]:  # its prefetched load is kept
                    self.marked[layer].discard(e)
                    self.stats["prefetch_used"] += 1
            else:
                fetched.append(e)
                self.stats["repin_fetches"] += 1
        dropped = sorted(old - new)
        self.pinned[layer] = new
        return fetched, dropped

    def autopin(self, layer):
        """Start-up pinning from the learned usage heat ("colibrì 架构概述" §5 autopin;
        ai4coding.ru "Обучающийся кэш"; README "統一記憶體階層").
        -> (fetched ids, dropped ids), each ascending"""
        return self._pin_by(layer, self.heat[layer])

    def repin(self, layer):
        """Live repin by the decayed session heat ("colibrì 架构概述" §4 tier.h, §5 repin_pass;
        ai4coding.ru "Обучающийся кэш", --repin N). -> (fetched ids, dropped ids), ascending"""
        return self._pin_by(layer, self.session[layer])

    def decay(self):
        """Halve every session heat (rounding down): the decay of the session heat map."""
        if MUTANT == 7:
            return
        for row in self.session:
            for e in range(self.n_experts):
                row[e] //= 2

    def set_heat(self, layer, heat):
        """Restore a learned usage map (the .coli_usage file, "colibrì 架构概述" §5 start-up)."""
        if not 0 <= layer < self.n_layers or len(heat) != self.n_experts or min(heat) < 0:
            raise ValueError("bad usage map")
        self.heat[layer] = [int(v) for v in heat]

    def resident(self, layer):
        return self.pinned[layer] | set(self.lru[layer])

// Expert residency tiers: the host-side decisions of which expert records sit in which HBM
// slots of each MoE layer ("colibrì 架构概述" §4, expert cache and scheduling layer; §5, the moe
// step's pin -> LRU -> load order, autopin, repin_pass and pilot_prefetch; ai4coding.ru
// "Обучающийся кэш", the decaying session heat map).  The rules are stated in coli_tier.h.  Every call is O(ids + evictions) except repin and state (O(n_experts)).
#include <algorithm>
#include <cstdio>
#include <cstring>
#include <new>
#include <vector>

#include "coli_tier.h"

namespace {

enum : int8_t { kAbsent = 0, kPinned = 1, kInLru = 2 };

struct Layer {
  std::vector<int8_t> where;     // kAbsent / kPinned / kInLru, per expert
  std::vector<int32_t> slot;     // slot of a resident expert, else -1
  std::vector<int32_t> prev;     // LRU links by expert id (-1 = none); prev points to the
  std::vector<int32_t> next;     // more recently used neighbour
  int32_t head = -1, tail = -1;  // most and least recently used
  int lru_size = 0, pin_size = 0;
  std::vector<int64_t> heat;       // usage heat: cumulative use count
  std::vector<int64_t> session;    // session heat: use count, halved by coli_tier_decay
  std::vector<uint8_t> marked;     // loaded by a prefetch, not used yet
  std::vector<uint64_t> free_bits; // bit s set: slot s is free
  std::vector<uint32_t> stamp;     // == the tier's call counter: the expert is in this call
};

enum { kPinHits, kLruHits, kMisses, kEvictions, kPfFetches, kPfUsed, kPfWasted, kRepinFetches };

}  // namespace

struct coli_tier {
  int n_layers = 0, n_experts = 0, n_pin = 0, n_lru = 0, n_slots = 0;
  std::vector<Layer> layers;
  int64_t stats[COLI_TIER_N_STATS] = {};
  uint32_t call = 0;
};

namespace {

void unlink(Layer& L, int32_t e) {
  const int32_t p = L.prev[e], n = L.next[e];
  if (p >= 0) L.next[p] = n; else L.head = n;
  if (n >= 0) L.prev[n] = p; else L.tail = p;
  L.prev[e] = L.next[e] = -1;
  --L.lru_size;
}

void push_front(Layer& L, int32_t e) {
  L.prev[e] = -1;
  L.next[e] = L.head;
  if (L.head >= 0) L.prev[L.head] = e; else L.tail = e;
  L.head = e;
  ++L.lru_size;
}

int32_t take_slot(Layer& L) {  // lowest free slot
  for (size_t w = 0; w < L.free_bits.size(); ++w) {
    if (L.free_bits[w]) {
      const int b = __builtin_ctzll(L.free_bits[w]);
      L.free_bits[w] &= L.free_bits[w] - 1;
      return (int32_t)(w * 64 + b);
    }
  }
  // Not reached.  A layer has n_pin + n_lru slots; a load happens only after the same call's
  // evictions and drops, when at most n_pin pinned and n_lru listed experts remain with it.
  return -1;
}

void free_slot(Layer& L, int32_t s) { L.free_bits[s >> 6] |= 1ull << (s & 63); }

uint32_t next_call(coli_tier* t) {
  if (++t->call == 0) {  // the counter wrapped: clear every stamp once
    for (Layer& L : t->layers) std::fill(L.stamp.begin(), L.stamp.end(), 0u);
    t->call = 1;
  }
  return t->call;
}

bool ids_ok(const coli_tier* t, int layer, const int32_t* ids, int n) {
  if (layer < 0 || layer >= t->n_layers || n < 0 || (n > 0 && !ids)) return false;
  for (int i = 0; i < n; ++i) {
    if (ids[i] < 0 || ids[i] >= t->n_experts) return false;
    if (i > 0 && ids[i - 1] >= ids[i]) return false;
  }
  return true;
}

// Evicts the n_evict least recently used experts of L that are not in the current call,
// least recent first; enough of them exist because a call holds at most n_lru unpinned ids.
void evict_tail(coli_tier* t, Layer& L, int n_evict, uint32_t call, int32_t* ids, int32_t* slots,
                int* count) {
  int k = 0;
  int32_t e = L.tail;
  while (k < n_evict && e >= 0) {
    const int32_t before = L.prev[e];
    if (L.stamp[e] != call) {
      if (ids) ids[k] = e;
      if (slots) slots[k] = L.slot[e];
      unlink(L, e);
      free_slot(L, L.slot[e]);
      L.slot[e] = -1;
      L.where[e] = kAbsent;
      if (L.marked[e]) {
        L.marked[e] = 0;
        ++t->stats[kPfWasted];
      }
      ++t->stats[kEvictions];
      ++k;
    }
    e = before;
  }
  if (count) *count = k;
}

// The unpinned experts among ids (ascending) move to the front: the largest id ends in front.
void to_front(Layer& L, const int32_t* ids, int n) {
  for (int i = 0; i < n; ++i) {
    const int32_t e = ids[i];
    if (L.where[e] == kPinned) continue;
    if (L.where[e] == kInLru) unlink(L, e);
    push_front(L, e);
    L.where[e] = kInLru;
  }
}

void put_le(unsigned char* p, uint64_t v, int bytes) {
  for (int i = 0; i < bytes; ++i) p[i] = (unsigned char)(v >> (8 * i));
}

uint64_t get_le(const unsigned char* p, int bytes) {
  uint64_t v = 0;
  for (int i = 0; i < bytes; ++i) v |= (uint64_t)p[i] << (8 * i);
  return v;
}

const char kMagic[8] = {'C', 'O', 'L', 'I', 'U', 'S', 'E', '1'};

}  // namespace

extern "C" {

int coli_tier_create(const coli_tier_config* cfg, coli_tier** out) {
  if (!cfg || !out) return COLI_EINVAL;
  *out = nullptr;
  const coli_tier_config c = *cfg;
  if (c.n_layers < 1 || c.n_layers > 4096 || c.n_experts < 1 || c.n_experts > 65536 ||
      c.n_pin < 0 || c.n_pin > c.n_experts || c.n_lru < 1 || c.n_lru > c.n_experts ||
      (int64_t)c.n_layers * c.n_experts > (int64_t)1 << 24)
    return COLI_EINVAL;
  coli_tier* t = new (std::nothrow) coli_tier;
  if (!t) return COLI_ENOMEM;
  try {
    t->n_layers = c.n_layers;
    t->n_experts = c.n_experts;
    t->n_pin = c.n_pin;
    t->n_lru = c.n_lru;
    t->n_slots = c.n_pin + c.n_lru;
    t->layers.resize(c.n_layers);
    const size_t E = (size_t)c.n_experts, words = ((size_t)t->n_slots + 63) / 64;
    for (Layer& L : t->layers) {
      L.where.assign(E, kAbsent);
      L.slot.assign(E, -1);
      L.prev.assign(E, -1);
      L.next.assign(E, -1);
      L.heat.assign(E, 0);
      L.session.assign(E, 0);
      L.marked.assign(E, 0);
      L.stamp.assign(E, 0u);
      L.free_bits.assign(words, ~0ull);
      if (t->n_slots % 64) L.free_bits[words - 1] = (1ull << (t->n_slots % 64)) - 1;
    }
  } catch (const std::bad_alloc&) {
    delete t;
    return COLI_ENOMEM;
  }
  *out = t;
  return COLI_OK;
}

void coli_tier_destroy(coli_tier* t) { delete t; }

int coli_tier_lookup(coli_tier* t, int layer, const int32_t* ids, int n, int32_t* cls,
                     int32_t* slot, int32_t* fetch_ids, int32_t* fetch_slots, int* n_fetch,
                     int32_t* evict_ids, int32_t* evict_slots, int* n_evict) {
  if (!t || !ids_ok(t, layer, ids, n)) return COLI_EINVAL;
  Layer& L = t->layers[layer];
  int unpinned = 0, misses = 0;
  for (int i = 0; i < n; ++i) {
    unpinned += L.where[ids[i]] != kPinned;
    misses += L.where[ids[i]] == kAbsent;
  }
  if (unpinned > t->n_lru) return COLI_EINVAL;
  const uint32_t call = next_call(t);
  for (int i = 0; i < n; ++i) {
    const int32_t e = ids[i];
    L.stamp[e] = call;
    ++L.heat[e];
    ++L.session[e];
    const int c = L.where[e] == kPinned ? COLI_TIER_PIN_HIT
                : L.where[e] == kInLru  ? COLI_TIER_LRU_HIT
                                        : COLI_TIER_MISS;
    if (cls) cls[i] = c;
    ++t->stats[c == COLI_TIER_PIN_HIT ? kPinHits : c == COLI_TIER_LRU_HIT ? kLruHits : kMisses];
    if (c == COLI_TIER_LRU_HIT && L.marked[e]) {
      L.marked[e] = 0;
      ++t->stats[kPfUsed];
    }
  }
  evict_tail(t, L, std::max(0, L.lru_size + misses - t->n_lru), call, evict_ids, evict_slots,
             n_evict);
  int k = 0;
  for (int i = 0; i < n; ++i) {
    const int32_t e = ids[i];
    if (L.where[e] != kAbsent) continue;
    L.slot[e] = take_slot(L);
    if (fetch_ids) fetch_ids[k] = e;
    if (fetch_slots) fetch_slots[k] = L.slot[e];
    ++k;
  }
  if (n_fetch) *n_fetch = k;
  to_front(L, ids, n);
  if (slot)
    for (int i = 0; i < n; ++i) slot[i] = L.slot[ids[i]];
  return COLI_OK;
}

int coli_tier_prefetch(coli_tier* t, int layer, const int32_t* ids, int n, int32_t* fetch_ids,
                       int32_t* fetch_slots, int* n_fetch, int32_t* evict_ids,
                       int32_t* evict_slots, int* n_evict) {
  if (!t || !ids_ok(t, layer, ids, n) || n > t->n_lru) return COLI_EINVAL;
  Layer& L = t->layers[layer];
  const uint32_t call = next_call(t);
  int loads = 0;
  for (int i = 0; i < n; ++i) {
    L.stamp[ids[i]] = call;
    loads += L.where[ids[i]] == kAbsent;
  }
  evict_tail(t, L, std::max(0, L.lru_size + loads - t->n_lru), call, evict_ids, evict_slots,
             n_evict);
  int k = 0;
  for (int i = 0; i < n; ++i) {
    const int32_t e = ids[i];
    if (L.where[e] != kAbsent) continue;
    L.slot[e] = take_slot(L);
    L.marked[e] = 1;
    ++t->stats[kPfFetches];
    if (fetch_ids) fetch_ids[k] = e;
    if (fetch_slots) fetch_slots[k] = L.slot[e];
    ++k;
  }
  if (n_fetch) *n_fetch = k;
  to_front(L, ids, n);
  return COLI_OK;
}

}  // extern "C"

namespace {

// New pinned set of L: the n_pin first of the pinned experts and every expert with key > 0,
// ranked by key (higher first), then pinned before unpinned, then lower id.
int pin_by(coli_tier* t, Layer& L, const std::vector<int64_t>& key, int32_t* fetch_ids,
           int32_t* fetch_slots, int* n_fetch, int32_t* drop_ids, int32_t* drop_slots,
           int* n_drop) {
  std::vector<int32_t> hot;
  try {
    for (int32_t e = 0; e < t->n_experts; ++e)
      if (key[e] > 0 || L.where[e] == kPinned) hot.push_back(e);
  } catch (const std::bad_alloc&) {
    return COLI_ENOMEM;
  }
  const size_t keep = std::min(hot.size(), (size_t)t->n_pin);
  std::partial_sort(hot.begin(), hot.begin() + keep, hot.end(), [&L, &key](int32_t a, int32_t b) {
    if (key[a] != key[b]) return key[a] > key[b];
    const bool pa = L.where[a] == kPinned, pb = L.where[b] == kPinned;
    return pa != pb ? pa : a < b;
  });
  hot.resize(keep);
  std::sort(hot.begin(), hot.end());
  const uint32_t call = next_call(t);
  for (int32_t e : hot) L.stamp[e] = call;
  int k = 0;
  for (int32_t e = 0; e < t->n_experts; ++e) {  // drops first: they free slots
    if (L.where[e] != kPinned || L.stamp[e] == call) continue;
    if (drop_ids) drop_ids[k] = e;
    if (drop_slots) drop_slots[k] = L.slot[e];
    ++k;
    free_slot(L, L.slot[e]);
    L.slot[e] = -1;
    L.where[e] = kAbsent;
    --L.pin_size;
  }
  if (n_drop) *n_drop = k;
  k = 0;
  for (int32_t e : hot) {
    if (L.where[e] == kPinned) continue;
    if (L.where[e] == kInLru) {  // keeps its slot and its loaded record
      unlink(L, e);
      if (L.marked[e]) {
        L.marked[e] = 0;
        ++t->stats[kPfUsed];
      }
    } else {
      L.slot[e] = take_slot(L);
      ++t->stats[kRepinFetches];
      if (fetch_ids) fetch_ids[k] = e;
      if (fetch_slots) fetch_slots[k] = L.slot[e];
      ++k;
    }
    L.where[e] = kPinned;
    ++L.pin_size;
  }
  if (n_fetch) *n_fetch = k;
  return COLI_OK;
}

}  // namespace

extern "C" {

int coli_tier_repin(coli_tier* t, int layer, int32_t* fetch_ids, int32_t* fetch_slots,
                    int* n_fetch, int32_t* drop_ids, int32_t* drop_slots, int* n_drop) {
  if (!t || layer < 0 || layer >= t->n_layers) return COLI_EINVAL;
  Layer& L = t->layers[layer];
  return pin_by(t, L, L.session, fetch_ids, fetch_slots, n_fetch, drop_ids, drop_slots, n_drop);
}

int coli_tier_autopin(coli_tier* t, int layer, int32_t* fetch_ids, int32_t* fetch_slots,
                      int* n_fetch, int32_t* drop_ids, int32_t* drop_slots, int* n_drop) {
  if (!t || layer < 0 || layer >= t->n_layers) return COLI_EINVAL;
  Layer& L = t->layers[layer];
  return pin_by(t, L, L.heat, fetch_ids, fetch_slots, n_fetch, drop_ids, drop_slots, n_drop);
}

int coli_tier_decay(coli_tier* t) {
  if (!t) return COLI_EINVAL;
  for (Layer& L : t->layers)
    for (int64_t& v : L.session) v >>= 1;  // counts are never negative: this rounds down
  return COLI_OK;
}

int coli_tier_state(const coli_tier* t, int layer, int32_t* pinned, int* n_pinned,
                    int32_t* lru, int* n_lru_used, int32_t* slot_of) {
  if (!t || layer < 0 || layer >= t->n_layers) return COLI_EINVAL;
  const Layer& L = t->layers[layer];
  int k = 0;
  for (int32_t e = 0; e < t->n_experts; ++e) {
    if (L.where[e] == kPinned) {
      if (pinned) pinned[k] = e;
      ++k;
    }
    if (slot_of) slot_of[e] = L.slot[e];
  }
  if (n_pinned) *n_pinned = k;
  k = 0;
  for (int32_t e = L.head; e >= 0; e = L.next[e]) {
    if (lru) lru[k] = e;
    ++k;
  }
  if (n_lru_used) *n_lru_used = k;
  return COLI_OK;
}

int coli_tier_heat(const coli_tier* t, int layer, int64_t* heat) {
  if (!t || !heat || layer < 0 || layer >= t->n_layers) return COLI_EINVAL;
  std::memcpy(heat, t->layers[layer].heat.data(), sizeof(int64_t) * (size_t)t->n_experts);
  return COLI_OK;
}

int coli_tier_session_heat(const coli_tier* t, int layer, int64_t* heat) {
  if (!t || !heat || layer < 0 || layer >= t->n_layers) return COLI_EINVAL;
  std::memcpy(heat, t->layers[layer].session.data(), sizeof(int64_t) * (size_t)t->n_experts);
  return COLI_OK;
}

int coli_tier_set_heat(coli_tier* t, int layer, const int64_t* heat) {
  if (!t || !heat || layer < 0 || layer >= t->n_layers) return COLI_EINVAL;
  for (int e = 0; e < t->n_experts; ++e)
    if (heat[e] < 0) return COLI_EINVAL;
  std::memcpy(t->layers[layer].heat.data(), heat, sizeof(int64_t) * (size_t)t->n_experts);
  return COLI_OK;
}

int coli_tier_config_of(const coli_tier* t, coli_tier_config* out) {
  if (!t || !out) return COLI_EINVAL;
  *out = coli_tier_config{t->n_layers, t->n_experts, t->n_pin, t->n_lru};
  return COLI_OK;
}

int coli_tier_stats(const coli_tier* t, int64_t* stats) {
  if (!t || !stats) return COLI_EINVAL;
  std::memcpy(stats, t->stats, sizeof(t->stats));
  return COLI_OK;
}

int coli_tier_save_usage(const coli_tier* t, const char* path) {
  if (!t || !path) return COLI_EINVAL;
  std::vector<unsigned char> buf;
  try {
    buf.resize(16 + (size_t)8 * t->n_layers * t->n_experts);
  } catch (const std::bad_alloc&) {
    return COLI_ENOMEM;
  }
  std::memcpy(buf.data(), kMagic, 8);
  put_le(buf.data() + 8, (uint32_t)t->n_layers, 4);
  put_le(buf.data() + 12, (uint32_t)t->n_experts, 4);
  unsigned char* p = buf.data() + 16;
  for (const Layer& L : t->layers)
    for (int64_t v : L.heat) {
      put_le(p, (uint64_t)v, 8);
      p += 8;
    }
  FILE* f = std::fopen(path, "wb");
  if (!f) return COLI_EIO;
  const bool ok = std::fwrite(buf.data(), 1, buf.size(), f) == buf.size();
  return (std::fclose(f) == 0 && ok) ? COLI_OK : COLI_EIO;
}

int coli_tier_load_usage(coli_tier* t, const char* path) {
  if (!t || !path) return COLI_EINVAL;
  FILE* f = std::fopen(path, "rb");
  if (!f) return COLI_EIO;
  unsigned char head[16];
  int rc = COLI_OK;
  std::vector<unsigned char> body;
  if (std::fread(head, 1, 16, f) != 16) {
    rc = COLI_EIO;
  } else if (std::memcmp(head, kMagic, 8) != 0 || get_le(head + 8, 4) != (uint32_t)t->n_layers ||
             get_le(head + 12, 4) != (uint32_t)t->n_experts) {
    rc = COLI_EINVAL;
  } else {
    try {
      body.resize((size_t)8 * t->n_layers * t->n_experts);
    } catch (const std::bad_alloc&) {
      rc = COLI_ENOMEM;
    }
    if (rc == COLI_OK && std::fread(body.data(), 1, body.size(), f) != body.size()) rc = COLI_EIO;
    if (rc == COLI_OK && std::fgetc(f) != EOF) rc = COLI_EINVAL;  // trailing bytes
  }
  std::fclose(f);
  if (rc != COLI_OK) return rc;
  for (size_t i = 0; i < body.size(); i += 8)
    if ((int64_t)get_le(body.data() + i, 8) < 0) return COLI_EINVAL;
  const unsigned char* p = body.data();
  for (Layer& L : t->layers)
    for (int64_t& v : L.heat) {
      v = (int64_t)get_le(p, 8);
      p += 8;
    }
  return COLI_OK;
}

}  // extern "C"

/* coli_tier -- the expert residency tiers of the int4 routed-expert MoE layers, C ABI.
 *
 * Not every expert of a large model fits in HBM. On a GB300 all expert records live in the
 * Grace host memory, and each MoE layer owns a pool of HBM slots of n_pin + n_lru records.
 * This object decides which experts sit in which slots. It runs on the host, needs no GPU, and
 * moves no data: every call returns the loads and evictions it decided, and the caller copies
 * the records into the named slots. The decisions follow "colibrì 架构概述":
 *   - §4 (expert cache and scheduling layer): a per-layer LRU cache, a pinned hot store,
 *     heat-driven repinning and router-lookahead prefetch;
 *   - §5 (the life of a token): look up pin, then the LRU cache, and load on a miss, with LRU
 *     promotion after the expert computation; at start-up, pin the hottest experts learned in
 *     the usage file; repin at turn boundaries, swapping cold pinned experts for hot ones;
 *   - README "統一記憶體階層": a learning cache records where the workload routes and pins the
 *     hottest experts;
 *   - README "絕不為同一次硬碟讀取等待兩遍": the next layer's router predicts its experts
 *     one layer ahead;
 *   - ai4coding.ru "colibrì: движок GLM-5.2", "Обучающийся кэш": start-up pins the hottest
 *     experts of the usage file, and the optional live repin (--repin N) swaps cold pinned
 *     experts for hotter ones by a decaying session heat map.
 *
 * The rules below fix the steps the pages leave open:
 *   - Per layer there is a pinned set (at most n_pin experts) and an LRU list (at most n_lru
 *     experts, most recently used first). The two are disjoint. The shared expert is always
 *     resident and is not tracked here.
 *   - A lookup classifies each expert of a call as a pinned hit, an LRU hit or a miss, and
 *     adds 1 to its usage heat and its session heat.
 *   - The lookup then loads the misses and moves every unpinned expert of the call to the
 *     front of the list, in ascending id order, so the largest id ends in front. It cuts the
 *     list back to n_lru from its tail; those experts are evicted, least recent first.
 *   - So a call never evicts an expert it uses, and the recency order does not depend on
 *     n_lru.
 *   - A prefetch does the same for predicted experts, without heat or hits, and marks each
 *     expert it loads.
 *   - A marked expert later counts as a used prefetch (an LRU hit on it, or a repin that pins
 *     it) or as a wasted one (it is evicted).
 *   - Usage heat is a cumulative use count, and the usage file saves it. Session heat counts
 *     the same uses, but coli_tier_decay halves it (rounding down). The caller's interval
 *     between decays sets its half-life.
 *   - Autopin pins by usage heat (start-up); repin pins by session heat (live). Both rank the
 *     pinned experts and every expert with heat > 0: higher heat first, then pinned before
 *     unpinned, then the lower id. The top n_pin form the new pinned set. So an expert replaces
 *     a pinned one only if strictly hotter, and a map of zeros changes nothing.
 *   - Experts that leave the set are dropped. An entering expert found in the LRU list keeps
 *     its slot; any other entering expert is loaded.
 *
 * Slots are layer-local indices 0 .. n_pin+n_lru-1. Each resident expert holds exactly one
 * slot, and keeps it until it is evicted or dropped. A load takes the lowest free slot after
 * the same call's evictions and drops have freed theirs.
 *
 * Conventions are those of coli_moe.h. Every call returns COLI_OK or a negative COLI_E*
 * status. A rejected call changes nothing. All arrays are host memory owned by the caller.
 * One handle must not be used by two threads at once.
 */
#ifndef COLI_TIER_H
#define COLI_TIER_H

#include <stdint.h>

#include "coli_moe.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct coli_tier coli_tier;

typedef struct {
  int n_layers;  /* MoE layers, 1 .. 4096                                       */
  int n_experts; /* routed experts per layer, 1 .. 65536 (ids 0 .. n_experts-1) */
  int n_pin;     /* pinned slots per layer, 0 .. n_experts                      */
  int n_lru;     /* LRU slots per layer, 1 .. n_experts                         */
} coli_tier_config; /* and n_layers * n_experts <= 2^24 (about 30 bytes of state each) */

/* Hit classes written by coli_tier_lookup. */
#define COLI_TIER_PIN_HIT 0
#define COLI_TIER_LRU_HIT 1
#define COLI_TIER_MISS 2

/* Counters of coli_tier_stats, in this order. */
#define COLI_TIER_N_STATS 8 /* pin_hits, lru_hits, misses, evictions, prefetch_fetches,
                               prefetch_used, prefetch_wasted, repin_fetches */

/* Creates an empty tier: nothing is resident and all heat is 0.  EINVAL: NULL argument or a
 * configuration outside the limits above.  ENOMEM: host allocation failed. */
int coli_tier_create(const coli_tier_config* cfg, coli_tier** out);
void coli_tier_destroy(coli_tier* t);

/* One call's experts in `layer`: ids[n] distinct, ascending, in [0, n_experts), at most n_lru
 * of them outside the pinned set (the batch union of one forward satisfies this whenever
 * n_lru >= top_k * tokens).  Outputs, any of which may be NULL:
 *   cls[n]          COLI_TIER_PIN_HIT / _LRU_HIT / _MISS of each id;
 *   slot[n]         the slot of each id after the call;
 *   fetch_ids[n], fetch_slots[n], *n_fetch    the misses (ascending) and their new slots;
 *   evict_ids[n], evict_slots[n], *n_evict    the evicted experts (least recent first) and
 *                                             the slots they freed.
 * The caller copies each fetched record into its slot before the layer's kernels read it; an
 * evicted slot may be overwritten once no earlier work reads it.  EINVAL: NULL t or ids with
 * n > 0, a bad layer, or ids that break the rules above. */
int coli_tier_lookup(coli_tier* t, int layer, const int32_t* ids, int n, int32_t* cls,
                     int32_t* slot, int32_t* fetch_ids, int32_t* fetch_slots, int* n_fetch,
                     int32_t* evict_ids, int32_t* evict_slots, int* n_evict);

/* Predicted experts of `layer` (ids[n] distinct, ascending, in range, n <= n_lru): the
 * router-lookahead read-ahead.  Outputs as in coli_tier_lookup (fetch/evict arrays of n
 * entries, any may be NULL).  Counts no heat and no hits.  EINVAL as in coli_tier_lookup. */
int coli_tier_prefetch(coli_tier* t, int layer, const int32_t* ids, int n, int32_t* fetch_ids,
                       int32_t* fetch_slots, int* n_fetch, int32_t* evict_ids,
                       int32_t* evict_slots, int* n_evict);

/* Live repin of `layer` by its session heat (coli_tier_autopin: the same by usage heat, for
 * start-up after coli_tier_load_usage).  Outputs (any may be NULL; arrays of n_pin entries):
 * fetch_ids/fetch_slots/*n_fetch  the entering experts that must be loaded (ascending);
 * drop_ids/drop_slots/*n_drop     the experts that left the pinned set (ascending) and the
 *                                 slots they freed.
 * EINVAL: NULL t or a bad layer. */
int coli_tier_repin(coli_tier* t, int layer, int32_t* fetch_ids, int32_t* fetch_slots,
                    int* n_fetch, int32_t* drop_ids, int32_t* drop_slots, int* n_drop);
int coli_tier_autopin(coli_tier* t, int layer, int32_t* fetch_ids, int32_t* fetch_slots,
                      int* n_fetch, int32_t* drop_ids, int32_t* drop_slots, int* n_drop);

/* Halves every layer's session heat (rounding down).  EINVAL: NULL t. */
int coli_tier_decay(coli_tier* t);

/* State of `layer`: pinned[n_pin] ascending and *n_pinned; lru[n_lru] most recent first and
 * *n_lru_used; slot_of[n_experts] (-1 = not resident); any output may be NULL.
 * EINVAL: NULL t or a bad layer. */
int coli_tier_state(const coli_tier* t, int layer, int32_t* pinned, int* n_pinned,
                    int32_t* lru, int* n_lru_used, int32_t* slot_of);

/* Usage heat of `layer`: heat[n_experts], the number of lookups that used each expert (or
 * what coli_tier_set_heat / coli_tier_load_usage put there); coli_tier_session_heat gives the
 * decayed session heat.  EINVAL: NULL argument, bad layer, or (set) a negative count. */
int coli_tier_heat(const coli_tier* t, int layer, int64_t* heat);
int coli_tier_session_heat(const coli_tier* t, int layer, int64_t* heat);
int coli_tier_set_heat(coli_tier* t, int layer, const int64_t* heat);

/* The configuration the tier was created with.  EINVAL: NULL argument. */
int coli_tier_config_of(const coli_tier* t, coli_tier_config* out);

/* stats[COLI_TIER_N_STATS], the counters listed above, summed over all layers since create. */
int coli_tier_stats(const coli_tier* t, int64_t* stats);

/* The usage file: the usage heat of every layer, so a later process can pin the hottest
 * experts at start-up (coli_tier_load_usage, then coli_tier_autopin per layer).  Format: the 8
 * bytes "COLIUSE1", int32 n_layers, int32 n_experts, then int64 heat[n_layers][n_experts],
 * all little-endian.  save writes the whole file or reports an error.  load replaces every
 * layer's heat only after the whole file has been read and checked.  EINVAL: NULL argument,
 * or a file whose magic or shape does not match this tier.  EIO: the file cannot be opened,
 * read or written in full. */
int coli_tier_save_usage(const coli_tier* t, const char* path);
int coli_tier_load_usage(coli_tier* t, const char* path);

/* ---- The device side: tiered coli_moe layers (created with 0 < hbm_slots < n_experts) ----
 *
 * Such a layer keeps every expert record in pinned host (Grace) memory, in the layout its
 * kernels stream, and hbm_slots routed records plus the shared expert in HBM; its kernels find
 * each record through a slot table on the device.  Where an expert sits changes how fast a
 * forward runs, never what it computes: the tiered forward is bit-identical to the all-resident
 * layer's.  The tier passed to these calls must have n_experts equal to the layer's experts and
 * n_pin + n_lru equal to its hbm_slots; `layer` is the layer's index in the tier.  Placements
 * copy each record with one copy per part (gate/up rows, down rows, scales) and then update the
 * slot table, in the order of the given stream. */

/* Forward of T tokens with host-decided placement ("colibrì 架构概述" §5: pin, then LRU, then
 * load; README "統一記憶體階層"): the routing runs on `stream`, the call waits for its union,
 * coli_tier_lookup decides the loads and evictions, the missing records are copied to their
 * slots, and the expert kernels run.  Batches run in chunks of at most n_lru / top_k tokens so
 * that a chunk's union fits the LRU slots.  The call synchronises `stream` once per chunk (to
 * read the union); it waits (on the device) for placements made by the two calls below.
 * Arguments and errors as coli_moe_forward, plus EINVAL for a tier that does not match the
 * layer and EUNSUPPORTED when n_lru < top_k. */
int coli_moe_forward_tiered(coli_moe* h, coli_tier* tier, int layer, const float* x_dev, int T,
                            float* y_dev, void* stream);

/* Router-lookahead read-ahead ("colibrì 架构概述" §4 pilot_prefetch; README: the next layer's
 * router predicts its experts one layer ahead): coli_tier_prefetch on ids[n] (host memory, as
 * that call takes them), then the copies on `stream`, after the layer's last forward (an event
 * wait) and before its next one (the next forward waits for them).  Use one stream for the
 * prefetch and repin calls of a layer. */
int coli_moe_prefetch_tiered(coli_moe* h, coli_tier* tier, int layer, const int32_t* ids, int n,
                             void* stream);

/* coli_tier_repin (by_usage = 0: session heat, the live repin) or coli_tier_autopin (by_usage =
 * 1: usage heat, at start-up) of the layer, carried out like a prefetch: dropped experts leave
 * the slot table, entering ones are copied in. */
int coli_moe_repin_tiered(coli_moe* h, coli_tier* tier, int layer, int by_usage, void* stream);

/* Records and bytes copied from host memory into the layer's HBM slots since it was created
 * (the traffic over the host link that the placements caused).  EINVAL: NULL argument. */
int coli_moe_tier_copies(const coli_moe* h, int64_t* records, int64_t* bytes);

#ifdef __cplusplus
}
#endif

#endif /* COLI_TIER_H */

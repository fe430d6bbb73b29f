/*
 * moe_residency.h — host-side slot planner of the partially resident expert
 * pool (MOE_RESIDENCY_PARTIAL in moe_layer.h), exposed for tests and tools.
 * Pure host code: no CUDA call is made by these functions.
 *
 * Background (pages): the Horizon RunMap report, "Partial-residency
 * contract", keeps every routed expert in an immutable host copy and moves
 * only demanded compact copies to the GPU; eviction discards GPU copies and
 * never writes the host copy back. The F51 Nitro-MoE page, "Layer 1 - expert
 * persistence cache", describes the structure as a fixed pool of GPU slots
 * with expert_to_slot / slot_to_expert maps, a last-used time per slot and
 * hit/miss counters. The moe-stream page, "Findings", shows why plain LRU in a
 * fixed expert order gets no hits once the working set exceeds the pool.
 *
 * Planning one forward: the demanded experts are split into waves of at most
 * num_slots experts that are resident together. Wave 0 holds every demanded
 * expert already resident (hits) plus as many misses as fit in the slots not
 * holding a hit (empty slots first, then least recently used). Later waves
 * reuse all slots for the remaining misses in ascending expert id. With
 * MOE_PLAN_FIXED_ORDER_LRU the experts are instead visited in ascending id
 * order with plain LRU replacement (the baseline the moe-stream page
 * measures).
 */
#ifndef MOE_RESIDENCY_H
#define MOE_RESIDENCY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_slot_planner moe_slot_planner_t;

enum { MOE_PLAN_HITS_FIRST = 0, MOE_PLAN_FIXED_ORDER_LRU = 1 };

/* New planner with all slots empty; NULL if n_records < 1 or num_slots < 1. */
moe_slot_planner_t* moe_slot_planner_create(int32_t n_records, int32_t num_slots);

/* Plans one forward for `n` distinct demanded expert ids (any order, each in
 * [0, n_records)) and applies it to the planner state. For the i-th demanded
 * expert (in ascending id order) it writes: wave_of[i] (wave index), slot_of[i]
 * (slot the expert occupies during its wave), hit[i] (1 if it was resident
 * before the call). *n_waves receives the number of waves. Returns 0, or -1 on
 * an invalid argument (duplicate or out-of-range id, NULL pointer). */
int32_t moe_slot_planner_plan(moe_slot_planner_t* planner, const int32_t* demanded, int32_t n, int32_t policy,
                              int32_t* wave_of, int32_t* slot_of, int32_t* hit, int32_t* n_waves);

/* Slot currently holding `expert`, or -1. */
int32_t moe_slot_planner_slot_of(const moe_slot_planner_t* planner, int32_t expert);

/* Marks a slot empty (its contents are no longer trusted). */
void moe_slot_planner_invalidate(moe_slot_planner_t* planner, int32_t slot);

/* NULL is accepted. */
void moe_slot_planner_destroy(moe_slot_planner_t* planner);

/* ------------------------------------------------------------------------
 * Expert cache model (the partially resident pool's bookkeeping, pure host
 * code). Horizon RunMap report, "Partial-residency contract", steps 1-7: a
 * forward works on a complete published generation; misses are loaded into
 * unpublished rows (spare rows, or the rows of victims once their consumers
 * have retired) and become visible only when the whole routed group is
 * published as a new generation; a transaction that fails before
 * publication leaves the old generation authoritative; eviction discards
 * GPU copies. Policies (F51 Nitro-MoE, "Layer 1 - expert persistence
 * cache"; moe-stream, "Findings"): least recently used, least frequently
 * used (every access counted), and LRU-FREQ, scoring freq * 1000 - age with
 * all frequencies multiplied by 0.75 after every 2 x capacity misses; the
 * lowest score is evicted first, ties to the lower row. */
typedef struct moe_expert_cache moe_expert_cache_t;

enum { MOE_CACHE_LRU = 0, MOE_CACHE_LFU = 1, MOE_CACHE_LRU_FREQ = 2 };

/* A cache of `capacity` published rows plus `spare_rows` unpublished rows,
 * all empty; NULL on an invalid argument. */
moe_expert_cache_t* moe_expert_cache_create(int32_t n_records, int32_t capacity, int32_t spare_rows, int32_t policy);

/* One forward over n distinct demanded experts (any order): every access is
 * counted (in ascending id), then transactions of at most `capacity`
 * experts (the resident ones first, then misses in ascending id) are
 * planned and published one after another. For demanded[i] it writes
 * txn_of[i], row_of[i] (the row it is read from) and hit[i] (resident
 * before the call); *n_txn receives the number of transactions. If
 * abort_txn >= 0, that transaction fails before publication instead: the
 * state keeps the previous generation, *n_txn is set to abort_txn and the
 * call returns 1. Returns 0, or -1 on an invalid argument. */
int32_t moe_expert_cache_access(moe_expert_cache_t* cache, const int32_t* demanded, int32_t n, int32_t abort_txn,
                                int32_t* txn_of, int32_t* row_of, int32_t* hit, int32_t* n_txn);

/* Published row of `expert`, or -1. */
int32_t moe_expert_cache_row_of(const moe_expert_cache_t* cache, int32_t expert);

/* out5[0..4] = hits, misses, evictions, generations published, frequency
 * decays. Returns 0, or -1 on NULL. */
int32_t moe_expert_cache_stats(const moe_expert_cache_t* cache, uint64_t* out5);

/* A prefetch (moe-stream, "Findings": the next layer's router run early on
 * the current state guesses its experts): the n distinct guessed experts
 * (at most `capacity` are made resident; resident ones are kept) are planned
 * as one transaction without counting accesses, and published. Returns the
 * number of experts it loaded, or -1 on an invalid argument. */
int32_t moe_expert_cache_prefetch(moe_expert_cache_t* cache, const int32_t* guessed, int32_t n);

/* out2[0] = experts loaded by prefetches, out2[1] = those demanded by a
 * later access while still resident (each counted once). */
int32_t moe_expert_cache_prefetch_stats(const moe_expert_cache_t* cache, uint64_t* out2);

/* NULL is accepted. */
void moe_expert_cache_destroy(moe_expert_cache_t* cache);

#ifdef __cplusplus
}
#endif

#endif /* MOE_RESIDENCY_H */

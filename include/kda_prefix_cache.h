/*
 * kda_prefix_cache.h -- host prefix-cache index of libkda.so.
 *
 * A KDA layer keeps one fixed-size state per head.  A prompt prefix can therefore
 * be reused only where a state was saved ("Kimi K3 Tech Intro", section 2.1).
 * This index decides, for every new request, which saved state the prefill can
 * resume from.  It also decides which of the request's states to save.  Its plan
 * fills exactly the inputs kda_prefill_chunked() takes: start_pos, init_slot and
 * one row of snap_table.  The index runs on the host only.  It never touches
 * device memory and needs no GPU.
 *
 * What it implements ("Kimi K3 Tech Intro"):
 *  - section 2.2: prefixes match in units of `match_unit` tokens (256).  The unit
 *    is independent of the physical block.
 *  - section 2.4, chained hash row: unit n of a prompt is identified by
 *        h_n = SHA-256(h_{n-1} || tokens of unit n as int32 little-endian),
 *    with h_0 = 32 zero bytes.  h_n identifies the whole prefix (logical id),
 *    not only its last unit.
 *  - section 2.3, copy-on-write: a matched state is shared and read-only.  The
 *    prefill reads it through init_slot and writes only its own outputs and
 *    new snapshots.
 *  - section 2.4, same-step reuse row: states registered in a step become
 *    matchable only after kda_pcache_end_step() reports that step finished.
 *  - section 3.1, interval retention: keep a state every `retention_interval`
 *    tokens plus the state at the prompt boundary.  0 keeps only the prompt
 *    boundary.
 *  - section 3.2, second-hit admission (Marconi-style): with
 *    `admit_on_second_hit`, a request whose prefix an earlier request already
 *    produced also keeps the state at the end of the shared part.  A prefix
 *    seen only once keeps nothing but its prompt-boundary state.
 *
 * Readings where the pages are silent:
 *  - The prompt boundary is floor(L / unit) * unit.  States exist only at unit
 *    boundaries.
 *  - A match leaves at least one prompt token to compute:
 *    start_pos <= L - 1.
 *  - The index owns pool slots [slot_base, slot_base + n_slots).  A new state
 *    takes the lowest free slot.  When none is free, it evicts the least
 *    recently used published entry that no request has pinned; ties go to the
 *    lower slot.  With no such entry, the state is not saved.
 *  - A matched entry stays pinned until kda_pcache_release() for that request.
 *    The caller releases a request after the prefill that reads the entry has
 *    completed.
 *
 * Conventions: every pointer here is a HOST pointer, owned by the caller.
 * Calls on one index are serialised by a lock inside it.  Errors return a
 * status with a message in kda_last_error().  An argument error leaves the
 * index unchanged.  After KDA_ERR_NO_MEMORY the index may hold a partial
 * update and must be destroyed.
 */
#ifndef KDA_PREFIX_CACHE_H
#define KDA_PREFIX_CACHE_H

#include <stdint.h>

#include "kda.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kda_pcache kda_pcache; /* opaque */

typedef struct {
    int32_t match_unit;          /* tokens per hashed unit; must equal the prefill's snap_interval (256) */
    int32_t admit_on_second_hit; /* nonzero: second-hit admission (section 3.2) */
    int64_t retention_interval;  /* 0, or a positive multiple of match_unit (section 3.1) */
    int64_t slot_base;           /* first pool slot the index owns */
    int64_t n_slots;             /* slots it owns (>= 0) */
} kda_pcache_config;

typedef struct {
    int64_t request_id; /* identifies the request in kda_pcache_release() */
    int64_t start_pos;  /* tokens the prefill skips; a multiple of match_unit */
    int32_t init_slot;  /* pool slot of the matched state, -1 = start from zeros */
    int32_t n_units;    /* floor(L / match_unit): entries of snap_row written */
    int32_t n_saved;    /* entries of snap_row that name a slot */
    int32_t reserved;
} kda_pcache_plan;

typedef struct {
    int64_t entries;    /* states registered or published */
    int64_t published;  /* states a request can match */
    int64_t pinned;     /* published states pinned by unreleased requests */
    int64_t free_slots;
    int64_t seen_units; /* distinct chained hashes seen (second-hit admission) */
    int64_t requests, hits, misses, evictions, dropped; /* dropped: states not saved for want of a slot */
} kda_pcache_stats;

/* Create an index.  KDA_ERR_INVALID_ARG: cfg or out NULL, match_unit < 1,
 * retention_interval negative or not a multiple of match_unit, slot_base < 0,
 * n_slots < 0, or slot_base + n_slots > 2^31.  KDA_ERR_NO_MEMORY: host
 * allocation failed.  *out is set only on KDA_OK. */
kda_status_t kda_pcache_create(const kda_pcache_config* cfg, kda_pcache** out);

/* Destroy an index (NULL is a no-op).  Pool slots are the caller's and are not touched. */
void kda_pcache_destroy(kda_pcache* pc);

/* Plan one request with prompt tokens[0 .. n_tokens).
 * On KDA_OK:
 *  - out->start_pos and out->init_slot are the resume point: the deepest
 *    published state of the prompt's prefix, with start_pos <= n_tokens - 1.
 *  - snap_row[o], for o < out->n_units, is the slot that the prefill writes
 *    the state at absolute position p = (o + 1) * match_unit into.  It is -1
 *    where no state is kept.  Such a slot is registered (pending) until
 *    kda_pcache_end_step().
 *  - Entries o >= out->n_units are left untouched.
 * The call pins the matched state.  Release the request with
 * kda_pcache_release() once its prefill has completed.
 * KDA_ERR_INVALID_ARG: pc, tokens or out NULL, n_tokens < 1,
 * snap_row NULL with n_units > 0, or snap_row_len < n_units. */
kda_status_t kda_pcache_plan_request(kda_pcache* pc, const int32_t* tokens, int64_t n_tokens, int32_t* snap_row,
                                     int64_t snap_row_len, kda_pcache_plan* out);

/* The step whose requests were planned since the last call has finished.
 * succeeded != 0: publish the states it registered, so that later requests can
 * match them.  succeeded == 0 (for example, kda_check_status reported a
 * device error): discard those states and free their slots. */
kda_status_t kda_pcache_end_step(kda_pcache* pc, int32_t succeeded);

/* The request no longer reads its matched state (unpins it).
 * KDA_ERR_INVALID_ARG: unknown or already released request_id. */
kda_status_t kda_pcache_release(kda_pcache* pc, int64_t request_id);

/* Counters of the index.  KDA_ERR_INVALID_ARG: pc or out NULL. */
kda_status_t kda_pcache_get_stats(const kda_pcache* pc, kda_pcache_stats* out);

/* The published state with logical id `hash` (32 bytes): *slot = its pool slot
 * and *pos = its absolute position.  If the id is unknown or not yet
 * published, *slot = -1 and *pos = 0.  Workers exchange logical ids, not
 * slots (section 2.4, cross-worker transfer row).
 * KDA_ERR_INVALID_ARG: a NULL pointer. */
kda_status_t kda_pcache_lookup(const kda_pcache* pc, const uint8_t* hash, int32_t* slot, int64_t* pos);

/* Register a state received from another worker under its logical id `hash`
 * at absolute position `pos` (a positive multiple of match_unit).
 * *slot is set as follows:
 *  - a new slot (pending), which the caller fills (kda_snapshot_restore) before
 *    kda_pcache_end_step();
 *  - -1 when the id is already registered or no slot can be had.
 * *is_new is 1 only in the first case.
 * KDA_ERR_INVALID_ARG: a NULL pointer or a bad pos. */
kda_status_t kda_pcache_import(kda_pcache* pc, const uint8_t* hash, int64_t pos, int32_t* slot, int32_t* is_new);

/* The chained hashes h_1 .. h_m (m = n_tokens / match_unit) of a prompt, 32
 * bytes each, into out[0 .. 32 m).  Needs no index.
 * KDA_ERR_INVALID_ARG: tokens NULL with n_tokens > 0, n_tokens < 0,
 * match_unit < 1, out NULL with m > 0, or out_len < 32 m. */
kda_status_t kda_pcache_unit_hashes(const int32_t* tokens, int64_t n_tokens, int32_t match_unit, uint8_t* out,
                                    int64_t out_len);

/*
 * State transfer by logical id ("Kimi K3 Tech Intro", section 2.4: workers pass
 * logical prefix identifiers, not physical addresses; section 7: the tail of a
 * transfer is zeroed so that no stale data leaks).  On one GPU this is a
 * gather into a transfer buffer and a restore out of one.  The slot lists are
 * resolved on the host and copied into the caller's device scratch, so the
 * library still allocates nothing.
 */

/* Gather the published states named by ids[0 .. n) (32-byte chained hashes,
 * host memory) into dst[0 .. capacity) (device, [capacity, H, d_k, d_v] fp32).
 *  - Entry i < n gets the state of ids[i].  It is all zeros when the id is
 *    unknown or not yet published.
 *  - Entries n .. capacity-1 (the tail) are zeroed.
 *  - pos_out[i] (host, may be NULL) receives the state's absolute position, or
 *    0 when the id was not found.
 * slot_scratch: device int32 [capacity], caller-owned, overwritten.  The states
 * are read when the gather runs on `stream`, in stream order: do not let other
 * streams overwrite those slots before it completes.
 * Errors:
 *   - KDA_ERR_INVALID_ARG: a NULL pointer, n < 0, capacity < n, or
 *     n_slots < 0;
 *   - the shape errors of kda_snapshot_gather;
 *   - KDA_ERR_CUDA: the copy or the launch failed. */
kda_status_t kda_state_export(const kda_pcache *pc, const uint8_t *ids, int32_t n, int32_t capacity,
                              const float *pool, int64_t n_slots, int32_t n_heads, int32_t d_k, int32_t d_v,
                              float *dst, int32_t *slot_scratch, int64_t *pos_out, void *stream);

/* Register the states of ids[0 .. n) with positions pos[0 .. n) (host
 * memory, positive multiples of match_unit) in this index, and copy the new
 * ones from src[0 .. n) (device, [n, H, d_k, d_v] fp32) into the slots they
 * got.  An id that is already registered, or that finds no slot, is skipped.
 * slots_out[i] (host, may be NULL) is the slot taken, or -1.  The states
 * become matchable at the next kda_pcache_end_step(pc, 1).  Call it once the
 * restore has completed on `stream`.
 * slot_scratch: device int32 [n], caller-owned, overwritten.
 * Errors:
 *   - KDA_ERR_INVALID_ARG: a NULL pointer, n < 0, or a bad position.  A bad
 *     position stops the registration at that id: earlier ids stay registered,
 *     and nothing is copied.
 *   - the shape errors of kda_snapshot_restore;
 *   - KDA_ERR_CUDA. */
kda_status_t kda_state_import(kda_pcache *pc, const uint8_t *ids, const int64_t *pos, int32_t n,
                              const float *src, float *pool, int64_t n_slots, int32_t n_heads, int32_t d_k,
                              int32_t d_v, int32_t *slot_scratch, int32_t *slots_out, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_PREFIX_CACHE_H */

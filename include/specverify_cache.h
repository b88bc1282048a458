/*
 * specverify_cache.h — C ABI of the ready-distribution cache on GB300.
 *
 * A device-resident table of session slots holding each session's pre-positioned decision
 * point and the gated summary of its ready distribution, with the three operations of
 * "Speculative Pre-Positioning":
 *
 *   ready_cache_record      Algorithm 1 (section 3.2), for a batch of updated sessions: skip
 *                           when the entry would over-commit the cell budget, else record the
 *                           decision point and the ready logits' (argmax, gamma) — one scan
 *                           of each ready row, the gate's scan — and mark the slot valid.
 *   ready_cache_serve       Algorithm 2 (section 3.4), for a batch of requests: fall through
 *                           when the slot is not valid or the request's entry differs from
 *                           the pre-positioned one; else serve the cached argmax iff
 *                           gamma > tau and it lies in the fast-answer set A (Eq. (12)).
 *   ready_cache_invalidate  section 3.6 and Figure 3: a mutation of the session state clears
 *                           the slot and returns it to "no ready distribution".
 *
 * The conventions of specverify.h hold. The table (slots, entry store, statistics) is caller
 * memory on the device; a zero-filled table is the empty cache. Calls that touch one table
 * must be ordered on one stream (or by events): each call reads the state the previous one
 * left, which is how an invalidation stays coupled to the mutation it follows.
 */
#ifndef SPECVERIFY_CACHE_H_
#define SPECVERIFY_CACHE_H_

#include "specverify.h"

#ifdef __cplusplus
extern "C" {
#endif

#define SV_CACHE_VALID 1u    /* the slot holds a current ready distribution */
#define SV_CACHE_DECODED 2u  /* its entry has been decoded into the session */
#define SV_CACHE_CONSUMED 4u /* a request has reached it while valid (Eq. (8)'s hit) */

/* One session's cached decision point (32 bytes). */
typedef struct {
  int64_t position;   /* the decision point p = n_s + L_entry of the recorded entry */
  double gap;         /* gamma = l(1) - l(2) of the ready logits, in double (NaN: none) */
  int32_t token;      /* a_hat, the lowest index of the largest ready logit (-1: none) */
  int32_t entry_len;  /* L_entry; the tokens are in the entry store */
  uint32_t flags;     /* SV_CACHE_* */
  uint32_t epoch;     /* incremented by every record, skip and invalidation of the slot */
} sv_cache_slot;

/* Event counters of one table (9 x 8 bytes), incremented by the calls. */
typedef struct {
  uint64_t pre_positions;   /* records that made a slot valid */
  uint64_t skipped;         /* records skipped on the cell budget */
  uint64_t consumed;        /* pre-positions reached by a request while valid */
  uint64_t wasted;          /* pre-positions invalidated or replaced before that */
  uint64_t fast;            /* requests served from the cache */
  uint64_t fall_invalid;    /* requests that found no valid distribution */
  uint64_t fall_ineligible; /* requests whose entry differs from the pre-positioned one */
  uint64_t fall_gate;       /* eligible requests the gate did not pass */
  uint64_t bad;             /* rows or requests with an out-of-range argument */
} sv_cache_stats;

/* out_status of a record row / out_reason of a request. */
#define SV_RECORDED 0
#define SV_SKIPPED 1
#define SV_SERVE_FAST 0
#define SV_FALL_INVALID 1
#define SV_FALL_INELIGIBLE 2
#define SV_FALL_GATE 3
#define SV_CACHE_BAD (-1)

/* ----------------------------------------------------------------------------------------
 * Record (Algorithm 1, pre-position on idle), for M updated sessions (distinct ids).
 *
 * Row m: the session session[m] at end position end_pos[m] appended an entry of
 * entry_len[m] tokens (entry_tokens[m, 0..entry_len[m])) with cell-budget headroom
 * headroom[m], and its forward pass gave the ready logits ready_logits[m, :].
 *   entry_len > headroom: skipped: the slot leaves the valid state, nothing is read;
 *   else: position <- end_pos + entry_len, (token, gap) <- the gate's (a_hat, gamma) of the
 *         row (raw logits, l(2) from the multiset, gamma in double), the entry tokens are
 *         copied to the entry store, flags <- VALID | DECODED.
 * Either way a slot that was valid and unconsumed counts as wasted, and its epoch advances.
 * A ready row without a comparable logit (all NaN) is recorded with token -1 and gap NaN (the
 * gate never passes it); a row whose copy did not complete is reported as SV_CACHE_BAD and
 * leaves the slot invalid.
 * Arguments
 *   slots        [S] sv_cache_slot; entry_store [S, max_entry] int32; stats [1].
 *   S, max_entry S >= 1, 1 <= max_entry <= 4096.
 *   session, end_pos, entry_len, headroom  [M] (int32, int64, int32, int64).
 *   entry_tokens [M, max_entry] int32 (row m's first entry_len[m] tokens are read).
 *   M            >= 0 (0 is a no-op); M*ceil(V/S') < 2^31 (S' as for spec_verify_sample).
 *   ready_logits [M, V] dtype, V >= 2.
 *   dist_store   [S, V] dtype or NULL: when given, the whole ready row is also stored in
 *                the session's row (the full distribution of Algorithm 1, line 11).
 *   out_status   [M] int32 or NULL: SV_RECORDED, SV_SKIPPED or SV_CACHE_BAD (a session id
 *                outside [0, S), entry_len outside [0, max_entry] or end_pos < 0: the row
 *                touches no slot).
 *   workspace    >= ready_cache_record_workspace(M, V, dtype) bytes.
 * ---------------------------------------------------------------------------------------- */
size_t ready_cache_record_workspace(int M, int V, sv_dtype dtype);
sv_status ready_cache_record(sv_cache_slot* slots, int32_t* entry_store, int S, int max_entry,
                             sv_cache_stats* stats, const int32_t* session,
                             const int64_t* end_pos, const int32_t* entry_tokens,
                             const int32_t* entry_len, const int64_t* headroom, int M,
                             const void* ready_logits, sv_dtype dtype, int V,
                             void* dist_store, int32_t* out_status, void* workspace,
                             size_t workspace_bytes, sv_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * Serve (Algorithm 2, confidence-gated fast path), for R requests (ids may repeat).
 *
 * Request r targets session[r] with a realized entry of req_len[r] tokens
 * (req_tokens[r, 0..req_len[r])) starting at position start[r].
 *   slot not VALID                          -> SV_FALL_INVALID;
 *   exact != 0 and (req_len != entry_len or start != position - entry_len or a token
 *   differs from the entry store)           -> SV_FALL_INELIGIBLE (exact == 0 is the streaming
 *                                              ad-hoc path: any request reaching a valid slot
 *                                              is eligible);
 *   else the slot is consumed, and gap > tau (in double) with token in A -> SV_SERVE_FAST
 *   (out_token = the cached token), otherwise SV_FALL_GATE.
 * out_token is -1 whenever the request falls through.
 * Arguments
 *   req_tokens   [R, max_entry] int32; session, req_len [R] int32; start [R] int64.
 *   tau          the gate threshold (any float; compared in double).
 *   answer_set   [n_answer] int32 sorted ascending, or NULL when n_answer == 0.
 *   out_token, out_reason  [R] int32 (SV_CACHE_BAD for a session id outside [0, S) or a
 *                req_len outside [0, max_entry]).
 * One warp per request; no workspace.
 * ---------------------------------------------------------------------------------------- */
sv_status ready_cache_serve(sv_cache_slot* slots, const int32_t* entry_store, int S,
                            int max_entry, sv_cache_stats* stats, const int32_t* session,
                            const int64_t* start, const int32_t* req_tokens,
                            const int32_t* req_len, int R, float tau,
                            const int32_t* answer_set, int n_answer, int exact,
                            int32_t* out_token, int32_t* out_reason, sv_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * Invalidate (section 3.6): the sessions session[0..n) mutated. Each slot's flags are
 * cleared atomically (a valid, unconsumed pre-position counts as wasted once, however often
 * the id repeats) and its epoch advances once per occurrence. An id outside [0, S) counts
 * as bad and touches nothing.
 * ---------------------------------------------------------------------------------------- */
sv_status ready_cache_invalidate(sv_cache_slot* slots, int S, sv_cache_stats* stats,
                                 const int32_t* session, int n, sv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_CACHE_H_ */

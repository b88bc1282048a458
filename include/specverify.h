/*
 * specverify.h — C ABI of the speculative-decoding verify step on GB300 (sm_103a).
 *
 * Five device operations sit behind this boundary:
 *
 *   spec_verify_sample  the lossless modified-rejection verify: temperature softmax of the
 *                       target logits at k+1 positions and of the draft logits at k positions,
 *                       accept x_i with probability min(1, p_i(x_i)/q_i(x_i)) using caller
 *                       supplied uniforms, keep the longest accepted prefix, then draw one
 *                       correction token from norm(max(0, p_a - q_a)) or, when every draft
 *                       token is accepted, a bonus token from p_n.
 *   spec_verify_greedy  the temperature-0 variant: accept while the draft token equals the
 *                       target argmax, then emit the target argmax.
 *   logit_gap_gate      top-1/top-2 logit-gap confidence gate over cached distributions.
 *   draft_confidence_stop  variable-length drafting: the first draft position whose
 *                       top probability (or inverse entropy) falls below a floor.
 *   ngram_propose       prompt-lookup n-gram draft proposer.
 *
 * General conventions (all entry points)
 * --------------------------------------
 *  - Every array argument is caller-owned DEVICE memory on the current CUDA device, except
 *    where a comment says otherwise. Scalars are passed by value. The library allocates no
 *    device or host memory and keeps no state between calls apart from what the caller's
 *    workspace holds.
 *  - Calls are asynchronous on `stream` (0 = the legacy default stream). Nothing is
 *    synchronised inside the library: outputs are valid once the stream reaches the call.
 *  - Arguments are validated on the host before any launch. An invalid argument returns
 *    SV_ERR_INVALID_ARG (or SV_ERR_UNSUPPORTED for a legal but unsupported shape) and
 *    launches nothing. A failed launch returns SV_ERR_CUDA; sv_last_cuda_error() then gives
 *    the cudaError_t value.
 *  - Data errors that can only be seen on the device (a draft token outside [0, V), a
 *    per-request draft count outside [0, k], a used uniform outside [0, 1), a row whose
 *    logits contain NaN or +inf or are all -inf) never fault: the affected request (or
 *    gate row) gets the error sentinel described with each call, and the kernel never
 *    indexes memory with the bad value.
 *  - Logit rows are contiguous, row-major, V elements each; element j of a row is the logit
 *    of token j. -inf is a legal logit (a masked token: probability 0).
 *  - Workspaces: the sampled verify, the greedy verify and the gate need a caller-owned
 *    device workspace of at least the size their *_workspace() query returns, 256-byte
 *    aligned. It needs no initialisation and may be reused across calls of any shape: each
 *    call first clears the counters it uses (a small kernel on `stream`, ahead of the call's
 *    other launches). Two calls in flight at the same time must not share one.
 *  - Nothing here is thread-unsafe on the host; the only process-wide state is the value
 *    returned by sv_last_cuda_error(), which is per host thread.
 */
#ifndef SPECVERIFY_H_
#define SPECVERIFY_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* sv_stream_t; /* the same type as cudaStream_t */

typedef enum {
  SV_OK = 0,
  SV_ERR_INVALID_ARG = 1,  /* a null required pointer, a bad size, T <= 0, n_min > n_max ... */
  SV_ERR_UNSUPPORTED = 2,  /* a legal request this library does not handle (k > 16, huge grids) */
  SV_ERR_WORKSPACE = 3,    /* workspace pointer null, misaligned or smaller than the query */
  SV_ERR_CUDA = 4,         /* a CUDA launch or attribute call failed; see sv_last_cuda_error */
  SV_ERR_TIMEOUT = 5       /* reserved: no call returns it. The library's bounded device
                              waits (the copy waits of every streaming kernel, and the grid
                              barriers of conformal_quantile, whose CTAs wait on one another)
                              report a wait that ran out through the call's outputs instead:
                              see each call's error sentinel */
} sv_status;

typedef enum {
  SV_F32 = 0,  /* IEEE binary32 logits */
  SV_BF16 = 1  /* bfloat16 logits (upper 16 bits of a binary32) */
} sv_dtype;

/* Largest draft length k the verify calls accept. */
#define SV_MAX_K 16

/* Library version as 10000*major + 100*minor + patch. */
int sv_version(void);

/* Short human-readable name of a status value (static storage; never NULL). */
const char* sv_status_string(sv_status s);

/* cudaError_t value of the last SV_ERR_CUDA returned on this host thread (0 if none). */
int sv_last_cuda_error(void);

/* ------------------------------------------------------------------------------------------
 * Sampled verify.
 *
 * Defined by: "Speculative Decoding: The Physics of Stolen Time in Autoregressive
 * Inference", section 2 (the modified rejection sampling rule: acceptance probability
 * alpha = min(1, p/q), residual p' = norm(max(0, p - q))) and section 1, stage 3 (keep the
 * longest accepted prefix; a bonus token when all k are accepted); and by the
 * "speculative-decoding-plan.md" design note, section "The acceptance math (standard
 * speculative sampling)" (accept loop, resample on first rejection, bonus from p_{k+1}).
 *
 * For request r with n = num_draft[r] drafted tokens x_0..x_{n-1}:
 *   p_i = softmax(target[r, i, :] / T)   for i = 0..n   (one target row per draft + 1)
 *   q_i = softmax(draft[r, i, :] / T)    for i = 0..n-1
 *   accept_i  <=>  u[r, i] < p_i(x_i) / q_i(x_i)          (IEEE division; q = 0 accepts)
 *   a = the first i < n that is not accepted, else n
 *   if a < n : w = max(0, p_a - q_a), W = sum(w)       (the residual; W > 0 when rejected)
 *   else     : w = p_n, W = 1                          (the bonus distribution)
 *   t = the smallest token j with w_0 + ... + w_j > u[r, k] * W   (inverse CDF, ascending j)
 *   emitted tokens: x_0 .. x_{a-1}, t        accept length: a
 * u[r, k] (the LAST uniform of the row, whatever n is) is the one sampling uniform;
 * u[r, n..k-1] are unused when n < k.
 *
 * Arguments
 *   target_logits   [B, k+1, V] dtype. Rows past n_r + 1 of a request are not read.
 *   draft_logits    [B, k, V]   dtype. Rows past n_r of a request are not read.
 *   draft_tokens    [B, k] int32; entries past n_r are ignored (e.g. -1 padding).
 *   num_draft       [B] int32 per-request draft count n_r in [0, k], or NULL for all k.
 *   uniforms        [B, k+1] fp32 in [0, 1).
 *   B, k, V         B >= 0 (B = 0 is a no-op), 1 <= k <= SV_MAX_K, V >= 2, and
 *                   B*(2k+1)*ceil(V/S) < 2^31 with S = 65536 logits for SV_F32 and
 *                   131072 for SV_BF16 (one CTA per row piece of S logits); beyond that,
 *                   SV_ERR_UNSUPPORTED.
 *   temperature     T, finite, 1e-4 <= T <= 1e4 (the fp32 exponent scale log2(e)/T must
 *                   stay in range); greedy decoding is spec_verify_greedy, not T -> 0.
 *   out_tokens      [B, k+1] int32: x_0..x_{a-1}, t, then -1 padding.
 *   out_accept_len  [B] int32: a, or -1 for a request with a data error (its out_tokens
 *                   row is then all -1 and its optional outputs NaN).
 *   out_p_draft     [B, k] fp32 or NULL: p_i(x_i) for i < n_r, 0 beyond.
 *   out_q_draft     [B, k] fp32 or NULL: q_i(x_i) for i < n_r, 0 beyond.
 *   out_resid_mass  [B] fp32 or NULL: W when a < n_r (the rejection probability
 *                   1 - sum(min(p_a, q_a))), 0 when every draft token was accepted.
 *   workspace       >= spec_verify_sample_workspace(B, k, V, dtype) bytes (see above).
 * Returns SV_OK or an error status; see the general conventions.
 * ---------------------------------------------------------------------------------------- */
size_t spec_verify_sample_workspace(int B, int k, int V, sv_dtype dtype);

/* The number of kernel launches one spec_verify_sample call of this shape makes on the
 * current device: 2 (the clear of its counters and the verify), or 3 when the rows are long
 * enough (at least 8 chunks of 32 KiB, and at most 32) for the draws of the batch's last
 * requests to run in a third launch split over runs of their chunks; 0 for B = 0 or an invalid
 * shape. The outputs do not depend on it. A library query; the pages have no counterpart. */
int spec_verify_sample_launches(int B, int k, int V, sv_dtype dtype);

sv_status spec_verify_sample(const void* target_logits, const void* draft_logits,
                             sv_dtype dtype, const int32_t* draft_tokens,
                             const int32_t* num_draft, const float* uniforms, int B, int k,
                             int V, float temperature, int32_t* out_tokens,
                             int32_t* out_accept_len, float* out_p_draft, float* out_q_draft,
                             float* out_resid_mass, void* workspace, size_t workspace_bytes,
                             sv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Greedy verify.
 *
 * Defined by: "The Inference Wall, Part 7", section "How speculative decoding works" (walk
 * the positions in order, accept while the draft token matches the target's, at the first
 * mismatch take the target's own token) and section "Does it make the answers worse?" (at
 * temperature 0 a guess is accepted only if it is exactly the target's pick).
 *
 *   g_i = argmax_j target[r, i, j] (lowest j among equal maxima; NaN entries are skipped)
 *   a   = the first i < n with x_i != g_i, else n
 *   emitted tokens: x_0 .. x_{a-1}, g_a;  accept length a.
 * Temperature does not enter. Arguments as for spec_verify_sample (with B*(k+1)*ceil(V/S)
 * < 2^31); a request with a data error (bad n_r, a token outside [0, V), a needed row that
 * is all NaN) gets out_accept_len = -1 and an all -1 out_tokens row.
 * ---------------------------------------------------------------------------------------- */
size_t spec_verify_greedy_workspace(int B, int k, int V, sv_dtype dtype);
sv_status spec_verify_greedy(const void* target_logits, sv_dtype dtype,
                             const int32_t* draft_tokens, const int32_t* num_draft, int B,
                             int k, int V, int32_t* out_tokens, int32_t* out_accept_len,
                             void* workspace, size_t workspace_bytes, sv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Greedy verify for callers that cannot allocate device memory.
 *
 * The pages have no counterpart: this is a convenience of the library. Some callers cannot
 * allocate device memory at all, for example an engine that has handed the whole device to
 * its own memory pool, or code on a path where cudaMalloc's implicit synchronisation is not
 * allowed. This call computes exactly what spec_verify_greedy computes (same arguments,
 * outputs and error sentinels) but takes no workspace: it uses a fixed 8 MiB scratch array
 * that lives in the library's device image, which every GPU that loads the library keeps
 * until the process exits.
 *   - Limit: spec_verify_greedy_workspace(B, k, V, dtype) must be at most 8 MiB (8388608
 *     bytes); a larger shape returns SV_ERR_UNSUPPORTED and launches nothing.
 *   - The first call on a device (with that device current) looks up the array's device
 *     address with cudaGetSymbolAddress; make that first call before any stream capture.
 *     The address is kept for the life of the process, so resetting the device
 *     (cudaDeviceReset, or releasing and re-creating its primary context) after the first
 *     call is not supported.
 *   - The host checks are spec_verify_greedy's, in the same order (sizes and dtype, then the
 *     pointers and their alignment, then the grid size); the scratch limit is checked last.
 *   - Every call on a device shares the one array: it clears the counters it needs at the
 *     start (a small kernel on `stream`), and calls whose work overlaps on the GPU
 *     (on different streams, or from different host threads) race and give wrong results.
 *     Issue them on one stream, or order them.
 *   - No cudaMalloc, cudaFree or other allocating call is made.
 * ---------------------------------------------------------------------------------------- */
sv_status spec_verify_greedy_noalloc(const void* target_logits, sv_dtype dtype,
                                     const int32_t* draft_tokens, const int32_t* num_draft,
                                     int B, int k, int V, int32_t* out_tokens,
                                     int32_t* out_accept_len, sv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Logit-gap confidence gate.
 *
 * Defined by: "Speculative Pre-Positioning", section 2.4, Eq. (11) (gamma = l(1) - l(2), the
 * two largest logits) and Eq. (12) (fire iff gamma > tau and argmax in the fast-answer set
 * A), and section 3.4, Algorithm 2 (Top2 of the cached distribution, then serve the argmax
 * or fall through).
 *
 * For each of the N rows (raw, untempered logits):
 *   l1 = the largest logit, a_hat = the lowest index holding it;
 *   l2 = the largest logit of the row with ONE copy of l1 removed (a tied maximum gives
 *        gamma = 0); NaN entries are skipped;
 *   gamma = l1 - l2 (evaluated in double), fire = gamma > tau && a_hat in A.
 * Arguments
 *   logits      [N, V] dtype.  N >= 0 (N = 0 is a no-op), V >= 2, N*ceil(V/S) < 2^31
 *               (S as for spec_verify_sample; beyond that, SV_ERR_UNSUPPORTED).
 *   tau         threshold (any float; compared in double).
 *   answer_set  [n_answer] int32, sorted ascending (duplicates allowed); may be NULL when
 *               n_answer == 0 (then nothing fires). An unsorted set gives unspecified
 *               membership answers.
 *   out_token   [N] int32: a_hat (-1 for a row whose entries are all NaN).
 *   out_gap     [N] fp32: gamma rounded to fp32 (NaN for an all-NaN row).
 *   out_fire    [N] uint8: 1 if the gate fires, else 0.
 *   workspace   >= logit_gap_gate_workspace(N, V, dtype) bytes (see the conventions).
 * ---------------------------------------------------------------------------------------- */
size_t logit_gap_gate_workspace(int N, int V, sv_dtype dtype);
sv_status logit_gap_gate(const void* logits, sv_dtype dtype, int N, int V, float tau,
                         const int32_t* answer_set, int n_answer, int32_t* out_token,
                         float* out_gap, uint8_t* out_fire, void* workspace,
                         size_t workspace_bytes, sv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Draft-side confidence stop (variable-length drafting).
 *
 * Defined by: the "speculative-decoding-plan.md" design note, the variable-length drafting
 * paragraph after "The acceptance math (standard speculative sampling)" (the draft keeps
 * proposing while its own confidence stays above a floor, by top probability or an
 * inverse-entropy gate, and stops early when it gets unsure; the accept loop is unchanged).
 * The result feeds the num_draft argument of the verify calls.
 *
 * For request r, with n_in = num_draft[r] (k when num_draft is NULL) and
 * q_i = softmax(draft[r, i, :] / T) for i < n_in:
 *   SV_CONF_TOP_PROB:     c_i = max_j q_i(j)
 *   SV_CONF_INV_ENTROPY:  c_i = 1 / H_i, H_i = -sum_j q_i(j) ln q_i(j) in nats (+inf if 0)
 *   n_r = the first i < n_in with c_i < floor, else n_in.
 * Rows at or past n_in are not read. Accuracy: the top probability to a few 1e-7 relative;
 * H to a few 1e-7 nats absolute (the relative error of the fp32 exponentials), so 1/H to
 * 1e-5 relative while H is above ~0.05 nats. A near-certain row gets a large 1/H, or +inf
 * when the computed H is not positive.
 * Arguments
 *   draft_logits   [B, k, V] dtype.
 *   num_draft      [B] int32 in [0, k], or NULL for k.
 *   B, k, V        B >= 0 (0 is a no-op), 1 <= k <= SV_MAX_K, V >= 2, and
 *                  B*k*ceil(V/S) < 2^31 (S as for spec_verify_sample).
 *   temperature    T as for spec_verify_sample (the draft's own sampling temperature).
 *   mode           SV_CONF_TOP_PROB or SV_CONF_INV_ENTROPY.
 *   floor_val      the confidence floor (compared in double; any finite value).
 *   out_num_draft  [B] int32: n_r, or -1 for a request with a data error (n_in outside
 *                  [0, k], or a row it reads that holds NaN or +inf or is all -inf).
 *   out_conf       [B, k] fp32 or NULL: c_i for i < n_in, 0 beyond, NaN on a data error.
 *   workspace      >= draft_confidence_workspace(B, k, V, dtype) bytes (see the conventions).
 * The pages' drafting loop stops generating at the first unsure position; here the draft
 * logits of all k positions already exist, and one batched call finds that position.
 * ---------------------------------------------------------------------------------------- */
typedef enum { SV_CONF_TOP_PROB = 0, SV_CONF_INV_ENTROPY = 1 } sv_conf_mode;

size_t draft_confidence_workspace(int B, int k, int V, sv_dtype dtype);
sv_status draft_confidence_stop(const void* draft_logits, sv_dtype dtype,
                                const int32_t* num_draft, int B, int k, int V,
                                float temperature, sv_conf_mode mode, float floor_val,
                                int32_t* out_num_draft, float* out_conf, void* workspace,
                                size_t workspace_bytes, sv_stream_t stream);

/* ------------------------------------------------------------------------------------------
 * Prompt-lookup n-gram proposer.
 *
 * Defined by: "The Inference Wall, Part 7", section "What S is in this experiment, and what
 * 'ngram' actually means" (take the last few tokens, find the same phrase earlier in the
 * text the request holds, longest phrase first from prompt_lookup_max down to
 * prompt_lookup_min, and copy the k tokens that followed it; nothing earlier => no
 * proposal).
 *
 * For request r with history h = history[r, 0 .. L-1], L = hist_len[r]:
 *   for n = n_max down to n_min: the earliest start s with s + n <= L - 1 and
 *   h[s .. s+n-1] == h[L-n .. L-1]; the first n that has one wins and proposes
 *   h[s+n .. min(s+n+k-1, L-1)]  (so n_r = min(k, L - s - n) >= 1).
 *   With no such n, n_r = 0. The occurrence may overlap the suffix itself.
 * Arguments
 *   history        [B, L_max] int32 token ids (any int32 values).
 *   hist_len       [B] int32 in [0, L_max]; a length outside that range gives n_r = -1 and
 *                  an all -1 draft row (spec_verify_* then flag that request as an error).
 *   B, L_max       B >= 0 (0 is a no-op), 1 <= L_max < 2^24.
 *   n_max, n_min   1 <= n_min <= n_max <= 64.
 *   k              1 <= k <= 64: proposal length bound.
 *   out_draft      [B, k] int32: the proposal, -1 padded.
 *   out_num_draft  [B] int32: n_r.
 * No workspace is needed.
 * ---------------------------------------------------------------------------------------- */
sv_status ngram_propose(const int32_t* history, const int32_t* hist_len, int B, int L_max,
                        int n_max, int n_min, int k, int32_t* out_draft,
                        int32_t* out_num_draft, sv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H_ */

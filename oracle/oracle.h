/*
 * oracle.h — plain fp64 CPU oracle of the speculative-decoding verify step.
 *
 * TEST INFRASTRUCTURE ONLY. The tests, the smoke check and the benchmark's CPU-baseline leg
 * are the only callers; the product library never links, loads or calls it, and this code
 * shares no source, header, table or helper with the CUDA library.
 *
 * Every function works on host arrays laid out exactly like the device arguments of the
 * library, processes the half-open request (or row) range [r0, r1) of the batch so a caller
 * may split a batch across threads, and returns 0, or a negative value for an invalid
 * argument (nothing is written then).
 *
 * Logit dtype codes: 0 = binary32, 1 = bfloat16 (raw 16-bit patterns).
 */
#ifndef ORACLE_H_
#define ORACLE_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Near-tie threshold: a decision whose margin is below this is reported, not compared. */
#define ORACLE_TIE_MARGIN 1e-6

/* p = softmax(row / T) in double. Returns 0, or -1 if the row holds NaN or +inf or is all
 * -inf (not a distribution). */
int oracle_row_softmax(const void* row, int dtype, int V, double T, double* p_out);

/* Sampled verify (modified rejection rule). Outputs, per request r in [r0, r1):
 *   out_tokens[r, 0..k], out_accept_len[r]      as the library's spec_verify_sample;
 *   out_p[r, i], out_q[r, i]                    p_i(x_i), q_i(x_i) for i < n_r, else 0;
 *   out_resid[r]                                W when a < n_r, else 0;
 *   out_flag_pos[r]  the first position whose decision had a near tie (the accept test of
 *                    position i, or the draw that emitted token a), or -1;
 *   out_margin[r]    the smallest margin among the decisions that fixed the result;
 *   out_t_lo[r], out_t_hi[r]  the first and last token the draw selects for any target
 *                    within ORACLE_TIE_MARGIN * W of u[r, k] * W (equal when no near tie);
 *   out_tie_prob[r]  the chance that request r is flagged, given its path: for each accept
 *                    test it took, the probability over u[r, i] that |u - rho_i| < the
 *                    margin, plus the probability over u[r, k] that its draw is a near tie
 *                    (the sum of min(w_t / W, margin per interior boundary of token t));
 *                    0 for a data error. It sizes the expected count of flagged requests.
 * Every output pointer past out_accept_len may be NULL.
 * A request with a data error gets accept_len -1, tokens -1, p/q/resid NaN, flag -1. */
int oracle_spec_verify_sample(const void* target, const void* draft, int dtype,
                              const int32_t* draft_tokens, const int32_t* num_draft,
                              const float* uniforms, int B, int k, int V, double T,
                              int32_t* out_tokens, int32_t* out_accept_len, double* out_p,
                              double* out_q, double* out_resid, int32_t* out_flag_pos,
                              double* out_margin, int32_t* out_t_lo, int32_t* out_t_hi,
                              double* out_tie_prob, int r0, int r1);

/* Greedy verify; outputs as the library's spec_verify_greedy. */
int oracle_spec_verify_greedy(const void* target, int dtype, const int32_t* draft_tokens,
                              const int32_t* num_draft, int B, int k, int V,
                              int32_t* out_tokens, int32_t* out_accept_len, int r0, int r1);

/* Logit-gap gate over rows [i0, i1); out_gap is gamma in double; out_flag[i] = 1 when
 * |gamma - tau| < ORACLE_TIE_MARGIN. */
int oracle_logit_gap_gate(const void* logits, int dtype, int N, int V, double tau,
                          const int32_t* answer_set, int n_answer, int32_t* out_token,
                          double* out_gap, uint8_t* out_fire, uint8_t* out_flag, int i0,
                          int i1);

/* Relative near-tie threshold of the draft-confidence stop: |c - floor| <= this * floor. */
#define ORACLE_CONF_MARGIN 1e-5

/* Draft-side confidence and the variable-length stop ("speculative-decoding-plan.md", the
 * variable-length drafting paragraph after "The acceptance math": the draft keeps proposing
 * while its own confidence stays above a floor, by top probability or an inverse-entropy
 * gate, and stops when it gets unsure). For request r in [r0, r1), with n_in = num_draft[r]
 * (all k when num_draft is NULL) and q_i = softmax(draft[r, i] / T) for i < n_in:
 *   mode 0: c_i = max_j q_i(j)                                  (top probability)
 *   mode 1: c_i = 1 / H_i, H_i = -sum_j q_i(j) ln q_i(j) nats   (+inf when H_i = 0)
 *   out_num_draft[r] = the first i < n_in with c_i < floor, else n_in;
 *   out_conf[r, i]   = c_i for i < n_in, 0 beyond (may be NULL);
 *   out_flag[r]      = the first i up to the stop with |c_i - floor| <= ORACLE_CONF_MARGIN
 *                      * floor, else -1 (may be NULL).
 * A request with a data error (n_in outside [0, k], or a row it reads that is not a
 * distribution) gets out_num_draft -1, out_conf NaN and flag -1. H is the definition
 * evaluated in double: accurate to about 1e-17 nats absolute, so 1/H is accurate wherever
 * H is well above that (a floor on 1/H below 1e12, say). */
int oracle_draft_confidence(const void* draft, int dtype, const int32_t* num_draft, int B,
                            int k, int V, double T, int mode, double floor_val,
                            int32_t* out_num_draft, double* out_conf, int32_t* out_flag,
                            int r0, int r1);

/* ---- Gate calibration ("Speculative Pre-Positioning", section 2.4, Eq. (13) coverage and
 * Eq. (14) false-accept risk, the calibration "smallest tau with r(tau) <= r_max", and the
 * Wilson 95 % intervals reported with them in section 4, Figures 6 and 7) ---- */

/* Wilson score interval of k successes in n trials at the normal quantile z:
 *   centre = (k/n + z^2 / (2n)) / (1 + z^2 / n)
 *   half   = z / (1 + z^2 / n) * sqrt((k/n)(1 - k/n) / n + z^2 / (4 n^2))
 * lo = centre - half and hi = centre + half, clamped to [0, 1]; both NaN when n = 0. */
void oracle_wilson(int64_t k, int64_t n, double z, double* lo, double* hi);

/* Risk-coverage sweep over the thresholds taus[0..T) (non-decreasing, no NaN). For each t:
 *   accepted[t] = #{i : gap[i] > taus[t] and token[i] in A}   (compared in double; a NaN gap
 *                 is never accepted; answer_set sorted ascending)
 *   wrong[t]    = #{accepted i : token[i] != full_token[i]}   (the served token disagrees with
 *                 the model's own full-path output)
 *   stats[6t..6t+5] = coverage accepted/N, its Wilson interval, risk wrong/accepted, its
 *                 Wilson interval (the risk and its interval NaN when accepted = 0).
 * *tau_index = the smallest t with accepted[t] > 0 and risk <= r_max, else -1.
 * Returns -1 on bad arguments (taus unsorted or NaN, N < 0, T < 1). */
int oracle_risk_coverage(const float* gap, const int32_t* token, const int32_t* full_token,
                         int N, const int32_t* answer_set, int n_answer, const float* taus,
                         int T, double z, double r_max, int64_t* accepted, int64_t* wrong,
                         double* stats, int32_t* tau_index);

/* Conformal residual of draft logits against the true ones ("speculative-decoding-plan.md",
 * the conformal 2 tau <= gamma gate: a draft within tau of the truth in sup-norm cannot flip
 * an argmax whose runner-up margin is at least 2 tau). Row i of [N, V]:
 *   r_i = max_j d_j, d_j = 0 where the two logits are equal (a token masked, -inf, in both
 *         included), |draft_j - truth_j| elsewhere (+inf where only one is masked);
 *   NaN when either row holds a NaN. Evaluated in double, stored rounded to fp32. */
int oracle_conformal_residual(const void* draft, const void* truth, int dtype, int N, int V,
                              float* out, int i0, int i1);

/* Split-conformal quantile of n calibration residuals: Q = the ceil((n + 1) q)-th smallest
 * (ranks from 1; NaN orders above +inf), +inf when that rank exceeds n; the rank is computed
 * as ceil((double)(n + 1) * q). q in (0, 1], n >= 1. */
int oracle_conformal_quantile(const float* r, int n, double q, float* out_q);

/* Conformal admission over K layers: logits [N, K, V] (row n*K + k is step n's early-exit
 * logits at layer k), Q[K] the calibrated quantile of each layer.
 *   gamma_{n,k}, a_hat_{n,k} as in oracle_logit_gap_gate (double; NaN for an all-NaN row);
 *   admit_{n,k} = 2 Q[k] <= gamma_{n,k} (in double; a NaN gamma never admits);
 *   out_layer[n] = the first admitted k, else K; out_token[n] = a_hat at that layer, else -1;
 *   out_gap[n*K + k] = gamma_{n,k} (may be NULL);
 *   out_flag[n] = the first k <= out_layer[n] (k < K) with |gamma - 2 Q[k]| <
 *                 ORACLE_TIE_MARGIN, else -1 (may be NULL). Steps [n0, n1). */
int oracle_conformal_admit(const void* logits, int dtype, int N, int K, int V, const float* Q,
                           int32_t* out_layer, int32_t* out_token, double* out_gap,
                           int32_t* out_flag, int n0, int n1);

/* Prompt-lookup n-gram proposer; outputs as the library's ngram_propose. */
int oracle_ngram_propose(const int32_t* history, const int32_t* hist_len, int B, int L_max,
                         int n_max, int n_min, int k, int32_t* out_draft,
                         int32_t* out_num_draft, int r0, int r1);

#ifdef __cplusplus
}
#endif

#endif /* ORACLE_H_ */

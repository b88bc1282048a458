/*
 * specverify_calib.h — C ABI of the gate calibration and the conformal gate on GB300.
 *
 * Four device operations around the logit-gap gate of specverify.h:
 *
 *   gate_risk_coverage   the gate's coverage and false-accept risk over a grid of thresholds,
 *                        with Wilson intervals, and the calibrated threshold (the smallest
 *                        one whose risk meets a budget).
 *   conformal_residual   the sup-norm distance of draft logits from the true logits, row by
 *                        row: the calibration scores of the conformal gate.
 *   conformal_quantile   the split-conformal quantile Q of those scores.
 *   conformal_admit      the conformal gate: per decoding step, the earliest of K layers
 *                        whose logit gap gamma satisfies 2 Q_k <= gamma.
 *
 * The conventions of specverify.h hold (device pointers, asynchronous on `stream`, host-side
 * validation before any launch, no allocation, data errors reported in the outputs, the
 * workspace rules). These calls are the calibration side of the gate: they run once per
 * calibration set or per threshold grid, next to the per-token verify path.
 */
#ifndef SPECVERIFY_CALIB_H_
#define SPECVERIFY_CALIB_H_

#include "specverify.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Largest threshold grid gate_risk_coverage accepts. */
#define SV_MAX_TAUS 4096

/* One threshold of the risk-coverage sweep (64 bytes). */
typedef struct {
  int64_t accepted;  /* decision points the gate accepts: gamma > tau and a_hat in A */
  int64_t wrong;     /* accepted points whose served token differs from the full path's */
  double coverage;   /* c(tau) = accepted / N (NaN when N = 0) */
  double cov_lo, cov_hi;    /* its Wilson interval */
  double risk;       /* r(tau) = wrong / accepted (NaN when nothing is accepted) */
  double risk_lo, risk_hi;  /* its Wilson interval (NaN when nothing is accepted) */
} sv_calib_point;

/* ----------------------------------------------------------------------------------------
 * Risk-coverage sweep and threshold calibration.
 *
 * Defined by: "Speculative Pre-Positioning", section 2.4, Eq. (13) (coverage: the fraction
 * of decision points the gate accepts, gamma > tau and argmax in A) and Eq. (14) (risk: the
 * fraction of served fast-path answers that disagree with the model's own full-path output),
 * the calibration rule stated after them (the smallest tau with r(tau) <= r_max), and
 * section 4, Figures 6 and 7 (Wilson 95 % intervals on both rates).
 *
 * For each t < T, over the N decision points i:
 *   accepted[t] = #{i : gap[i] > taus[t] and token[i] in A}  (a NaN gap is never accepted)
 *   wrong[t]    = #{accepted i : token[i] != full_token[i]}
 *   Wilson interval of k successes in n trials at the normal quantile z:
 *     centre = (k/n + z^2/(2n)) / (1 + z^2/n),
 *     half   = z / (1 + z^2/n) * sqrt((k/n)(1 - k/n)/n + z^2/(4n^2)),
 *     [centre - half, centre + half] clamped to [0, 1].
 *   out_tau_index = the smallest t with accepted[t] > 0 and risk <= r_max, else -1.
 * Arguments
 *   gap          [N] fp32: the gate's gamma per decision point (logit_gap_gate's out_gap).
 *   token        [N] int32: the gate's a_hat (the token the fast path would serve).
 *   full_token   [N] int32: the model's own full-path output at the same point.
 *   N            >= 0.
 *   answer_set   [n_answer] int32 sorted ascending (duplicates allowed), or NULL when
 *                n_answer == 0 (then nothing is accepted).
 *   taus         [T] fp32, non-decreasing, no NaN (+-inf allowed); 1 <= T <= SV_MAX_TAUS.
 *                A grid that breaks this order is a data error: every point gets
 *                accepted = wrong = -1 and NaN rates, and out_tau_index = -2.
 *   z            the normal quantile of the intervals (1.959964 for 95 %); finite, >= 0.
 *   r_max        the risk budget (NaN: no threshold qualifies).
 *   out_points   [T] sv_calib_point.
 *   out_tau_index  [1] int32.
 *   workspace    >= gate_risk_coverage_workspace(N, T) bytes.
 * Counts are exact; the rates are evaluated in double on the device, each operation rounded on
 * its own in the order written above (no fused multiply-add).
 * ---------------------------------------------------------------------------------------- */
size_t gate_risk_coverage_workspace(int N, int T);
sv_status gate_risk_coverage(const float* gap, const int32_t* token, const int32_t* full_token,
                             int N, const int32_t* answer_set, int n_answer, const float* taus,
                             int T, double z, double r_max, sv_calib_point* out_points,
                             int32_t* out_tau_index, void* workspace, size_t workspace_bytes,
                             sv_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * Conformal residual (calibration score of the conformal gate).
 *
 * Defined by: the "speculative-decoding-plan.md" design note, "Axis 1 reuses the gate we
 * already have: 2*tau <= gamma" (a draft that differs from the true logits by less than tau
 * in sup-norm cannot flip an argmax whose runner-up margin is at least 2 tau; the residual is
 * calibrated once and its conformal quantile stands in for tau).
 *
 * For each of the N row pairs:
 *   r = max_j d_j, d_j = 0 where draft_j == truth_j (a token masked, -inf, in both included),
 *       |draft_j - truth_j| elsewhere (+inf where only one of the two is masked);
 *   r = NaN when either row holds a NaN.
 * The difference is formed in fp32 (exact for bf16 inputs whose magnitudes are within 2^16
 * of each other; otherwise rounded once).
 * Arguments
 *   draft_logits, true_logits  [N, V] dtype each.  N >= 0 (0 is a no-op), V >= 1.
 *   out_resid    [N] fp32.
 * No workspace: each CTA folds its piece into out_resid with an atomic maximum after the
 * call has cleared it (an asynchronous memset on `stream`).
 * ---------------------------------------------------------------------------------------- */
sv_status conformal_residual(const void* draft_logits, const void* true_logits,
                             sv_dtype dtype, int N, int V, float* out_resid,
                             sv_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * Split-conformal quantile.
 *
 * Defined by: the same passage ("calibrate the residual once, take the conformal
 * q-quantile Q_q"), read as the standard split-conformal quantile: with n calibration
 * scores, Q = the ceil((n + 1) q)-th smallest (ranks from 1, NaN ordered above +inf), and
 * Q = +inf when that rank exceeds n. The rank is ceil((double)(n + 1) * q), on the host.
 * Arguments
 *   resid        [n] fp32 scores (any values; -0 orders below +0).
 *   n            >= 1.
 *   q            in (0, 1].
 *   out_q        [1] fp32: Q, one of the scores bit for bit (or +inf).
 *   workspace    >= conformal_quantile_workspace(n) bytes.
 * Three passes of a radix select over the scores' order-preserving 32-bit keys (11, 11 and 10
 * bits). Up to 8192 scores: one CTA, the keys in shared memory. Beyond that: one cooperative
 * launch (cudaLaunchCooperativeKernel; every CTA resident at once) whose passes meet at grid
 * barriers (the CTA that arrives last picks the pass's digit and publishes it to the others).
 * A barrier wait is bounded (2 s, never reached when the launch is cooperative); if one runs
 * out, out_q is the quiet NaN with payload 1 (bits 0x7fc00001), which no score produces (a
 * NaN score gives 0x7fc00000).
 * ---------------------------------------------------------------------------------------- */
size_t conformal_quantile_workspace(int n);
sv_status conformal_quantile(const float* resid, int n, double q, float* out_q,
                             void* workspace, size_t workspace_bytes, sv_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * Self-test of the quantile's bounded grid barriers.
 *
 * A library diagnostic; the pages have no counterpart. It makes the one launch of this
 * library whose CTAs wait on one another give up, on purpose, so that a test can see the
 * wait end and the timeout reported, with no fault and no hang: the same cooperative
 * select launch as conformal_quantile over n > 8192 scores, except that every grid barrier
 * waits for one arrival more than the grid has. No barrier can complete; each CTA waits
 * wait_us microseconds, gives up and returns. out_q then holds the timeout sentinel, the
 * quiet NaN with payload 1 (bits 0x7fc00001), and the device stays usable (the workspace
 * too: conformal_quantile clears it at every call).
 * Arguments
 *   resid, out_q, workspace   as for conformal_quantile (the scores are read, not ranked).
 *   n                         > 8192 (smaller sets take the one-CTA path, which never waits).
 *   wait_us                   1 .. 100000: how long each barrier waits before giving up.
 * Returns SV_ERR_INVALID_ARG / SV_ERR_WORKSPACE on bad arguments, else the launch status.
 * ---------------------------------------------------------------------------------------- */
sv_status conformal_quantile_barrier_selftest(const float* resid, int n, float* out_q,
                                              void* workspace, size_t workspace_bytes,
                                              unsigned int wait_us, sv_stream_t stream);

/* ----------------------------------------------------------------------------------------
 * Conformal gate over K layers.
 *
 * Defined by: the same note, "conformal_admit(cal_k, q, gamma)": per decoding step, the
 * earliest layer k whose 2 Q_q(k) <= gamma, where gamma is that layer's logit gap; with
 * K = 1 it is the plain rule "admit iff 2 Q_q <= gamma". gamma and a_hat are those of
 * logit_gap_gate (raw logits, l(2) from the multiset, the lowest index of the maximum).
 *
 * For step n and layer k (row n*K + k of the logits):
 *   admit_{n,k} = 2 * Q[k] <= gamma_{n,k}, in double; a row with no comparable logit
 *                 (all NaN) never admits.
 *   out_layer[n] = the first admitted k, else K; out_token[n] = a_hat at that layer, else -1.
 * Arguments
 *   logits       [N, K, V] dtype: step n's early-exit logits at each of the K layers.
 *   N, K, V      N >= 0 (0 is a no-op), K >= 1, V >= 2, N*K*ceil(V/S) < 2^31 (S as for
 *                spec_verify_sample).
 *   Q            [K] fp32 on the device: the calibrated quantile of each layer (as written
 *                by conformal_quantile).
 *   out_layer    [N] int32.
 *   out_token    [N] int32.
 *   out_gap      [N, K] fp32 or NULL: gamma_{n,k} rounded to fp32 (NaN for an all-NaN row).
 *   workspace    >= conformal_admit_workspace(N, K, V, dtype) bytes.
 * ---------------------------------------------------------------------------------------- */
size_t conformal_admit_workspace(int N, int K, int V, sv_dtype dtype);
sv_status conformal_admit(const void* logits, sv_dtype dtype, int N, int K, int V,
                          const float* Q, int32_t* out_layer, int32_t* out_token,
                          float* out_gap, void* workspace, size_t workspace_bytes,
                          sv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_CALIB_H_ */

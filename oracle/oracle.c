/*
 * oracle.c — plain fp64 CPU oracle of the speculative-decoding verify step.
 *
 * TEST INFRASTRUCTURE ONLY: called by the tests, the smoke check and the benchmark's
 * CPU-baseline leg, never by the product library, with which it shares no code.
 *
 * It is written to be read against the pages, not to be fast: every row is rescanned when
 * it is needed, every sum runs in ascending token order in double, and the steps follow the
 * order in which the pages state them.
 *
 *  - Sampled verify: "Speculative Decoding: The Physics of Stolen Time in Autoregressive
 *    Inference", section 1 (stage 2 gives p at every draft position; stage 3 keeps the
 *    longest accepted prefix and resamples after the first rejection, or adds a bonus token
 *    when all k are accepted) and section 2 (alpha = min(1, p/q); residual
 *    p' = norm(max(0, p - q)); Z = 1 - sum(min(p, q))); and the "speculative-decoding-plan.md"
 *    design note, section "The acceptance math (standard speculative sampling)", which
 *    states the same loop (accept x_i with min(1, p_i(x_i)/q_i(x_i)); on the first rejection
 *    resample from norm(max(0, p_i - q_i)) and stop; bonus from p_{gamma+1}).
 *  - Greedy verify: "The Inference Wall, Part 7", section "How speculative decoding works"
 *    (walk the positions in order, accept while the draft matches the target, at the first
 *    mismatch take the target's token).
 *  - Gate: "Speculative Pre-Positioning", section 2.4, Eq. (11) and Eq. (12), and section 3.4,
 *    Algorithm 2 (Top2, gap, argmax, fire or fall through).
 *  - Draft-confidence stop: the "speculative-decoding-plan.md" design note, the
 *    variable-length drafting paragraph (keep drafting while the draft's top probability, or
 *    the inverse of its entropy, stays above a floor).
 *  - Gate calibration: "Speculative Pre-Positioning", section 2.4, Eq. (13) and Eq. (14)
 *    (coverage and false-accept risk of the gate as tau sweeps; calibration takes the
 *    smallest tau whose risk meets a budget) and section 4 (Wilson 95 % intervals); the
 *    "speculative-decoding-plan.md" conformal gate (sup-norm residual, its conformal
 *    q-quantile Q, admit iff 2 Q <= gamma, per layer the earliest admitting one).
 *  - N-gram proposer: "The Inference Wall, Part 7", section "What S is in this experiment,
 *    and what 'ngram' actually means" (four-word phrase first, then three, then two; copy
 *    what followed the phrase; nothing earlier means no proposal).
 *
 * Readings where the pages are silent (each one is listed with its reason in the design
 * document): temperature T scales both p and q; the accept test is the strict u < p/q; the
 * sampling uniform is the last of the k+1 supplied per request; the inverse CDF runs in
 * ascending token order and falls back to the last token with positive weight when rounding
 * leaves the target past the total; a zero residual falls back to p_a; the gate works on
 * raw logits with a strict ">" and l(2) is taken from the multiset (a tied maximum gives a
 * zero gap); the n-gram match is the earliest occurrence that ends before the last token.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* Largest draft length k the oracle handles (rows per request: k + 1). */
#define ORACLE_MAX_K 64
#define ORACLE_MAX_ROWS (ORACLE_MAX_K + 1)

/* ---- input decoding (bf16 is the upper half of a binary32) ---- */
static double logit_at(const void* base, int dtype, size_t idx) {
  if (dtype == 0) return (double)((const float*)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* Tempered-softmax statistics of one row: m = max_j z_j and S = sum_j exp((z_j - m)/T),
 * so p(j) = exp((z_j - m)/T) / S. Returns -1 when the row is not a distribution. */
static int softmax_stats(const void* base, int dtype, size_t off, int V, double T, double* m,
                         double* S) {
  double mx = -INFINITY;
  for (int j = 0; j < V; ++j) {
    double z = logit_at(base, dtype, off + (size_t)j);
    if (isnan(z) || z == INFINITY) return -1;
    if (z > mx) mx = z;
  }
  if (mx == -INFINITY) return -1;
  double s = 0.0;
  for (int j = 0; j < V; ++j) s += exp((logit_at(base, dtype, off + (size_t)j) - mx) / T);
  *m = mx;
  *S = s;
  return 0;
}

static double prob_at(const void* base, int dtype, size_t off, double m, double S, double T,
                      int j) {
  return exp((logit_at(base, dtype, off + (size_t)j) - m) / T) / S;
}

int oracle_row_softmax(const void* row, int dtype, int V, double T, double* p_out) {
  if (!row || !p_out || V < 1 || !(T > 0.0) || !isfinite(T) || (dtype != 0 && dtype != 1))
    return -2;
  double m, S;
  if (softmax_stats(row, dtype, 0, V, T, &m, &S) != 0) return -1;
  for (int j = 0; j < V; ++j) p_out[j] = prob_at(row, dtype, 0, m, S, T, j);
  return 0;
}

/* Inverse-CDF draw from unnormalised weights w (total W): the smallest j whose running sum
 * exceeds u*W. If rounding leaves no such j, the last j with positive weight. *margin is
 * the distance from u*W to the nearest boundary of the chosen token's interval that has
 * mass on its far side, divided by W (0 for the rounding fallback). */
static int inverse_cdf(const double* w, int V, double W, double u, double* margin) {
  const double target = u * W;
  double run = 0.0;
  for (int j = 0; j < V; ++j) {
    const double before = run;
    run += w[j];
    if (run > target) {
      double mg = INFINITY;
      if (before > 0.0) mg = target - before;
      int later = 0;
      for (int i = j + 1; i < V; ++i)
        if (w[i] > 0.0) { later = 1; break; }
      if (later && run - target < mg) mg = run - target;
      *margin = mg / W;
      return j;
    }
  }
  int last = -1;
  for (int j = 0; j < V; ++j)
    if (w[j] > 0.0) last = j;
  *margin = 0.0;
  return last;
}

/* The token the inverse-CDF draw selects for an absolute target (clamped to the first or
 * last token with positive weight at either end). */
static int select_at(const double* w, int V, double target) {
  double run = 0.0;
  int last = -1;
  for (int j = 0; j < V; ++j) {
    run += w[j];
    if (w[j] > 0.0) last = j;
    if (run > target && w[j] > 0.0) return j;
  }
  return last;
}

static int uniform_ok(float u) { return u >= 0.0f && u < 1.0f; }

/* The probability, over a target u*W with u uniform on [0, 1), that the inverse-CDF draw over
 * w is flagged as a near tie: that the target lies within ORACLE_TIE_MARGIN * W of a boundary
 * between two tokens of positive weight. The chosen token t covers [C_{t-1}, C_t); inside it,
 * the flagged targets are the first margin*W (unless t is the first token of positive weight)
 * and the last margin*W (unless t is the last), or all of it when it is shorter. */
static double draw_tie_probability(const double* w, int V, double W) {
  int first = -1, last = -1;
  for (int j = 0; j < V; ++j)
    if (w[j] > 0.0) {
      if (first < 0) first = j;
      last = j;
    }
  double prob = 0.0;
  for (int j = 0; j < V; ++j) {
    if (!(w[j] > 0.0)) continue;
    const double window = ORACLE_TIE_MARGIN * ((j != first) + (j != last));
    const double m = w[j] / W;
    prob += m < window ? m : window;
  }
  return prob;
}

/* The probability, over u uniform on [0, 1), that |u - rho| < ORACLE_TIE_MARGIN. */
static double accept_tie_probability(double rho) {
  const double lo = rho - ORACLE_TIE_MARGIN > 0.0 ? rho - ORACLE_TIE_MARGIN : 0.0;
  const double hi = rho + ORACLE_TIE_MARGIN < 1.0 ? rho + ORACLE_TIE_MARGIN : 1.0;
  return hi > lo ? hi - lo : 0.0;
}

int oracle_spec_verify_sample(const void* target, const void* draft, int dtype,
                              const int32_t* draft_tokens, const int32_t* num_draft,
                              const float* uniforms, int B, int k, int V, double T,
                              int32_t* out_tokens, int32_t* out_accept_len, double* out_p,
                              double* out_q, double* out_resid, int32_t* out_flag_pos,
                              double* out_margin, int32_t* out_t_lo, int32_t* out_t_hi,
                              double* out_tie_prob, int r0, int r1) {
  if (B < 0 || k < 1 || k > ORACLE_MAX_K || V < 2 || !(T > 0.0) || !isfinite(T) ||
      (dtype != 0 && dtype != 1))
    return -1;
  if (r0 < 0 || r1 > B || r0 > r1) return -1;
  if (r0 == r1) return 0;
  if (!target || !draft || !draft_tokens || !uniforms || !out_tokens || !out_accept_len)
    return -1;
  double* w = (double*)malloc((size_t)V * sizeof(double));
  if (!w) return -3;

  for (int r = r0; r < r1; ++r) {
    int32_t* tok = out_tokens + (size_t)r * (k + 1);
    const int32_t* x = draft_tokens + (size_t)r * k;
    const float* u = uniforms + (size_t)r * (k + 1);
    for (int i = 0; i <= k; ++i) tok[i] = -1;
    if (out_p) for (int i = 0; i < k; ++i) out_p[(size_t)r * k + i] = 0.0;
    if (out_q) for (int i = 0; i < k; ++i) out_q[(size_t)r * k + i] = 0.0;
    if (out_resid) out_resid[r] = 0.0;
    if (out_flag_pos) out_flag_pos[r] = -1;
    if (out_margin) out_margin[r] = INFINITY;
    if (out_t_lo) out_t_lo[r] = -1;
    if (out_t_hi) out_t_hi[r] = -1;
    if (out_tie_prob) out_tie_prob[r] = 0.0;

    const int n = num_draft ? num_draft[r] : k;
    int err = (n < 0 || n > k);
    for (int i = 0; !err && i < n; ++i)
      if (x[i] < 0 || x[i] >= V || !uniform_ok(u[i])) err = 1;
    if (!err && !uniform_ok(u[k])) err = 1;

    /* Stage 2: the target distribution at positions 0..n, the draft's at 0..n-1. Every
     * needed row must be a distribution. */
    double mp[ORACLE_MAX_ROWS], Sp[ORACLE_MAX_ROWS], mq[ORACLE_MAX_ROWS],
        Sq[ORACLE_MAX_ROWS];
    for (int i = 0; !err && i <= n; ++i) {
      size_t off = ((size_t)r * (k + 1) + i) * (size_t)V;
      if (softmax_stats(target, dtype, off, V, T, &mp[i], &Sp[i]) != 0) err = 1;
    }
    for (int i = 0; !err && i < n; ++i) {
      size_t off = ((size_t)r * k + i) * (size_t)V;
      if (softmax_stats(draft, dtype, off, V, T, &mq[i], &Sq[i]) != 0) err = 1;
    }
    if (err) {
      out_accept_len[r] = -1;
      if (out_p) for (int i = 0; i < k; ++i) out_p[(size_t)r * k + i] = NAN;
      if (out_q) for (int i = 0; i < k; ++i) out_q[(size_t)r * k + i] = NAN;
      if (out_resid) out_resid[r] = NAN;
      continue;
    }

    /* p_i(x_i) and q_i(x_i) at every drafted position. */
    double px[ORACLE_MAX_ROWS], qx[ORACLE_MAX_ROWS];
    for (int i = 0; i < n; ++i) {
      px[i] = prob_at(target, dtype, ((size_t)r * (k + 1) + i) * (size_t)V, mp[i], Sp[i], T,
                      x[i]);
      qx[i] = prob_at(draft, dtype, ((size_t)r * k + i) * (size_t)V, mq[i], Sq[i], T, x[i]);
      if (out_p) out_p[(size_t)r * k + i] = px[i];
      if (out_q) out_q[(size_t)r * k + i] = qx[i];
    }

    /* Stage 3: accept x_i while u_i < p_i(x_i)/q_i(x_i); stop at the first rejection. */
    int flag = -1;
    double min_margin = INFINITY;
    double tie_prob = 0.0;
    int a = n;
    for (int i = 0; i < n; ++i) {
      const double rho = px[i] / qx[i];
      tie_prob += accept_tie_probability(rho);
      const double mg = fabs((double)u[i] - rho);
      if (mg < min_margin) min_margin = mg;
      if (mg < ORACLE_TIE_MARGIN && flag < 0) flag = i;
      if (!((double)u[i] < rho)) {
        a = i;
        break;
      }
    }

    /* The correction token from norm(max(0, p_a - q_a)) after a rejection, else the bonus
     * token from p_n. */
    double W = 0.0;
    int from_residual = 0;
    if (a < n) {
      const size_t offp = ((size_t)r * (k + 1) + a) * (size_t)V;
      const size_t offq = ((size_t)r * k + a) * (size_t)V;
      for (int j = 0; j < V; ++j) {
        const double p = prob_at(target, dtype, offp, mp[a], Sp[a], T, j);
        const double q = prob_at(draft, dtype, offq, mq[a], Sq[a], T, j);
        w[j] = p > q ? p - q : 0.0;
        W += w[j];
      }
      from_residual = W > 0.0;
      if (out_resid) out_resid[r] = W;
    }
    const int bonus_row = from_residual ? -1 : a; /* a == n: the bonus row; else fallback */
    if (bonus_row >= 0) {
      const size_t off = ((size_t)r * (k + 1) + bonus_row) * (size_t)V;
      W = 0.0;
      for (int j = 0; j < V; ++j) {
        w[j] = prob_at(target, dtype, off, mp[bonus_row], Sp[bonus_row], T, j);
        W += w[j];
      }
    }
    double smg;
    const int t = inverse_cdf(w, V, W, (double)u[k], &smg);
    if (smg < min_margin) min_margin = smg;
    if (smg < ORACLE_TIE_MARGIN && flag < 0) flag = a;
    /* every token a target within the tie margin of u*W could select */
    if (out_t_lo) out_t_lo[r] = select_at(w, V, (double)u[k] * W - ORACLE_TIE_MARGIN * W);
    if (out_t_hi) out_t_hi[r] = select_at(w, V, (double)u[k] * W + ORACLE_TIE_MARGIN * W);

    for (int i = 0; i < a; ++i) tok[i] = x[i];
    tok[a] = t;
    out_accept_len[r] = a;
    if (out_flag_pos) out_flag_pos[r] = flag;
    if (out_margin) out_margin[r] = min_margin;
    if (out_tie_prob) out_tie_prob[r] = tie_prob + draw_tie_probability(w, V, W);
  }
  free(w);
  return 0;
}

/* Index of the largest logit of a row, the lowest index among equal maxima, NaN skipped;
 * -1 if every entry is NaN. */
static int row_argmax(const void* base, int dtype, size_t off, int V) {
  int best = -1;
  double bv = 0.0;
  for (int j = 0; j < V; ++j) {
    const double z = logit_at(base, dtype, off + (size_t)j);
    if (isnan(z)) continue;
    if (best < 0 || z > bv) {
      best = j;
      bv = z;
    }
  }
  return best;
}

int oracle_spec_verify_greedy(const void* target, int dtype, const int32_t* draft_tokens,
                              const int32_t* num_draft, int B, int k, int V,
                              int32_t* out_tokens, int32_t* out_accept_len, int r0, int r1) {
  if (B < 0 || k < 1 || k > ORACLE_MAX_K || V < 2 || (dtype != 0 && dtype != 1)) return -1;
  if (r0 < 0 || r1 > B || r0 > r1) return -1;
  if (r0 == r1) return 0;
  if (!target || !draft_tokens || !out_tokens || !out_accept_len) return -1;
  for (int r = r0; r < r1; ++r) {
    int32_t* tok = out_tokens + (size_t)r * (k + 1);
    const int32_t* x = draft_tokens + (size_t)r * k;
    for (int i = 0; i <= k; ++i) tok[i] = -1;
    const int n = num_draft ? num_draft[r] : k;
    int err = (n < 0 || n > k);
    for (int i = 0; !err && i < n; ++i)
      if (x[i] < 0 || x[i] >= V) err = 1;
    int g[ORACLE_MAX_ROWS];
    for (int i = 0; !err && i <= n; ++i) {
      g[i] = row_argmax(target, dtype, ((size_t)r * (k + 1) + i) * (size_t)V, V);
      if (g[i] < 0) err = 1;
    }
    if (err) {
      out_accept_len[r] = -1;
      continue;
    }
    int a = n;
    for (int i = 0; i < n; ++i)
      if (x[i] != g[i]) {
        a = i;
        break;
      }
    for (int i = 0; i < a; ++i) tok[i] = x[i];
    tok[a] = g[a];
    out_accept_len[r] = a;
  }
  return 0;
}

static int in_answer_set(const int32_t* set, int n, int32_t v) {
  for (int i = 0; i < n; ++i)
    if (set[i] == v) return 1;
  return 0;
}

/* ---- draft-side confidence stop ---- */

/* c of one draft row: its top probability (mode 0) or the inverse of its entropy in nats
 * (mode 1), from q = softmax(row / T) written out term by term in ascending token order.
 * Returns -1 when the row is not a distribution. */
static int row_confidence(const void* base, int dtype, size_t off, int V, double T, int mode,
                          double* c) {
  double m, S;
  if (softmax_stats(base, dtype, off, V, T, &m, &S) != 0) return -1;
  if (mode == 0) {
    double top = 0.0;
    for (int j = 0; j < V; ++j) {
      const double q = prob_at(base, dtype, off, m, S, T, j);
      if (q > top) top = q;
    }
    *c = top;
    return 0;
  }
  double H = 0.0;
  for (int j = 0; j < V; ++j) {
    const double q = prob_at(base, dtype, off, m, S, T, j);
    if (q > 0.0) H -= q * log(q);
  }
  *c = H > 0.0 ? 1.0 / H : INFINITY;
  return 0;
}

int oracle_draft_confidence(const void* draft, int dtype, const int32_t* num_draft, int B,
                            int k, int V, double T, int mode, double floor_val,
                            int32_t* out_num_draft, double* out_conf, int32_t* out_flag,
                            int r0, int r1) {
  if (B < 0 || k < 1 || k > ORACLE_MAX_K || V < 2 || (dtype != 0 && dtype != 1)) return -1;
  if (!(T > 0.0) || !isfinite(T) || (mode != 0 && mode != 1) || isnan(floor_val)) return -1;
  if (r0 < 0 || r1 > B || r0 > r1) return -1;
  if (r0 == r1) return 0;
  if (!draft || !out_num_draft) return -1;
  for (int r = r0; r < r1; ++r) {
    const int n_in = num_draft ? num_draft[r] : k;
    double c[ORACLE_MAX_K];
    int bad = n_in < 0 || n_in > k;
    for (int i = 0; !bad && i < n_in; ++i) {
      const size_t off = ((size_t)r * (size_t)k + (size_t)i) * (size_t)V;
      if (row_confidence(draft, dtype, off, V, T, mode, &c[i]) != 0) bad = 1;
    }
    if (bad) {
      out_num_draft[r] = -1;
      if (out_conf)
        for (int i = 0; i < k; ++i) out_conf[(size_t)r * k + i] = NAN;
      if (out_flag) out_flag[r] = -1;
      continue;
    }
    int n = n_in, flag = -1;
    for (int i = 0; i < n_in; ++i) {
      if (flag < 0 && fabs(c[i] - floor_val) <= ORACLE_CONF_MARGIN * fabs(floor_val)) flag = i;
      if (c[i] < floor_val) {
        n = i;
        break;
      }
    }
    out_num_draft[r] = n;
    if (out_conf)
      for (int i = 0; i < k; ++i) out_conf[(size_t)r * k + i] = i < n_in ? c[i] : 0.0;
    if (out_flag) out_flag[r] = flag;
  }
  return 0;
}

int oracle_logit_gap_gate(const void* logits, int dtype, int N, int V, double tau,
                          const int32_t* answer_set, int n_answer, int32_t* out_token,
                          double* out_gap, uint8_t* out_fire, uint8_t* out_flag, int i0,
                          int i1) {
  if (N < 0 || V < 2 || n_answer < 0 || (dtype != 0 && dtype != 1)) return -1;
  if (i0 < 0 || i1 > N || i0 > i1) return -1;
  if (i0 == i1) return 0;
  if (!logits || !out_token || !out_gap || !out_fire || (n_answer > 0 && !answer_set))
    return -1;
  for (int row = i0; row < i1; ++row) {
    const size_t off = (size_t)row * (size_t)V;
    /* Top2 of the row as a multiset, and the lowest index of the largest value. */
    double l1 = -INFINITY, l2 = -INFINITY;
    int ahat = -1;
    for (int j = 0; j < V; ++j) {
      const double z = logit_at(logits, dtype, off + (size_t)j);
      if (isnan(z)) continue;
      if (ahat < 0) {
        l1 = z;
        ahat = j;
      } else if (z > l1) {
        l2 = l1;
        l1 = z;
        ahat = j;
      } else if (z > l2) {
        l2 = z;
      }
    }
    if (out_flag) out_flag[row] = 0;
    if (ahat < 0) {
      out_token[row] = -1;
      out_gap[row] = NAN;
      out_fire[row] = 0;
      continue;
    }
    const double gap = l1 - l2;
    out_token[row] = ahat;
    out_gap[row] = gap;
    out_fire[row] = (uint8_t)((gap > tau) && in_answer_set(answer_set, n_answer, ahat));
    if (out_flag) out_flag[row] = (uint8_t)(fabs(gap - tau) < ORACLE_TIE_MARGIN);
  }
  return 0;
}

/* ---------------------------------------------------------------------- gate calibration */

void oracle_wilson(int64_t k, int64_t n, double z, double* lo, double* hi) {
  if (n <= 0) {
    *lo = NAN;
    *hi = NAN;
    return;
  }
  const double nn = (double)n;
  const double p = (double)k / nn;
  const double z2 = z * z;
  const double denom = 1.0 + z2 / nn;
  const double centre = (p + z2 / (2.0 * nn)) / denom;
  const double half = z / denom * sqrt(p * (1.0 - p) / nn + z2 / (4.0 * nn * nn));
  double a = centre - half, b = centre + half;
  if (a < 0.0) a = 0.0;
  if (b > 1.0) b = 1.0;
  *lo = a;
  *hi = b;
}

int oracle_risk_coverage(const float* gap, const int32_t* token, const int32_t* full_token,
                         int N, const int32_t* answer_set, int n_answer, const float* taus,
                         int T, double z, double r_max, int64_t* accepted, int64_t* wrong,
                         double* stats, int32_t* tau_index) {
  if (N < 0 || T < 1 || n_answer < 0 || !taus || !accepted || !wrong || !stats || !tau_index)
    return -1;
  if (N > 0 && (!gap || !token || !full_token)) return -1;
  for (int t = 0; t < T; ++t) {
    if (isnan(taus[t])) return -1;
    if (t > 0 && taus[t] < taus[t - 1]) return -1;
  }
  *tau_index = -1;
  /* Eq. (13) and Eq. (14), one threshold at a time, straight from the definitions. */
  for (int t = 0; t < T; ++t) {
    const double tau = (double)taus[t];
    int64_t acc = 0, bad = 0;
    for (int i = 0; i < N; ++i) {
      const double g = (double)gap[i];
      if (!(g > tau)) continue;
      if (!in_answer_set(answer_set, n_answer, token[i])) continue;
      ++acc;
      if (token[i] != full_token[i]) ++bad;
    }
    accepted[t] = acc;
    wrong[t] = bad;
    double* st = stats + 6 * (size_t)t;
    st[0] = N > 0 ? (double)acc / (double)N : NAN;
    oracle_wilson(acc, N, z, &st[1], &st[2]);
    if (acc > 0) {
      st[3] = (double)bad / (double)acc;
      oracle_wilson(bad, acc, z, &st[4], &st[5]);
    } else {
      st[3] = st[4] = st[5] = NAN;
    }
    if (*tau_index < 0 && acc > 0 && st[3] <= r_max) *tau_index = t;
  }
  return 0;
}

int oracle_conformal_residual(const void* draft, const void* truth, int dtype, int N, int V,
                              float* out, int i0, int i1) {
  if (N < 0 || V < 1 || (dtype != 0 && dtype != 1)) return -1;
  if (i0 < 0 || i1 > N || i0 > i1) return -1;
  if (i0 == i1) return 0;
  if (!draft || !truth || !out) return -1;
  for (int i = i0; i < i1; ++i) {
    const size_t off = (size_t)i * (size_t)V;
    double r = 0.0;
    int nan = 0;
    for (int j = 0; j < V; ++j) {
      const double a = logit_at(draft, dtype, off + (size_t)j);
      const double b = logit_at(truth, dtype, off + (size_t)j);
      if (isnan(a) || isnan(b)) {
        nan = 1;
        break;
      }
      const double d = a == b ? 0.0 : fabs(a - b);
      if (d > r) r = d;
    }
    out[i] = nan ? NAN : (float)r;
  }
  return 0;
}

/* Ascending order with every NaN after +inf. */
static int cmp_nan_last(const void* x, const void* y) {
  const float a = *(const float*)x, b = *(const float*)y;
  const int na = isnan(a), nb = isnan(b);
  if (na || nb) return na - nb;
  return (a > b) - (a < b);
}

int oracle_conformal_quantile(const float* r, int n, double q, float* out_q) {
  if (n < 1 || !r || !out_q || !(q > 0.0) || !(q <= 1.0)) return -1;
  const double rank = ceil((double)(n + 1) * q);
  if (rank > (double)n) {
    *out_q = INFINITY;
    return 0;
  }
  float* s = (float*)malloc(sizeof(float) * (size_t)n);
  if (!s) return -1;
  memcpy(s, r, sizeof(float) * (size_t)n);
  qsort(s, (size_t)n, sizeof(float), cmp_nan_last);
  *out_q = s[(size_t)rank - 1];
  free(s);
  return 0;
}

int oracle_conformal_admit(const void* logits, int dtype, int N, int K, int V, const float* Q,
                           int32_t* out_layer, int32_t* out_token, double* out_gap,
                           int32_t* out_flag, int n0, int n1) {
  if (N < 0 || K < 1 || V < 2 || (dtype != 0 && dtype != 1)) return -1;
  if (n0 < 0 || n1 > N || n0 > n1) return -1;
  if (n0 == n1) return 0;
  if (!logits || !Q || !out_layer || !out_token) return -1;
  for (int n = n0; n < n1; ++n) {
    int layer = K, tok = -1, flag = -1;
    for (int k = 0; k < K; ++k) {
      int32_t ahat;
      double gamma;
      uint8_t fire, tie;
      const int row = n * K + k;
      /* gamma and a_hat of the row exactly as the gate defines them (no answer set) */
      if (oracle_logit_gap_gate((const char*)logits + (size_t)row * (size_t)V *
                                                          (dtype == 0 ? 4u : 2u),
                                dtype, 1, V, 0.0, NULL, 0, &ahat, &gamma, &fire, &tie, 0, 1))
        return -1;
      if (out_gap) out_gap[row] = gamma;
      const double thr = 2.0 * (double)Q[k];
      if (layer == K && flag < 0 && !isnan(gamma) && fabs(gamma - thr) < ORACLE_TIE_MARGIN)
        flag = k;
      if (layer == K && !isnan(gamma) && thr <= gamma) {
        layer = k;
        tok = ahat;
      }
    }
    out_layer[n] = layer;
    out_token[n] = tok;
    if (out_flag) out_flag[n] = flag;
  }
  return 0;
}

int oracle_ngram_propose(const int32_t* history, const int32_t* hist_len, int B, int L_max,
                         int n_max, int n_min, int k, int32_t* out_draft,
                         int32_t* out_num_draft, int r0, int r1) {
  if (B < 0 || L_max < 1 || n_min < 1 || n_max < n_min || k < 1) return -1;
  if (r0 < 0 || r1 > B || r0 > r1) return -1;
  if (r0 == r1) return 0;
  if (!history || !hist_len || !out_draft || !out_num_draft) return -1;
  for (int r = r0; r < r1; ++r) {
    int32_t* d = out_draft + (size_t)r * k;
    for (int i = 0; i < k; ++i) d[i] = -1;
    const int L = hist_len[r];
    if (L < 0 || L > L_max) {
      out_num_draft[r] = -1;
      continue;
    }
    const int32_t* h = history + (size_t)r * L_max;
    int cnt = 0;
    /* Longest phrase first; for each length, the earliest earlier occurrence. */
    for (int n = n_max; n >= n_min && cnt == 0; --n) {
      if (n > L - 1) continue;
      for (int s = 0; s + n <= L - 1; ++s) {
        int same = 1;
        for (int t = 0; t < n; ++t)
          if (h[s + t] != h[L - n + t]) {
            same = 0;
            break;
          }
        if (!same) continue;
        const int start = s + n;
        cnt = L - start < k ? L - start : k;
        for (int i = 0; i < cnt; ++i) d[i] = h[start + i];
        break;
      }
    }
    out_num_draft[r] = cnt;
  }
  return 0;
}

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
 *                    within ORACLE_TIE_MARGIN * W of u[r, k] * W (equal when no near tie).
 * Every output pointer past out_accept_len may be NULL.
 * A request with a data error gets accept_len -1, tokens -1, p/q/resid NaN, flag -1. */
int oracle_spec_verify_sample(const void* target, const void* draft, int dtype,
                              const int32_t* draft_tokens, const int32_t* num_draft,
                              const float* uniforms, int B, int k, int V, double T,
                              int32_t* out_tokens, int32_t* out_accept_len, double* out_p,
                              double* out_q, double* out_resid, int32_t* out_flag_pos,
                              double* out_margin, int32_t* out_t_lo, int32_t* out_t_hi, int r0,
                              int r1);

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

/* Prompt-lookup n-gram proposer; outputs as the library's ngram_propose. */
int oracle_ngram_propose(const int32_t* history, const int32_t* hist_len, int B, int L_max,
                         int n_max, int n_min, int k, int32_t* out_draft,
                         int32_t* out_num_draft, int r0, int r1);

#ifdef __cplusplus
}
#endif

#endif /* ORACLE_H_ */

"""Planted mistakes in the oracle must fail its pins.

Each case edits one expression of a copy of ``oracle.c`` (a transposed operand, a wrong
index, a dropped term, a flipped comparison), compiles the copy on the CPU, routes the
oracle through it and runs the pins that should catch that kind of mistake: at least one
of them has to fail. This shows that the pins constrain the oracle rather than restate it.
"""
import os
import tempfile

import pytest

import oracle
import test_oracle_calibration as K
import test_oracle_confidence as C
import test_oracle_ready_cache as RC
import test_oracle_rules as R
import test_oracle_sample as S


def _enum_small():
    S.test_exact_enumeration_is_lossless(5, 2, 1.3, 3)


def _enum_bonus():
    S.test_exact_enumeration_is_lossless(3, 2, 0.7, 2)


MUTANTS = [
    ("residual operands transposed",
     "w[j] = p > q ? p - q : 0.0;", "w[j] = q > p ? q - p : 0.0;",
     [_enum_small, S.test_residual_mass_identity_and_searchsorted]),
    ("sampling uniform taken at the rejected position",
     "(double)u[k], &smg", "(double)u[a], &smg", [_enum_small]),
    ("temperature dropped",
     "exp((logit_at(base, dtype, off + (size_t)j) - m) / T)",
     "exp((logit_at(base, dtype, off + (size_t)j) - m))",
     [lambda: R.test_softmax_matches_torch(1000, 0.7, 3.0), _enum_small]),
    ("accept ratio inverted", "const double rho = px[i] / qx[i];",
     "const double rho = qx[i] / px[i];", [_enum_small]),
    ("non-strict accept test", "if (!((double)u[i] < rho)) {", "if (!((double)u[i] <= rho)) {",
     [S.test_accept_is_strict_at_an_exact_ratio]),
    ("non-strict inverse CDF", "if (run > target) {", "if (run >= target) {",
     [S.test_inverse_cdf_boundaries]),
    ("bonus drawn from the previous row", "const int bonus_row = from_residual ? -1 : a;",
     "const int bonus_row = from_residual ? -1 : (a > 0 ? a - 1 : a);",
     [_enum_bonus, S.test_q_equal_p_accepts_everything]),
    ("target row stride of the draft array",
     "size_t off = ((size_t)r * (k + 1) + i) * (size_t)V;\n      if (softmax_stats(target",
     "size_t off = ((size_t)r * k + i) * (size_t)V;\n      if (softmax_stats(target",
     [S.test_q_equal_p_accepts_everything, S.test_residual_mass_identity_and_searchsorted]),
    ("tie window on both sides of every token",
     "const double window = ORACLE_TIE_MARGIN * ((j != first) + (j != last));",
     "const double window = 2.0 * ORACLE_TIE_MARGIN;",
     [S.test_tie_probability_is_the_measure_of_flagged_uniforms]),
    ("tie probability without the token's own mass as a bound",
     "prob += m < window ? m : window;", "prob += window;",
     [S.test_tie_probability_is_the_measure_of_flagged_uniforms]),
    ("accept tie window one-sided",
     "const double hi = rho + ORACLE_TIE_MARGIN < 1.0 ? rho + ORACLE_TIE_MARGIN : 1.0;",
     "const double hi = rho < 1.0 ? rho : 1.0;",
     [S.test_tie_probability_is_the_measure_of_flagged_uniforms]),
    ("greedy emits the draft token at the mismatch", "tok[a] = g[a];",
     "tok[a] = a < n ? x[a] : g[a];", [R.test_greedy_argmax_and_walk]),
    ("greedy argmax keeps the last tie", "if (best < 0 || z > bv) {",
     "if (best < 0 || z >= bv) {", [R.test_greedy_argmax_and_walk]),
    ("gate argmax keeps the last tie", "} else if (z > l1) {", "} else if (z >= l1) {",
     [R.test_gate_truth_table]),
    ("gate fires at gap == tau", "(gap > tau)", "(gap >= tau)", [R.test_gate_truth_table]),
    ("gate forgets the old maximum", "l2 = l1;\n        l1 = z;", "l1 = z;",
     [R.test_gate_matches_topk]),
    ("n-gram tries the shortest phrase first",
     "for (int n = n_max; n >= n_min && cnt == 0; --n) {",
     "for (int n = n_min; n <= n_max && cnt == 0; ++n) {",
     [lambda: R.test_ngram_brute_force(3)]),
    ("n-gram takes the latest occurrence", "for (int s = 0; s + n <= L - 1; ++s) {",
     "for (int s = L - 1 - n; s >= 0; --s) {", [lambda: R.test_ngram_brute_force(2)]),
    ("entropy in bits", "if (q > 0.0) H -= q * log(q);", "if (q > 0.0) H -= q * log2(q);",
     [C.test_uniform_rows_have_closed_forms, C.test_inverse_entropy_stop_uses_the_entropy_in_nats]),
    ("confidence stop at c == floor", "if (c[i] < floor_val) {", "if (c[i] <= floor_val) {",
     [C.test_near_tie_is_flagged]),
    ("top probability of the first token", "if (q > top) top = q;", "if (j == 0) top = q;",
     [C.test_stop_is_the_first_position_below_the_floor,
      lambda: C.test_random_rows_match_scipy(1.0)]),
    ("draft count ignored", "const int n_in = num_draft ? num_draft[r] : k;",
     "const int n_in = k;", [C.test_stop_respects_the_input_draft_count]),
    ("Wilson half-width without the z^2/(4n^2) term",
     "sqrt(p * (1.0 - p) / nn + z2 / (4.0 * nn * nn))", "sqrt(p * (1.0 - p) / nn)",
     [K.test_wilson_matches_the_pages_printed_intervals,
      lambda: K.test_wilson_matches_scipy(0, 37)]),
    ("risk over all decision points", "st[3] = (double)bad / (double)acc;",
     "st[3] = (double)bad / (double)N;", [K.test_the_pages_operating_point]),
    ("gate calibration accepts gap == tau", "if (!(g > tau)) continue;",
     "if (!(g >= tau)) continue;", [K.test_the_pages_operating_point,
                                     K.test_sweep_matches_sort_and_count]),
    ("calibration ignores the answer set",
     "if (!in_answer_set(answer_set, n_answer, token[i])) continue;", "",
     [K.test_the_pages_operating_point]),
    ("calibration keeps the last qualifying tau", "if (*tau_index < 0 && acc > 0",
     "if (acc > 0", [K.test_selection_picks_the_smallest_qualifying_tau_not_a_monotone_one]),
    ("conformal rank without the +1", "ceil((double)(n + 1) * q)", "ceil((double)n * q)",
     [K.test_quantile_rank_rule_and_edges,
      lambda: K.test_quantile_has_the_split_conformal_coverage(19, 0.9)]),
    ("residual without the absolute value", "a == b ? 0.0 : fabs(a - b)", "a == b ? 0.0 : a - b",
     [K.test_residual_hand_built_rows,
      K.test_residual_bounds_the_argmax_no_flip_theorem]),
    ("conformal admission without the factor 2", "const double thr = 2.0 * (double)Q[k];",
     "const double thr = (double)Q[k];", [K.test_admit_takes_the_earliest_admitting_layer]),
    ("conformal admission keeps the last layer", "if (layer == K && !isnan(gamma) && thr <= gamma)",
     "if (!isnan(gamma) && thr <= gamma)", [K.test_admit_takes_the_earliest_admitting_layer]),
]


@pytest.fixture(scope="module")
def workdir():
    with tempfile.TemporaryDirectory(prefix="oracle_mutants_") as d:
        yield d


@pytest.mark.parametrize("name,old,new,pins", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(workdir, name, old, new, pins):
    src = oracle.source()
    assert src.count(old) == 1, f"mutation site not unique: {old!r}"
    path = os.path.join(workdir, name.replace(" ", "_") + ".so")
    oracle.compile_variant(src.replace(old, new), path)
    failures = 0
    with oracle.library(path):
        for pin in pins:
            try:
                pin()
            except (AssertionError, ValueError):
                failures += 1
    assert failures >= 1, f"no pin caught the planted mistake: {name}"


# The ready-distribution cache oracle is Python: its mutants are edits of that module's source,
# executed as a fresh module whose ReadyCache class the pins then use.
PY_MUTANTS = [
    ("gate fires at gamma == tau", 'if s["gap"] > float(np.float32(tau))',
     'if s["gap"] >= float(np.float32(tau))',
     [RC.test_gate_falls_through_on_a_small_gap_or_outside_the_answer_set]),
    ("eligibility ignores the decision point",
     'int(start[r]) == s["position"] - L and', "",
     [RC.test_eligibility_is_an_exact_entry_match]),
    ("skip keeps the old pre-position", 's["valid"] = s["decoded"] = s["consumed"] = False\n'
     '                self.stats["skipped"] += 1', 'self.stats["skipped"] += 1',
     [RC.test_budget_skip_leaves_no_ready_distribution]),
    ("invalidation keeps the distribution", 's["valid"] = s["decoded"] = s["consumed"] = False\n'
     '            s["epoch"] += 1', 's["epoch"] += 1',
     [RC.test_invalidation_returns_to_no_ready_distribution,
      RC.test_served_tokens_are_never_stale]),
    ("every eligible request counts as a consumption", 'if not s["consumed"]:\n'
     '                s["consumed"] = True\n                self.stats["consumed"] += 1',
     's["consumed"] = True\n            self.stats["consumed"] += 1',
     [lambda: RC.test_hit_rate_matches_eq8_for_memoryless_sessions(4.0)]),
    ("decision point without the entry length", 's["position"] = n_s + L', 's["position"] = n_s',
     [RC.test_record_then_fast_serve, RC.test_served_tokens_are_never_stale]),
]


@pytest.mark.parametrize("name,old,new,pins", PY_MUTANTS, ids=[m[0] for m in PY_MUTANTS])
def test_planted_mistake_in_the_cache_oracle_is_caught(monkeypatch, name, old, new, pins):
    import types

    import oracle.ready_cache as mod

    src = open(mod.__file__).read()
    assert src.count(old) == 1, f"mutation site not unique: {old!r}"
    m = types.ModuleType("ready_cache_mutant")
    m.__dict__["__package__"] = "oracle"
    exec(compile(src.replace(old, new), "ready_cache_mutant", "exec"), m.__dict__)
    monkeypatch.setattr(RC, "ReadyCache", m.ReadyCache)
    failures = 0
    for pin in pins:
        try:
            pin()
        except (AssertionError, ValueError, IndexError, TypeError):
            failures += 1
    assert failures >= 1, f"no pin caught the planted mistake: {name}"

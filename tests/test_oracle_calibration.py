"""Pins of the oracle's gate calibration and conformal gate.

Each pin fixes a value by something other than the oracle's own formula:
- the operating point the pre-positioning page prints (121 of 128 served at tau = 2.0, 16 of
  them false accepts, with Wilson 95 % intervals), from tests/golden;
- scipy's independent Wilson interval and the interval's closed-form special cases;
- a sort-and-count restatement of coverage and risk, and designed threshold sequences;
- for the conformal gate: the split-conformal coverage law P(r_new <= Q) = rank / (n + 1)
  checked by simulation, the argmax no-flip theorem it rests on, and hand-built rows.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden")
Z95 = 1.959963984540054


def _gold():
    with open(os.path.join(GOLD, "gate_calibration_operating_point.json")) as f:
        return json.load(f)


# --------------------------------------------------------------------------- Wilson interval
def test_wilson_matches_the_pages_printed_intervals():
    g = _gold()
    lo, hi = oracle.wilson(g["served"], g["decision_points"], g["z"])
    for got, want in zip((lo, hi), g["coverage_ci_printed"]):
        assert abs(got - want) <= 0.005 + 1e-12, (got, want)
    lo, hi = oracle.wilson(g["false_accepts"], g["served"], g["z"])
    for got, want in zip((lo, hi), g["risk_ci_printed"]):
        assert abs(got - want) <= 0.0005 + 1e-12, (got, want)


@pytest.mark.parametrize("k,n", [(0, 1), (1, 1), (3, 10), (121, 128), (16, 121), (500, 1000),
                                 (0, 37), (37, 37), (1, 100000)])
def test_wilson_matches_scipy(k, n):
    stats = pytest.importorskip("scipy.stats")
    ci = stats.binomtest(k, n).proportion_ci(confidence_level=0.95, method="wilson")
    lo, hi = oracle.wilson(k, n, Z95)
    assert lo == pytest.approx(ci.low, abs=1e-12)
    assert hi == pytest.approx(ci.high, abs=1e-12)


def test_wilson_special_cases():
    # k = 0 gives lo = 0 and hi = z^2 / (n + z^2); k = n mirrors it; n = 0 is undefined
    for n in (1, 5, 128):
        lo, hi = oracle.wilson(0, n, Z95)
        assert lo == 0.0 and hi == pytest.approx(Z95 ** 2 / (n + Z95 ** 2), rel=1e-14)
        lo2, hi2 = oracle.wilson(n, n, Z95)
        assert hi2 == 1.0 and lo2 == pytest.approx(1.0 - hi, rel=1e-13)
    assert all(math.isnan(v) for v in oracle.wilson(0, 0, Z95))
    # symmetry k <-> n - k, and z = 0 collapses to the point estimate
    lo, hi = oracle.wilson(7, 30, Z95)
    lo2, hi2 = oracle.wilson(23, 30, Z95)
    assert lo == pytest.approx(1 - hi2, rel=1e-13) and hi == pytest.approx(1 - lo2, rel=1e-13)
    assert oracle.wilson(7, 30, 0.0) == pytest.approx((7 / 30, 7 / 30), rel=1e-15)


# ------------------------------------------------------------------------ risk and coverage
def _operating_point_fixture(seed=0):
    """128 decision points built to the page's counts: at tau = 2.0, 121 fire with 16 of them
    disagreeing with the full path; 7 fall through (three by a small gap, two by a gap of
    exactly tau, two with the argmax outside A)."""
    g = _gold()
    rng = np.random.default_rng(seed)
    A = np.sort(rng.choice(1000, g["answer_set_size"], replace=False)).astype(np.int32)
    outside = np.setdiff1d(np.arange(1000), A)
    N = g["decision_points"]
    gap = rng.uniform(2.05, 9.0, N).astype(np.float32)
    token = rng.choice(A, N).astype(np.int32)
    gap[:3] = [0.3, 1.2, 1.99]
    gap[3:5] = 2.0                       # not strictly above tau
    token[5:7] = rng.choice(outside, 2)  # argmax outside the fast-answer set
    full = token.copy()
    served = np.arange(7, N)
    wrong = rng.choice(served, g["false_accepts"], replace=False)
    full[wrong] = (full[wrong] + 1) % 1000
    full[:7] = (full[:7] + 3) % 1000     # falls through: its correctness does not count
    return gap, token, full, A


def test_the_pages_operating_point():
    g = _gold()
    gap, token, full, A = _operating_point_fixture()
    out = oracle.risk_coverage(gap, token, full, A, [g["tau"]], g["z"], r_max=0.15)
    assert out["accepted"][0] == g["served"] and out["wrong"][0] == g["false_accepts"]
    # the printed rates: coverage over all decision points, risk over the served ones
    assert abs(out["coverage"][0] - g["coverage_printed"]) <= 0.0005
    assert abs(out["risk"][0] - g["risk_printed"]) <= 0.0005
    assert abs(out["cov_lo"][0] - 0.89) <= 0.005 and abs(out["cov_hi"][0] - 0.97) <= 0.005
    assert abs(out["risk_lo"][0] - 0.083) <= 0.0005
    assert abs(out["risk_hi"][0] - 0.204) <= 0.0005
    assert out["tau_index"] == 0


def _sort_and_count(gap, token, full, A, taus):
    """An independent restatement: sort the admissible gaps once, count by binary search."""
    ok = np.isin(token, A) & ~np.isnan(gap)
    g = np.sort(gap[ok].astype(np.float64))
    gw = np.sort(gap[ok & (token != full)].astype(np.float64))
    acc = len(g) - np.searchsorted(g, np.asarray(taus, np.float64), side="right")
    bad = len(gw) - np.searchsorted(gw, np.asarray(taus, np.float64), side="right")
    return acc, bad


def test_sweep_matches_sort_and_count():
    rng = np.random.default_rng(3)
    N = 2000
    A = np.arange(0, 400, 3, dtype=np.int32)
    token = rng.integers(0, 400, N).astype(np.int32)
    gap = np.abs(rng.standard_normal(N) * 3).astype(np.float32)
    gap[::97] = np.nan
    gap[5:40] = 1.5  # ties on a threshold
    full = np.where(rng.random(N) < 0.8 * (1 - np.exp(-gap.astype(np.float64))), token,
                    token + 1).astype(np.int32)
    taus = np.concatenate([[-np.inf, -1.0, 0.0], np.linspace(0, 10, 41), [1.5, 1.5, np.inf]])
    taus = np.sort(taus).astype(np.float32)
    out = oracle.risk_coverage(gap, token, full, A, taus, Z95, r_max=0.3)
    acc, bad = _sort_and_count(gap, token, full, A, taus)
    np.testing.assert_array_equal(out["accepted"], acc)
    np.testing.assert_array_equal(out["wrong"], bad)
    # coverage is monotone non-increasing in tau (the page's Eq. (13) remark)
    assert (np.diff(out["accepted"]) <= 0).all()
    np.testing.assert_allclose(out["coverage"], acc / N, rtol=1e-15)
    has = acc > 0
    np.testing.assert_allclose(out["risk"][has], bad[has] / acc[has], rtol=1e-15)
    assert np.isnan(out["risk"][~has]).all() and np.isnan(out["risk_lo"][~has]).all()
    # the selection: smallest tau whose risk meets the budget, among taus that serve anything
    ok = np.flatnonzero(has & (out["risk"] <= 0.3))
    assert out["tau_index"] == (ok[0] if ok.size else -1)


def test_selection_picks_the_smallest_qualifying_tau_not_a_monotone_one():
    # risk is not monotone in tau (the page's Figure 7 remark): the selection takes the first
    # tau that meets the budget even if a larger one breaks it again
    gap = np.array([1, 2, 3, 4, 5, 6], np.float32)
    token = np.zeros(6, np.int32)
    full = np.array([1, 0, 0, 0, 1, 0], np.int32)   # wrong at gaps 1 and 5
    taus = np.array([0.5, 1.5, 4.5, 5.5], np.float32)
    out = oracle.risk_coverage(gap, token, full, [0], taus, Z95, r_max=0.2)
    np.testing.assert_array_equal(out["accepted"], [6, 5, 2, 1])
    np.testing.assert_array_equal(out["wrong"], [2, 1, 1, 0])
    assert out["tau_index"] == 1  # risk 1/5 = 0.2 <= 0.2; tau 4.5 has 1/2, tau 5.5 has 0
    assert oracle.risk_coverage(gap, token, full, [0], taus, Z95, 0.1)["tau_index"] == 3
    assert oracle.risk_coverage(gap, token, full, [0], taus[:3], Z95, 0.1)["tau_index"] == -1


def test_sweep_argument_checks():
    g = np.ones(3, np.float32)
    t = np.zeros(3, np.int32)
    with pytest.raises(ValueError):
        oracle.risk_coverage(g, t, t, [0], np.array([2.0, 1.0], np.float32))  # unsorted
    with pytest.raises(ValueError):
        oracle.risk_coverage(g, t, t, [0], np.array([np.nan], np.float32))


# ------------------------------------------------------------------------ conformal gate
def test_residual_hand_built_rows():
    V = 7
    t = np.zeros((5, V), np.float32)
    d = t.copy()
    d[0, 3] = 0.75                       # one logit moved: r = 0.75
    d[1] = t[1] - 2.5                    # a constant shift: r = 2.5
    t[2, 1] = d[2, 1] = -np.inf          # masked in both: no contribution
    d[2, 4] = -1.0
    d[3, 5] = -np.inf                    # masked in one only: r = inf
    t[4, 6] = np.nan                     # NaN: r = NaN
    r = oracle.conformal_residual(d[None], t[None])
    assert r[0] == 0.75 and r[1] == 2.5 and r[2] == 1.0
    assert r[3] == np.inf and np.isnan(r[4])


def test_residual_bounds_the_argmax_no_flip_theorem():
    # if 2 * sup|d - t| <= the draft's runner-up margin, argmax(t) = argmax(d) (or ties it);
    # and the theorem is tight: a residual of just over half the margin can flip it
    rng = np.random.default_rng(11)
    N, V = 400, 64
    t = (rng.standard_normal((N, V)) * 2).astype(np.float32)
    d = (t + rng.uniform(-1, 1, (N, 1)).astype(np.float32) *
         rng.standard_normal((N, V)).astype(np.float32) * 0.3).astype(np.float32)
    r = oracle.conformal_residual(d, t).astype(np.float64)
    g = oracle.logit_gap_gate(d, 0.0, None)
    admitted = 2.0 * r <= g["gap"]
    assert admitted.sum() > 50
    tt = t.astype(np.float64)
    ahat = g["token"]
    assert (tt[admitted, ahat[admitted]] >= tt[admitted].max(axis=1)).all()
    # tightness: margin gamma, residual gamma/2 + eps on the two leading logits flips it
    d1 = np.zeros((1, V), np.float32)
    d1[0, 0], d1[0, 1] = 3.0, 1.0        # gamma = 2
    t1 = d1.copy()
    t1[0, 0], t1[0, 1] = 1.9, 2.1        # each moved by 1.1 > gamma / 2
    assert oracle.conformal_residual(d1, t1)[0] == np.float32(1.1)
    assert np.argmax(t1[0]) != np.argmax(d1[0])


def test_quantile_rank_rule_and_edges():
    r = np.array([5, 1, 4, 2, 3], np.float32)
    # ranks ceil(6 q): q = 0.5 -> 3rd smallest; q = 0.8 -> 5th; q = 0.9 -> 6 > n -> +inf
    assert oracle.conformal_quantile(r, 0.5) == 3.0
    assert oracle.conformal_quantile(r, 0.8) == 5.0
    assert oracle.conformal_quantile(r, 0.9) == np.inf
    assert oracle.conformal_quantile(r, 1e-9) == 1.0
    rn = np.array([np.nan, 1.0, np.inf, 0.5], np.float32)  # NaN above +inf
    assert oracle.conformal_quantile(rn, 0.4) == 1.0       # rank 2 of (0.5, 1, inf, NaN)
    assert oracle.conformal_quantile(rn, 0.6) == np.inf    # rank 3
    assert np.isnan(oracle.conformal_quantile(rn, 0.8))    # rank 4
    with pytest.raises(ValueError):
        oracle.conformal_quantile(r, 0.0)


@pytest.mark.parametrize("n,q", [(19, 0.9), (49, 0.8), (9, 0.5)])
def test_quantile_has_the_split_conformal_coverage(n, q):
    # exchangeable continuous residuals: P(r_new <= Q) = ceil((n+1) q) / (n + 1) exactly
    rng = np.random.default_rng(n)
    trials = 20000
    cal = rng.exponential(1.0, (trials, n)).astype(np.float32)
    new = rng.exponential(1.0, trials).astype(np.float32)
    Q = np.array([oracle.conformal_quantile(c, q) for c in cal])
    want = math.ceil((n + 1) * q) / (n + 1)
    got = float(np.mean(new <= Q))
    sd = math.sqrt(want * (1 - want) / trials)
    assert abs(got - want) < 5 * sd, (got, want)
    assert 1.0 / (n + 1) > 5 * sd  # an off-by-one rank would fail


def test_admit_takes_the_earliest_admitting_layer():
    V, K = 16, 4
    z = np.zeros((3, K, V), np.float32)
    # step 0: gaps 0.5, 1.0, 3.0, 5.0 at layers 0..3 (argmax 2, 3, 4, 5)
    for k, (gam, a) in enumerate([(0.5, 2), (1.0, 3), (3.0, 4), (5.0, 5)]):
        z[0, k, a] = gam
    z[1] = z[0]
    z[2, :, :] = np.nan                   # no finite logit anywhere: never admits
    Q = np.array([0.2, 0.6, 1.5, 1.0], np.float32)  # 2Q = 0.4, 1.2, 3.0, 2.0
    out = oracle.conformal_admit(z, Q)
    # layer 0: 0.4 <= 0.5 admits at once
    assert out["layer"][0] == 0 and out["token"][0] == 2
    Q2 = np.array([0.3, 0.6, 1.5, 1.0], np.float32)  # 2Q = 0.6 > 0.5, 1.2 > 1, 3.0 <= 3.0
    out = oracle.conformal_admit(z, Q2)
    assert out["layer"][0] == 2 and out["token"][0] == 4   # non-strict: 2Q = gamma admits
    assert out["flag"][0] == 2                             # and it is a near tie
    assert out["layer"][2] == K and out["token"][2] == -1
    np.testing.assert_allclose(out["gap"][0], [0.5, 1.0, 3.0, 5.0])
    Q3 = np.full(K, 10.0, np.float32)
    out = oracle.conformal_admit(z, Q3)
    assert (out["layer"][:2] == K).all() and (out["flag"] == -1).all()

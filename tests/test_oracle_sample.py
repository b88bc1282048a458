"""Pins of the oracle's sampled verify against what the pages and the mathematics fix.

- Exact enumeration of the emitted-token law on tiny vocabularies equals the target
  softmax: the losslessness result of "Speculative Decoding: The Physics of Stolen Time in
  Autoregressive Inference", section 2. Uniforms are the 2^-24 grid the inputs use, so
  the law is computed exactly over that grid and may differ from p by the grid step only.
- q = p accepts every draft token (ratio 1 > u) and the bonus token follows p_k.
- A chi-square test of 1e5 seeded trials of the first emitted token against p_0.
- The rejection probability identity Z = 1 - sum(min(p, q)) (same page, section 2).
- E[tokens/step] = (1 - alpha^(k+1)) / (1 - alpha) for iid acceptance, and the page's own
  printed value of about 1.6 at alpha = 0.4, k = 4 (same page, sections 3 and 4).
- The inverse-CDF draw equals numpy.searchsorted over the CDF of the distribution.
The reference probabilities come from torch.softmax in double, not from the oracle.
"""
import json
import os

import numpy as np
import pytest
import torch
from scipy import stats

import oracle

GRID = 1 << 24  # uniforms are multiples of 2^-24 in [0, 1)
HERE = os.path.dirname(os.path.abspath(__file__))


def softmax64(z, T):
    return torch.softmax(torch.as_tensor(np.asarray(z, np.float64)) / T, dim=-1).numpy()


def _batch(zt, zd, tokens, uniforms, T, num_draft=None):
    """Run the oracle on P probes that share the rows zt [k+1, V], zd [k, V]."""
    P = tokens.shape[0]
    t = np.ascontiguousarray(np.broadcast_to(zt, (P,) + zt.shape), np.float32)
    d = np.ascontiguousarray(np.broadcast_to(zd, (P,) + zd.shape), np.float32)
    nd = None if num_draft is None else np.full(P, num_draft, np.int32)
    return oracle.spec_verify_sample(t, d, tokens.astype(np.int32),
                                     nd, uniforms.astype(np.float32), T)


def _first_true(pred_at, n_probe):
    """Vectorised integer bisection: for each probe the smallest i in [0, GRID] with
    pred_at(i)[probe] True, given each predicate is False then True along i."""
    lo = np.zeros(n_probe, np.int64)      # pred False at lo-1 (or lo == 0)
    hi = np.full(n_probe, GRID, np.int64)  # pred True at hi (GRID stands for "never")
    while True:
        active = lo < hi
        if not active.any():
            return hi
        mid = (lo + hi) // 2
        res = pred_at(mid)
        hi = np.where(active & res, mid, hi)
        lo = np.where(active & ~res, mid + 1, lo)


def _sampler_law(zt, zd, T, tokens, u_prefix, pos, V, k):
    """Law of the token the oracle emits at index ``pos`` as u[k] sweeps the grid, the other
    uniforms held at u_prefix. Returns (law over V tokens, emitted tokens are monotone)."""
    ys = np.arange(1, V)

    def pred(i):
        u = np.repeat(u_prefix[None, :], ys.size, 0)
        u[:, k] = i / GRID
        out = _batch(zt, zd, np.repeat(tokens[None, :], ys.size, 0), u, T)
        return out["tokens"][:, pos] >= ys

    c = np.concatenate([[0], _first_true(pred, ys.size), [GRID]])
    return np.diff(c) / GRID


def emitted_law(zt, zd, T, j):
    """Law of the token emitted at position j given positions < j were accepted, taken
    only from the oracle's decisions (bisection over the uniform grid)."""
    k, V = zd.shape
    q = softmax64(zd, T)
    tokens = np.argmax(zd, axis=1).astype(np.int32)  # any token: u_i = 0 accepts it
    u0 = np.zeros(k + 1)
    if j == k:  # every draft accepted: the bonus draw
        return _sampler_law(zt, zd, T, tokens, u0, k, V, k)
    law = np.zeros(V)
    xs = np.arange(V)

    def rejects(i):
        u = np.repeat(u0[None, :], V, 0)
        u[:, j] = i / GRID
        tk = np.repeat(tokens[None, :], V, 0)
        tk[:, j] = xs
        out = _batch(zt, zd, tk, u, T)
        assert (out["accept_len"] >= j).all()
        return out["accept_len"] == j

    A = _first_true(rejects, V) / GRID  # measure of u_j that accepts x
    for x in range(V):
        law[x] += q[j, x] * A[x]
        if A[x] < 1.0:
            tk = tokens.copy()
            tk[j] = x
            u = u0.copy()
            u[j] = round(A[x] * GRID) / GRID  # the smallest grid uniform that rejects x
            law += q[j, x] * (1.0 - A[x]) * _sampler_law(zt, zd, T, tk, u, j, V, k)
    return law


@pytest.mark.parametrize("V,k,T,seed", [(2, 1, 1.0, 1), (3, 2, 0.7, 2), (5, 2, 1.3, 3),
                                        (8, 3, 0.9, 4), (6, 3, 2.0, 5)])
def test_exact_enumeration_is_lossless(V, k, T, seed):
    rng = np.random.default_rng(seed)
    zt = rng.normal(0, 1.5, (k + 1, V)).astype(np.float32)
    zd = (zt[:k] + rng.normal(0, 1.0, (k, V))).astype(np.float32)
    p = softmax64(zt, T)
    for j in range(k + 1):
        law = emitted_law(zt, zd, T, j)
        # grid discretisation: each interval end moves by < 2^-24, and the accept measure
        # of every draft token too; the bound below covers all of them
        assert np.abs(law - p[j]).max() <= (2 * V + 2) / GRID, (j, law, p[j])
        assert abs(law.sum() - 1.0) < 1e-12


def test_q_equal_p_accepts_everything():
    rng = np.random.default_rng(11)
    B, k, V, T = 4000, 4, 12, 0.8
    zt = rng.normal(0, 2.0, (B, k + 1, V)).astype(np.float32)
    zd = zt[:, :k].copy()
    q = softmax64(zd, T)
    x = np.array([[rng.choice(V, p=q[b, i]) for i in range(k)] for b in range(B)], np.int32)
    u = rng.integers(0, GRID, (B, k + 1)) / GRID
    out = oracle.spec_verify_sample(zt, zd, x, None, u.astype(np.float32), T)
    assert (out["accept_len"] == k).all()
    assert (out["tokens"][:, :k] == x).all()
    assert np.allclose(out["p"], out["q"], rtol=0, atol=0)
    assert (out["resid"] == 0).all()
    # the bonus token follows p_k of its own request: compare with searchsorted
    pk = softmax64(zt[:, k], T)
    cdf = np.cumsum(pk, axis=1)
    want = [np.searchsorted(cdf[b], u[b, k] * cdf[b, -1], side="right") for b in range(B)]
    assert (out["tokens"][:, k] == np.array(want)).all()


def test_chi_square_first_token():
    rng = np.random.default_rng(2024)
    trials, k, V, T = 100_000, 3, 16, 1.1
    zt1 = rng.normal(0, 1.5, (k + 1, V)).astype(np.float32)
    zd1 = (0.7 * zt1[:k] + rng.normal(0, 1.0, (k, V))).astype(np.float32)
    p = softmax64(zt1, T)
    q = softmax64(zd1, T)
    x = np.stack([rng.choice(V, size=trials, p=q[i]) for i in range(k)], 1).astype(np.int32)
    u = (rng.integers(0, GRID, (trials, k + 1)) / GRID).astype(np.float32)
    zt = np.ascontiguousarray(np.broadcast_to(zt1, (trials, k + 1, V)))
    zd = np.ascontiguousarray(np.broadcast_to(zd1, (trials, k, V)))
    out = oracle.spec_verify_sample(zt, zd, x, None, u, T, threads=4)
    a = out["accept_len"]
    assert (a >= 0).all()
    for j in range(k + 1):
        reached = a >= j
        obs = np.bincount(out["tokens"][reached, j], minlength=V)
        exp = p[j] * reached.sum()
        keep = exp > 5
        stat = ((obs[keep] - exp[keep]) ** 2 / exp[keep]).sum()
        pval = stats.chi2.sf(stat, keep.sum() - 1)
        assert pval > 1e-3, (j, stat, pval)


def test_residual_mass_identity_and_searchsorted():
    rng = np.random.default_rng(7)
    B, k, V, T = 300, 3, 40, 0.9
    zt = rng.normal(0, 2.0, (B, k + 1, V)).astype(np.float32)
    zd = (0.5 * zt[:, :k] + rng.normal(0, 1.5, (B, k, V))).astype(np.float32)
    q = softmax64(zd, T)
    x = np.array([[rng.choice(V, p=q[b, i]) for i in range(k)] for b in range(B)], np.int32)
    u = (rng.integers(0, GRID, (B, k + 1)) / GRID).astype(np.float32)
    out = oracle.spec_verify_sample(zt, zd, x, None, u, T)
    p = softmax64(zt, T)
    rejected = 0
    for b in range(B):
        a = out["accept_len"][b]
        assert 0 <= a <= k
        for i in range(k):
            assert abs(out["p"][b, i] - p[b, i, x[b, i]]) < 1e-15
            assert abs(out["q"][b, i] - q[b, i, x[b, i]]) < 1e-15
        if a < k:
            rejected += 1
            Z = 1.0 - np.minimum(p[b, a], q[b, a]).sum()
            assert abs(out["resid"][b] - Z) < 1e-12
            w = np.maximum(p[b, a] - q[b, a], 0.0)
        else:
            assert out["resid"][b] == 0.0
            w = p[b, k]
        cdf = np.cumsum(w)
        tgt = float(u[b, k]) * cdf[-1]
        t = np.searchsorted(cdf, tgt, side="right")
        if np.min(np.abs(cdf - tgt)) > 1e-9:
            assert out["tokens"][b, a] == t
        assert (out["tokens"][b, :a] == x[b, :a]).all()
        assert (out["tokens"][b, a + 1:] == -1).all()
    assert rejected > B // 4


def _iid_rows(p_logits, q_logits, trials, k, rng):
    V = len(p_logits)
    zt = np.ascontiguousarray(np.broadcast_to(np.float32(p_logits), (trials, k + 1, V)))
    zd = np.ascontiguousarray(np.broadcast_to(np.float32(q_logits), (trials, k, V)))
    q = softmax64(q_logits, 1.0)
    x = rng.choice(V, size=(trials, k), p=q).astype(np.int32)
    u = (rng.integers(0, GRID, (trials, k + 1)) / GRID).astype(np.float32)
    return zt, zd, x, u


def test_expected_tokens_per_step_closed_form():
    rng = np.random.default_rng(99)
    trials, k, V = 200_000, 5, 10
    pl = rng.normal(0, 1.2, V)
    ql = pl + rng.normal(0, 1.0, V)
    zt, zd, x, u = _iid_rows(pl, ql, trials, k, rng)
    out = oracle.spec_verify_sample(zt, zd, x, None, u, 1.0, threads=4)
    p, q = softmax64(np.float32(pl), 1.0), softmax64(np.float32(ql), 1.0)
    alpha = np.minimum(p, q).sum()
    want = (1 - alpha ** (k + 1)) / (1 - alpha)
    n = out["accept_len"] + 1
    sigma = n.std() / np.sqrt(trials)
    assert abs(n.mean() - want) < 4 * sigma, (n.mean(), want, sigma)
    # acceptance frequency at position 0 estimates alpha
    acc0 = (out["accept_len"] >= 1).mean()
    assert abs(acc0 - alpha) < 4 * np.sqrt(alpha * (1 - alpha) / trials)


def test_expected_tokens_per_step_printed_value():
    with open(os.path.join(HERE, "golden", "expected_tokens_per_step.json")) as f:
        g = json.load(f)
    alpha, k = g["alpha"], g["k"]
    # two-token rows with sum(min(p, q)) = alpha: p = (1 - alpha/2, alpha/2), q reversed
    pl = np.log([1 - alpha / 2, alpha / 2])
    ql = pl[::-1].copy()
    rng = np.random.default_rng(5)
    trials = 200_000
    zt, zd, x, u = _iid_rows(pl, ql, trials, k, rng)
    out = oracle.spec_verify_sample(zt, zd, x, None, u, 1.0, threads=4)
    n = out["accept_len"] + 1
    assert abs(n.mean() - g["tokens_per_step_printed"]) < g["printed_precision"]
    closed = (1 - alpha ** (k + 1)) / (1 - alpha)
    assert abs(n.mean() - closed) < 4 * n.std() / np.sqrt(trials)


def test_accept_is_strict_at_an_exact_ratio():
    # p(x) = 1/4 (four equal logits), q(x) = 1/2 (two live tokens): ratio exactly 0.5
    zt = np.zeros((1, 2, 4), np.float32)
    zd = np.array([[[0.0, 0.0, -np.inf, -np.inf]]], np.float32)
    x = np.array([[0]], np.int32)
    for u0, want in [(0.5, 0), (np.nextafter(np.float32(0.5), np.float32(0)), 1), (0.0, 1)]:
        u = np.array([[u0, 0.3]], np.float32)
        out = oracle.spec_verify_sample(zt, zd, x, None, u, 1.0)
        assert out["accept_len"][0] == want, u0


def test_inverse_cdf_boundaries():
    # num_draft = 0: the bonus draw from p_0 = (1/4, 1/4, 1/4, 1/4)
    zt = np.zeros((1, 2, 4), np.float32)
    zd = np.zeros((1, 1, 4), np.float32)
    x = np.array([[0]], np.int32)
    nd = np.array([0], np.int32)
    for uk, want in [(0.0, 0), (0.25, 1), (np.nextafter(np.float32(0.25), np.float32(0)), 0),
                     (0.5, 2), (0.75, 3), (np.nextafter(np.float32(1), np.float32(0)), 3)]:
        u = np.array([[0.9, uk]], np.float32)
        out = oracle.spec_verify_sample(zt, zd, x, nd, u, 1.0)
        assert out["accept_len"][0] == 0 and out["tokens"][0, 0] == want, uk
        assert out["tokens"][0, 1] == -1
        # the tie window spans both neighbours exactly at a CDF boundary
        lo, hi = out["t_lo"][0], out["t_hi"][0]
        near = min(abs(float(uk) - b) for b in (0.25, 0.5, 0.75)) < 1e-6
        if near:
            assert lo <= want <= hi and hi - lo == 1 and out["flag_pos"][0] == 0, uk
        else:
            assert (lo, hi) == (want, want) and out["flag_pos"][0] == -1, uk


def test_masked_tokens_are_never_drawn():
    rng = np.random.default_rng(3)
    B, k, V = 2000, 2, 9
    zt = rng.normal(0, 1, (B, k + 1, V)).astype(np.float32)
    zt[:, :, ::2] = -np.inf  # even tokens masked in the target
    zd = rng.normal(0, 1, (B, k, V)).astype(np.float32)
    x = rng.integers(0, V, (B, k)).astype(np.int32)
    u = (rng.integers(0, GRID, (B, k + 1)) / GRID).astype(np.float32)
    out = oracle.spec_verify_sample(zt, zd, x, None, u, 1.0)
    a = out["accept_len"]
    emitted = out["tokens"][np.arange(B), a]
    assert (emitted % 2 == 1).all()
    # an accepted draft token must have target probability > 0
    for b in range(B):
        assert (out["tokens"][b, :a[b]] % 2 == 1).all()


def test_data_errors_give_the_sentinel():
    rng = np.random.default_rng(1)
    B, k, V = 6, 3, 10
    zt = rng.normal(0, 1, (B, k + 1, V)).astype(np.float32)
    zd = rng.normal(0, 1, (B, k, V)).astype(np.float32)
    x = rng.integers(0, V, (B, k)).astype(np.int32)
    u = np.full((B, k + 1), 0.5, np.float32)
    nd = np.full(B, k, np.int32)
    x[0, 1] = V          # token out of range
    nd[1] = k + 1        # count out of range
    u[2, k] = 1.0        # sampling uniform out of [0, 1)
    zt[3, 2, 4] = np.nan  # NaN in a needed row
    zd[4, 0, :] = -np.inf  # draft row with no finite logit
    nd[5] = 1
    zt[5, 3, 0] = np.nan  # NaN in a row past n_r + 1: not read, not an error
    out = oracle.spec_verify_sample(zt, zd, x, nd, u, 1.0)
    assert list(out["accept_len"][:5]) == [-1] * 5
    assert (out["tokens"][:5] == -1).all()
    assert np.isnan(out["p"][:5]).all() and np.isnan(out["resid"][:5]).all()
    assert out["accept_len"][5] in (0, 1)


def test_argument_validation():
    z = np.zeros((1, 2, 4), np.float32)
    d = np.zeros((1, 1, 4), np.float32)
    x = np.zeros((1, 1), np.int32)
    u = np.zeros((1, 2), np.float32)
    for T in (0.0, -1.0, np.inf, np.nan):
        with pytest.raises(ValueError):
            oracle.spec_verify_sample(z, d, x, None, u, T)


def _flag_edge(flagged, lo, hi, iters=80):
    """The point in [lo, hi] where flagged(u) changes (flagged(lo) != flagged(hi)), by
    bisection over float32 values."""
    f_lo = flagged(lo)
    assert flagged(hi) != f_lo
    for _ in range(iters):
        mid = np.float32((np.float64(lo) + np.float64(hi)) / 2)
        if mid in (lo, hi):
            break
        if flagged(mid) == f_lo:
            lo = mid
        else:
            hi = mid
    return (np.float64(lo) + np.float64(hi)) / 2


def test_tie_probability_is_the_measure_of_flagged_uniforms():
    """out_tie_prob is the chance, over the uniforms, that the oracle flags a near tie. Here
    it is compared with the measure of the uniforms the oracle actually flags, found by
    bisection on its own flag output: (1) a bonus draw whose first four tokens are tinier
    than the margin (each flagged whole, the first one only at its upper boundary) ahead of
    one large last token (flagged only at its lower boundary); (2) an accept test at
    rho ~ 0.3 (flagged within the margin on either side)."""
    # (1) n = 0: the bonus draw from p_0; every flagged target lies below ~5e-6
    m = np.array([3e-7, 4e-7, 2e-6, 1e-6, 1.0], np.float64)
    zt = np.log(m).astype(np.float32)[None, None, :].repeat(2, axis=1)
    zd = np.zeros((1, 1, 5), np.float32)
    x, nd = np.array([[0]], np.int32), np.array([0], np.int32)

    def draw_flag(uk):
        u = np.array([[0.5, uk]], np.float32)
        return oracle.spec_verify_sample(zt, zd, x, nd, u, 1.0)["flag_pos"][0] >= 0

    assert draw_flag(np.float32(0.0)) and not draw_flag(np.float32(0.5))
    edge = _flag_edge(draw_flag, np.float32(0.0), np.float32(1e-4))
    u = np.array([[0.5, 0.5]], np.float32)
    tp = oracle.spec_verify_sample(zt, zd, x, nd, u, 1.0)["tie_prob"][0]
    assert abs(tp - edge) < 1e-11, (tp, edge)
    # nothing else is flagged: the last token has no upper boundary
    for uk in (0.1, 0.9, np.nextafter(np.float32(1), np.float32(0))):
        assert not draw_flag(np.float32(uk))

    # (2) one accept test: p_0 uniform over 3 tokens, q_0(0) = 3/5, so rho = 5/9; a
    # rejection draws from the residual over tokens 1 and 2 (one boundary, at W/2), an
    # acceptance from the uniform p_1 (boundaries at 1/3 and 2/3)
    V = 3
    zt = np.zeros((1, 2, V), np.float32)
    zd = np.zeros((1, 1, V), np.float32)
    zd[0, 0, 0] = np.float32(np.log(3.0))
    x, nd = np.array([[0]], np.int32), np.array([1], np.int32)

    def run(u0, uk):
        return oracle.spec_verify_sample(zt, zd, x, nd, np.array([[u0, uk]], np.float32), 1.0)

    o = run(0.0, 0.25)
    rho = o["p"][0, 0] / o["q"][0, 0]
    assert abs(rho - 5.0 / 9.0) < 1e-6

    def acc_flag(u0):
        return run(u0, 0.25)["flag_pos"][0] == 0

    lo = _flag_edge(acc_flag, np.float32(rho - 1e-5), np.float32(rho))
    hi = _flag_edge(acc_flag, np.float32(rho), np.float32(rho + 1e-5))
    accept_part = hi - lo
    assert abs(accept_part - 2e-6) < 2 * np.spacing(np.float32(rho)), accept_part

    def draw_width(u0, b):
        """Measure of the flagged draw targets around the boundary b (in units of u_k)."""
        def f(uk):
            return run(u0, uk)["flag_pos"][0] >= 0
        return (_flag_edge(f, np.float32(b), np.float32(b + 1e-5))
                - _flag_edge(f, np.float32(b - 1e-5), np.float32(b)))

    # rejected (u0 above rho): one residual boundary
    u0 = np.float32(rho + 0.2)
    want = accept_part + draw_width(u0, 0.5)
    assert abs(run(u0, 0.25)["tie_prob"][0] - want) < 1e-12 + 4 * np.spacing(np.float32(0.5))
    # accepted (u0 below rho): two bonus boundaries
    u0 = np.float32(rho - 0.2)
    want = accept_part + draw_width(u0, 1.0 / 3.0) + draw_width(u0, 2.0 / 3.0)
    assert abs(run(u0, 0.25)["tie_prob"][0] - want) < 1e-12 + 8 * np.spacing(np.float32(0.7))

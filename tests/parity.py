"""Comparison rules between the CUDA path and the oracle (used by the GPU tests).

Tokens, accept lengths and gate decisions must be identical. The one exception is a
decision whose margin in the oracle's own fp64 arithmetic is below 1e-6 (an accept ratio
within 1e-6 of its uniform, a sampling target within 1e-6*W of a CDF boundary, a gate gap
within 1e-6 of tau): such a position, and everything after it in its request, is counted
and reported, not compared. Probabilities and residual masses must agree within 1e-5
absolute wherever both sides took the same path.
"""
from __future__ import annotations

import numpy as np

PROB_ATOL = 1e-5


def compare_sample(gpu: dict, orc: dict, requests) -> dict:
    """gpu: numpy arrays tokens, accept_len, p, q, resid and n (the per-request draft
    counts) over the full batch; orc: the oracle's output."""
    stats = dict(requests=0, flagged=0, flagged_differ=0, errors=0, max_p_err=0.0,
                 max_resid_err=0.0)
    for r in requests:
        stats["requests"] += 1
        oa, ga = int(orc["accept_len"][r]), int(gpu["accept_len"][r])
        if oa == -1:
            stats["errors"] += 1
            assert ga == -1, f"request {r}: oracle flags a data error, GPU a={ga}"
            assert (gpu["tokens"][r] == -1).all(), f"request {r}: error row not all -1"
            continue
        f = int(orc["flag_pos"][r])
        k = gpu["tokens"].shape[1] - 1
        if f < 0:
            assert ga == oa, f"request {r}: accept length GPU {ga} oracle {oa}"
            assert np.array_equal(gpu["tokens"][r], orc["tokens"][r]), (
                f"request {r}: tokens GPU {gpu['tokens'][r]} oracle {orc['tokens'][r]}")
        else:
            stats["flagged"] += 1
            assert np.array_equal(gpu["tokens"][r, :f], orc["tokens"][r, :f]), f"request {r}"
            assert ga >= f and oa >= f, f"request {r}: flagged at {f}, a GPU {ga} oracle {oa}"
            if f == oa and ga == oa:
                # a near tie in the draw: the GPU token must be one the tie window allows
                t = int(gpu["tokens"][r, oa])
                assert orc["t_lo"][r] <= t <= orc["t_hi"][r], (
                    f"request {r}: drawn {t} outside the tie window "
                    f"[{orc['t_lo'][r]}, {orc['t_hi'][r]}]")
            if ga != oa or not np.array_equal(gpu["tokens"][r], orc["tokens"][r]):
                stats["flagged_differ"] += 1
        n = int(gpu["n"][r])
        for key in ("p", "q"):
            if gpu.get(key) is not None:
                e = np.abs(gpu[key][r, :n].astype(np.float64) - orc[key][r, :n])
                if e.size:
                    stats["max_p_err"] = max(stats["max_p_err"], float(e.max()))
                    assert e.max() <= PROB_ATOL, f"request {r}: {key} error {e.max()}"
                assert (gpu[key][r, n:k] == 0).all()
        if gpu.get("resid") is not None and (f < 0 or ga == oa):
            e = abs(float(gpu["resid"][r]) - orc["resid"][r])
            stats["max_resid_err"] = max(stats["max_resid_err"], e)
            assert e <= PROB_ATOL, f"request {r}: residual mass error {e}"
    return stats


def flag_bound(orc: dict, requests) -> tuple[float, int]:
    """The expected number of flagged requests and a cap on the count, from the 1e-6 rule.

    The oracle's tie_prob[r] is the chance, over the uniforms, that request r is flagged
    given its path (accept tests within 1e-6 of rho, or a draw target within 1e-6*W of a
    boundary between tokens of positive weight; a token lighter than the margin is flagged
    wherever the target falls in it, so long-tailed rows raise it). Requests draw their
    uniforms independently, so the flagged count is a sum of independent Bernoulli(p_r)
    terms: mean E = sum p_r, variance sum p_r(1 - p_r). The cap is E + 5 standard deviations
    + 3 (the +3 covers tiny batches, where the normal tail bound is loose)."""
    p = np.array([orc["tie_prob"][r] for r in requests if orc["accept_len"][r] >= 0],
                 dtype=np.float64)
    mean = float(p.sum())
    sd = float(np.sqrt((p * (1.0 - p)).sum()))
    return mean, int(np.floor(mean + 5.0 * sd + 3.0))


def check_flags(name: str, stats: dict, orc: dict, requests) -> None:
    """Report a sampled-verify comparison on one line (pytest -s shows it) and check the
    flagged count against flag_bound."""
    mean, cap = flag_bound(orc, requests)
    print(f"PARITY {name}: requests={stats['requests']} errors={stats['errors']} "
          f"flagged={stats['flagged']} flagged_differ={stats['flagged_differ']} "
          f"expected_flagged={mean:.2f} cap={cap} max_p_err={stats['max_p_err']:.2e} "
          f"max_resid_err={stats['max_resid_err']:.2e}")
    assert stats["flagged"] <= cap, (name, stats, mean, cap)


def compare_greedy(gpu_tokens, gpu_accept, orc) -> None:
    assert np.array_equal(gpu_accept, orc["accept_len"]), "greedy accept lengths differ"
    assert np.array_equal(gpu_tokens, orc["tokens"]), "greedy tokens differ"


def compare_gate(token, gap, fire, orc) -> int:
    assert np.array_equal(token, orc["token"]), "gate tokens differ"
    og = orc["gap"].astype(np.float32)
    same = (gap == og) | (np.isnan(gap) & np.isnan(og))
    assert same.all(), "gate gaps differ"
    keep = orc["flag"] == 0
    assert np.array_equal(fire[keep], orc["fire"][keep]), "gate decisions differ"
    return int((~keep).sum())


def compare_confidence(nd, conf, nin, orc, floor: float, mode: int, requests,
                       rel: float = 1e-5, h_abs: float = 5e-7) -> dict:
    """Draft-confidence stop. nd [B] and conf [B, k] from the CUDA path, nin [B] the input
    draft counts. Top probabilities agree within ``rel``; for the inverse entropy, H = 1/c
    agrees within rel * H + h_abs nats (the CUDA path's H carries an absolute error of a few
    1e-7 nats from its fp32 exponentials, see the library header). The stop agrees exactly
    unless a position up to the oracle's stop is a near tie (the oracle's flag, or a
    confidence within this tolerance of the floor) at f; then the CUDA stop is at least f
    and is the first position whose own confidence is below the floor."""
    stats = dict(requests=0, flagged=0, errors=0, max_rel=0.0)

    def inv(c):
        return 0.0 if c == np.inf else 1.0 / c

    for r in requests:
        stats["requests"] += 1
        on = int(orc["num_draft"][r])
        if on == -1:
            stats["errors"] += 1
            assert nd[r] == -1, (r, nd[r])
            assert np.isnan(conf[r]).all(), r
            continue
        n = int(nin[r])
        assert (conf[r, n:] == 0).all(), r
        f = int(orc["flag"][r])
        for i in range(n):
            g, o = float(conf[r, i]), float(orc["conf"][r, i])
            if mode == 0:
                err = abs(g - o) / o
                assert err <= rel, (r, i, g, o)
                tie = abs(o - floor) <= rel * max(o, floor)
            else:
                hg, ho = inv(g), inv(o)
                err = abs(hg - ho) / ho if ho > 0 else 0.0
                assert abs(hg - ho) <= rel * ho + h_abs, (r, i, g, o)
                tie = abs(ho - inv(floor)) <= rel * ho + h_abs
            stats["max_rel"] = max(stats["max_rel"], err)
            if tie and i <= on and (f == -1 or i < f):
                f = i
        if f == -1:
            assert nd[r] == on, (r, nd[r], on)
        else:
            stats["flagged"] += 1
            below = [i for i in range(n) if conf[r, i] < floor]
            assert nd[r] >= f and nd[r] == (below[0] if below else n), (r, nd[r], f)
    return stats

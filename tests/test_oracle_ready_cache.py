"""Pins of the oracle's ready-distribution cache (pre-positioning page, Algorithms 1 and 2,
Figure 3, Eq. (8)).

- Each branch of the two algorithms on a designed scenario: record and fast serve, the
  cell-budget skip, an ineligible entry, the gate's two fall-through causes, the ad-hoc path.
- The invalidation invariant against an independent model: over random event sequences, a
  served token is always numpy's argmax of the latest ready logits recorded for that session,
  with no mutation since, and the request's entry equals the recorded one.
- The hit rate against Eq. (8)'s closed form h = rho / (1 + rho) for memoryless queries and
  updates (each update mutates the state and pre-positions again).
"""
import math

import numpy as np
import pytest

from oracle.ready_cache import (BAD_REQUEST, FALL_GATE, FALL_INELIGIBLE, FALL_INVALID, FAST,
                                RECORDED, SKIPPED, ReadyCache)


def _logits(rows, V=50, seed=0, peak=6.0, at=None):
    rng = np.random.default_rng(seed)
    z = rng.standard_normal((rows, V)).astype(np.float32)
    at = rng.integers(0, V, rows) if at is None else np.asarray(at)
    z[np.arange(rows), at] += peak
    return z, at


def test_record_then_fast_serve():
    c = ReadyCache(4, 8)
    z, at = _logits(1, at=[7])
    assert c.record([2], [100], [[5, 6, 9]], [3], [10], z) == [RECORDED]
    s = c.slots[2]
    assert s["valid"] and s["decoded"] and s["position"] == 103 and s["token"] == 7
    # the gap is the top-1 minus top-2 logit of the row
    top = np.sort(z[0].astype(np.float64))[::-1]
    assert s["gap"] == top[0] - top[1]
    tok, why = c.serve([2], [100], [[5, 6, 9]], [3], 2.0, [1, 7, 40])
    assert tok == [7] and why == [FAST]
    assert c.stats["fast"] == 1 and c.stats["consumed"] == 1


def test_budget_skip_leaves_no_ready_distribution():
    c = ReadyCache(2, 8)
    z, _ = _logits(1)
    assert c.record([0], [6], [[1, 2, 3, 4]], [4], [9], z) == [RECORDED]
    # the next update's entry no longer fits: the pre-position is skipped, the old one dropped
    assert c.record([0], [10], [[1, 2, 3, 4]], [4], [3], z) == [SKIPPED]  # L_entry > B
    assert not c.slots[0]["valid"] and not c.slots[0]["decoded"]
    for start in (6, 10):
        tok, why = c.serve([0], [start], [[1, 2, 3, 4]], [4], 0.0, [0])
        assert why == [FALL_INVALID] and tok == [-1]
    assert c.stats["wasted"] == 1 and c.stats["skipped"] == 1
    # L_entry == B fits
    assert c.record([0], [10], [[1, 2, 3, 4]], [4], [4], z) == [RECORDED]


def test_eligibility_is_an_exact_entry_match():
    c = ReadyCache(1, 8)
    z, at = _logits(1, at=[3])
    c.record([0], [20], [[4, 4, 8]], [3], [100], z)
    A = [3]
    assert c.serve([0], [20], [[4, 4, 8]], [3], 1.0, A)[1] == [FAST]
    assert c.serve([0], [20], [[4, 4, 9]], [3], 1.0, A)[1] == [FALL_INELIGIBLE]  # a token
    assert c.serve([0], [20], [[4, 4, 8, 1]], [4], 1.0, A)[1] == [FALL_INELIGIBLE]  # a length
    assert c.serve([0], [21], [[4, 4, 8]], [3], 1.0, A)[1] == [FALL_INELIGIBLE]  # a position
    # the streaming ad-hoc path serves the question-independent token whatever the entry
    assert c.serve([0], [21], [[7]], [1], 1.0, A, exact=False)[1] == [FAST]


def test_gate_falls_through_on_a_small_gap_or_outside_the_answer_set():
    c = ReadyCache(1, 4)
    z = np.zeros((1, 10), np.float32)
    z[0, 4], z[0, 6] = 3.0, 1.0  # gamma = 2
    c.record([0], [0], [[1]], [1], [5], z)
    assert c.serve([0], [0], [[1]], [1], 1.99, [4])[1] == [FAST]
    assert c.serve([0], [0], [[1]], [1], 2.0, [4])[1] == [FALL_GATE]  # gamma > tau is strict
    assert c.serve([0], [0], [[1]], [1], 1.0, [6])[1] == [FALL_GATE]  # argmax not in A
    assert c.stats["consumed"] == 1  # one pre-position, consumed once


def test_invalidation_returns_to_no_ready_distribution():
    c = ReadyCache(3, 4)
    z, at = _logits(2, seed=1, at=[1, 2])
    c.record([0, 1], [0, 0], [[9], [9]], [1, 1], [4, 4], z)
    c.serve([0], [0], [[9]], [1], 0.0, [1])       # consumes slot 0
    c.invalidate([0, 1])                          # slot 1 was never consumed: wasted
    assert c.stats["wasted"] == 1 and c.stats["consumed"] == 1
    assert c.serve([0, 1], [0, 0], [[9], [9]], [1, 1], 0.0, [1, 2])[1] == [FALL_INVALID] * 2
    assert c.slots[0]["epoch"] == 2 and c.slots[2]["epoch"] == 0
    # a record over a live, unconsumed pre-position replaces it and wastes it
    c.record([2], [0], [[9]], [1], [4], z[:1])
    c.record([2], [5], [[9]], [1], [4], z[1:])
    assert c.stats["wasted"] == 2 and c.slots[2]["position"] == 6
    assert c.serve([7], [0], [[9]], [1], 0.0, [1])[1] == [BAD_REQUEST]


def test_served_tokens_are_never_stale():
    rng = np.random.default_rng(5)
    S, V, E = 6, 40, 4
    c = ReadyCache(S, E)
    truth = {}  # sid -> (argmax, entry, start) of the latest record, or None after a mutation
    for step in range(600):
        kind = rng.integers(0, 3)
        sids = rng.choice(S, rng.integers(1, 4), replace=False)
        if kind == 0:
            M = len(sids)
            z, _ = _logits(M, V, seed=step, peak=float(rng.uniform(0, 8)))
            L = rng.integers(1, E + 1, M)
            ent = rng.integers(0, 5, (M, E))
            n_s = rng.integers(0, 50, M)
            B = rng.integers(0, E + 2, M)
            st = c.record(sids, n_s, ent, L, B, z)
            for m, sid in enumerate(sids):
                truth[int(sid)] = ((int(np.argmax(z[m])), list(ent[m, :L[m]]), int(n_s[m]))
                                   if st[m] == RECORDED else None)
        elif kind == 1:
            c.invalidate(sids)
            for sid in sids:
                truth[int(sid)] = None
        else:
            reqs = []
            for sid in sids:
                t = truth.get(int(sid))
                if t is not None and rng.random() < 0.7:
                    reqs.append((int(sid), t[2], t[1]))  # the recorded entry itself
                else:
                    reqs.append((int(sid), int(rng.integers(0, 50)), list(rng.integers(0, 5, 2))))
            toks, why = c.serve([r[0] for r in reqs], [r[1] for r in reqs],
                                [r[2] + [0] * (E - len(r[2])) for r in reqs],
                                [len(r[2]) for r in reqs], 1.0, list(range(V)))
            for (sid, start, ent), tok, w in zip(reqs, toks, why):
                t = truth.get(sid)
                if w == FAST:
                    assert t is not None and tok == t[0] and ent == t[1] and start == t[2]
                if t is None:
                    assert w == FALL_INVALID


@pytest.mark.parametrize("rho", [0.25, 1.0, 4.0])
def test_hit_rate_matches_eq8_for_memoryless_sessions(rho):
    # queries at rate rho, updates at rate 1: after each update the session is invalidated and
    # pre-positioned again; the next event is a query with probability rho / (1 + rho)
    rng = np.random.default_rng(int(rho * 100))
    c = ReadyCache(1, 2)
    z, at = _logits(1, at=[0])
    c.record([0], [0], [[1]], [1], [2], z)
    n_events = 40000
    for _ in range(n_events):
        if rng.random() < rho / (1 + rho):
            c.serve([0], [0], [[1]], [1], 0.0, [0])
        else:
            c.invalidate([0])
            c.record([0], [0], [[1]], [1], [2], z)
    h = c.hit_rate()
    want = rho / (1 + rho)
    n = c.stats["consumed"] + c.stats["wasted"]
    assert abs(h - want) < 5 * math.sqrt(want * (1 - want) / n), (h, want)
    # counting every query as a consumption instead would exceed the bound at rho = 4
    assert c.stats["consumed"] <= c.stats["pre_positions"]

"""Pins of the oracle's draft-confidence stop against closed forms and library routines.

The design note on variable-length drafting ("speculative-decoding-plan.md", after "The
acceptance math") has the draft keep proposing while its own confidence stays above a floor,
by top probability or an inverse-entropy gate. The oracle reads that as c = max_j q(j) or
c = 1/H (H in nats) of q = softmax(z/T), and n_r = the first position with c < floor. Each pin
below fixes the value by something other than the oracle's own formula: a uniform or
two-point distribution (closed forms), scipy's softmax and entropy, or a stop sequence built
so that every confidence sits far from the floor.
"""
import math

import numpy as np
import pytest

import oracle

TOP, ENT = oracle.CONF_TOP_PROB, oracle.CONF_INV_ENTROPY


def _run(z, T, mode, floor, num_draft=None):
    z = np.ascontiguousarray(z, dtype=np.float32)
    return oracle.draft_confidence(z, num_draft, T, mode, floor)


def test_uniform_rows_have_closed_forms():
    for V in (2, 7, 1000, 50257):
        z = np.full((1, 1, V), 0.375, np.float32)
        top = _run(z, 0.9, TOP, 0.0)["conf"][0, 0]
        ent = _run(z, 0.9, ENT, 0.0)["conf"][0, 0]
        assert top == pytest.approx(1.0 / V, rel=1e-13)
        assert ent == pytest.approx(1.0 / math.log(V), rel=1e-12)


@pytest.mark.parametrize("d,T", [(0.0, 1.0), (1.0, 1.0), (3.5, 0.7), (-2.0, 2.5), (12.0, 1.0)])
def test_two_point_rows_match_the_binary_entropy(d, T):
    # two finite logits (0 and d), the rest masked: q = (1 - s, s) with s = 1/(1 + e^(-d/T))
    V = 9
    z = np.full((1, 1, V), -np.inf, np.float32)
    z[0, 0, 2] = 0.0
    z[0, 0, 6] = d
    # with a = |d|/T: top = 1/(1 + e^-a), H = ln(1 + e^-a) + a e^-a / (1 + e^-a)
    a = abs(float(np.float32(d))) / T
    e = math.exp(-a)
    top = 1.0 / (1.0 + e)
    H = math.log1p(e) + a * e / (1.0 + e)
    assert _run(z, T, TOP, 0.0)["conf"][0, 0] == pytest.approx(top, rel=1e-13)
    assert _run(z, T, ENT, 0.0)["conf"][0, 0] == pytest.approx(1.0 / H, rel=1e-9)


def test_near_certain_row_has_a_huge_inverse_entropy():
    # q = (e^-40, 1 - e^-40): H ~ 1.7e-16 nats, below what double resolves around 1 (the
    # definition evaluated in double keeps H to ~1e-17 absolute), so only its size is pinned
    z = np.full((1, 1, 4), -np.inf, np.float32)
    z[0, 0, 0] = 0.0
    z[0, 0, 1] = 40.0
    assert 1e15 < _run(z, 1.0, ENT, 0.0)["conf"][0, 0] < 1e16


def test_one_hot_row_has_zero_entropy():
    z = np.full((1, 1, 5), -np.inf, np.float32)
    z[0, 0, 3] = 1.25
    assert _run(z, 1.0, TOP, 0.0)["conf"][0, 0] == 1.0
    assert _run(z, 1.0, ENT, 0.0)["conf"][0, 0] == math.inf


@pytest.mark.parametrize("T", [0.3, 1.0, 4.0])
def test_random_rows_match_scipy(T):
    special = pytest.importorskip("scipy.special")
    stats = pytest.importorskip("scipy.stats")
    rng = np.random.default_rng(7)
    z = (rng.standard_normal((3, 4, 300)) * 2.5).astype(np.float32)
    top = _run(z, T, TOP, 0.0)["conf"]
    ent = _run(z, T, ENT, 0.0)["conf"]
    for r in range(3):
        for i in range(4):
            q = special.softmax(z[r, i].astype(np.float64) / T)
            assert top[r, i] == pytest.approx(q.max(), rel=1e-12)
            assert ent[r, i] == pytest.approx(1.0 / stats.entropy(q), rel=1e-10)


def _designed(tops, V=64):
    """One request whose draft row i has top probability tops[i] (one raised logit)."""
    k = len(tops)
    z = np.zeros((1, k, V), np.float32)
    for i, t in enumerate(tops):
        # e^a / (e^a + V - 1) = t  =>  a = ln(t (V - 1) / (1 - t))
        z[0, i, 5] = math.log(t * (V - 1) / (1.0 - t))
    return z


def test_stop_is_the_first_position_below_the_floor():
    tops = [0.9, 0.8, 0.3, 0.95, 0.2]
    z = _designed(tops)
    for floor, want in [(0.5, 2), (0.1, 5), (0.85, 1), (0.99, 0), (0.25, 4)]:
        out = _run(z, 1.0, TOP, floor)
        assert out["num_draft"][0] == want, (floor, out)
        assert out["flag"][0] == -1
    np.testing.assert_allclose(_run(z, 1.0, TOP, 0.5)["conf"][0], tops, rtol=1e-6)


def test_stop_respects_the_input_draft_count():
    z = np.concatenate([_designed([0.9, 0.8, 0.3, 0.95])] * 3)
    nd = np.array([1, 4, 0], np.int32)
    out = _run(z, 1.0, TOP, 0.5, nd)
    assert list(out["num_draft"]) == [1, 2, 0]
    # rows at or past n_in are not read: reported as 0
    assert out["conf"][0, 1] == 0.0 and out["conf"][2, 0] == 0.0


def test_inverse_entropy_stop_uses_the_entropy_in_nats():
    # uniform rows over w finite logits have H = ln w: c = 1/ln w
    V = 32
    widths = [2, 3, 20, 4]
    z = np.full((1, len(widths), V), -np.inf, np.float32)
    for i, w in enumerate(widths):
        z[0, i, :w] = 0.0
    floor = 1.0 / math.log(10)  # stop once H > ln 10 nats
    assert _run(z, 1.0, ENT, floor)["num_draft"][0] == 2
    assert _run(z, 1.0, ENT, 1.0 / math.log(21))["num_draft"][0] == len(widths)


def test_data_errors_and_unread_rows():
    z = np.concatenate([_designed([0.9, 0.8, 0.7])] * 4)
    z[0, 1, 7] = np.nan        # a NaN in a row that is read
    z[1, 2, 3] = np.inf        # +inf in a row past the request's n_in: not read
    z[2, 0, :] = -np.inf       # a row with no finite logit
    nd = np.array([3, 2, 3, 5], np.int32)  # request 3: n_in beyond k
    out = _run(z, 1.0, TOP, 0.5, nd)
    assert list(out["num_draft"]) == [-1, 2, -1, -1]
    assert np.isnan(out["conf"][0]).all() and np.isnan(out["conf"][3]).all()
    assert out["flag"][1] == -1


def test_near_tie_is_flagged():
    tops = [0.9, 0.6, 0.3]
    z = _designed(tops)
    c = _run(z, 1.0, TOP, 0.0)["conf"][0]
    out = _run(z, 1.0, TOP, float(c[1]))  # the floor sits on position 1's confidence
    assert out["flag"][0] == 1
    assert out["num_draft"][0] == 2  # c_1 is not below the floor; c_2 is


def test_argument_checks():
    z = _designed([0.9, 0.8])
    with pytest.raises(ValueError):
        _run(z, 0.0, TOP, 0.5)   # T must be positive
    with pytest.raises(ValueError):
        _run(z, 1.0, 2, 0.5)     # unknown mode

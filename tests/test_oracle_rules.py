"""Pins of the oracle's softmax, greedy verify, logit-gap gate and n-gram proposer.

- Softmax: torch.softmax in double (a library routine) and sum to one; bf16 decoding
  against known bit patterns.
- Greedy verify ("The Inference Wall, Part 7", "How speculative decoding works"): the
  argmax is numpy.argmax (first occurrence on ties); and at temperature 0 a draft token is
  kept only if it is exactly the target's pick ("Does it make the answers worse?"), so the
  sampled verify on rows made near one-hot must give exactly the greedy result.
- Gate ("Speculative Pre-Positioning", section 2.4, Eq. (11)-(12)): torch.topk values,
  numpy.argmax, and a hand-made truth table with the page's tau = 2.0.
- N-gram proposer ("The Inference Wall, Part 7", the prompt-lookup worked example): the
  page's own example and a brute force written as a per-end-position match length.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


# ---------------------------------------------------------------- softmax and bf16 decoding
@pytest.mark.parametrize("V,T,std", [(7, 1.0, 1.0), (1000, 0.7, 3.0), (32000, 1.3, 5.0)])
def test_softmax_matches_torch(V, T, std):
    rng = np.random.default_rng(V)
    z = rng.normal(0, std, V).astype(np.float32)
    p = oracle.row_softmax(z, T)
    ref = torch.softmax(torch.from_numpy(z).double() / T, 0).numpy()
    assert np.allclose(p, ref, rtol=1e-13, atol=1e-300)
    assert abs(p.sum() - 1) < 1e-13


def test_softmax_bf16_and_special_values():
    bits = np.array([0x3F80, 0xC000, 0x0000, 0xFF80], np.uint16)  # 1, -2, 0, -inf
    p = oracle.row_softmax(bits, 1.0)
    e = np.exp([1.0, -2.0, 0.0])
    assert np.allclose(p, np.append(e / e.sum(), 0.0), rtol=1e-15)
    assert oracle.row_softmax(np.array([0.0, np.nan], np.float32), 1.0) is None
    assert oracle.row_softmax(np.array([0.0, np.inf], np.float32), 1.0) is None
    assert oracle.row_softmax(np.array([-np.inf, -np.inf], np.float32), 1.0) is None
    t = torch.randn(300).to(torch.bfloat16)
    p = oracle.row_softmax(t, 0.8)
    ref = torch.softmax(t.double() / 0.8, 0).numpy()
    assert np.allclose(p, ref, rtol=1e-13)


# ---------------------------------------------------------------- greedy verify
def test_greedy_argmax_and_walk():
    rng = np.random.default_rng(4)
    B, k, V = 400, 4, 50
    z = rng.integers(-3, 4, (B, k + 1, V)).astype(np.float32)  # many ties
    g = np.argmax(z, axis=2)  # first occurrence
    x = np.where(rng.random((B, k)) < 0.7, g[:, :k], rng.integers(0, V, (B, k))).astype(np.int32)
    nd = rng.integers(0, k + 1, B).astype(np.int32)
    out = oracle.spec_verify_greedy(z, x, nd)
    for b in range(B):
        n = nd[b]
        mism = [i for i in range(n) if x[b, i] != g[b, i]]
        a = mism[0] if mism else n
        assert out["accept_len"][b] == a
        assert list(out["tokens"][b, :a]) == list(x[b, :a])
        assert out["tokens"][b, a] == g[b, a]
        assert (out["tokens"][b, a + 1:] == -1).all()


def test_greedy_pages_cases():
    # "If all k guesses are right, one weight-stream bought k+1 tokens. If the first is
    # wrong, the pass bought one token." (How speculative decoding works)
    k, V = 5, 20
    z = np.zeros((2, k + 1, V), np.float32)
    targets = np.array([[3, 1, 4, 1, 5, 9], [2, 7, 1, 8, 2, 8]])
    for b in range(2):
        for i in range(k + 1):
            z[b, i, targets[b, i]] = 1.0
    x = np.array([targets[0, :k], [0, 7, 1, 8, 2]], np.int32)
    out = oracle.spec_verify_greedy(z, x, None)
    assert out["accept_len"][0] == k and list(out["tokens"][0]) == list(targets[0])
    assert out["accept_len"][1] == 0 and list(out["tokens"][1]) == [2, -1, -1, -1, -1, -1]


def test_sampled_verify_on_one_hot_rows_is_greedy():
    rng = np.random.default_rng(8)
    B, k, V, T = 300, 4, 64, 0.5
    g = rng.integers(0, V, (B, k + 1))
    zt = rng.normal(0, 1, (B, k + 1, V)).astype(np.float32)
    zt[np.arange(B)[:, None], np.arange(k + 1)[None, :], g] += 200.0 * T
    x = np.where(rng.random((B, k)) < 0.6, g[:, :k], rng.integers(0, V, (B, k))).astype(np.int32)
    zd = rng.normal(0, 1, (B, k, V)).astype(np.float32)
    zd[np.arange(B)[:, None], np.arange(k)[None, :], x] += 200.0 * T
    nd = rng.integers(0, k + 1, B).astype(np.int32)
    u = rng.uniform(1e-3, 1 - 1e-3, (B, k + 1)).astype(np.float32)
    s = oracle.spec_verify_sample(zt, zd, x, nd, u, T)
    gr = oracle.spec_verify_greedy(zt, x, nd)
    assert (s["accept_len"] == gr["accept_len"]).all()
    assert (s["tokens"] == gr["tokens"]).all()


def test_greedy_data_errors():
    z = np.zeros((3, 3, 5), np.float32)
    x = np.array([[0, 1], [5, 0], [0, 0]], np.int32)
    nd = np.array([3, 2, 1], np.int32)
    z[2, 1, :] = np.nan  # a needed row with no comparable entry
    out = oracle.spec_verify_greedy(z, x, nd)
    assert list(out["accept_len"]) == [-1, -1, -1]
    assert (out["tokens"] == -1).all()


# ---------------------------------------------------------------- gate
def test_gate_truth_table():
    with open(os.path.join(HERE, "golden", "gate_truth_table.json")) as f:
        g = json.load(f)
    z = np.array([r["logits"] for r in g["rows"]], np.float32)
    out = oracle.logit_gap_gate(z, g["tau"], np.array(g["answer_set"], np.int32))
    for i, r in enumerate(g["rows"]):
        assert out["token"][i] == r["token"], r["why"]
        assert out["gap"][i] == r["gap"], r["why"]
        assert out["fire"][i] == r["fire"], r["why"]


def test_gate_matches_topk():
    rng = np.random.default_rng(12)
    N, V = 200, 3000
    z = rng.normal(0, 3, (N, V)).astype(np.float32)
    A = np.sort(rng.choice(V, 300, replace=False)).astype(np.int32)
    tau = 4.0
    out = oracle.logit_gap_gate(z, tau, A)
    top = torch.topk(torch.from_numpy(z).double(), 2, dim=1).values.numpy()
    gap = top[:, 0] - top[:, 1]
    assert np.array_equal(out["gap"], gap)
    assert np.array_equal(out["token"], np.argmax(z, 1))
    want = (gap > tau) & np.isin(np.argmax(z, 1), A)
    assert np.array_equal(out["fire"].astype(bool), want)
    # bf16 rows with many exact ties: argmax is the first occurrence, gap from topk
    zb = torch.from_numpy(rng.integers(-4, 5, (N, 64)).astype(np.float32)).to(torch.bfloat16)
    ob = oracle.logit_gap_gate(zb, 0.5, A)
    tb = torch.topk(zb.double(), 2, dim=1).values.numpy()
    assert np.array_equal(ob["gap"], tb[:, 0] - tb[:, 1])
    assert np.array_equal(ob["token"], np.argmax(zb.float().numpy(), 1))


def test_gate_special_rows():
    z = np.array([[np.nan, np.nan, np.nan], [np.nan, 1.0, np.nan], [-np.inf, 2.0, -np.inf],
                  [-np.inf, -np.inf, -np.inf], [np.inf, 1.0, 0.0]], np.float32)
    out = oracle.logit_gap_gate(z, 1.0, np.array([0, 1, 2], np.int32))
    assert out["token"][0] == -1 and np.isnan(out["gap"][0]) and out["fire"][0] == 0
    assert out["token"][1] == 1 and out["gap"][1] == np.inf and out["fire"][1] == 1
    assert out["token"][2] == 1 and out["gap"][2] == np.inf and out["fire"][2] == 1
    assert out["token"][3] == 0 and np.isnan(out["gap"][3]) and out["fire"][3] == 0
    assert out["token"][4] == 0 and out["gap"][4] == np.inf and out["fire"][4] == 1
    empty = oracle.logit_gap_gate(np.zeros((2, 4), np.float32), -1.0, None)
    assert (empty["fire"] == 0).all()


# ---------------------------------------------------------------- n-gram proposer
def _ids(words, vocab):
    return [vocab.setdefault(w, len(vocab)) for w in words]


def test_ngram_worked_example():
    with open(os.path.join(HERE, "golden", "ngram_worked_example.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        vocab = {}
        words = case["text"].split()
        h = np.array([_ids(words, vocab)], np.int32)
        want = _ids(case["expected_proposal"].split(), vocab)
        out = oracle.ngram_propose(h, np.array([len(words)], np.int32), case["n_max"],
                                   case["n_min"], case["k"])
        assert out["num_draft"][0] == len(want), case["name"]
        assert list(out["draft"][0, :len(want)]) == want, case["name"]
        assert (out["draft"][0, len(want):] == -1).all()


def _brute_force(h, n_max, n_min, k):
    """Per end position e < L-1: the length of the common suffix of h[:e+1] and h,
    capped at n_max; take the longest (>= n_min), then the smallest e."""
    L = len(h)
    best_len, best_e = 0, -1
    for e in range(L - 1):
        m = 0
        while m < n_max and m <= e and h[e - m] == h[L - 1 - m]:
            m += 1
        if m > best_len:
            best_len, best_e = m, e
    if best_len < n_min:
        return []
    return list(h[best_e + 1: best_e + 1 + k])


@pytest.mark.parametrize("alphabet", [2, 3, 5, 50])
def test_ngram_brute_force(alphabet):
    rng = np.random.default_rng(alphabet)
    B, L_max = 300, 40
    h = rng.integers(0, alphabet, (B, L_max)).astype(np.int32)
    lens = rng.integers(0, L_max + 1, B).astype(np.int32)
    for n_max, n_min, k in [(4, 2, 5), (3, 3, 2), (6, 1, 7), (1, 1, 1)]:
        out = oracle.ngram_propose(h, lens, n_max, n_min, k)
        for b in range(B):
            want = _brute_force(list(h[b, :lens[b]]), n_max, n_min, k)
            assert out["num_draft"][b] == len(want)
            assert list(out["draft"][b, :len(want)]) == want
            assert (out["draft"][b, len(want):] == -1).all()


def test_ngram_edge_cases():
    h = np.array([[7, 7, 7, 7], [1, 2, 3, 4], [5, 5, 0, 0], [9, 9, 9, 9]], np.int32)
    lens = np.array([4, 4, 0, 5], np.int32)  # the last length is outside [0, L_max]
    out = oracle.ngram_propose(h, lens, 3, 2, 4)
    # [7 7 7 7]: the suffix 7 7 7 first occurs at 0..2, overlapping itself; copies h[3]
    assert out["num_draft"][0] == 1 and out["draft"][0, 0] == 7
    assert out["num_draft"][1] == 0 and out["num_draft"][2] == 0
    assert out["num_draft"][3] == -1 and (out["draft"][3] == -1).all()
    with pytest.raises(ValueError):
        oracle.ngram_propose(h, lens, 2, 3, 4)

"""CUDA path vs the oracle, through the C ABI (via the thin binding), on seeded inputs.

Small cases span several chunks, ragged tails, unaligned rows and ragged draft counts; the
five workloads run at full size in the launch configuration the benchmark times. The oracle
runs on every request of every case. Near ties (the 1e-6 rule) are counted, printed on a
PARITY line and bounded by the count the rule itself predicts (parity.flag_bound).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_17_gb300 as sv
import synth
from parity import check_flags, compare_gate, compare_greedy, compare_sample

pytestmark = pytest.mark.gpu
DEV = "cuda"


def run_sample(d, requests=None, threads=os.cpu_count() or 16):
    tok, acc, p, q, W = sv.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"],
                                              d["uniforms"], d["T"], d["num_draft"])
    torch.cuda.synchronize()
    B, k = d["B"], d["k"]
    nd = d["num_draft"]
    gpu = dict(tokens=tok.cpu().numpy(), accept_len=acc.cpu().numpy(), p=p.cpu().numpy(),
               q=q.cpu().numpy(), resid=W.cpu().numpy(),
               n=np.full(B, k) if nd is None else nd.cpu().numpy())
    orc = oracle.spec_verify_sample(d["target"].cpu(), d["draft"].cpu(), d["draft_tokens"].cpu(),
                                    None if nd is None else nd.cpu(), d["uniforms"].cpu(), d["T"],
                                    requests=requests, threads=threads)
    reqs = range(B) if requests is None else requests
    return compare_sample(gpu, orc, reqs), gpu, orc


SMALL = [
    # B, k, V, dtype, T, ragged, target_std, draft_noise, draft_scale
    (1, 4, 1000, "f32", 1.0, False, 2.0, 0.5, 1.0),
    (37, 3, 40000, "bf16", 0.8, True, 2.0, 1.0, 1.0),      # 3 chunks, partial last one
    (20, 2, 8191, "f32", 1.2, True, 3.0, 1.0, 0.8),        # rows not 16-byte aligned
    (16, 5, 16385, "bf16", 0.6, False, 2.5, 1.5, 0.6),     # one logit into a second chunk
    (12, 1, 2, "f32", 1.0, False, 1.0, 1.0, 1.0),          # V = 2
    (9, 16, 3001, "bf16", 1.0, True, 1.5, 0.8, 1.0),       # k = 16 (maximum)
    (64, 4, 24577, "f32", 0.9, True, 4.0, 2.0, 0.5),       # 4 chunks (fp32), ragged tail
    (7, 8, 50001, "bf16", 1e-2, False, 2.0, 1.0, 1.0),     # very low temperature
    (5, 3, 777, "bf16", 50.0, True, 2.0, 1.0, 1.0),        # very high temperature
    (6, 3, 151936, "bf16", 0.8, True, 2.0, 1.0, 1.0),      # 10 chunks: two segments per row
    (4, 2, 200003, "bf16", 1.0, False, 2.0, 0.7, 1.0),     # two segments, rows not aligned
    (3, 2, 600000, "bf16", 1.0, True, 2.0, 1.0, 1.0),      # 37 chunks: the draw's masses in
    (2, 3, 300001, "f32", 0.7, False, 2.0, 0.8, 1.0),      # the workspace (aligned / not)
    (3, 2, 262144, "f32", 1.0, True, 2.0, 1.0, 1.0),       # 32 chunks: the most whose masses
    (3, 2, 262145, "f32", 1.0, True, 2.0, 1.0, 1.0),       # stay in shared memory; 33
]


@pytest.mark.parametrize("case", SMALL, ids=[f"B{c[0]}k{c[1]}V{c[2]}{c[3]}" for c in SMALL])
def test_sample_small(case):
    B, k, V, dt, T, ragged, ts, dn, ds = case
    d = synth.sample_inputs(B, k, V, dt, T, device=DEV, seed=V + B, ragged=ragged,
                            target_std=ts, draft_noise=dn, draft_scale=ds)
    stats, _, orc = run_sample(d)
    check_flags(f"B={B} k={k} V={V} {dt} T={T}", stats, orc, range(B))


@pytest.mark.parametrize("B,k,V,dt", [(32, 6, 20000, "bf16"), (6, 3, 151936, "bf16"),
                                      (3, 2, 600000, "bf16"), (32, 6, 20000, "f32"),
                                      (6, 3, 151936, "f32"), (3, 2, 300001, "f32")])
def test_sample_draft_equals_target_accepts_all(B, k, V, dt):
    # every draft accepted: the bonus draw from row k (one to five segments per row; for fp32
    # from the sub-range masses pass 1 kept, rows aligned and not)
    d = synth.sample_inputs(B, k, V, dt, 0.9, device=DEV, seed=3)
    d["draft"] = d["target"][:, :k].contiguous()
    g = torch.Generator(device=DEV).manual_seed(4)
    zq = d["draft"].float() / 0.9
    d["draft_tokens"] = torch.argmax(zq - torch.log(-torch.log(
        torch.rand(zq.shape, generator=g, device=DEV).clamp_(1e-20, 1 - 1e-7))), -1).to(torch.int32)
    stats, gpu, _ = run_sample(d)
    assert (gpu["accept_len"] == k).all()
    assert (gpu["resid"] == 0).all()


def test_sample_masked_draft_token_accepts():
    # a drafted token the draft itself masks (q(x) = 0): the ratio p/q is +inf and the
    # position accepts whatever u is; one the target masks (p(x) = 0) rejects
    B, k, V = 6, 3, 3000
    d = synth.sample_inputs(B, k, V, "f32", 1.0, device=DEV, seed=41)
    x = d["draft_tokens"]
    for r in range(3):
        d["draft"][r, 0, x[r, 0]] = float("-inf")
    for r in range(3, 6):
        d["target"][r, 1, x[r, 1]] = float("-inf")
    d["uniforms"][:, :k] = 0.999
    stats, gpu, orc = run_sample(d)
    assert (gpu["accept_len"][:3] >= 1).all()
    assert (gpu["accept_len"][3:] <= 1).all()
    assert (gpu["q"][:3, 0] == 0).all() and (gpu["p"][3:, 1] == 0).all()


def test_sample_data_errors_and_masks():
    B, k, V = 8, 3, 5000
    d = synth.sample_inputs(B, k, V, "f32", 1.0, device=DEV, seed=11)
    nd = torch.full((B,), k, dtype=torch.int32, device=DEV)
    d["draft_tokens"][0, 1] = V          # token out of range
    nd[1] = k + 1                        # count out of range
    d["uniforms"][2, k] = 1.0            # sampling uniform out of [0, 1)
    d["target"][3, 2, 17] = float("nan")  # NaN in a needed row
    d["draft"][4, 0, :] = float("-inf")  # a draft row with no finite logit
    d["target"][5, :, ::2] = float("-inf")  # masked tokens: legal
    d["draft_tokens"][5] = 1
    nd[6] = 0                             # nothing drafted: a bonus draw only
    d["uniforms"][7, 0] = float("nan")   # NaN accept uniform
    d["num_draft"] = nd
    stats, gpu, orc = run_sample(d)
    assert list(gpu["accept_len"][:5]) == [-1] * 5 and gpu["accept_len"][7] == -1
    assert gpu["accept_len"][6] == 0 and gpu["tokens"][6, 0] >= 0
    assert gpu["tokens"][5, gpu["accept_len"][5]] % 2 == 1


def test_sample_empty_batch_and_repeat_calls():
    d = synth.sample_inputs(0, 3, 100, "f32", 1.0, device=DEV, seed=1)
    out = sv.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], 1.0)
    torch.cuda.synchronize()
    assert out[0].shape == (0, 4)
    # the workspace counters return to zero: two calls in a row agree, on another stream too
    d = synth.sample_inputs(40, 4, 30000, "bf16", 0.7, device=DEV, seed=2, ragged=True)
    a = sv.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], 0.7,
                              d["num_draft"])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        b = sv.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], 0.7,
                                  d["num_draft"], stream=s)
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_sample_concurrent_streams_keep_their_own_workspaces():
    # two batches verified at the same time on two streams, each with the binding's cached
    # workspace: the cache gives each stream its own, so both equal their one-at-a-time runs
    ds = [synth.sample_inputs(48, 4, 30000, "bf16", 0.8, device=DEV, seed=s, ragged=True)
          for s in (31, 32)]
    ref = []
    for d in ds:
        ref.append(sv.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"],
                                         d["uniforms"], d["T"], d["num_draft"]))
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    for st in streams:
        st.wait_stream(torch.cuda.current_stream())
    got = [None, None]
    for rep in range(4):
        for i, (d, st) in enumerate(zip(ds, streams)):
            with torch.cuda.stream(st):
                got[i] = sv.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"],
                                               d["uniforms"], d["T"], d["num_draft"],
                                               stream=st)
    torch.cuda.synchronize()
    for a, b in zip(ref, got):
        for x, y in zip(a, b):
            assert torch.equal(x, y)


@pytest.mark.parametrize("off", [0, 1])
def test_sample_deferred_draws(off):
    # rows of 15 fp32 chunks: the batch's last requests draw in the second launch, split over
    # their chunks; among them bonus draws (q = p), a bad token and a NaN row. off = 1 puts
    # the rows off the 16-byte grid (plain loads instead of the TMA ring)
    B, k, V = 160, 3, 120000
    assert sv.spec_verify_sample_launches(B, k, V, sv.SV_F32) == 3  # clear, verify, draws
    d = synth.sample_inputs(B, k, V, "f32", 0.9, device=DEV, seed=21, ragged=True,
                            target_std=2.5, draft_noise=0.8)
    d["draft"][140:145] = d["target"][140:145, :k]  # every draft accepted: bonus draws
    d["draft_tokens"][150, 0] = V                    # a token out of range
    d["num_draft"][150] = k
    d["target"][155, 0, 7] = float("nan")            # NaN in a needed row
    if off:
        for key in ("target", "draft"):
            flat = torch.empty(d[key].numel() + 1, dtype=d[key].dtype, device=DEV)
            view = flat[1:].view(d[key].shape)
            view.copy_(d[key])
            d[key] = view
    stats, gpu, orc = run_sample(d)
    check_flags(f"deferred draws off={off}", stats, orc, range(B))
    assert gpu["accept_len"][150] == -1 and gpu["accept_len"][155] == -1
    nd = d["num_draft"].cpu().numpy()
    assert (gpu["accept_len"][140:145] == nd[140:145]).all()


def test_sample_and_greedy_in_a_cuda_graph():
    # serving loops replay captured graphs: one sampled-verify call (the clear of its counters,
    # the verify, and the draws of the last requests, chained with programmatic dependencies)
    # and one greedy call, captured together and replayed twice, give what eager calls give
    B, k, V = 32, 4, 131072  # 8 chunks of bf16: the draws run in their own launch
    assert sv.spec_verify_sample_launches(B, k, V, sv.SV_BF16) == 3
    d = synth.sample_inputs(B, k, V, "bf16", 0.8, device=DEV, seed=17, ragged=True)
    sws = torch.zeros(sv.spec_verify_sample_workspace(B, k, V, sv.SV_BF16), dtype=torch.uint8,
                      device=DEV)
    gws = torch.zeros(sv.spec_verify_greedy_workspace(B, k, V, sv.SV_BF16), dtype=torch.uint8,
                      device=DEV)

    def outs():
        return dict(out_tokens=torch.full((B, k + 1), -7, dtype=torch.int32, device=DEV),
                    out_accept_len=torch.full((B,), -7, dtype=torch.int32, device=DEV),
                    out_p_draft=torch.zeros((B, k), device=DEV),
                    out_q_draft=torch.zeros((B, k), device=DEV),
                    out_resid_mass=torch.zeros((B,), device=DEV))

    def calls(o, go, stream=None):
        sv.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], 0.8,
                              d["num_draft"], workspace=sws, stream=stream, **o)
        sv.spec_verify_greedy(d["target"], d["draft_tokens"], d["num_draft"],
                              out_tokens=go[0], out_accept_len=go[1], workspace=gws,
                              stream=stream)

    eager, geager = outs(), (torch.empty((B, k + 1), dtype=torch.int32, device=DEV),
                             torch.empty((B,), dtype=torch.int32, device=DEV))
    calls(eager, geager)
    torch.cuda.synchronize()
    captured, gcap = outs(), (torch.full((B, k + 1), -7, dtype=torch.int32, device=DEV),
                              torch.full((B,), -7, dtype=torch.int32, device=DEV))
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # a warm-up outside the capture, as graph users do
        calls(outs(), (torch.empty_like(gcap[0]), torch.empty_like(gcap[1])))
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        calls(captured, gcap)
    for _ in range(2):
        for t in list(captured.values()) + list(gcap):
            t.fill_(float("nan") if t.is_floating_point() else -9)
        graph.replay()
        torch.cuda.synchronize()
        for name in eager:
            a, b = captured[name], eager[name]
            if a.is_floating_point():
                a, b = a.nan_to_num(-1.0), b.nan_to_num(-1.0)
            assert torch.equal(a, b), name
        assert torch.equal(gcap[0], geager[0]) and torch.equal(gcap[1], geager[1])
    assert (eager["out_accept_len"] >= 0).all()


@pytest.mark.parametrize("w", [0, 1, 2])
def test_sample_workloads_full(w):
    d = synth.workload_inputs(w, device=DEV)
    stats, gpu, orc = run_sample(d)
    # near ties are a property of the data (long-tailed rows put many draws within 1e-6 of
    # a CDF boundary); they are counted against the rule's own expectation, reported, and
    # checked against the oracle's tie window
    check_flags(f"workload {w}", stats, orc, range(d["B"]))


def test_sample_workload3_full_every_request():
    d = synth.workload_inputs(3, device=DEV)
    stats, gpu, orc = run_sample(d)
    check_flags("workload 3", stats, orc, range(d["B"]))
    assert stats["requests"] == d["B"]
    # every request: a well-formed result (prefix of drafts, one drawn token, -1 padding)
    a = gpu["accept_len"]
    assert ((a >= 0) & (a <= d["k"])).all()
    x = d["draft_tokens"].cpu().numpy()
    for r in range(d["B"]):
        assert (gpu["tokens"][r, :a[r]] == x[r, :a[r]]).all()
        assert 0 <= gpu["tokens"][r, a[r]] < d["V"]
        assert (gpu["tokens"][r, a[r] + 1:] == -1).all()


# ------------------------------------------------------------------------------ greedy
@pytest.mark.parametrize("B,k,V,dt,ties", [(64, 5, 32000, "bf16", False), (30, 4, 8191, "f32", True),
                                          (10, 16, 40000, "bf16", True), (3, 1, 2, "f32", True),
                                          (8, 4, 151936, "bf16", False),   # two segments per row
                                          (5, 2, 300001, "f32", True)])    # five, not aligned
def test_greedy_small(B, k, V, dt, ties):
    g = torch.Generator(device=DEV).manual_seed(V)
    if ties:
        z = torch.randint(-3, 4, (B, k + 1, V), generator=g, device=DEV).float()
    else:
        z = torch.randn((B, k + 1, V), generator=g, device=DEV) * 3
    z = z.to(torch.float32 if dt == "f32" else torch.bfloat16)
    am = torch.argmax(z.float(), -1)  # any tie-break: the test only uses it to make matches
    x = torch.where(torch.rand((B, k), generator=g, device=DEV) < 0.7, am[:, :k],
                    torch.randint(0, V, (B, k), generator=g, device=DEV)).to(torch.int32)
    nd = torch.randint(0, k + 1, (B,), generator=g, device=DEV, dtype=torch.int32)
    tok, acc = sv.spec_verify_greedy(z, x, nd)
    torch.cuda.synchronize()
    orc = oracle.spec_verify_greedy(z.cpu(), x.cpu(), nd.cpu())
    compare_greedy(tok.cpu().numpy(), acc.cpu().numpy(), orc)


def test_greedy_special_rows():
    B, k, V = 6, 3, 3000
    z = torch.randn((B, k + 1, V), device=DEV)
    x = torch.zeros((B, k), dtype=torch.int32, device=DEV)
    nd = torch.full((B,), k, dtype=torch.int32, device=DEV)
    z[0, 1, :] = float("nan")        # a needed row with nothing comparable: error
    z[1, :, :] = float("-inf")       # all -inf: argmax is token 0, matches x = 0
    z[2, 0, 5:] = float("nan")       # NaN entries are skipped
    nd[3] = -1                       # bad count
    x[4, 2] = V                      # bad token
    z[5, 3, :] = float("nan")        # row past n_r + 1 is not read
    nd[5] = 2
    tok, acc = sv.spec_verify_greedy(z, x, nd)
    torch.cuda.synchronize()
    orc = oracle.spec_verify_greedy(z.cpu(), x.cpu(), nd.cpu())
    compare_greedy(tok.cpu().numpy(), acc.cpu().numpy(), orc)
    assert acc[0].item() == -1 and acc[1].item() == k


def test_greedy_workload1_full():
    d = synth.workload_inputs(1, device=DEV)
    tok, acc = sv.spec_verify_greedy(d["target"], d["draft_tokens"], d["num_draft"])
    torch.cuda.synchronize()
    orc = oracle.spec_verify_greedy(d["target"].cpu(), d["draft_tokens"].cpu(), None)
    compare_greedy(tok.cpu().numpy(), acc.cpu().numpy(), orc)


def test_sampled_on_one_hot_rows_equals_greedy():
    B, k, V, T = 50, 5, 32000, 0.5
    d = synth.sample_inputs(B, k, V, "bf16", T, device=DEV, seed=9, ragged=True)
    g = torch.randint(0, V, (B, k + 1), device=DEV)
    t = d["target"].float()
    t.scatter_add_(2, g[:, :, None], torch.full((B, k + 1, 1), 200.0 * T, device=DEV))
    x = torch.where(torch.rand((B, k), device=DEV) < 0.6, g[:, :k],
                    torch.randint(0, V, (B, k), device=DEV))
    q = d["draft"].float()
    q.scatter_add_(2, x[:, :, None], torch.full((B, k, 1), 200.0 * T, device=DEV))
    d["target"], d["draft"] = t.to(torch.bfloat16), q.to(torch.bfloat16)
    d["draft_tokens"] = x.to(torch.int32)
    d["uniforms"] = d["uniforms"].clamp(1e-3, 1 - 1e-3)
    s_tok, s_acc, *_ = sv.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"],
                                             d["uniforms"], T, d["num_draft"])
    g_tok, g_acc = sv.spec_verify_greedy(d["target"], d["draft_tokens"], d["num_draft"])
    torch.cuda.synchronize()
    assert torch.equal(s_acc, g_acc) and torch.equal(s_tok, g_tok)


# ------------------------------------------------------------------------------ gate
@pytest.mark.parametrize("N,V,dt", [(40, 151936, "f32"), (33, 50001, "bf16"), (17, 8191, "f32"),
                                    (5, 2, "bf16"), (9, 262145, "bf16")])
def test_gate_small(N, V, dt):
    g = torch.Generator(device=DEV).manual_seed(N)
    z = torch.randn((N, V), generator=g, device=DEV) * 3
    idx = torch.randint(0, V, (N,), generator=g, device=DEV)
    z[torch.arange(N, device=DEV), idx] += torch.rand(N, generator=g, device=DEV) * 10
    z = z.to(torch.float32 if dt == "f32" else torch.bfloat16)
    A = torch.unique(torch.cat([idx[: N // 2], torch.randint(0, V, (20,), device=DEV)])).to(torch.int32)
    tk, gap, fire = sv.logit_gap_gate(z, 4.0, A)
    torch.cuda.synchronize()
    orc = oracle.logit_gap_gate(z.cpu(), 4.0, A.cpu())
    compare_gate(tk.cpu().numpy(), gap.cpu().numpy(), fire.cpu().numpy(), orc)


def test_gate_ties_and_special_rows():
    V = 40000
    z = torch.zeros((6, V), device=DEV)
    z[0, 100] = 5.0
    z[0, 30000] = 5.0                   # tied maximum across chunks: lowest index, gap 0
    z[1, :] = float("nan")              # nothing comparable
    z[2, :] = float("-inf")
    z[2, 39999] = 1.0                   # one finite logit: gap +inf
    z[3, 7] = float("inf")
    z[4, 16383] = 3.0
    z[4, 16384] = 3.0                   # tie across the bf16 chunk edge
    z[5, :] = torch.arange(V, device=DEV, dtype=torch.float32) * 1e-3
    for dt in (torch.float32, torch.bfloat16):
        zz = z.to(dt)
        A = torch.tensor([7, 100, 16383, 39999], dtype=torch.int32, device=DEV)
        tk, gap, fire = sv.logit_gap_gate(zz, 0.5, A)
        torch.cuda.synchronize()
        orc = oracle.logit_gap_gate(zz.cpu(), 0.5, A.cpu())
        compare_gate(tk.cpu().numpy(), gap.cpu().numpy(), fire.cpu().numpy(), orc)
    tk, gap, fire = sv.logit_gap_gate(z, -1.0, None)  # empty answer set: nothing fires
    torch.cuda.synchronize()
    assert fire.sum().item() == 0


def test_gate_workload2_full():
    d = synth.workload_inputs(2, device=DEV)
    rows = d["target"].reshape(-1, d["V"])
    tk, gap, fire = sv.logit_gap_gate(rows, d["tau"], d["answer_set"])
    torch.cuda.synchronize()
    orc = oracle.logit_gap_gate(rows.cpu(), d["tau"], d["answer_set"].cpu(), threads=16)
    flagged = compare_gate(tk.cpu().numpy(), gap.cpu().numpy(), fire.cpu().numpy(), orc)
    print(f"gate: {fire.sum().item()} of {rows.shape[0]} rows fire, {flagged} near ties")


# ------------------------------------------------------------------------------ n-gram
def test_ngram_worked_example_on_gpu():
    words = "Repeat this sentence : The quick brown fox jumps over the lazy dog . The quick brown".split()
    vocab = {}
    ids = [vocab.setdefault(w, len(vocab)) for w in words]
    h = torch.tensor([ids, ids[-3:] + [-1] * (len(ids) - 3)], dtype=torch.int32, device=DEV)
    hl = torch.tensor([len(ids), 3], dtype=torch.int32, device=DEV)
    d, n = sv.ngram_propose(h, hl, 4, 2, 5)
    torch.cuda.synchronize()
    want = [vocab[w] for w in "fox jumps over the lazy".split()]
    assert n.tolist() == [5, 0]
    assert d[0].tolist() == want and d[1].tolist() == [-1] * 5


@pytest.mark.parametrize("alphabet,nmax,nmin,k", [(2, 4, 2, 5), (3, 3, 3, 2), (7, 6, 1, 7),
                                                  (50, 1, 1, 1), (1000, 4, 2, 64)])
def test_ngram_random(alphabet, nmax, nmin, k):
    rng = np.random.default_rng(alphabet)
    B, L_max = 300, 700
    h = rng.integers(0, alphabet, (B, L_max)).astype(np.int32)
    lens = rng.integers(0, L_max + 1, B).astype(np.int32)
    lens[:3] = [0, 1, L_max + 1]  # empty, one token, out of range
    d, n = sv.ngram_propose(torch.from_numpy(h).to(DEV), torch.from_numpy(lens).to(DEV),
                            nmax, nmin, k)
    torch.cuda.synchronize()
    orc = oracle.ngram_propose(h, lens, nmax, nmin, k)
    assert np.array_equal(n.cpu().numpy(), orc["num_draft"])
    assert np.array_equal(d.cpu().numpy(), orc["draft"])


@pytest.mark.parametrize("nmax,nmin", [(4, 2), (6, 1), (64, 3)])
def test_ngram_long_histories_across_tiles(nmax, nmin):
    # histories past one 8192-position shared-memory tile, with the suffix phrase planted so
    # that its earliest earlier occurrence ends at, or just before, a tile boundary (its
    # first tokens then come from the previous tile's halo)
    rng = np.random.default_rng(100 * nmax + nmin)
    B, L_max, tile = 12, 20000, 8192
    h = rng.integers(0, 5000, (B, L_max)).astype(np.int32)
    lens = np.array([8192, 8193, 8194, 16385, 20000, 19999, 9000, 12000, 20000, 16384, 8191,
                     17000], np.int32)
    planted = []
    for b in range(B):
        L = int(lens[b])
        n = min(nmax, L // 4)
        e = (nmin - 1) + tile * (1 + b % 2) - (b % 3)  # a tile's first end position, or before
        if e <= L - 2 - n and e - n + 1 >= 0:
            h[b, e - n + 1:e + 1] = h[b, L - n:L]
            planted.append(b)
    d, cnt = sv.ngram_propose(torch.from_numpy(h).to(DEV), torch.from_numpy(lens).to(DEV),
                              nmax, nmin, 5)
    torch.cuda.synchronize()
    orc = oracle.ngram_propose(h, lens, nmax, nmin, 5)
    assert len(planted) >= 5 and (orc["num_draft"][planted] > 0).all()  # found by the oracle
    assert np.array_equal(cnt.cpu().numpy(), orc["num_draft"])
    assert np.array_equal(d.cpu().numpy(), orc["draft"])


def test_ngram_greedy_workload4_full():
    w = synth.workload_inputs(4, device=DEV)
    d, n = sv.ngram_propose(w["history"], w["hist_len"], w["n_max"], w["n_min"], w["k"])
    torch.cuda.synchronize()
    orc = oracle.ngram_propose(w["history"].cpu(), w["hist_len"].cpu(), w["n_max"], w["n_min"],
                               w["k"])
    assert np.array_equal(n.cpu().numpy(), orc["num_draft"])
    assert np.array_equal(d.cpu().numpy(), orc["draft"])
    tgt = synth.greedy_targets(torch.from_numpy(orc["draft"]).to(DEV),
                               torch.from_numpy(orc["num_draft"]).to(DEV), w["V"], k=w["k"],
                               seed=w["seed"])
    tok, acc = sv.spec_verify_greedy(tgt, d, n)
    torch.cuda.synchronize()
    og = oracle.spec_verify_greedy(tgt.cpu(), orc["draft"], orc["num_draft"])
    compare_greedy(tok.cpu().numpy(), acc.cpu().numpy(), og)
    print(f"workload 4: {int((orc['num_draft'] > 0).sum())} of {w['B']} requests proposed, "
          f"mean accepted {acc.float().mean().item():.2f}")

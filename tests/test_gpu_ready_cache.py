"""CUDA ready-distribution cache vs the oracle's state machine, through the C ABI.

The same seeded sequence of record, serve and invalidate batches drives both the device
table and the oracle's ReadyCache; every call's outputs (record statuses, served tokens and
reasons) must agree exactly, and at checkpoints so must every slot's state (flags, decision
point, argmax, gamma in double, entry, epoch) and the event counters. Rows of one and two
segments, fp32 and bf16, aligned and unaligned rows, the stored full distributions, the
cell-budget skip, bad arguments and repeated ids are covered.
"""
import numpy as np
import pytest
import torch

import speculative_decoding_verification_17_gb300 as sv
from oracle.ready_cache import ReadyCache

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _t(a, dtype):
    return torch.as_tensor(np.asarray(a), dtype=dtype).to(DEV)


def compare_state(table, ref):
    st = table.state()
    for sid, s in enumerate(ref.slots):
        f = int(st["flags"][sid])
        assert bool(f & sv.SV_CACHE_VALID) == s["valid"], sid
        assert bool(f & sv.SV_CACHE_DECODED) == s["decoded"], sid
        assert bool(f & sv.SV_CACHE_CONSUMED) == (s["consumed"] and s["valid"]), sid
        assert int(st["epoch"][sid]) == s["epoch"], sid
        if s["valid"]:
            assert int(st["position"][sid]) == s["position"], sid
            assert int(st["token"][sid]) == s["token"], sid
            g, o = float(st["gap"][sid]), s["gap"]
            assert (g == o) or (np.isnan(g) and np.isnan(o)), (sid, g, o)
            assert int(st["entry_len"][sid]) == len(s["entry"]), sid
            ent = table.entry_store[sid, : len(s["entry"])].cpu().tolist()
            assert ent == s["entry"], sid
    assert table.counters() == ref.stats, (table.counters(), ref.stats)


def run_sequence(S, V, dt, steps, seed, E=6, keep_dist=False, bad_every=0):
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    rng = np.random.default_rng(seed)
    table = sv.ReadyCacheTable(S, E, DEV, V=V, dist_dtype=tdt, keep_dist=keep_dist)
    ref = ReadyCache(S, E)
    recorded = {}  # sid -> (start, entry) of the latest successful record
    last_rows = {}
    A = np.sort(rng.choice(V, max(2, V // 3), replace=False)).astype(np.int32)
    for step in range(steps):
        kind = rng.choice(3, p=[0.35, 0.2, 0.45])
        if kind == 0:
            M = int(rng.integers(1, min(S, 12) + 1))
            sids = rng.choice(S, M, replace=False).astype(np.int32)
            z = torch.randn((M, V), generator=torch.Generator().manual_seed(seed * 1000 + step))
            at = torch.randint(0, V, (M,))
            z[torch.arange(M), at] += torch.rand(M) * 8
            if step % 7 == 3:
                z[0, : V // 2] = float("nan")             # NaN entries are skipped
            if step % 11 == 5 and M > 1:
                z[1, :] = float("nan")                    # no comparable logit
            z = z.to(tdt)
            L = rng.integers(0, E + 1, M).astype(np.int32)
            ent = rng.integers(0, 4, (M, E)).astype(np.int32)
            n_s = rng.integers(0, 100, M).astype(np.int64)
            B = rng.integers(0, E + 2, M).astype(np.int64)
            if bad_every and step % bad_every == 0:
                sids[0] = S + 3                           # out of range: touches nothing
            got = table.record(_t(sids, torch.int32), _t(n_s, torch.int64),
                               _t(ent, torch.int32), _t(L, torch.int32), _t(B, torch.int64),
                               z.to(DEV)).cpu().tolist()
            want = ref.record(sids, n_s, ent, L, B, z)
            assert got == want, (step, got, want)
            for m, sid in enumerate(sids):
                if want[m] == 0:
                    recorded[int(sid)] = (int(n_s[m]), list(ent[m, : L[m]]))
                    last_rows[int(sid)] = z[m]
        elif kind == 1:
            n = int(rng.integers(1, 5))
            sids = rng.choice(S, n).astype(np.int32)      # repeats allowed
            table.invalidate(_t(sids, torch.int32))
            ref.invalidate(sids)
        else:
            R = int(rng.integers(1, 24))
            sids = rng.choice(S, R).astype(np.int32)      # repeats allowed
            start = np.zeros(R, np.int64)
            toks = np.zeros((R, E), np.int32)
            lens = np.zeros(R, np.int32)
            for r, sid in enumerate(sids):
                rec = recorded.get(int(sid))
                if rec is not None and rng.random() < 0.7:
                    start[r], lens[r] = rec[0], len(rec[1])
                    toks[r, : lens[r]] = rec[1]
                    if rng.random() < 0.15 and lens[r] > 0:
                        toks[r, int(rng.integers(0, lens[r]))] += 1  # one token differs
                else:
                    start[r] = rng.integers(0, 100)
                    lens[r] = rng.integers(0, E + 1)
                    toks[r, : lens[r]] = rng.integers(0, 4, lens[r])
            tau = float(rng.choice([0.0, 1.5, 3.0]))
            exact = bool(rng.random() < 0.8)
            tok, why = table.serve(_t(sids, torch.int32), _t(start, torch.int64),
                                   _t(toks, torch.int32), _t(lens, torch.int32), tau,
                                   _t(A, torch.int32), exact=exact)
            wt, ww = ref.serve(sids, start, toks, lens, tau, A, exact=exact)
            assert tok.cpu().tolist() == wt and why.cpu().tolist() == ww, step
        if step % 25 == 24:
            torch.cuda.synchronize()
            compare_state(table, ref)
    torch.cuda.synchronize()
    compare_state(table, ref)
    if keep_dist:
        for sid, row in last_rows.items():
            got = table.dist[sid].cpu()
            assert torch.equal(got.view(torch.int16 if dt == "bf16" else torch.int32),
                               row.view(torch.int16 if dt == "bf16" else torch.int32)), sid
    return table, ref


@pytest.mark.parametrize("S,V,dt,keep", [(16, 1000, "f32", False), (40, 32000, "bf16", True),
                                         (12, 8191, "f32", True), (8, 151936, "bf16", True),
                                         (24, 3001, "bf16", False)])
def test_cache_matches_the_oracle(S, V, dt, keep):
    table, ref = run_sequence(S, V, dt, 150, seed=S + V, keep_dist=keep, bad_every=13)
    c = table.counters()
    assert c["pre_positions"] > 0 and c["fast"] > 0 and c["skipped"] > 0
    assert c["fall_invalid"] > 0 and c["fall_ineligible"] > 0 and c["bad"] > 0


def test_hit_rate_of_a_memoryless_session_stream():
    # one session, queries at rate rho = 1 per update: the device counters give Eq. (8)'s h
    rng = np.random.default_rng(3)
    table = sv.ReadyCacheTable(1, 2, DEV)
    ref = ReadyCache(1, 2)
    z = torch.zeros((1, 64))
    z[0, 5] = 4.0
    args = (_t([0], torch.int32), _t([0], torch.int64), _t([[1, 0]], torch.int32),
            _t([1], torch.int32), _t([2], torch.int64), z.to(DEV))
    table.record(*args)
    ref.record([0], [0], [[1, 0]], [1], [2], z)
    q = (_t([0], torch.int32), _t([0], torch.int64), _t([[1, 0]], torch.int32),
         _t([1], torch.int32))
    A = _t([5], torch.int32)
    for _ in range(1500):
        if rng.random() < 0.5:
            table.serve(*q, 1.0, A)
            ref.serve([0], [0], [[1, 0]], [1], 1.0, [5])
        else:
            table.invalidate(_t([0], torch.int32))
            table.record(*args)
            ref.invalidate([0])
            ref.record([0], [0], [[1, 0]], [1], [2], z)
    torch.cuda.synchronize()
    c = table.counters()
    assert c == ref.stats
    h = c["consumed"] / (c["consumed"] + c["wasted"])
    assert abs(h - 0.5) < 0.06


def test_large_batch_record_and_serve():
    # 1024 sessions recorded at once from V=128256 bf16 rows, then 8192 requests
    S, V, E = 1024, 128256, 8
    g = torch.Generator(device=DEV).manual_seed(9)
    z = torch.randn((S, V), generator=g, device=DEV)
    at = torch.randint(0, V, (S,), generator=g, device=DEV)
    z[torch.arange(S, device=DEV), at] += 12.0
    z = z.to(torch.bfloat16)
    table = sv.ReadyCacheTable(S, E, DEV)
    ent = torch.randint(0, 50, (S, E), generator=g, device=DEV, dtype=torch.int32)
    n_s = torch.randint(0, 1000, (S,), generator=g, device=DEV)
    L = torch.full((S,), E, dtype=torch.int32, device=DEV)
    B = torch.full((S,), 64, dtype=torch.int64, device=DEV)
    sid = torch.arange(S, dtype=torch.int32, device=DEV)
    st = table.record(sid, n_s, ent, L, B, z)
    torch.cuda.synchronize()
    assert (st == 0).all()
    state = table.state()
    want_tok = torch.argmax(z.float(), dim=1).cpu().numpy()  # distinct maxima: +12 peaks
    np.testing.assert_array_equal(state["token"], want_tok)
    top2 = torch.topk(z.float(), 2, dim=1).values.double().cpu().numpy()
    np.testing.assert_array_equal(state["gap"], top2[:, 0] - top2[:, 1])
    R = 8192
    rs = torch.randint(0, S, (R,), generator=g, device=DEV, dtype=torch.int32)
    tok, why = table.serve(rs, n_s[rs.long()], ent[rs.long()], L[rs.long()], 2.0, None,
                           exact=True)
    torch.cuda.synchronize()
    assert (why == 3).all()  # eligible everywhere; the empty answer set never fires
    A = torch.arange(V, dtype=torch.int32, device=DEV)
    tok, why = table.serve(rs, n_s[rs.long()], ent[rs.long()], L[rs.long()], 2.0, A)
    torch.cuda.synchronize()
    assert (why == 0).all() and torch.equal(tok.cpu(), torch.from_numpy(want_tok)[rs.cpu().long()].int())

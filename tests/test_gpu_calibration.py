"""CUDA gate calibration and conformal gate vs the oracle, through the C ABI (via the binding).

- gate_risk_coverage: exact counts, selected threshold and rates (bit for bit), on the
  pre-positioning page's operating point, random decision points with NaN gaps and tied
  thresholds, the largest grid, an empty set, an unsorted grid, answer sets of every span
  (negative, int32 extremes, repeated answers, past the membership bitmap), and a million
  points.
- conformal_residual: bit-exact fp32 residuals on rows with masked tokens, one-sided masks,
  NaN and infinities, aligned and unaligned rows, both dtypes, and the sampled-verify
  benchmark batch's draft rows against its target rows (sampled rows).
- conformal_quantile: the exact order statistic on ties, NaN, infinities and negative
  scores, at sizes from 1 to four million.
- conformal_admit: exact layers and tokens outside near ties and the fp32 gaps bit for bit,
  K from 1 to 8, both dtypes, rows of two segments, all-NaN rows; and the whole calibration
  pipeline (residuals -> quantile -> admission) on the device against the oracle's.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_17_gb300 as sv
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda"
Z95 = 1.959963984540054


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def run_sweep(gap, token, full, A, taus, z=Z95, r_max=0.15):
    pts, idx = sv.gate_risk_coverage(_dev(gap), _dev(token), _dev(full),
                                     None if A is None else _dev(A), _dev(taus), z, r_max)
    torch.cuda.synchronize()
    return sv.gate_points_dict(pts), int(idx.item())


def check_sweep(gap, token, full, A, taus, z=Z95, r_max=0.15):
    got, idx = run_sweep(gap, token, full, A, taus, z, r_max)
    want = oracle.risk_coverage(gap, token, full, A, taus, z, r_max)
    np.testing.assert_array_equal(got["accepted"].numpy(), want["accepted"])
    np.testing.assert_array_equal(got["wrong"].numpy(), want["wrong"])
    for name in ("coverage", "cov_lo", "cov_hi", "risk", "risk_lo", "risk_hi"):
        # the same operations in the same order, each rounded on its own: bit for bit
        np.testing.assert_array_equal(got[name].numpy(), want[name], err_msg=name)
    assert idx == want["tau_index"], (idx, want["tau_index"])
    return got, idx


def _points(N, seed, n_vocab=500, nan_every=0):
    rng = np.random.default_rng(seed)
    A = np.sort(rng.choice(n_vocab, n_vocab // 6, replace=False)).astype(np.int32)
    token = rng.integers(0, n_vocab, N).astype(np.int32)
    token[: N // 2] = rng.choice(A, N // 2)
    gap = np.abs(rng.standard_normal(N) * 3).astype(np.float32)
    if nan_every:
        gap[::nan_every] = np.nan
    p_ok = 1 - 0.5 * np.exp(-np.nan_to_num(gap.astype(np.float64)))
    full = np.where(rng.random(N) < p_ok, token, token + 1).astype(np.int32)
    return gap, token, full, A


def test_sweep_pages_operating_point():
    import test_oracle_calibration as K

    gap, token, full, A = K._operating_point_fixture()
    taus = np.linspace(0.0, 6.0, 25).astype(np.float32)
    got, idx = check_sweep(gap, token, full, A, taus, r_max=0.15)
    t = int(np.flatnonzero(taus == 2.0)[0])
    assert int(got["accepted"][t]) == 121 and int(got["wrong"][t]) == 16


@pytest.mark.parametrize("N,T,seed", [(1, 1, 0), (37, 5, 1), (10000, 61, 2), (5000, 4096, 3),
                                      (300, 4095, 4)])
def test_sweep_random(N, T, seed):
    gap, token, full, A = _points(N, seed, nan_every=13)
    rng = np.random.default_rng(seed + 100)
    taus = np.sort(rng.uniform(-1, 9, T)).astype(np.float32)
    if T > 3:
        taus[1] = taus[2]             # a repeated threshold
        taus[0] = -np.inf
        taus[-1] = np.inf
        gap[: min(N, 8)] = taus[T // 2]  # gaps sitting exactly on a threshold
    check_sweep(gap, token, full, A, taus, r_max=0.2)


def test_sweep_edges():
    gap, token, full, A = _points(200, 9)
    taus = np.array([0.5, 1.0, 2.0], np.float32)
    # empty answer set: nothing accepted, no threshold qualifies
    got, idx = check_sweep(gap, token, full, None, taus)
    assert (got["accepted"].numpy() == 0).all() and idx == -1
    # no decision points at all
    e = np.zeros(0, np.float32)
    ei = np.zeros(0, np.int32)
    got, idx = check_sweep(e, ei, ei, A, taus)
    assert np.isnan(got["coverage"].numpy()).all() and idx == -1
    # r_max NaN: nothing qualifies
    got, idx = check_sweep(gap, token, full, A, taus, r_max=float("nan"))
    assert idx == -1
    # an unsorted grid is reported, not guessed at
    got, idx = run_sweep(gap, token, full, A, np.array([1.0, 0.5, 2.0], np.float32))
    assert idx == -2 and (got["accepted"].numpy() == -1).all()
    assert np.isnan(got["risk"].numpy()).all()
    got, idx = run_sweep(gap, token, full, A, np.array([0.5, np.nan], np.float32))
    assert idx == -2


def test_sweep_inputs_off_the_16_byte_grid():
    # views one element into their buffers: the four-at-a-time loads give way to single ones
    gap, token, full, A = _points(5003, 17, nan_every=7)
    taus = np.linspace(0, 6, 33).astype(np.float32)
    g = torch.empty(gap.size + 1, dtype=torch.float32, device=DEV)[1:]
    t = torch.empty(gap.size + 1, dtype=torch.int32, device=DEV)[1:]
    f = torch.empty(gap.size + 1, dtype=torch.int32, device=DEV)[1:]
    g.copy_(torch.from_numpy(gap))
    t.copy_(torch.from_numpy(token))
    f.copy_(torch.from_numpy(full))
    assert g.data_ptr() % 16 != 0
    pts, idx = sv.gate_risk_coverage(g, t, f, _dev(A), _dev(taus), Z95, 0.2)
    torch.cuda.synchronize()
    got = sv.gate_points_dict(pts)
    want = oracle.risk_coverage(gap, token, full, A, taus, Z95, 0.2)
    np.testing.assert_array_equal(got["accepted"].numpy(), want["accepted"])
    np.testing.assert_array_equal(got["wrong"].numpy(), want["wrong"])
    np.testing.assert_array_equal(got["risk"].numpy(), want["risk"])
    assert int(idx.item()) == want["tau_index"]


@pytest.mark.parametrize("grid", ["clustered", "infinite_ends", "largest", "one_value"])
def test_sweep_threshold_grids(grid):
    # the bin of a gap comes from a bucket table over [taus[0], taus[-1]]: dense clusters and
    # exact duplicates (many thresholds in one bucket), gaps equal to thresholds, a grid with
    # infinite ends (the table gives way to a search over the whole grid), the largest grid
    # and a grid of one value
    gap, token, full, A = _points(60000, 31, nan_every=11)
    rng = np.random.default_rng(32)
    if grid == "clustered":
        taus = np.sort(np.concatenate([np.linspace(0, 1, 8), np.full(500, 2.5),
                                       np.linspace(2.5, 2.5001, 300),
                                       np.linspace(3, 9, 200)])).astype(np.float32)
    elif grid == "infinite_ends":
        taus = np.concatenate([[-np.inf], np.linspace(0, 8, 61), [np.inf]]).astype(np.float32)
    elif grid == "largest":
        taus = np.sort(rng.uniform(-1, 12, 4096)).astype(np.float32)
    else:
        taus = np.full(17, 1.5, np.float32)
    gap[:3000] = rng.choice(taus[np.isfinite(taus)], 3000)  # gaps equal to thresholds
    gap[3000:3010] = np.inf
    check_sweep(gap, token, full, A, taus, r_max=0.3)


def test_sweep_large_answer_set():
    # 6000 answers over a 50000-token span: more than the shared-memory copy holds, but within
    # the membership bitmap's span
    gap, token, full, _ = _points(40000, 41, n_vocab=50000)
    A = np.sort(np.random.default_rng(42).choice(50000, 6000, replace=False)).astype(np.int32)
    token[:20000] = np.random.default_rng(43).choice(A, 20000)
    check_sweep(gap, token, full, A, np.linspace(0, 9, 257).astype(np.float32), r_max=0.2)


I32_MIN, I32_MAX = -(1 << 31), (1 << 31) - 1
SPAN = 1 << 18  # the widest answer set whose membership is a bitmap


SPAN_CASES = ["negative", "span_at_bitmap_limit", "span_past_bitmap_small",
              "span_past_bitmap_large", "duplicates", "near_int32_max", "near_int32_min"]


@pytest.mark.parametrize("case", SPAN_CASES)
def test_sweep_answer_set_spans(case):
    # membership is a bitmap over [A[0], A[-1]] up to SPAN tokens, a search beyond: both
    # ends of each span, tokens just outside it, the int32 extremes, repeated answers, and
    # sets wider than the bitmap held in shared memory (<= 4096 entries) or searched in
    # global memory
    rng = np.random.default_rng(50 + SPAN_CASES.index(case))
    if case == "negative":
        A = np.array([-70000, -5, -3, 0, 7, 100], np.int64)
    elif case == "span_at_bitmap_limit":
        A = np.concatenate([[1000, 1000 + SPAN - 1], rng.integers(1001, 1000 + SPAN - 1, 200)])
    elif case == "span_past_bitmap_small":
        A = np.concatenate([[1000, 1000 + SPAN], rng.integers(1001, 1000 + SPAN, 200)])
    elif case == "span_past_bitmap_large":
        A = rng.choice(1 << 22, 6000, replace=False)
    elif case == "duplicates":
        A = np.repeat(np.array([3, 9, 9, 40, 41, 500]), 3)
    elif case == "near_int32_max":
        A = np.array([I32_MAX - 40, I32_MAX - 3, I32_MAX], np.int64)
    else:
        A = np.array([I32_MIN, I32_MIN + 2, I32_MIN + 77], np.int64)
    A = np.sort(A).astype(np.int32)
    N = 30000
    near = np.concatenate([A.astype(np.int64) + d for d in (-1, 0, 1)])
    near = near[(near >= I32_MIN) & (near <= I32_MAX)]
    extremes = np.array([I32_MIN, I32_MIN + 1, -1, 0, 1, I32_MAX - 1, I32_MAX], np.int64)
    token = rng.choice(np.concatenate([near, extremes]), N)
    token[: N // 3] = rng.choice(A, N // 3)
    token = token.astype(np.int32)
    gap = np.abs(rng.standard_normal(N) * 3).astype(np.float32)
    full = np.where(rng.random(N) < 0.8, token, token ^ 1).astype(np.int32)
    check_sweep(gap, token, full, A, np.linspace(0, 9, 300).astype(np.float32), r_max=0.2)


def test_sweep_reuses_its_workspace():
    # one workspace across calls of one CTA (no workspace state at all for grids of at most
    # 256 thresholds) and of many CTAs (histograms and counters cleared first), with a
    # broken grid in between: every call equals the oracle
    ws = torch.zeros(sv.gate_risk_coverage_workspace(200000, 300), dtype=torch.uint8,
                     device=DEV)
    calls = [(200000, np.linspace(0, 6, 64)), (300, np.linspace(0, 6, 64)),
             (300, np.array([1.0, 0.5, 2.0])), (200000, np.linspace(0, 6, 300)),
             (700, np.linspace(0, 6, 300)), (0, np.linspace(0, 6, 5)),
             (2000, np.linspace(0, 6, 64))]
    for i, (N, taus) in enumerate(calls):
        gap, token, full, A = _points(N, 60 + i, nan_every=9)
        taus = taus.astype(np.float32)
        pts, idx = sv.gate_risk_coverage(_dev(gap), _dev(token), _dev(full), _dev(A),
                                         _dev(taus), Z95, 0.2, workspace=ws)
        torch.cuda.synchronize()
        got = sv.gate_points_dict(pts)
        if np.all(np.diff(taus) >= 0):
            want = oracle.risk_coverage(gap, token, full, A, taus, Z95, 0.2)
            np.testing.assert_array_equal(got["accepted"].numpy(), want["accepted"])
            np.testing.assert_array_equal(got["wrong"].numpy(), want["wrong"])
            np.testing.assert_array_equal(got["risk_hi"].numpy(), want["risk_hi"])
            assert int(idx.item()) == want["tau_index"], (i, N)
        else:
            assert int(idx.item()) == -2 and (got["accepted"].numpy() == -1).all()


def test_sweep_a_million_points():
    gap, token, full, A = _points(1 << 20, 21, n_vocab=120, nan_every=1001)
    taus = np.linspace(0.0, 8.0, 64).astype(np.float32)
    check_sweep(gap, token, full, A, taus, r_max=0.3)


# ------------------------------------------------------------------------------ residual
def _bits(x):
    return np.asarray(x, np.float32).view(np.uint32)


def _same_f32(a, b):
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    both_nan = np.isnan(a) & np.isnan(b)
    return bool(((_bits(a) == _bits(b)) | both_nan).all())


@pytest.mark.parametrize("N,V,dt", [(5, 1, "f32"), (7, 1000, "f32"), (9, 1001, "bf16"),
                                    (6, 40000, "bf16"), (4, 8191, "f32"), (3, 151936, "bf16"),
                                    (2, 200003, "f32")])
def test_residual_small(N, V, dt):
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    g = torch.Generator().manual_seed(N * V)
    t = (torch.randn((N, V), generator=g) * 3).to(tdt)
    d = (t.float() + torch.randn((N, V), generator=g) * 0.2).to(tdt)
    if N >= 4 and V >= 8:
        d[0] = t[0]                                   # identical rows: 0
        t[1, : V // 2] = d[1, : V // 2] = float("-inf")  # masked in both
        d[2, V - 1] = float("-inf")                   # masked in one: inf
        t[3, V // 3] = float("nan")                   # NaN: NaN
    got = sv.conformal_residual(d.to(DEV), t.to(DEV))
    torch.cuda.synchronize()
    want = oracle.conformal_residual(d, t)
    assert _same_f32(got.cpu().numpy(), want), (got.cpu().numpy(), want)


def test_residual_unaligned_views_and_inf():
    V = 3000
    base_t = torch.randn((5, V + 1)) * 2
    base_d = base_t + torch.randn((5, V + 1)) * 0.1
    base_d[1, 7] = float("inf")
    base_t[1, 7] = float("inf")                      # +inf in both: equal, 0
    base_d[2, 9] = float("inf")                      # +inf against a finite value: inf
    # views 4 bytes into device buffers: the rows are off the 16-byte grid
    bt = base_t.to(DEV).reshape(-1)[1: 1 + 4 * V].reshape(4, V)
    bd = base_d.to(DEV).reshape(-1)[1: 1 + 4 * V].reshape(4, V)
    assert bt.data_ptr() % 16 != 0 and bt.is_contiguous()
    got = sv.conformal_residual(bd, bt)
    torch.cuda.synchronize()
    want = oracle.conformal_residual(bd.cpu(), bt.cpu())
    assert _same_f32(got.cpu().numpy(), want)


def test_residual_benchmark_rows_sampled():
    # the sampled-verify benchmark batch (B=512, k=8, V=128256 bf16): draft rows against the
    # target rows at the same positions, 4096 row pairs in one launch
    d = synth.workload_inputs(3, device=DEV)
    B, k, V = d["B"], d["k"], d["V"]
    tgt = d["target"][:, :k].contiguous()
    got = sv.conformal_residual(d["draft"], tgt).cpu().numpy()
    torch.cuda.synchronize()
    rows = sorted(np.random.default_rng(5).choice(B * k, 64, replace=False).tolist())
    want = oracle.conformal_residual(d["draft"].reshape(-1, V).cpu(), tgt.reshape(-1, V).cpu(),
                                     rows=rows, threads=16)
    assert _same_f32(got[rows], want[rows])
    assert (got > 0).all() and np.isfinite(got).all()


# ------------------------------------------------------------------------------ quantile
@pytest.mark.parametrize("n", [1, 2, 5, 19, 4096, 100003, 1 << 22])
@pytest.mark.parametrize("q", [1e-6, 0.5, 0.9, 0.95, 1.0])
def test_quantile_random(n, q):
    rng = np.random.default_rng(n)
    r = rng.exponential(1.0, n).astype(np.float32)
    if n >= 19:
        r[:5] = r[5]                  # ties
        r[6] = np.inf
        r[7] = np.nan
        r[8] = -1.5                   # negative scores order below zero
    got = sv.conformal_quantile(_dev(r), q)
    torch.cuda.synchronize()
    want = oracle.conformal_quantile(r, q)
    assert _same_f32(got.cpu().numpy(), [want]), (got.item(), want)


@pytest.mark.parametrize("kind", ["all_equal", "two_values", "sorted", "all_nan", "all_inf",
                                  "denormals"])
def test_quantile_degenerate_score_sets(kind):
    # more than 8192 scores: the cooperative radix select, where every pass's digit comes
    # from the CTA whose arrival completes the pass; here one bin holds every key (or most)
    n = 50021
    rng = np.random.default_rng(17)
    r = {"all_equal": np.full(n, 0.25, np.float32),
         "two_values": np.where(rng.random(n) < 0.3, 1.0, 2.0).astype(np.float32),
         "sorted": np.sort(rng.standard_normal(n)).astype(np.float32),
         "all_nan": np.full(n, np.nan, np.float32),
         "all_inf": np.full(n, np.inf, np.float32),
         "denormals": (rng.integers(1, 1 << 20, n) * np.float32(1e-45)).astype(np.float32),
         }[kind]
    for q in (1e-6, 0.3, 0.9, 1.0):
        got = sv.conformal_quantile(_dev(r), q)
        torch.cuda.synchronize()
        want = oracle.conformal_quantile(r, q)
        assert _same_f32(got.cpu().numpy(), [want]), (kind, q, got.item(), want)


def test_quantile_of_scores_off_the_16_byte_grid():
    rng = np.random.default_rng(4)
    r = rng.exponential(1.0, 100003).astype(np.float32)
    buf = torch.empty(r.size + 3, dtype=torch.float32, device=DEV)
    v = buf[3:]
    v.copy_(torch.from_numpy(r))
    assert v.data_ptr() % 16 != 0
    for q in (0.5, 0.9, 0.999):
        got = sv.conformal_quantile(v, q)
        torch.cuda.synchronize()
        assert _same_f32(got.cpu().numpy(), [oracle.conformal_quantile(r, q)])


def test_quantile_reuses_its_workspace():
    r = np.arange(1000, dtype=np.float32)[::-1].copy()
    ws = torch.zeros(sv.conformal_quantile_workspace(1000), dtype=torch.uint8, device=DEV)
    for q in (0.1, 0.5, 0.99, 0.999):
        got = sv.conformal_quantile(_dev(r), q, workspace=ws).item()
        assert got == oracle.conformal_quantile(r, q)


def test_quantile_barrier_wait_runs_out_and_reports_it():
    """The quantile's cooperative launch is the one place where CTAs wait on one another.
    Its self-test entry sets every grid barrier's arrival target one above the grid, so no
    barrier completes: each wait must give up after its limit (here 1 ms), the launch must
    end on its own, and out_q must carry the timeout sentinel (quiet NaN, payload 1). The
    device, and the same workspace, must then serve a normal call."""
    import ctypes

    n = 1 << 20
    rng = np.random.default_rng(11)
    r = rng.exponential(1.0, n).astype(np.float32)
    d = _dev(r)
    ws = torch.zeros(sv.conformal_quantile_workspace(n), dtype=torch.uint8, device=DEV)
    out = torch.zeros(1, dtype=torch.float32, device=DEV)
    P = ctypes.c_void_p
    L = sv.library()
    h = torch.cuda.current_stream().cuda_stream
    for wait_us in (1000, 200):
        out.fill_(0.0)
        st = L.conformal_quantile_barrier_selftest(P(d.data_ptr()), n, P(out.data_ptr()),
                                                   P(ws.data_ptr()), ws.numel(), wait_us, P(h))
        assert st == 0, L.sv_status_string(st)
        torch.cuda.synchronize()
        assert out.view(torch.int32).item() == 0x7FC00001
    # bad arguments are refused on the host
    assert L.conformal_quantile_barrier_selftest(P(d.data_ptr()), 8192, P(out.data_ptr()),
                                                 P(ws.data_ptr()), ws.numel(), 1000, P(h)) == 1
    assert L.conformal_quantile_barrier_selftest(P(d.data_ptr()), n, P(out.data_ptr()),
                                                 P(ws.data_ptr()), ws.numel(), 0, P(h)) == 1
    # the context and the workspace still serve a normal call
    got = sv.conformal_quantile(d, 0.9, workspace=ws)
    torch.cuda.synchronize()
    assert _same_f32(got.cpu().numpy(), [oracle.conformal_quantile(r, 0.9)])


# ------------------------------------------------------------------------------ admission
def _layer_logits(N, K, V, dt, seed, peak_hi=8.0):
    g = torch.Generator().manual_seed(seed)
    z = torch.randn((N, K, V), generator=g)
    idx = torch.randint(0, V, (N, K, 1), generator=g)
    scale = torch.linspace(0.3, 1.0, K) if K > 1 else torch.ones(1)
    amp = torch.rand((N, K, 1), generator=g) * peak_hi * scale[None, :, None]
    z.scatter_add_(2, idx, amp)
    return z.to(torch.float32 if dt == "f32" else torch.bfloat16)


def check_admit(z, Q):
    lay, tok, gap = sv.conformal_admit(z.to(DEV), _dev(Q))
    torch.cuda.synchronize()
    o = oracle.conformal_admit(z, Q)
    lay, tok, gap = lay.cpu().numpy(), tok.cpu().numpy(), gap.cpu().numpy()
    assert _same_f32(gap, o["gap"].astype(np.float32))
    keep = o["flag"] == -1
    np.testing.assert_array_equal(lay[keep], o["layer"][keep])
    np.testing.assert_array_equal(tok[keep], o["token"][keep])
    return lay, tok, o


@pytest.mark.parametrize("N,K,V,dt", [(64, 1, 1000, "f32"), (40, 2, 32000, "bf16"),
                                      (25, 4, 8191, "f32"), (16, 8, 3001, "bf16"),
                                      (6, 3, 151936, "bf16")])
def test_admit_random(N, K, V, dt):
    z = _layer_logits(N, K, V, dt, seed=N * K + V)
    Q = np.linspace(1.2, 0.4, K).astype(np.float32)
    lay, tok, o = check_admit(z, Q)
    assert len(set(lay.tolist())) > 1  # several layers actually taken


def test_admit_nan_rows_and_edges():
    N, K, V = 5, 3, 700
    z = _layer_logits(N, K, V, "f32", seed=3)
    z[0, :, :] = float("nan")           # never admits
    z[1, 0, :] = float("nan")           # layer 0 of step 1 cannot admit
    z[2, :, :] = float("-inf")
    z[2, :, 11] = 1.0                   # one finite logit: gamma = +inf admits at layer 0
    Q = np.array([0.5, 0.5, 0.5], np.float32)
    lay, tok, o = check_admit(z, Q)
    assert lay[0] == K and tok[0] == -1
    assert lay[2] == 0 and tok[2] == 11
    lay, tok, o = check_admit(z, np.full(K, np.inf, np.float32))  # +inf Q admits only +inf gaps
    assert lay[2] == 0 and (lay[[0, 1, 3, 4]] == K).all()
    lay, tok, o = check_admit(z, np.full(K, -1.0, np.float32))    # negative Q admits any gap
    assert (lay[1:] <= 1).all() and lay[1] == 1


def test_calibration_pipeline_on_the_device():
    # calibrate on draft/true row pairs, then admit fresh steps: residuals -> Q -> admission
    n_cal, V = 512, 32000
    g = torch.Generator().manual_seed(77)
    t = torch.randn((n_cal, V), generator=g) * 2
    d = (t + torch.randn((n_cal, V), generator=g) * torch.rand((n_cal, 1), generator=g) * 0.5)
    t, d = t.to(torch.bfloat16), d.to(torch.bfloat16)
    r = sv.conformal_residual(d.to(DEV), t.to(DEV))
    Q = sv.conformal_quantile(r, 0.9)
    torch.cuda.synchronize()
    r_o = oracle.conformal_residual(d, t)
    assert _same_f32(r.cpu().numpy(), r_o)
    Q_o = oracle.conformal_quantile(r_o, 0.9)
    assert Q.item() == Q_o
    z = _layer_logits(64, 1, V, "bf16", seed=78, peak_hi=12.0)
    lay, tok, gap = sv.conformal_admit(z.to(DEV), Q)
    torch.cuda.synchronize()
    o = oracle.conformal_admit(z, np.array([Q_o], np.float32))
    keep = o["flag"] == -1
    np.testing.assert_array_equal(lay.cpu().numpy()[keep], o["layer"][keep])
    assert 0 < int((o["layer"] == 0).sum()) < 64

"""CUDA draft-confidence stop vs the oracle, through the C ABI (via the thin binding).

Both confidence measures (top probability, inverse entropy) on seeded draft rows whose
peakedness varies from row to row, so that the stop lands at many positions. The floor of a
case sits between two of the oracle's own confidences (never on one). Small cases span several
chunks, ragged tails, unaligned rows, two segments per row and ragged or invalid draft counts;
the sampled-verify benchmark batch's draft rows run at full size on a seeded sample of
requests.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_17_gb300 as sv
import synth
from parity import compare_confidence

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOP, ENT = sv.SV_CONF_TOP_PROB, sv.SV_CONF_INV_ENTROPY


def _floor_between(conf: np.ndarray, q: float) -> float:
    """A floor halfway (geometrically) between two neighbouring confidences near quantile q."""
    c = np.sort(conf[np.isfinite(conf) & (conf > 0)])
    if c.size < 2:
        return 0.5
    i = min(max(int(q * c.size), 1), c.size - 1)
    return float(math.sqrt(c[i - 1] * c[i])) if c[i] > c[i - 1] else float(c[i] * 1.5)


def run_case(z, nd, T, mode, floor=None, q=0.4, requests=None, threads=16):
    nin = (np.full(z.shape[0], z.shape[1]) if nd is None else nd.cpu().numpy())
    zc = z.cpu()
    ndc = None if nd is None else nd.cpu()
    if floor is None:
        probe = oracle.draft_confidence(zc, ndc, T, mode, 0.0, requests=requests,
                                        threads=threads)
        floor = _floor_between(probe["conf"][np.isfinite(probe["conf"])], q)
    out_nd, out_c = sv.draft_confidence_stop(z, T, mode, floor, nd)
    torch.cuda.synchronize()
    orc = oracle.draft_confidence(zc, ndc, T, mode, floor, requests=requests, threads=threads)
    reqs = range(z.shape[0]) if requests is None else requests
    stats = compare_confidence(out_nd.cpu().numpy(), out_c.cpu().numpy(), nin, orc, floor,
                               mode, reqs)
    return stats, out_nd.cpu().numpy(), out_c.cpu().numpy(), orc


SMALL = [
    # B, k, V, dtype, T, ragged, peak
    (1, 4, 1000, "f32", 1.0, False, (0.0, 12.0)),
    (37, 3, 40000, "bf16", 0.8, True, (0.0, 20.0)),     # 3 chunks, partial last one
    (20, 2, 8191, "f32", 1.2, True, (0.0, 16.0)),       # rows not 16-byte aligned
    (16, 5, 16385, "bf16", 0.6, False, (0.0, 14.0)),    # one logit into a second chunk
    (12, 1, 2, "f32", 1.0, False, (0.0, 3.0)),          # V = 2
    (9, 16, 3001, "bf16", 1.0, True, (0.0, 12.0)),      # k = 16 (maximum)
    (64, 4, 24577, "f32", 0.9, True, (0.0, 18.0)),      # 4 chunks (fp32), ragged tail
    (7, 8, 50001, "bf16", 0.05, False, (0.0, 2.0)),     # low temperature: near-certain rows
    (5, 3, 777, "bf16", 50.0, True, (0.0, 200.0)),      # high temperature: near-uniform rows
    (6, 3, 151936, "bf16", 0.8, True, (0.0, 22.0)),     # two segments per row
    (4, 2, 200003, "bf16", 1.0, False, (0.0, 22.0)),    # two segments, rows not aligned
]


@pytest.mark.parametrize("mode", [TOP, ENT], ids=["top", "inv_entropy"])
@pytest.mark.parametrize("case", SMALL, ids=[f"B{c[0]}k{c[1]}V{c[2]}{c[3]}" for c in SMALL])
def test_confidence_small(case, mode):
    B, k, V, dt, T, ragged, peak = case
    d = synth.sample_inputs(B, k, V, dt, T, device=DEV, seed=7 * V + B, ragged=ragged,
                            target_std=2.0, draft_noise=0.5, peak=peak)
    stats, nd, _, _ = run_case(d["draft"], d["num_draft"], T, mode)
    print(f"B={B} k={k} V={V} {dt} T={T} mode={mode}: {stats}")
    assert stats["flagged"] <= max(1, B // 8), stats


@pytest.mark.parametrize("mode", [TOP, ENT], ids=["top", "inv_entropy"])
def test_confidence_stops_land_everywhere(mode):
    # a floor at the lower quartile of the confidences: stops at 0, at 1 and at k all occur
    B, k, V = 64, 6, 12000
    d = synth.sample_inputs(B, k, V, "bf16", 1.0, device=DEV, seed=5, target_std=1.0,
                            draft_noise=0.3, peak=(0.0, 16.0))
    stats, nd, _, _ = run_case(d["draft"], None, 1.0, mode, q=0.25)
    assert set(np.unique(nd)) >= {0, 1, k}, np.unique(nd)


@pytest.mark.parametrize("mode", [TOP, ENT], ids=["top", "inv_entropy"])
def test_confidence_data_errors_and_counts(mode):
    B, k, V = 8, 4, 5000
    d = synth.sample_inputs(B, k, V, "f32", 1.0, device=DEV, seed=19, peak=(0.0, 12.0))
    z = d["draft"]
    nd = torch.tensor([4, 2, 4, 5, -1, 0, 3, 4], dtype=torch.int32, device=DEV)
    z[0, 1, 77] = float("nan")       # NaN in a row that is read
    z[1, 3, 5] = float("inf")        # +inf past the request's count: not read
    z[2, 0, :] = float("-inf")       # no finite logit
    z[6, 2, 4999] = float("inf")     # +inf in the last logit of a read row
    stats, got, c, orc = run_case(z, nd, 1.0, mode, floor=0.05 if mode == TOP else 0.2)
    assert list(orc["num_draft"][[0, 2, 3, 4, 6]]) == [-1, -1, -1, -1, -1]
    assert got[5] == 0 and (c[5] == 0).all()
    assert stats["errors"] == 5


def test_confidence_one_hot_and_masked_rows():
    # one finite logit: top probability 1, entropy 0 (inverse +inf); two segments per row
    B, k, V = 3, 3, 140001
    z = torch.full((B, k, V), float("-inf"), dtype=torch.bfloat16, device=DEV)
    for r in range(B):
        for i in range(k):
            z[r, i, (r * 7919 + i * 104729) % V] = 1.5
    z[2, 2, 5] = 1.5  # two equal finite logits: top 1/2, entropy ln 2
    nd, c = sv.draft_confidence_stop(z, 1.0, TOP, 0.75)
    torch.cuda.synchronize()
    assert list(nd.cpu().numpy()) == [3, 3, 2]
    np.testing.assert_allclose(c.cpu().numpy()[:2], 1.0, rtol=1e-6)
    assert c[2, 2].item() == pytest.approx(0.5, rel=1e-6)
    nd, c = sv.draft_confidence_stop(z, 1.0, ENT, 5.0)
    torch.cuda.synchronize()
    assert list(nd.cpu().numpy()) == [3, 3, 2]
    # H = 0 up to the fp32 exponentials' few 1e-7 nats: 1/H is +inf or above 1e6
    assert (c.cpu().numpy()[:2] > 1e6).all()
    assert c[2, 2].item() == pytest.approx(1.0 / math.log(2.0), rel=1e-6)


def test_confidence_without_conf_output_and_reused_workspace():
    B, k, V = 24, 5, 33000
    d = synth.sample_inputs(B, k, V, "bf16", 0.9, device=DEV, seed=23, ragged=True,
                            peak=(0.0, 18.0))
    ws = torch.zeros(sv.draft_confidence_workspace(B, k, V, sv.SV_BF16), dtype=torch.uint8,
                     device=DEV)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a, ca = sv.draft_confidence_stop(d["draft"], 0.9, TOP, 0.02, d["num_draft"],
                                         workspace=ws, stream=s)
        b, cb = sv.draft_confidence_stop(d["draft"], 0.9, TOP, 0.02, d["num_draft"],
                                         workspace=ws, stream=s, want_conf=False)
    s.synchronize()
    assert cb is None
    assert torch.equal(a, b)
    orc = oracle.draft_confidence(d["draft"].cpu(), d["num_draft"].cpu(), 0.9, TOP, 0.02)
    keep = orc["flag"] == -1
    np.testing.assert_array_equal(a.cpu().numpy()[keep], orc["num_draft"][keep])


@pytest.mark.parametrize("mode", [TOP, ENT], ids=["top", "inv_entropy"])
def test_confidence_benchmark_draft_rows_sampled(mode):
    # the sampled-verify benchmark batch (B=512, k=8, V=128256 bf16), all requests on the
    # GPU in one launch; the oracle on a seeded sample of 48 requests
    d = synth.workload_inputs(3, device=DEV)
    B, k, V, T = d["B"], d["k"], d["V"], d["T"]
    reqs = sorted(np.random.default_rng(31).choice(B, 48, replace=False).tolist())
    stats, nd, c, _ = run_case(d["draft"], None, T, mode, requests=reqs, q=0.3)
    print(f"benchmark draft rows mode={mode}: {stats}")
    assert stats["requests"] == 48 and stats["flagged"] <= 2
    # properties over every request: counts in range, confidences in their ranges
    assert ((nd >= 0) & (nd <= k)).all()
    if mode == TOP:
        assert ((c > 0) & (c <= 1)).all()
    else:
        assert (c >= 1.0 / math.log(V) * (1 - 1e-5)).all()

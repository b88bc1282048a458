"""Seeded random shapes for every call of the verify step, CUDA path vs the oracle.

Each case draws its own B, k, V, dtype, temperature, draft counts, alignment (a view one element
into a buffer) and a sprinkle of masked, NaN and +inf logits, so the cases cross chunk and
segment boundaries, ragged tails, unaligned rows and the data-error paths that fixed tests
may miss. The comparisons are those of the fixed parity tests.
"""
import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_17_gb300 as sv
import synth
from parity import check_flags, compare_confidence, compare_gate, compare_greedy, compare_sample

pytestmark = pytest.mark.gpu
DEV = "cuda"
CASES = 24


def _shape(rng):
    V = int(rng.choice([2, 3, 17, 999, 4096, 16383, 16385, 40000, 131073, 150001]))
    k = int(rng.integers(1, 17))
    B = int(rng.integers(1, 12 if V > 100000 else 40))
    dt = "bf16" if rng.random() < 0.5 else "f32"
    T = float(rng.choice([0.05, 0.5, 1.0, 2.0, 20.0]))
    return B, k, V, dt, T


def _offset_view(x, off):
    """x's values in a buffer `off` elements past an aligned start (rows off the 16-byte grid
    when off is not a multiple of the vector width)."""
    if off == 0:
        return x
    flat = torch.empty(x.numel() + off, dtype=x.dtype, device=x.device)
    v = flat[off:].view(x.shape)
    v.copy_(x)
    return v


def _sprinkle(z, rng, masked=0.02, nan_rows=0, inf_rows=0):
    """Mask a few logits per row with -inf; put NaN or +inf in a few chosen rows."""
    flat = z.view(-1, z.shape[-1])
    n, V = flat.shape
    if V > 2 and masked > 0:
        m = torch.from_numpy(rng.random((n, V)) < masked).to(z.device)
        flat.masked_fill_(m, float("-inf"))
    for _ in range(nan_rows):
        flat[int(rng.integers(0, n)), int(rng.integers(0, V))] = float("nan")
    for _ in range(inf_rows):
        flat[int(rng.integers(0, n)), int(rng.integers(0, V))] = float("inf")
    return z


@pytest.mark.parametrize("seed", range(CASES))
def test_fuzz_sample(seed):
    rng = np.random.default_rng(1000 + seed)
    B, k, V, dt, T = _shape(rng)
    d = synth.sample_inputs(B, k, V, dt, T, device=DEV, seed=seed, ragged=bool(rng.random() < .6),
                            target_std=float(rng.uniform(0.5, 4)),
                            draft_noise=float(rng.uniform(0, 2)), draft_scale=1.0)
    _sprinkle(d["target"], rng, nan_rows=int(rng.random() < 0.3), inf_rows=int(rng.random() < .2))
    _sprinkle(d["draft"], rng, nan_rows=int(rng.random() < 0.2))
    off = int(rng.choice([0, 0, 1, 3]))
    tgt, dft = _offset_view(d["target"], off), _offset_view(d["draft"], off)
    tok, acc, p, q, W = sv.spec_verify_sample(tgt, dft, d["draft_tokens"], d["uniforms"], T,
                                              d["num_draft"])
    torch.cuda.synchronize()
    nd = d["num_draft"]
    gpu = dict(tokens=tok.cpu().numpy(), accept_len=acc.cpu().numpy(), p=p.cpu().numpy(),
               q=q.cpu().numpy(), resid=W.cpu().numpy(),
               n=np.full(B, k) if nd is None else nd.cpu().numpy())
    orc = oracle.spec_verify_sample(d["target"].cpu(), d["draft"].cpu(), d["draft_tokens"].cpu(),
                                    None if nd is None else nd.cpu(), d["uniforms"].cpu(), T,
                                    threads=16)
    stats = compare_sample(gpu, orc, range(B))
    # near ties are the oracle's to flag (tiny V and extreme temperatures make many); every
    # unflagged position matched exactly above, and the count stays within the rule's bound
    check_flags(f"fuzz seed={seed} B={B} k={k} V={V} {dt} T={T:.3g}", stats, orc, range(B))


@pytest.mark.parametrize("seed", range(CASES))
def test_fuzz_greedy_and_gate(seed):
    rng = np.random.default_rng(2000 + seed)
    B, k, V, dt, _ = _shape(rng)
    tdt = torch.float32 if dt == "f32" else torch.bfloat16
    g = torch.Generator(device=DEV).manual_seed(seed)
    z = (torch.randn((B, k + 1, V), generator=g, device=DEV) * 2).to(tdt)
    if V > 3 and rng.random() < 0.5:
        z[..., : V // 3] = z[..., V // 3: 2 * (V // 3)]  # repeated values: ties
    _sprinkle(z, rng, nan_rows=int(rng.random() < 0.3), inf_rows=int(rng.random() < 0.2))
    x = torch.argmax(z[:, :k].float(), dim=-1).to(torch.int32)
    flip = torch.from_numpy(rng.random((B, k)) < 0.3).to(DEV)
    x = torch.where(flip, (x + 1) % V, x)
    nd = torch.from_numpy(rng.integers(0, k + 1, B).astype(np.int32)).to(DEV)
    off = int(rng.choice([0, 0, 1, 5]))
    zz = _offset_view(z, off)
    gt, ga = sv.spec_verify_greedy(zz, x, nd)
    torch.cuda.synchronize()
    og = oracle.spec_verify_greedy(z.cpu(), x.cpu(), nd.cpu())
    compare_greedy(gt.cpu().numpy(), ga.cpu().numpy(), og)
    rows = zz.reshape(-1, V)
    A = torch.from_numpy(np.sort(rng.choice(V, max(1, V // 4), replace=False)).astype(np.int32))
    tau = float(rng.choice([0.0, 0.5, 2.0]))
    tk, gap, fire = sv.logit_gap_gate(rows, tau, A.to(DEV))
    torch.cuda.synchronize()
    oz = oracle.logit_gap_gate(rows.cpu(), tau, A)
    compare_gate(tk.cpu().numpy(), gap.cpu().numpy(), fire.cpu().numpy(), oz)


@pytest.mark.parametrize("seed", range(CASES // 2))
def test_fuzz_confidence(seed):
    rng = np.random.default_rng(3000 + seed)
    B, k, V, dt, T = _shape(rng)
    d = synth.sample_inputs(B, k, V, dt, T, device=DEV, seed=seed, ragged=True,
                            peak=(0.0, float(rng.uniform(4, 24))))
    z = _sprinkle(d["draft"], rng, nan_rows=int(rng.random() < 0.3))
    mode = int(rng.integers(0, 2))
    floor = float(rng.choice([0.05, 0.3, 0.8])) if mode == 0 else float(rng.choice([0.2, 1.0]))
    off = int(rng.choice([0, 0, 1]))
    zz = _offset_view(z, off)
    nd_out, c = sv.draft_confidence_stop(zz, T, mode, floor, d["num_draft"])
    torch.cuda.synchronize()
    orc = oracle.draft_confidence(z.cpu(), d["num_draft"].cpu(), T, mode, floor, threads=16)
    compare_confidence(nd_out.cpu().numpy(), c.cpu().numpy(), d["num_draft"].cpu().numpy(), orc,
                       floor, mode, range(B))

"""Seeded synthetic inputs for the speculative-decoding verify step.

This module only draws random inputs; it holds none of the verify arithmetic, and both the
CUDA library's callers (tests, benchmark) and the oracle's callers take their inputs from
here. Every draw comes from a ``torch.Generator`` (or a numpy ``Generator`` for token
histories) seeded per workload, so the same call on the same device gives the same tensors.
Values differ between CPU and CUDA generators, which is harmless: a parity check always
hands the very same tensor to both sides.

The five workloads mirror the pages' settings (no page measures on a public suite, so these
shapes and value distributions stand in for real logits):

  0  sampled verify, B=1,   k=4, V=1000,   fp32, T=1.0; z_p ~ N(0, 2^2), z_q = z_p + N(0, 0.5^2)
  1  sampled + greedy, B=64, k=5, V=32000, bf16, T=0.8; z_p ~ N(0, 3^2) + a Zipf(s=1.1)-shaped
     log-bias over a random permutation of the vocabulary, z_q = z_p + N(0, 1)
  2  sampled + gate, B=256, k=4, V=151936, fp32, T=1.0; z_p ~ N(0, 3^2) plus one planted peak
     +U(2, 10) per row, z_q = z_p + N(0, 0.7^2); gate tau = 4.0 over all B*(k+1) target rows,
     fast-answer set of 64 distinct random tokens
  3  sampled verify with residual, B=512, k=8, V=128256, bf16, T=0.7; z_p ~ N(0, 2.5^2),
     z_q = 0.6 z_p + N(0, 1.5^2)
  4  n-gram proposal + greedy verify, B=128 histories of length 8192 over V=32000 built from
     a random base in which ~30% of the spans (length 8..64) are copied from earlier offsets;
     n_max=4, n_min=2, k=5; bf16 target rows N(0, 1) with a +8 peak that agrees with the
     proposal at 60% of drafted positions

Draft tokens are drawn from q = softmax(z_q / T) with the Gumbel-max trick
(argmax(z_q/T + Gumbel noise)), on the rounded logits the verifier sees; uniforms are
``torch.rand`` values in [0, 1).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    index: int
    name: str
    kind: str  # "sample", "sample+greedy", "sample+gate", "ngram+greedy"
    B: int
    k: int
    V: int
    dtype: str  # "f32" | "bf16"
    T: float = 1.0
    extra: dict = field(default_factory=dict)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2


WORKLOADS = [
    Workload(0, "b1_k4_v1000_f32", "sample", 1, 4, 1000, "f32", 1.0,
             dict(target_std=2.0, draft_noise=0.5, draft_scale=1.0)),
    Workload(1, "b64_k5_v32000_bf16_zipf", "sample+greedy", 64, 5, 32000, "bf16", 0.8,
             dict(target_std=3.0, draft_noise=1.0, draft_scale=1.0, zipf_s=1.1)),
    Workload(2, "b256_k4_v151936_f32_peak_gate", "sample+gate", 256, 4, 151936, "f32", 1.0,
             dict(target_std=3.0, draft_noise=0.7, draft_scale=1.0, peak=(2.0, 10.0),
                  tau=4.0, n_answer=64)),
    Workload(3, "b512_k8_v128256_bf16_resid", "sample", 512, 8, 128256, "bf16", 0.7,
             dict(target_std=2.5, draft_noise=1.5, draft_scale=0.6)),
    Workload(4, "ngram_b128_l8192_v32000_bf16", "ngram+greedy", 128, 5, 32000, "bf16", 1.0,
             dict(L=8192, n_max=4, n_min=2, copy_frac=0.3, span=(8, 64), agree=0.6,
                  peak=8.0)),
]

SEED_BASE = 1000


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _gumbel_argmax(logits_f32: torch.Tensor, T: float, g: torch.Generator) -> torch.Tensor:
    """Index drawn from softmax(logits/T) along the last axis (Gumbel-max trick)."""
    u = torch.rand(logits_f32.shape, generator=g, device=logits_f32.device,
                   dtype=torch.float32)
    u = u.clamp_(min=1e-20)
    gumbel = -torch.log(-torch.log(u).clamp_(max=-1e-20))
    return torch.argmax(logits_f32 / T + gumbel, dim=-1).to(torch.int32)


def sample_inputs(B: int, k: int, V: int, dtype: str, T: float, *, device="cpu", seed: int = 0,
                  target_std: float = 2.0, draft_noise: float = 0.5, draft_scale: float = 1.0,
                  zipf_s: float | None = None, peak=None, ragged: bool = False,
                  block: int = 32) -> dict:
    """Inputs of one sampled-verify batch.

    Returns ``target`` [B, k+1, V], ``draft`` [B, k, V] (dtype), ``draft_tokens`` [B, k]
    int32 drawn from q, ``num_draft`` [B] int32 (None unless ``ragged``: then uniform in
    0..k) and ``uniforms`` [B, k+1] fp32. Generated ``block`` requests at a time so the
    fp32 intermediates stay small.
    """
    tdt = torch.float32 if dtype == "f32" else torch.bfloat16
    g = _gen(device, seed)
    target = torch.empty((B, k + 1, V), dtype=tdt, device=device)
    draft = torch.empty((B, k, V), dtype=tdt, device=device)
    tokens = torch.empty((B, k), dtype=torch.int32, device=device)
    bias = None
    if zipf_s is not None:
        perm = torch.randperm(V, generator=g, device=device)
        bias = -zipf_s * torch.log(perm.to(torch.float64) + 1.0).to(torch.float32)
    for b0 in range(0, B, block):
        b1 = min(B, b0 + block)
        zp = torch.randn((b1 - b0, k + 1, V), generator=g, device=device) * target_std
        if bias is not None:
            zp += bias
        if peak is not None:
            lo, hi = peak
            idx = torch.randint(0, V, (b1 - b0, k + 1, 1), generator=g, device=device)
            amp = lo + (hi - lo) * torch.rand((b1 - b0, k + 1, 1), generator=g, device=device)
            zp.scatter_add_(2, idx, amp)
        zq = draft_scale * zp[:, :k] + draft_noise * torch.randn(
            (b1 - b0, k, V), generator=g, device=device)
        target[b0:b1] = zp.to(tdt)
        draft[b0:b1] = zq.to(tdt)
        tokens[b0:b1] = _gumbel_argmax(draft[b0:b1].float(), T, g)
        del zp, zq
    uniforms = torch.rand((B, k + 1), generator=g, device=device, dtype=torch.float32)
    num_draft = None
    if ragged:
        num_draft = torch.randint(0, k + 1, (B,), generator=g, device=device, dtype=torch.int32)
        pad = torch.arange(k, device=device)[None, :] >= num_draft[:, None]
        tokens = tokens.masked_fill(pad, -1)
    return dict(target=target, draft=draft, draft_tokens=tokens, num_draft=num_draft,
                uniforms=uniforms, B=B, k=k, V=V, T=T, dtype=dtype)


def answer_set(V: int, n: int, *, device="cpu", seed: int = 0) -> torch.Tensor:
    """``n`` distinct random token ids, sorted ascending (the gate's fast-answer set)."""
    g = _gen("cpu", seed)
    ids = torch.randperm(V, generator=g)[:n].sort().values.to(torch.int32)
    return ids.to(device)


def histories(B: int, L: int, V: int, *, seed: int = 0, copy_frac: float = 0.3,
              span=(8, 64), lengths=None) -> tuple[np.ndarray, np.ndarray]:
    """Token histories [B, L] int32 and their lengths [B] int32.

    Each history is a sequence of spans with lengths uniform in ``span``; a span is, with
    probability ``copy_frac``, a token-by-token copy starting at a uniformly random earlier
    offset (so it may overlap itself), else fresh uniform tokens. ``lengths`` (optional)
    gives per-request lengths <= L; the tail past a length is filled with -1.
    """
    rng = np.random.default_rng(seed)
    H = rng.integers(0, V, size=(B, L), dtype=np.int64).astype(np.int32)
    for b in range(B):
        h = H[b]
        pos = 0
        while pos < L:
            n = int(rng.integers(span[0], span[1] + 1))
            n = min(n, L - pos)
            if pos > 0 and rng.random() < copy_frac:
                src = int(rng.integers(0, pos))
                if src + n <= pos:
                    h[pos:pos + n] = h[src:src + n]
                else:
                    for t in range(n):
                        h[pos + t] = h[src + t]
            pos += n
    if lengths is None:
        lens = np.full(B, L, np.int32)
    else:
        lens = np.asarray(lengths, np.int32)
        for b in range(B):
            H[b, lens[b]:] = -1
    return H, lens


def greedy_targets(drafts: torch.Tensor, num_draft: torch.Tensor, V: int, *, k: int,
                   agree: float = 0.6, peak: float = 8.0, seed: int = 0,
                   dtype=torch.bfloat16) -> torch.Tensor:
    """Target logits [B, k+1, V] for a greedy verify of given proposals.

    Rows are N(0, 1). Drafted row i < n_r gets +``peak`` at the proposed token with
    probability ``agree``, else at a uniformly random other token; row n_r (the bonus row)
    gets +``peak`` at a random token; later rows stay plain noise. ``drafts`` and
    ``num_draft`` are inputs here (the proposal the verify will check), not results.
    """
    device = drafts.device
    g = _gen(device, seed)
    B = drafts.shape[0]
    z = torch.randn((B, k + 1, V), generator=g, device=device)
    nd = num_draft.to(torch.int64).clamp(min=0, max=k)
    d = drafts.to(torch.int64)
    agree_mask = torch.rand((B, k), generator=g, device=device) < agree
    other = torch.randint(0, V - 1, (B, k), generator=g, device=device)
    other = other + (other >= d.clamp(min=0)).to(torch.int64)
    col = torch.where(agree_mask & (d >= 0), d.clamp(min=0), other)
    rows = torch.arange(k, device=device)[None, :]
    live = rows < nd[:, None]
    amp = torch.where(live, torch.full_like(col, 0, dtype=torch.float32) + peak,
                      torch.zeros_like(col, dtype=torch.float32))
    z[:, :k].scatter_add_(2, col[:, :, None], amp[:, :, None])
    bonus_tok = torch.randint(0, V, (B,), generator=g, device=device)
    z[torch.arange(B, device=device), nd, bonus_tok] += peak
    return z.to(dtype)


def workload_inputs(w: Workload | int, *, device="cpu", seed: int | None = None,
                    B: int | None = None) -> dict:
    """Inputs of one of the five workloads (optionally with a smaller batch ``B``)."""
    if isinstance(w, int):
        w = WORKLOADS[w]
    seed = SEED_BASE + w.index if seed is None else seed
    Bn = w.B if B is None else B
    e = w.extra
    if w.kind == "ngram+greedy":
        H, lens = histories(Bn, e["L"], w.V, seed=seed, copy_frac=e["copy_frac"],
                            span=e["span"])
        return dict(history=torch.from_numpy(H).to(device), hist_len=torch.from_numpy(lens).to(device),
                    B=Bn, k=w.k, V=w.V, L=e["L"], n_max=e["n_max"], n_min=e["n_min"],
                    agree=e["agree"], peak=e["peak"], seed=seed, dtype=w.dtype)
    d = sample_inputs(Bn, w.k, w.V, w.dtype, w.T, device=device, seed=seed,
                      target_std=e["target_std"], draft_noise=e["draft_noise"],
                      draft_scale=e["draft_scale"], zipf_s=e.get("zipf_s"), peak=e.get("peak"))
    if w.kind == "sample+gate":
        d["tau"] = e["tau"]
        d["answer_set"] = answer_set(w.V, e["n_answer"], device=device, seed=seed + 77)
    return d

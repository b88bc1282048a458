"""The greedy verify for callers that cannot allocate device memory.

Some callers cannot allocate device memory at all: an engine that has handed the whole
device to its own pool, or code on a path where cudaMalloc's implicit synchronisation is not
allowed. spec_verify_greedy_noalloc serves them from a fixed 8 MiB scratch array that lives
in the library itself. Here it is called through the C ABI and must give exactly what the
regular spec_verify_greedy gives, and what the CPU oracle gives, on two calls in a row with
different shapes (the second call must not see what the first left in the shared scratch),
and on a shape whose scratch need is just under the limit. Shapes just over the limit, and
calls with bad pointers, are refused on the host.

This file sorts last so that a run that stops at the first failure has already run every
other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import speculative_decoding_verification_17_gb300 as sv

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_UNSUPPORTED = 0, 1, 2
SCRATCH_BYTES = 8 << 20  # the library's fixed scratch array
FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: every call below returns on the host


def _noalloc(z, x, nd, stream):
    """One call of the allocation-free entry point through ctypes."""
    B, k1, V = z.shape
    k = k1 - 1
    code = sv.SV_F32 if z.dtype == torch.float32 else sv.SV_BF16
    tok = torch.full((B, k1), -7, dtype=torch.int32, device=z.device)
    acc = torch.full((B,), -7, dtype=torch.int32, device=z.device)
    P = ctypes.c_void_p
    status = sv.library().spec_verify_greedy_noalloc(
        P(z.data_ptr()), code, P(x.data_ptr()), None if nd is None else P(nd.data_ptr()), B, k, V,
        P(tok.data_ptr()), P(acc.data_ptr()), P(stream.cuda_stream))
    assert status == SV_OK, sv.library().sv_status_string(status)
    return tok, acc


def _case(B, k, V, dtype, seed, ragged):
    g = torch.Generator(device="cuda").manual_seed(seed)
    z = (torch.randn((B, k + 1, V), generator=g, device="cuda") * 3).to(dtype)
    am = torch.argmax(z.float(), -1)
    x = torch.where(torch.rand((B, k), generator=g, device="cuda") < 0.6, am[:, :k],
                    torch.randint(0, V, (B, k), generator=g, device="cuda")).to(torch.int32)
    nd = torch.randint(0, k + 1, (B,), generator=g, device="cuda", dtype=torch.int32) if ragged else None
    return z, x, nd


def _check(z, x, nd, tok, acc):
    """Equal to spec_verify_greedy (the workspace path) and to the CPU oracle."""
    ref_tok, ref_acc = sv.spec_verify_greedy(z, x, nd)
    torch.cuda.synchronize()
    assert torch.equal(acc, ref_acc)
    assert torch.equal(tok, ref_tok)
    o = oracle.spec_verify_greedy(z.cpu(), x.cpu(), None if nd is None else nd.cpu(), threads=8)
    assert np.array_equal(acc.cpu().numpy(), o["accept_len"])
    assert np.array_equal(tok.cpu().numpy(), o["tokens"])
    assert (acc >= 0).all()


def _largest_batch_within(k, V, code, limit):
    """The largest B whose greedy workspace fits in `limit` bytes (bisection on the query)."""
    lo, hi = 1, 1 << 24
    while sv.spec_verify_greedy_workspace(hi, k, V, code) <= limit:
        hi *= 2
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if sv.spec_verify_greedy_workspace(mid, k, V, code) <= limit:
            lo = mid
        else:
            hi = mid
    return lo


@pytest.mark.gpu
def test_noalloc_matches_greedy_and_oracle_on_two_calls_in_a_row():
    stream = torch.cuda.current_stream()
    for B, k, V, dtype, seed, ragged in [(64, 5, 32000, torch.bfloat16, 1, False),
                                         (37, 3, 40001, torch.float32, 2, True)]:
        z, x, nd = _case(B, k, V, dtype, seed, ragged)
        tok, acc = _noalloc(z, x, nd, stream)
        torch.cuda.synchronize()
        _check(z, x, nd, tok, acc)


@pytest.mark.gpu
def test_noalloc_just_under_its_scratch_limit():
    # short rows (k = 1, V = 64 bf16) so that the batch, not the logits, fills the scratch
    k, V = 1, 64
    B = _largest_batch_within(k, V, sv.SV_BF16, SCRATCH_BYTES)
    need = sv.spec_verify_greedy_workspace(B, k, V, sv.SV_BF16)
    assert SCRATCH_BYTES - 4096 < need <= SCRATCH_BYTES
    stream = torch.cuda.current_stream()
    z, x, nd = _case(B, k, V, torch.bfloat16, 3, True)
    for _ in range(2):  # twice in a row on the same scratch
        tok, acc = _noalloc(z, x, nd, stream)
        torch.cuda.synchronize()
        _check(z, x, nd, tok, acc)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # refused on the host before any CUDA call: no GPU needed, nothing is launched
    L = sv.library()
    k, V = 1, 64
    B = _largest_batch_within(k, V, sv.SV_BF16, SCRATCH_BYTES) + 1
    assert sv.spec_verify_greedy_workspace(B, k, V, sv.SV_BF16) > SCRATCH_BYTES
    assert L.spec_verify_greedy_noalloc(FAKE, sv.SV_BF16, FAKE, None, B, k, V, FAKE, FAKE,
                                        None) == SV_ERR_UNSUPPORTED
    assert L.spec_verify_greedy_noalloc(FAKE, sv.SV_F32, FAKE, None, 4096, 16, 1 << 20, FAKE,
                                        FAKE, None) == SV_ERR_UNSUPPORTED


def test_noalloc_checks_its_arguments_before_the_limit():
    # the same host checks, in the same order, as spec_verify_greedy: a bad pointer is an
    # invalid argument even on a shape the scratch could not hold
    L = sv.library()
    big = (4096, 16, 1 << 20)
    odd = ctypes.c_void_p(0x10001)
    assert L.spec_verify_greedy_noalloc(None, sv.SV_F32, FAKE, None, *big, FAKE, FAKE,
                                        None) == SV_ERR_INVALID_ARG
    assert L.spec_verify_greedy_noalloc(FAKE, sv.SV_F32, FAKE, None, *big, None, FAKE,
                                        None) == SV_ERR_INVALID_ARG
    assert L.spec_verify_greedy_noalloc(odd, sv.SV_F32, FAKE, None, *big, FAKE, FAKE,
                                        None) == SV_ERR_INVALID_ARG
    assert L.spec_verify_greedy_noalloc(FAKE, 7, FAKE, None, *big, FAKE, FAKE,
                                        None) == SV_ERR_INVALID_ARG
    assert L.spec_verify_greedy_noalloc(FAKE, sv.SV_F32, FAKE, None, 4, 17, 100, FAKE, FAKE,
                                        None) == SV_ERR_UNSUPPORTED
    assert L.spec_verify_greedy_noalloc(None, sv.SV_F32, None, None, 0, 4, 100, None, None,
                                        None) == SV_OK  # B = 0: a no-op

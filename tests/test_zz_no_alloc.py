"""The greedy verify for callers that cannot allocate device memory.

Some callers cannot allocate device memory at all: an engine that has handed the whole
device to its own pool, or code on a path where cudaMalloc's implicit synchronisation is not
allowed. spec_verify_greedy_noalloc serves them from a fixed scratch array that lives in the
library itself. Here it is called through the C ABI and must give exactly what the regular
spec_verify_greedy gives, on two calls in a row with different shapes (the second call must
not see what the first left in the shared scratch).

This file sorts last so that a run that stops at the first failure has already run every
other test; it also passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

import speculative_decoding_verification_17_gb300 as sv

SV_ERR_UNSUPPORTED = 2


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
    assert status == 0, sv.library().sv_status_string(status)
    return tok, acc


def _case(B, k, V, dtype, seed, ragged):
    g = torch.Generator(device="cuda").manual_seed(seed)
    z = (torch.randn((B, k + 1, V), generator=g, device="cuda") * 3).to(dtype)
    am = torch.argmax(z.float(), -1)
    x = torch.where(torch.rand((B, k), generator=g, device="cuda") < 0.6, am[:, :k],
                    torch.randint(0, V, (B, k), generator=g, device="cuda")).to(torch.int32)
    nd = torch.randint(0, k + 1, (B,), generator=g, device="cuda", dtype=torch.int32) if ragged else None
    return z, x, nd


@pytest.mark.gpu
def test_noalloc_matches_greedy_on_two_calls_in_a_row():
    stream = torch.cuda.current_stream()
    for B, k, V, dtype, seed, ragged in [(64, 5, 32000, torch.bfloat16, 1, False),
                                         (37, 3, 40001, torch.float32, 2, True)]:
        z, x, nd = _case(B, k, V, dtype, seed, ragged)
        tok, acc = _noalloc(z, x, nd, stream)
        ref_tok, ref_acc = sv.spec_verify_greedy(z, x, nd)
        torch.cuda.synchronize()
        assert torch.equal(acc, ref_acc), (B, k, V, dtype)
        assert torch.equal(tok, ref_tok), (B, k, V, dtype)
        assert (acc >= 0).all()


def test_noalloc_rejects_shapes_beyond_its_scratch():
    # rejected on the host before any CUDA call: no GPU needed, nothing is launched
    fake = ctypes.c_void_p(0x10000)
    status = sv.library().spec_verify_greedy_noalloc(fake, sv.SV_F32, fake, None, 4096, 16, 1 << 20,
                                                     fake, fake, None)
    assert status == SV_ERR_UNSUPPORTED

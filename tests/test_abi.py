"""The C-ABI library loads, exports every function include/*.h declares, and validates its
arguments on the host (no GPU needed: every call here returns before any CUDA call)."""
import ctypes
import glob
import os
import re

import pytest

import speculative_decoding_verification_17_gb300 as sv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, WORKSPACE = 0, 1, 2, 3
FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: validation fails or returns first


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b([A-Za-z_]\w*)\s*\(([^;{}()]|\([^()]*\))*\)\s*;", text):
            if m.group(1) not in ("sizeof",):
                names.add(m.group(1))
    return names


def test_every_declared_function_is_exported():
    L = sv.library()
    names = declared_functions()
    assert {"spec_verify_sample", "spec_verify_greedy", "logit_gap_gate", "ngram_propose"} <= names
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"


def test_version_and_status_strings():
    L = sv.library()
    assert L.sv_version() > 0
    for s in range(6):
        assert L.sv_status_string(s)
    assert L.sv_last_cuda_error() == 0


def test_workspace_queries():
    assert sv.spec_verify_sample_workspace(512, 8, 128256, sv.SV_BF16) > 0
    assert sv.spec_verify_sample_workspace(1, 17, 100, sv.SV_F32) == 0
    # the clear of the counters and the verify, plus draw_kernel for rows of 8 to 32 chunks
    assert sv.spec_verify_sample_launches(512, 8, 128256, sv.SV_BF16) == 3
    assert sv.spec_verify_sample_launches(64, 5, 32000, sv.SV_BF16) == 2
    assert sv.spec_verify_sample_launches(256, 4, 151936, sv.SV_F32) == 3
    assert sv.spec_verify_sample_launches(1, 4, 1000, sv.SV_F32) == 2
    assert sv.spec_verify_sample_launches(0, 4, 1000, sv.SV_F32) == 0
    assert sv.spec_verify_sample_launches(4, 2, 600000, sv.SV_BF16) == 2  # 37 chunks
    assert sv.spec_verify_greedy_workspace(128, 5, 32000, sv.SV_BF16) > 0
    assert sv.logit_gap_gate_workspace(1280, 151936, sv.SV_F32) > 0
    for q in (sv.spec_verify_sample_workspace(0, 4, 1000, 0),
              sv.spec_verify_greedy_workspace(0, 4, 1000, 0), sv.logit_gap_gate_workspace(0, 10, 0)):
        assert q >= 0
    assert sv.spec_verify_sample_workspace(1, 4, 1, 0) == 0  # V < 2


def _sample(**kw):
    a = dict(t=FAKE, d=FAKE, dtype=0, x=FAKE, nd=None, u=FAKE, B=4, k=3, V=100, T=1.0, ot=FAKE,
             oa=FAKE, op=None, oq=None, orm=None, ws=ctypes.c_void_p(0x100000), wsb=1 << 30,
             st=None)
    a.update(kw)
    return sv.library().spec_verify_sample(a["t"], a["d"], a["dtype"], a["x"], a["nd"], a["u"],
                                           a["B"], a["k"], a["V"], a["T"], a["ot"], a["oa"],
                                           a["op"], a["oq"], a["orm"], a["ws"], a["wsb"], a["st"])


@pytest.mark.parametrize("kw,status", [
    (dict(B=-1), INVALID), (dict(k=0), INVALID), (dict(V=1), INVALID), (dict(dtype=7), INVALID),
    (dict(T=0.0), INVALID), (dict(T=-1.0), INVALID), (dict(T=float("nan")), INVALID),
    (dict(T=float("inf")), INVALID), (dict(T=1e-5), INVALID), (dict(k=17), UNSUPPORTED),
    (dict(t=None), INVALID), (dict(x=None), INVALID), (dict(u=None), INVALID),
    (dict(ot=None), INVALID), (dict(t=ctypes.c_void_p(0x10001)), INVALID),
    (dict(ws=None), WORKSPACE), (dict(wsb=16), WORKSPACE), (dict(ws=ctypes.c_void_p(0x100010)), WORKSPACE),
    (dict(B=0, t=None, d=None), OK),
])
def test_sample_validation(kw, status):
    assert _sample(**kw) == status


def test_greedy_gate_ngram_validation():
    L = sv.library()
    ws = ctypes.c_void_p(0x100000)
    g = lambda **kw: L.spec_verify_greedy(kw.get("t", FAKE), kw.get("dtype", 1), FAKE, None,
                                          kw.get("B", 2), kw.get("k", 3), kw.get("V", 50), FAKE,
                                          FAKE, kw.get("ws", ws), kw.get("wsb", 1 << 30), None)
    assert g(B=-1) == INVALID and g(k=0) == INVALID and g(V=1) == INVALID
    assert g(k=17) == UNSUPPORTED and g(t=None) == INVALID and g(wsb=0) == WORKSPACE
    assert g(B=0, t=None) == OK
    gt = lambda **kw: L.logit_gap_gate(kw.get("z", FAKE), kw.get("dtype", 0), kw.get("N", 3),
                                       kw.get("V", 10), 1.0, kw.get("A", FAKE), kw.get("nA", 2),
                                       FAKE, FAKE, FAKE, kw.get("ws", ws), kw.get("wsb", 1 << 30),
                                       None)
    assert gt(N=-1) == INVALID and gt(V=1) == INVALID and gt(nA=-1) == INVALID
    assert gt(A=None) == INVALID and gt(z=None) == INVALID and gt(wsb=8) == WORKSPACE
    assert gt(N=0, z=None) == OK
    ng = lambda **kw: L.ngram_propose(kw.get("h", FAKE), FAKE, kw.get("B", 2), kw.get("L", 64),
                                      kw.get("nmax", 4), kw.get("nmin", 2), kw.get("k", 5),
                                      FAKE, FAKE, None)
    assert ng(nmin=0) == INVALID and ng(nmax=1, nmin=2) == INVALID and ng(nmax=65) == INVALID
    assert ng(k=0) == INVALID and ng(k=65) == INVALID and ng(L=0) == INVALID
    assert ng(L=1 << 24) == INVALID and ng(h=None) == INVALID and ng(B=-1) == INVALID
    assert ng(B=0, h=None) == OK


def test_confidence_stop_validation():
    L = sv.library()
    ws = ctypes.c_void_p(0x100000)
    dc = lambda **kw: L.draft_confidence_stop(
        kw.get("z", FAKE), kw.get("dtype", 1), None, kw.get("B", 4), kw.get("k", 5),
        kw.get("V", 1000), kw.get("T", 1.0), kw.get("mode", 0), kw.get("floor", 0.5),
        kw.get("out", FAKE), None, kw.get("ws", ws), kw.get("wsb", 1 << 30), None)
    assert dc(B=-1) == INVALID and dc(k=0) == INVALID and dc(V=1) == INVALID
    assert dc(dtype=7) == INVALID and dc(T=0.0) == INVALID and dc(mode=2) == INVALID
    assert dc(floor=float("nan")) == INVALID and dc(floor=float("inf")) == INVALID
    assert dc(k=17) == UNSUPPORTED and dc(z=None) == INVALID and dc(out=None) == INVALID
    assert dc(wsb=8) == WORKSPACE and dc(ws=None) == WORKSPACE
    assert dc(B=0, z=None) == OK
    assert L.draft_confidence_workspace(4, 5, 1000, 1) > 0
    assert L.draft_confidence_workspace(4, 17, 1000, 1) == 0


def test_calibration_validation():
    L = sv.library()
    ws = ctypes.c_void_p(0x100000)
    rc = lambda **kw: L.gate_risk_coverage(
        FAKE, FAKE, FAKE, kw.get("N", 10), kw.get("A", FAKE), kw.get("nA", 3),
        kw.get("taus", FAKE), kw.get("T", 5), kw.get("z", 1.96), 0.1, kw.get("out", FAKE), FAKE,
        kw.get("ws", ws), kw.get("wsb", 1 << 30), None)
    assert rc(N=-1) == INVALID and rc(T=0) == INVALID and rc(nA=-1) == INVALID
    assert rc(T=4097) == UNSUPPORTED and rc(z=float("nan")) == INVALID and rc(z=-1.0) == INVALID
    assert rc(taus=None) == INVALID and rc(out=None) == INVALID and rc(A=None) == INVALID
    assert rc(wsb=16) == WORKSPACE and rc(ws=None) == WORKSPACE
    assert L.gate_risk_coverage_workspace(10, 5) > 0
    assert L.gate_risk_coverage_workspace(10, 4097) == 0

    cr = lambda **kw: L.conformal_residual(kw.get("a", FAKE), kw.get("b", FAKE),
                                           kw.get("dtype", 1), kw.get("N", 4), kw.get("V", 100),
                                           kw.get("out", FAKE), None)
    assert cr(N=-1) == INVALID and cr(V=0) == INVALID and cr(dtype=3) == INVALID
    assert cr(a=None) == INVALID and cr(out=None) == INVALID
    assert cr(N=0, a=None) == OK
    assert cr(a=ctypes.c_void_p(0x10001)) == INVALID  # misaligned for bf16

    cq = lambda **kw: L.conformal_quantile(kw.get("r", FAKE), kw.get("n", 10), kw.get("q", 0.9),
                                           kw.get("out", FAKE), kw.get("ws", ws),
                                           kw.get("wsb", 1 << 30), None)
    assert cq(n=0) == INVALID and cq(q=0.0) == INVALID and cq(q=1.5) == INVALID
    assert cq(q=float("nan")) == INVALID and cq(r=None) == INVALID and cq(out=None) == INVALID
    assert cq(wsb=64) == WORKSPACE
    assert L.conformal_quantile_workspace(0) == 0 and L.conformal_quantile_workspace(5) > 0

    bs = lambda **kw: L.conformal_quantile_barrier_selftest(
        kw.get("r", FAKE), kw.get("n", 10000), kw.get("out", FAKE), kw.get("ws", ws),
        kw.get("wsb", 1 << 30), kw.get("us", 1000), None)
    assert bs(n=8192) == INVALID and bs(us=0) == INVALID and bs(us=100001) == INVALID
    assert bs(r=None) == INVALID and bs(out=None) == INVALID and bs(wsb=64) == WORKSPACE
    assert bs(r=ctypes.c_void_p(0x10002)) == INVALID

    ca = lambda **kw: L.conformal_admit(kw.get("z", FAKE), kw.get("dtype", 1), kw.get("N", 3),
                                        kw.get("K", 2), kw.get("V", 50), kw.get("Q", FAKE),
                                        kw.get("lay", FAKE), FAKE, None, kw.get("ws", ws),
                                        kw.get("wsb", 1 << 30), None)
    assert ca(N=-1) == INVALID and ca(K=0) == INVALID and ca(V=1) == INVALID
    assert ca(Q=None) == INVALID and ca(lay=None) == INVALID and ca(z=None) == INVALID
    assert ca(wsb=16) == WORKSPACE and ca(N=0, z=None) == OK
    assert L.conformal_admit_workspace(3, 0, 50, 1) == 0


def test_ready_cache_validation():
    L = sv.library()
    ws = ctypes.c_void_p(0x100000)
    SL = ctypes.c_void_p(0x200000)  # 32-byte aligned
    rec = lambda **kw: L.ready_cache_record(
        kw.get("slots", SL), kw.get("store", FAKE), kw.get("S", 8), kw.get("E", 4),
        kw.get("stats", FAKE), FAKE, FAKE, FAKE, FAKE, FAKE, kw.get("M", 3), kw.get("z", FAKE),
        kw.get("dtype", 1), kw.get("V", 100), None, None, kw.get("ws", ws),
        kw.get("wsb", 1 << 30), None)
    assert rec(M=-1) == INVALID and rec(V=1) == INVALID and rec(dtype=5) == INVALID
    assert rec(S=0) == INVALID and rec(E=0) == INVALID and rec(E=5000) == INVALID
    assert rec(slots=None) == INVALID and rec(slots=ctypes.c_void_p(0x200010)) == INVALID
    assert rec(z=None) == INVALID and rec(wsb=8) == WORKSPACE and rec(M=0, z=None) == OK
    srv = lambda **kw: L.ready_cache_serve(
        SL, FAKE, kw.get("S", 8), 4, FAKE, FAKE, FAKE, FAKE, FAKE, kw.get("R", 5), 1.0,
        kw.get("A", None), kw.get("nA", 0), 1, kw.get("out", FAKE), FAKE, None)
    assert srv(R=-1) == INVALID and srv(S=0) == INVALID and srv(nA=2) == INVALID
    assert srv(out=None) == INVALID and srv(R=0, out=None) == OK
    inv = lambda **kw: L.ready_cache_invalidate(SL, kw.get("S", 8), FAKE, kw.get("sess", FAKE),
                                                kw.get("n", 2), None)
    assert inv(n=-1) == INVALID and inv(S=0) == INVALID and inv(sess=None) == INVALID
    assert inv(n=0, sess=None) == OK
    assert L.ready_cache_record_workspace(4, 1000, 1) > 0
    assert L.ready_cache_record_workspace(4, 1, 1) == 0


def test_binding_raises_on_bad_input():
    import torch

    with pytest.raises((TypeError, ValueError)):
        sv.spec_verify_greedy(torch.zeros(2, 3, 10), torch.zeros(2, 2, dtype=torch.int32))


def test_product_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "speculative_decoding_verification_17_gb300")
    for path in glob.glob(os.path.join(pkg, "**", "*.*"), recursive=True):
        if path.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
            text = open(path).read()
            assert "oracle" not in text.lower(), path

"""Plain fp64 CPU oracle of the speculative-decoding verify step.

TEST INFRASTRUCTURE ONLY. The tests, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg are its only callers. The product library never imports, links or runs
anything here, and the two share no code: the arithmetic lives in ``oracle.c`` (plain C,
double precision, ascending-order sums), this module only builds it and marshals numpy
arrays through ``ctypes``. ``ready_cache.py`` holds the ready-distribution cache as a plain
sequential Python state machine over those functions.

Logit arrays are numpy ``float32`` (dtype code 0) or ``uint16`` holding raw bfloat16 bit
patterns (dtype code 1); :func:`as_logits` converts torch CPU tensors.

Parity pins of each function (what fixes it other than itself) are in ``tests/test_oracle_*.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from contextlib import contextmanager

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_SRC = os.path.join(_HERE, "oracle.c")
_lock = threading.Lock()
_lib = None

TIE_MARGIN = 1e-6


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``_build/liboracle.so`` (gcc, -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "oracle.h"))
    ):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    subprocess.run(
        ["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"],
        check=True,
    )
    os.replace(tmp, _SO)
    return _SO


def _bind(lib):
    P = ctypes.c_void_p
    I = ctypes.c_int
    D = ctypes.c_double
    lib.oracle_row_softmax.argtypes = [P, I, I, D, P]
    lib.oracle_spec_verify_sample.argtypes = [P, P, I, P, P, P, I, I, I, D,
                                              P, P, P, P, P, P, P, P, P, P, I, I]
    lib.oracle_spec_verify_greedy.argtypes = [P, I, P, P, I, I, I, P, P, I, I]
    lib.oracle_logit_gap_gate.argtypes = [P, I, I, I, D, P, I, P, P, P, P, I, I]
    lib.oracle_ngram_propose.argtypes = [P, P, I, I, I, I, I, P, P, I, I]
    lib.oracle_draft_confidence.argtypes = [P, I, P, I, I, I, D, I, D, P, P, P, I, I]
    lib.oracle_wilson.argtypes = [ctypes.c_int64, ctypes.c_int64, D, P, P]
    lib.oracle_wilson.restype = None
    lib.oracle_risk_coverage.argtypes = [P, P, P, I, P, I, P, I, D, D, P, P, P, P]
    lib.oracle_conformal_residual.argtypes = [P, P, I, I, I, P, I, I]
    lib.oracle_conformal_quantile.argtypes = [P, I, D, P]
    lib.oracle_conformal_admit.argtypes = [P, I, I, I, I, P, P, P, P, P, I, I]
    for f in (lib.oracle_row_softmax, lib.oracle_spec_verify_sample,
              lib.oracle_spec_verify_greedy, lib.oracle_logit_gap_gate,
              lib.oracle_ngram_propose, lib.oracle_draft_confidence,
              lib.oracle_risk_coverage, lib.oracle_conformal_residual,
              lib.oracle_conformal_quantile, lib.oracle_conformal_admit):
        f.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


@contextmanager
def library(path: str):
    """Route every call through another build of ``oracle.c`` while the block runs.

    The mutation tests use it to show that the pins fail when a mistake is planted in the
    oracle. Not thread-safe; tests only.
    """
    global _lib
    _load()
    old = _lib
    _lib = _bind(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib = old


def compile_variant(src_text: str, out_path: str) -> str:
    """Compile an edited copy of ``oracle.c`` to ``out_path`` (mutation tests only)."""
    d = os.path.dirname(out_path)
    os.makedirs(d, exist_ok=True)
    c_path = out_path + ".c"
    with open(c_path, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-I", _HERE, c_path, "-o",
                    out_path, "-lm"], check=True)
    return out_path


def source() -> str:
    with open(_SRC) as f:
        return f.read()


def as_logits(x):
    """(contiguous numpy array, dtype code) from a numpy array or a torch CPU tensor."""
    try:
        import torch

        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), 1
            if x.dtype == torch.float32:
                return x.numpy(), 0
            raise TypeError(f"unsupported logit dtype {x.dtype}")
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, 0
    if x.dtype == np.uint16:
        return x, 1
    raise TypeError(f"unsupported logit dtype {x.dtype}")


def _i32(x):
    if x is None:
        return None
    try:
        import torch

        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x, dtype=np.int32)


def _f32(x):
    try:
        import torch

        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(x, dtype=np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _ranges(items, threads):
    """Split a sorted list of indices into (r0, r1) runs, grouped for ``threads`` workers."""
    runs = []
    start = prev = None
    for r in items:
        if start is None:
            start = prev = r
        elif r == prev + 1:
            prev = r
        else:
            runs.append((start, prev + 1))
            start = prev = r
    if start is not None:
        runs.append((start, prev + 1))
    # split long runs so every worker gets work
    if threads > 1:
        total = sum(b - a for a, b in runs)
        piece = max(1, total // (threads * 4))
        out = []
        for a, b in runs:
            while b - a > piece:
                out.append((a, a + piece))
                a += piece
            out.append((a, b))
        runs = out
    return runs


def _run(fn, runs, threads):
    if threads <= 1 or len(runs) <= 1:
        for a, b in runs:
            rc = fn(a, b)
            if rc != 0:
                raise ValueError(f"oracle rejected the arguments (code {rc})")
        return
    with ThreadPoolExecutor(max_workers=threads) as ex:
        for rc in ex.map(lambda ab: fn(*ab), runs):
            if rc != 0:
                raise ValueError(f"oracle rejected the arguments (code {rc})")


def row_softmax(row, T: float) -> np.ndarray | None:
    """softmax(row / T) in double, or None when the row is not a distribution."""
    z, code = as_logits(row)
    z = z.reshape(-1)
    out = np.empty(z.size, dtype=np.float64)
    rc = _load().oracle_row_softmax(_ptr(z), code, z.size, float(T), _ptr(out))
    if rc == -1:
        return None
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out


def spec_verify_sample(target, draft, draft_tokens, num_draft, uniforms, T: float,
                       requests=None, threads: int = 1) -> dict:
    """Sampled verify over the requests listed in ``requests`` (default: all).

    Returns full-batch arrays; rows of requests not listed are left at -2 / NaN.
    """
    tz, code = as_logits(target)
    dz, code2 = as_logits(draft)
    assert code == code2, "target and draft logits must share a dtype"
    B, k1, V = tz.shape
    k = k1 - 1
    assert dz.shape == (B, k, V)
    x = _i32(draft_tokens)
    nd = _i32(num_draft)
    u = _f32(uniforms)
    assert x.shape == (B, k) and u.shape == (B, k + 1)
    out = dict(
        tokens=np.full((B, k + 1), -2, np.int32),
        accept_len=np.full(B, -2, np.int32),
        p=np.full((B, k), np.nan),
        q=np.full((B, k), np.nan),
        resid=np.full(B, np.nan),
        flag_pos=np.full(B, -2, np.int32),
        margin=np.full(B, np.nan),
        t_lo=np.full(B, -2, np.int32),
        t_hi=np.full(B, -2, np.int32),
        tie_prob=np.full(B, np.nan),
    )
    lib = _load()
    reqs = sorted(range(B) if requests is None else {int(r) for r in requests})

    def fn(a, b):
        return lib.oracle_spec_verify_sample(
            _ptr(tz), _ptr(dz), code, _ptr(x), _ptr(nd), _ptr(u), B, k, V, float(T),
            _ptr(out["tokens"]), _ptr(out["accept_len"]), _ptr(out["p"]), _ptr(out["q"]),
            _ptr(out["resid"]), _ptr(out["flag_pos"]), _ptr(out["margin"]), _ptr(out["t_lo"]),
            _ptr(out["t_hi"]), _ptr(out["tie_prob"]), a, b)

    _run(fn, _ranges(reqs, threads), threads)
    return out


def spec_verify_greedy(target, draft_tokens, num_draft, requests=None, threads: int = 1) -> dict:
    tz, code = as_logits(target)
    B, k1, V = tz.shape
    k = k1 - 1
    x = _i32(draft_tokens)
    nd = _i32(num_draft)
    assert x.shape == (B, k)
    out = dict(tokens=np.full((B, k + 1), -2, np.int32), accept_len=np.full(B, -2, np.int32))
    lib = _load()
    reqs = sorted(range(B) if requests is None else {int(r) for r in requests})

    def fn(a, b):
        return lib.oracle_spec_verify_greedy(_ptr(tz), code, _ptr(x), _ptr(nd), B, k, V,
                                             _ptr(out["tokens"]), _ptr(out["accept_len"]), a, b)

    _run(fn, _ranges(reqs, threads), threads)
    return out


def logit_gap_gate(logits, tau: float, answer_set, rows=None, threads: int = 1) -> dict:
    z, code = as_logits(logits)
    z = z.reshape(-1, z.shape[-1])
    N, V = z.shape
    A = _i32(answer_set if answer_set is not None else np.zeros(0, np.int32)).reshape(-1)
    out = dict(token=np.full(N, -2, np.int32), gap=np.full(N, np.nan),
               fire=np.zeros(N, np.uint8), flag=np.zeros(N, np.uint8))
    lib = _load()
    idx = sorted(range(N) if rows is None else {int(r) for r in rows})

    def fn(a, b):
        return lib.oracle_logit_gap_gate(_ptr(z), code, N, V, float(tau), _ptr(A), A.size,
                                         _ptr(out["token"]), _ptr(out["gap"]), _ptr(out["fire"]),
                                         _ptr(out["flag"]), a, b)

    _run(fn, _ranges(idx, threads), threads)
    return out


CONF_TOP_PROB = 0
CONF_INV_ENTROPY = 1


def draft_confidence(draft, num_draft, T: float, mode: int, floor: float, requests=None,
                     threads: int = 1) -> dict:
    """Draft-side confidence c[B, k] and the variable-length stop num_draft[B] (see
    oracle.h); flag[B] is the first near-tie position up to the stop, or -1."""
    z, code = as_logits(draft)
    B, k, V = z.shape
    nd = _i32(num_draft)
    out = dict(num_draft=np.full(B, -2, np.int32), conf=np.full((B, k), np.nan),
               flag=np.full(B, -2, np.int32))
    lib = _load()
    reqs = sorted(range(B) if requests is None else {int(r) for r in requests})

    def fn(a, b):
        return lib.oracle_draft_confidence(_ptr(z), code, _ptr(nd), B, k, V, float(T),
                                           int(mode), float(floor), _ptr(out["num_draft"]),
                                           _ptr(out["conf"]), _ptr(out["flag"]), a, b)

    _run(fn, _ranges(reqs, threads), threads)
    return out


def ngram_propose(history, hist_len, n_max: int, n_min: int, k: int, requests=None,
                  threads: int = 1) -> dict:
    h = _i32(history)
    B, L_max = h.shape
    hl = _i32(hist_len).reshape(-1)
    assert hl.size == B
    out = dict(draft=np.full((B, k), -2, np.int32), num_draft=np.full(B, -2, np.int32))
    lib = _load()
    reqs = sorted(range(B) if requests is None else {int(r) for r in requests})

    def fn(a, b):
        return lib.oracle_ngram_propose(_ptr(h), _ptr(hl), B, L_max, n_max, n_min, k,
                                        _ptr(out["draft"]), _ptr(out["num_draft"]), a, b)

    _run(fn, _ranges(reqs, threads), threads)
    return out


# ------------------------------------------------------------------------ gate calibration
def wilson(k: int, n: int, z: float = 1.959963984540054) -> tuple[float, float]:
    """Wilson score interval of k successes in n trials (see oracle.h)."""
    lo, hi = ctypes.c_double(), ctypes.c_double()
    _load().oracle_wilson(int(k), int(n), float(z), ctypes.byref(lo), ctypes.byref(hi))
    return lo.value, hi.value


def risk_coverage(gap, token, full_token, answer_set, taus, z: float = 1.959963984540054,
                  r_max: float = 0.0) -> dict:
    """Coverage c(tau) and false-accept risk r(tau) with Wilson intervals over a threshold
    grid, and the index of the smallest tau with r <= r_max (-1 if none)."""
    g = _f32(gap).reshape(-1)
    t = _i32(token).reshape(-1)
    f = _i32(full_token).reshape(-1)
    A = _i32(answer_set if answer_set is not None else np.zeros(0, np.int32)).reshape(-1)
    tau = _f32(taus).reshape(-1)
    N, T = g.size, tau.size
    assert t.size == N and f.size == N
    acc = np.zeros(T, np.int64)
    bad = np.zeros(T, np.int64)
    st = np.zeros((T, 6), np.float64)
    idx = ctypes.c_int32(-3)
    rc = _load().oracle_risk_coverage(_ptr(g), _ptr(t), _ptr(f), N, _ptr(A), A.size, _ptr(tau),
                                      T, float(z), float(r_max), _ptr(acc), _ptr(bad), _ptr(st),
                                      ctypes.byref(idx))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return dict(accepted=acc, wrong=bad, coverage=st[:, 0], cov_lo=st[:, 1], cov_hi=st[:, 2],
                risk=st[:, 3], risk_lo=st[:, 4], risk_hi=st[:, 5], tau_index=idx.value)


def conformal_residual(draft, truth, rows=None, threads: int = 1) -> np.ndarray:
    """Sup-norm residual of each draft row against the true row, fp32 [N] (see oracle.h)."""
    a, code = as_logits(draft)
    b, code_b = as_logits(truth)
    assert code == code_b and a.shape == b.shape
    a = a.reshape(-1, a.shape[-1])
    b = b.reshape(-1, b.shape[-1])
    N, V = a.shape
    out = np.full(N, np.nan, np.float32)
    lib = _load()
    idx = sorted(range(N) if rows is None else {int(r) for r in rows})

    def fn(i0, i1):
        return lib.oracle_conformal_residual(_ptr(a), _ptr(b), code, N, V, _ptr(out), i0, i1)

    _run(fn, _ranges(idx, threads), threads)
    return out


def conformal_quantile(r, q: float) -> np.float32:
    """The ceil((n+1) q)-th smallest residual, +inf past n (see oracle.h)."""
    x = _f32(r).reshape(-1)
    out = np.zeros(1, np.float32)
    rc = _load().oracle_conformal_quantile(_ptr(x), x.size, float(q), _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (code {rc})")
    return out[0]


def conformal_admit(logits, Q, steps=None, threads: int = 1) -> dict:
    """Earliest layer whose 2 Q[k] <= gamma over logits [N, K, V] (see oracle.h)."""
    z, code = as_logits(logits)
    N, K, V = z.shape
    q = _f32(Q).reshape(-1)
    assert q.size == K
    out = dict(layer=np.full(N, -2, np.int32), token=np.full(N, -2, np.int32),
               gap=np.full((N, K), np.nan), flag=np.full(N, -2, np.int32))
    lib = _load()
    idx = sorted(range(N) if steps is None else {int(r) for r in steps})

    def fn(a, b):
        return lib.oracle_conformal_admit(_ptr(z), code, N, K, V, _ptr(q), _ptr(out["layer"]),
                                          _ptr(out["token"]), _ptr(out["gap"]),
                                          _ptr(out["flag"]), a, b)

    _run(fn, _ranges(idx, threads), threads)
    return out

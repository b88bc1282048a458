"""GB300-native speculative-decoding verify step.

A thin Python binding over ``libspecverify.so`` (C ABI declared in
``include/specverify.h``). Every function here only checks and marshals arguments: the
work runs in the library's sm_103a kernels on the caller's CUDA stream. Tensors are torch
CUDA tensors (PyTorch provides device memory and streams); the binding never computes a
result itself and raises :class:`SVError` on any non-OK status.

Calls (same names as the C ABI):

- :func:`spec_verify_sample` — modified-rejection verify with residual/bonus draw.
- :func:`spec_verify_greedy` — greedy (temperature-0) verify.
- :func:`spec_verify_greedy_noalloc` — the same without a workspace (fixed library scratch).
- :func:`logit_gap_gate`     — top-1/top-2 logit-gap confidence gate.
- :func:`draft_confidence_stop` — variable-length drafting: the first draft position whose
  top probability (or inverse entropy) is below a floor.
- :func:`ngram_propose`      — prompt-lookup n-gram draft proposer.

Gate calibration and the conformal gate (C ABI in ``include/specverify_calib.h``):

- :func:`gate_risk_coverage` — coverage and false-accept risk of the gate over a threshold
  grid, with Wilson intervals, and the smallest threshold within a risk budget.
- :func:`conformal_residual` — sup-norm distance of draft rows from the true rows.
- :func:`conformal_quantile` — the split-conformal quantile of those residuals.
- :func:`conformal_admit`    — the earliest of K layers whose gap clears 2 Q.

Ready-distribution cache (C ABI in ``include/specverify_cache.h``), through
:class:`ReadyCacheTable`, which owns a device-resident table of session slots:

- :meth:`ReadyCacheTable.record`     — pre-position on idle for a batch of sessions.
- :meth:`ReadyCacheTable.serve`      — the confidence-gated fast path for a batch of requests.
- :meth:`ReadyCacheTable.invalidate` — a mutation of the listed sessions' state.

Workspaces: pass ``workspace=`` (a uint8 CUDA tensor of at least the size the matching
``*_workspace`` query returns, 256-byte aligned, not shared by calls in flight at the same
time; it needs no initialisation), or let the binding keep one cached per (device, stream,
call) that it grows as needed: calls in flight on different streams never share one.
"""
from __future__ import annotations

import ctypes
import threading

import torch

from . import _native

__all__ = [
    "SVError", "SV_F32", "SV_BF16", "SV_MAX_K", "build", "library", "version",
    "spec_verify_sample_workspace", "spec_verify_sample_launches", "spec_verify_sample",
    "spec_verify_greedy_workspace", "spec_verify_greedy", "spec_verify_greedy_noalloc",
    "logit_gap_gate_workspace", "logit_gap_gate", "ngram_propose",
    "SV_CONF_TOP_PROB", "SV_CONF_INV_ENTROPY", "draft_confidence_workspace",
    "draft_confidence_stop", "SV_MAX_TAUS", "CALIB_POINT", "gate_risk_coverage_workspace",
    "gate_risk_coverage", "conformal_residual", "conformal_quantile_workspace",
    "conformal_quantile", "conformal_admit_workspace", "conformal_admit", "gate_points_dict",
    "ReadyCacheTable", "ready_cache_record_workspace", "SV_CACHE_VALID", "SV_CACHE_DECODED",
    "SV_CACHE_CONSUMED", "CACHE_STATS",
]

SV_F32 = 0
SV_BF16 = 1
SV_MAX_K = 16
SV_CONF_TOP_PROB = 0
SV_CONF_INV_ENTROPY = 1
SV_MAX_TAUS = 4096
# sv_calib_point as a row of 8 float64-sized fields: the two counts are int64, the six rates
# float64 (view the int64 columns with .view(torch.int64)).
CALIB_POINT = ("accepted", "wrong", "coverage", "cov_lo", "cov_hi", "risk", "risk_lo",
               "risk_hi")

_STATUS = {0: "SV_OK", 1: "SV_ERR_INVALID_ARG", 2: "SV_ERR_UNSUPPORTED", 3: "SV_ERR_WORKSPACE",
           4: "SV_ERR_CUDA", 5: "SV_ERR_TIMEOUT"}


class SVError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        L = _native.lib()
        msg = f"{where}: {_STATUS.get(status, status)} ({L.sv_status_string(status).decode()})"
        if status == 4:
            msg += f", cudaError {L.sv_last_cuda_error()}"
        super().__init__(msg)


def build(force: bool = False, verbose: bool = False) -> str:
    return _native.build(force=force, verbose=verbose)


def library():
    return _native.lib()


def version() -> int:
    return library().sv_version()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SV_F32
    if t.dtype == torch.bfloat16:
        return SV_BF16
    raise TypeError(f"logits must be float32 or bfloat16, got {t.dtype}")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _check_cuda(name, t, dtype=None, shape=None, device=None):
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream), stream


_ws_lock = threading.Lock()
_ws_cache: dict = {}


def _workspace(kind: str, nbytes: int, device, stream):
    """Cached zero-filled workspace for (device, stream, kind) of at least ``nbytes`` bytes.
    Calls on one stream run in order, so they may share it; calls on two streams may overlap,
    so each stream has its own."""
    key = (kind, device, stream.cuda_stream)
    with _ws_lock:
        ws = _ws_cache.get(key)
        if ws is None or ws.numel() < nbytes:
            with torch.cuda.stream(stream):
                ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
            _ws_cache[key] = ws
    return ws


def _ok(status, where):
    if status != 0:
        raise SVError(status, where)


# ------------------------------------------------------------------------------ sampled
def spec_verify_sample_workspace(B: int, k: int, V: int, dtype: int) -> int:
    return int(library().spec_verify_sample_workspace(B, k, V, dtype))


def spec_verify_sample_launches(B: int, k: int, V: int, dtype: int) -> int:
    return int(library().spec_verify_sample_launches(B, k, V, dtype))


def spec_verify_sample(target_logits, draft_logits, draft_tokens, uniforms, temperature: float,
                       num_draft=None, *, out_tokens=None, out_accept_len=None,
                       out_p_draft=None, out_q_draft=None, out_resid_mass=None,
                       want_probs: bool = True, workspace=None, stream=None):
    """Sampled verify. Returns (tokens [B,k+1], accept_len [B], p_draft [B,k] | None,
    q_draft [B,k] | None, resid_mass [B] | None)."""
    B, k1, V = target_logits.shape
    k = k1 - 1
    dev = target_logits.device
    code = _dtype_code(target_logits)
    _check_cuda("target_logits", target_logits)
    _check_cuda("draft_logits", draft_logits, target_logits.dtype, (B, k, V), dev)
    _check_cuda("draft_tokens", draft_tokens, torch.int32, (B, k), dev)
    _check_cuda("uniforms", uniforms, torch.float32, (B, k + 1), dev)
    _check_cuda("num_draft", num_draft, torch.int32, (B,), dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    if out_accept_len is None:
        out_accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
    if want_probs:
        if out_p_draft is None:
            out_p_draft = torch.empty((B, k), dtype=torch.float32, device=dev)
        if out_q_draft is None:
            out_q_draft = torch.empty((B, k), dtype=torch.float32, device=dev)
        if out_resid_mass is None:
            out_resid_mass = torch.empty((B,), dtype=torch.float32, device=dev)
    _check_cuda("out_tokens", out_tokens, torch.int32, (B, k + 1), dev)
    _check_cuda("out_accept_len", out_accept_len, torch.int32, (B,), dev)
    _check_cuda("out_p_draft", out_p_draft, torch.float32, (B, k), dev)
    _check_cuda("out_q_draft", out_q_draft, torch.float32, (B, k), dev)
    _check_cuda("out_resid_mass", out_resid_mass, torch.float32, (B,), dev)
    h, st = _stream_handle(stream)
    need = spec_verify_sample_workspace(B, k, V, code)
    ws = workspace if workspace is not None else _workspace("sample", need, dev, st)
    _ok(library().spec_verify_sample(
        _ptr(target_logits), _ptr(draft_logits), code, _ptr(draft_tokens), _ptr(num_draft),
        _ptr(uniforms), B, k, V, float(temperature), _ptr(out_tokens), _ptr(out_accept_len),
        _ptr(out_p_draft), _ptr(out_q_draft), _ptr(out_resid_mass), _ptr(ws), ws.numel(), h),
        "spec_verify_sample")
    return out_tokens, out_accept_len, out_p_draft, out_q_draft, out_resid_mass


# ------------------------------------------------------------------------------ greedy
def spec_verify_greedy_workspace(B: int, k: int, V: int, dtype: int) -> int:
    return int(library().spec_verify_greedy_workspace(B, k, V, dtype))


def spec_verify_greedy(target_logits, draft_tokens, num_draft=None, *, out_tokens=None,
                       out_accept_len=None, workspace=None, stream=None):
    """Greedy verify. Returns (tokens [B,k+1], accept_len [B])."""
    B, k1, V = target_logits.shape
    k = k1 - 1
    dev = target_logits.device
    code = _dtype_code(target_logits)
    _check_cuda("target_logits", target_logits)
    _check_cuda("draft_tokens", draft_tokens, torch.int32, (B, k), dev)
    _check_cuda("num_draft", num_draft, torch.int32, (B,), dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    if out_accept_len is None:
        out_accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
    _check_cuda("out_tokens", out_tokens, torch.int32, (B, k + 1), dev)
    _check_cuda("out_accept_len", out_accept_len, torch.int32, (B,), dev)
    h, st = _stream_handle(stream)
    need = spec_verify_greedy_workspace(B, k, V, code)
    ws = workspace if workspace is not None else _workspace("greedy", need, dev, st)
    _ok(library().spec_verify_greedy(
        _ptr(target_logits), code, _ptr(draft_tokens), _ptr(num_draft), B, k, V,
        _ptr(out_tokens), _ptr(out_accept_len), _ptr(ws), ws.numel(), h), "spec_verify_greedy")
    return out_tokens, out_accept_len


def spec_verify_greedy_noalloc(target_logits, draft_tokens, num_draft=None, *, out_tokens=None,
                               out_accept_len=None, stream=None):
    """Greedy verify without a workspace, for callers that cannot allocate device memory:
    it uses the library's fixed 8 MiB scratch array (shapes needing more are rejected).
    Calls that overlap on the GPU share that array and race. Returns (tokens, accept_len)."""
    B, k1, V = target_logits.shape
    k = k1 - 1
    dev = target_logits.device
    code = _dtype_code(target_logits)
    _check_cuda("target_logits", target_logits)
    _check_cuda("draft_tokens", draft_tokens, torch.int32, (B, k), dev)
    _check_cuda("num_draft", num_draft, torch.int32, (B,), dev)
    if out_tokens is None:
        out_tokens = torch.empty((B, k + 1), dtype=torch.int32, device=dev)
    if out_accept_len is None:
        out_accept_len = torch.empty((B,), dtype=torch.int32, device=dev)
    _check_cuda("out_tokens", out_tokens, torch.int32, (B, k + 1), dev)
    _check_cuda("out_accept_len", out_accept_len, torch.int32, (B,), dev)
    h, _ = _stream_handle(stream)
    _ok(library().spec_verify_greedy_noalloc(
        _ptr(target_logits), code, _ptr(draft_tokens), _ptr(num_draft), B, k, V,
        _ptr(out_tokens), _ptr(out_accept_len), h), "spec_verify_greedy_noalloc")
    return out_tokens, out_accept_len


# ------------------------------------------------------------------------------ gate
def logit_gap_gate_workspace(N: int, V: int, dtype: int) -> int:
    return int(library().logit_gap_gate_workspace(N, V, dtype))


def logit_gap_gate(logits, tau: float, answer_set=None, *, out_token=None, out_gap=None,
                   out_fire=None, workspace=None, stream=None):
    """Gate over the rows of ``logits`` [..., V]. Returns (token [N], gap [N], fire [N])."""
    V = logits.shape[-1]
    N = logits.numel() // V if V else 0
    dev = logits.device
    code = _dtype_code(logits)
    _check_cuda("logits", logits)
    if answer_set is not None:
        _check_cuda("answer_set", answer_set, torch.int32, None, dev)
    n_answer = 0 if answer_set is None else answer_set.numel()
    if out_token is None:
        out_token = torch.empty((N,), dtype=torch.int32, device=dev)
    if out_gap is None:
        out_gap = torch.empty((N,), dtype=torch.float32, device=dev)
    if out_fire is None:
        out_fire = torch.empty((N,), dtype=torch.uint8, device=dev)
    _check_cuda("out_token", out_token, torch.int32, (N,), dev)
    _check_cuda("out_gap", out_gap, torch.float32, (N,), dev)
    _check_cuda("out_fire", out_fire, torch.uint8, (N,), dev)
    h, st = _stream_handle(stream)
    need = logit_gap_gate_workspace(N, V, code)
    ws = workspace if workspace is not None else _workspace("gate", need, dev, st)
    _ok(library().logit_gap_gate(
        _ptr(logits), code, N, V, float(tau), _ptr(answer_set), n_answer, _ptr(out_token),
        _ptr(out_gap), _ptr(out_fire), _ptr(ws), ws.numel(), h), "logit_gap_gate")
    return out_token, out_gap, out_fire


# ------------------------------------------------------------------------ gate calibration
def gate_risk_coverage_workspace(N: int, T: int) -> int:
    return int(library().gate_risk_coverage_workspace(N, T))


def gate_risk_coverage(gap, token, full_token, answer_set, taus, z: float = 1.959963984540054,
                       r_max: float = 0.0, *, out_points=None, out_tau_index=None,
                       workspace=None, stream=None):
    """Risk-coverage sweep. Returns (points [T, 8] float64 whose columns are CALIB_POINT, the
    first two holding int64 bits, tau_index [1] int32). ``gate_points_dict`` unpacks them."""
    N = gap.numel()
    T = taus.numel()
    dev = gap.device
    _check_cuda("gap", gap, torch.float32, (N,), dev)
    _check_cuda("token", token, torch.int32, (N,), dev)
    _check_cuda("full_token", full_token, torch.int32, (N,), dev)
    _check_cuda("taus", taus, torch.float32, (T,), dev)
    if answer_set is not None:
        _check_cuda("answer_set", answer_set, torch.int32, None, dev)
    n_answer = 0 if answer_set is None else answer_set.numel()
    if out_points is None:
        out_points = torch.empty((T, 8), dtype=torch.float64, device=dev)
    if out_tau_index is None:
        out_tau_index = torch.empty((1,), dtype=torch.int32, device=dev)
    _check_cuda("out_points", out_points, torch.float64, (T, 8), dev)
    _check_cuda("out_tau_index", out_tau_index, torch.int32, (1,), dev)
    h, st = _stream_handle(stream)
    need = gate_risk_coverage_workspace(N, T)
    ws = workspace if workspace is not None else _workspace("sweep", need, dev, st)
    _ok(library().gate_risk_coverage(
        _ptr(gap), _ptr(token), _ptr(full_token), N, _ptr(answer_set), n_answer, _ptr(taus), T,
        float(z), float(r_max), _ptr(out_points), _ptr(out_tau_index), _ptr(ws), ws.numel(), h),
        "gate_risk_coverage")
    return out_points, out_tau_index


def gate_points_dict(points) -> dict:
    """Columns of gate_risk_coverage's points as CPU tensors (counts as int64)."""
    p = points.detach().cpu()
    out = {}
    for i, name in enumerate(CALIB_POINT):
        col = p[:, i].contiguous()
        out[name] = col.view(torch.int64) if i < 2 else col
    return out


def conformal_residual(draft_logits, true_logits, *, out_resid=None, stream=None):
    """Sup-norm residual of each draft row [..., V] against the true row. Returns [N] fp32."""
    V = draft_logits.shape[-1]
    N = draft_logits.numel() // V if V else 0
    dev = draft_logits.device
    code = _dtype_code(draft_logits)
    _check_cuda("draft_logits", draft_logits)
    _check_cuda("true_logits", true_logits, draft_logits.dtype, tuple(draft_logits.shape), dev)
    if out_resid is None:
        out_resid = torch.empty((N,), dtype=torch.float32, device=dev)
    _check_cuda("out_resid", out_resid, torch.float32, (N,), dev)
    h, _ = _stream_handle(stream)
    _ok(library().conformal_residual(_ptr(draft_logits), _ptr(true_logits), code, N, V,
                                     _ptr(out_resid), h), "conformal_residual")
    return out_resid


def conformal_quantile_workspace(n: int) -> int:
    return int(library().conformal_quantile_workspace(n))


def conformal_quantile(resid, q: float, *, out_q=None, workspace=None, stream=None):
    """Split-conformal quantile of the residuals [n]. Returns Q as a [1] fp32 tensor."""
    n = resid.numel()
    dev = resid.device
    _check_cuda("resid", resid, torch.float32, (n,), dev)
    if out_q is None:
        out_q = torch.empty((1,), dtype=torch.float32, device=dev)
    _check_cuda("out_q", out_q, torch.float32, (1,), dev)
    h, st = _stream_handle(stream)
    need = conformal_quantile_workspace(n)
    ws = workspace if workspace is not None else _workspace("select", need, dev, st)
    _ok(library().conformal_quantile(_ptr(resid), n, float(q), _ptr(out_q), _ptr(ws),
                                     ws.numel(), h), "conformal_quantile")
    return out_q


def conformal_admit_workspace(N: int, K: int, V: int, dtype: int) -> int:
    return int(library().conformal_admit_workspace(N, K, V, dtype))


def conformal_admit(logits, Q, *, out_layer=None, out_token=None, out_gap=None,
                    want_gap: bool = True, workspace=None, stream=None):
    """Conformal gate over logits [N, K, V] and per-layer quantiles Q [K]. Returns (layer [N],
    token [N], gap [N, K] or None)."""
    N, K, V = logits.shape
    dev = logits.device
    code = _dtype_code(logits)
    _check_cuda("logits", logits)
    _check_cuda("Q", Q, torch.float32, (K,), dev)
    if out_layer is None:
        out_layer = torch.empty((N,), dtype=torch.int32, device=dev)
    if out_token is None:
        out_token = torch.empty((N,), dtype=torch.int32, device=dev)
    if out_gap is None and want_gap:
        out_gap = torch.empty((N, K), dtype=torch.float32, device=dev)
    _check_cuda("out_layer", out_layer, torch.int32, (N,), dev)
    _check_cuda("out_token", out_token, torch.int32, (N,), dev)
    _check_cuda("out_gap", out_gap, torch.float32, (N, K), dev)
    h, st = _stream_handle(stream)
    need = conformal_admit_workspace(N, K, V, code)
    ws = workspace if workspace is not None else _workspace("admit", need, dev, st)
    _ok(library().conformal_admit(_ptr(logits), code, N, K, V, _ptr(Q), _ptr(out_layer),
                                  _ptr(out_token), _ptr(out_gap), _ptr(ws), ws.numel(), h),
        "conformal_admit")
    return out_layer, out_token, out_gap


# ---------------------------------------------------------------- ready-distribution cache
SV_CACHE_VALID, SV_CACHE_DECODED, SV_CACHE_CONSUMED = 1, 2, 4
CACHE_STATS = ("pre_positions", "skipped", "consumed", "wasted", "fast", "fall_invalid",
               "fall_ineligible", "fall_gate", "bad")


def ready_cache_record_workspace(M: int, V: int, dtype: int) -> int:
    return int(library().ready_cache_record_workspace(M, V, dtype))


class ReadyCacheTable:
    """A device-resident table of S session slots (32 bytes each), entries of at most
    max_entry tokens, and the table's event counters; with ``keep_dist`` also one stored
    ready row of V logits per session. A new table is empty (zero-filled)."""

    def __init__(self, S: int, max_entry: int, device, *, V: int | None = None,
                 dist_dtype=None, keep_dist: bool = False):
        self.S, self.max_entry = S, max_entry
        self.slots = torch.zeros((S, 4), dtype=torch.int64, device=device)
        self.device = self.slots.device  # with its index ("cuda" -> "cuda:0")
        self.entry_store = torch.zeros((S, max_entry), dtype=torch.int32, device=self.device)
        self.stats = torch.zeros((len(CACHE_STATS),), dtype=torch.int64, device=self.device)
        self.dist = None
        if keep_dist:
            if V is None or dist_dtype is None:
                raise ValueError("keep_dist needs V and dist_dtype")
            self.dist = torch.zeros((S, V), dtype=dist_dtype, device=self.device)

    def record(self, session, end_pos, entry_tokens, entry_len, headroom, ready_logits, *,
               out_status=None, workspace=None, stream=None):
        """Algorithm 1 for M sessions (distinct ids). Returns out_status [M] int32."""
        M, V = ready_logits.shape
        dev = self.device
        code = _dtype_code(ready_logits)
        _check_cuda("ready_logits", ready_logits, None, None, dev)
        _check_cuda("session", session, torch.int32, (M,), dev)
        _check_cuda("end_pos", end_pos, torch.int64, (M,), dev)
        _check_cuda("entry_tokens", entry_tokens, torch.int32, (M, self.max_entry), dev)
        _check_cuda("entry_len", entry_len, torch.int32, (M,), dev)
        _check_cuda("headroom", headroom, torch.int64, (M,), dev)
        if self.dist is not None:
            _check_cuda("dist", self.dist, ready_logits.dtype, (self.S, V), dev)
        if out_status is None:
            out_status = torch.empty((M,), dtype=torch.int32, device=dev)
        _check_cuda("out_status", out_status, torch.int32, (M,), dev)
        h, st = _stream_handle(stream)
        need = ready_cache_record_workspace(M, V, code)
        ws = workspace if workspace is not None else _workspace("record", need, dev, st)
        _ok(library().ready_cache_record(
            _ptr(self.slots), _ptr(self.entry_store), self.S, self.max_entry, _ptr(self.stats),
            _ptr(session), _ptr(end_pos), _ptr(entry_tokens), _ptr(entry_len), _ptr(headroom),
            M, _ptr(ready_logits), code, V, _ptr(self.dist), _ptr(out_status), _ptr(ws),
            ws.numel(), h), "ready_cache_record")
        return out_status

    def serve(self, session, start, req_tokens, req_len, tau: float, answer_set=None, *,
              exact: bool = True, out_token=None, out_reason=None, stream=None):
        """Algorithm 2 for R requests. Returns (token [R], reason [R]) int32."""
        R = session.numel()
        dev = self.device
        _check_cuda("session", session, torch.int32, (R,), dev)
        _check_cuda("start", start, torch.int64, (R,), dev)
        _check_cuda("req_tokens", req_tokens, torch.int32, (R, self.max_entry), dev)
        _check_cuda("req_len", req_len, torch.int32, (R,), dev)
        if answer_set is not None:
            _check_cuda("answer_set", answer_set, torch.int32, None, dev)
        n_answer = 0 if answer_set is None else answer_set.numel()
        if out_token is None:
            out_token = torch.empty((R,), dtype=torch.int32, device=dev)
        if out_reason is None:
            out_reason = torch.empty((R,), dtype=torch.int32, device=dev)
        _check_cuda("out_token", out_token, torch.int32, (R,), dev)
        _check_cuda("out_reason", out_reason, torch.int32, (R,), dev)
        h, _ = _stream_handle(stream)
        _ok(library().ready_cache_serve(
            _ptr(self.slots), _ptr(self.entry_store), self.S, self.max_entry, _ptr(self.stats),
            _ptr(session), _ptr(start), _ptr(req_tokens), _ptr(req_len), R, float(tau),
            _ptr(answer_set), n_answer, 1 if exact else 0, _ptr(out_token), _ptr(out_reason),
            h), "ready_cache_serve")
        return out_token, out_reason

    def invalidate(self, session, *, stream=None):
        """Section 3.6: the listed sessions' state mutated."""
        n = session.numel()
        _check_cuda("session", session, torch.int32, (n,), self.device)
        h, _ = _stream_handle(stream)
        _ok(library().ready_cache_invalidate(_ptr(self.slots), self.S, _ptr(self.stats),
                                             _ptr(session), n, h), "ready_cache_invalidate")

    def state(self) -> dict:
        """The slots' fields as CPU numpy arrays (a device-to-host copy)."""
        import numpy as np

        raw = self.slots.detach().cpu().numpy().tobytes()
        rec = np.frombuffer(raw, dtype=np.dtype([
            ("position", "<i8"), ("gap", "<f8"), ("token", "<i4"), ("entry_len", "<i4"),
            ("flags", "<u4"), ("epoch", "<u4")]))
        return {k: rec[k].copy() for k in rec.dtype.names}

    def counters(self) -> dict:
        vals = self.stats.detach().cpu().tolist()
        return dict(zip(CACHE_STATS, vals))


# ------------------------------------------------------------------------------ confidence
def draft_confidence_workspace(B: int, k: int, V: int, dtype: int) -> int:
    return int(library().draft_confidence_workspace(B, k, V, dtype))


def draft_confidence_stop(draft_logits, temperature: float, mode: int, floor: float,
                          num_draft=None, *, out_num_draft=None, out_conf=None,
                          want_conf: bool = True, workspace=None, stream=None):
    """Variable-length drafting over draft logits [B, k, V]. Returns (num_draft [B] int32,
    conf [B, k] fp32 or None)."""
    B, k, V = draft_logits.shape
    dev = draft_logits.device
    code = _dtype_code(draft_logits)
    _check_cuda("draft_logits", draft_logits)
    _check_cuda("num_draft", num_draft, torch.int32, (B,), dev)
    if out_num_draft is None:
        out_num_draft = torch.empty((B,), dtype=torch.int32, device=dev)
    if out_conf is None and want_conf:
        out_conf = torch.empty((B, k), dtype=torch.float32, device=dev)
    _check_cuda("out_num_draft", out_num_draft, torch.int32, (B,), dev)
    _check_cuda("out_conf", out_conf, torch.float32, (B, k), dev)
    h, st = _stream_handle(stream)
    need = draft_confidence_workspace(B, k, V, code)
    ws = workspace if workspace is not None else _workspace("conf", need, dev, st)
    _ok(library().draft_confidence_stop(
        _ptr(draft_logits), code, _ptr(num_draft), B, k, V, float(temperature), int(mode),
        float(floor), _ptr(out_num_draft), _ptr(out_conf), _ptr(ws), ws.numel(), h),
        "draft_confidence_stop")
    return out_num_draft, out_conf


# ------------------------------------------------------------------------------ n-gram
def ngram_propose(history, hist_len, n_max: int, n_min: int, k: int, *, out_draft=None,
                  out_num_draft=None, stream=None):
    """Prompt-lookup proposer. Returns (draft [B,k] int32, num_draft [B] int32)."""
    B, L_max = history.shape
    dev = history.device
    _check_cuda("history", history, torch.int32)
    _check_cuda("hist_len", hist_len, torch.int32, (B,), dev)
    if out_draft is None:
        out_draft = torch.empty((B, k), dtype=torch.int32, device=dev)
    if out_num_draft is None:
        out_num_draft = torch.empty((B,), dtype=torch.int32, device=dev)
    _check_cuda("out_draft", out_draft, torch.int32, (B, k), dev)
    _check_cuda("out_num_draft", out_num_draft, torch.int32, (B,), dev)
    h, _ = _stream_handle(stream)
    _ok(library().ngram_propose(_ptr(history), _ptr(hist_len), B, L_max, n_max, n_min, k,
                                _ptr(out_draft), _ptr(out_num_draft), h), "ngram_propose")
    return out_draft, out_num_draft

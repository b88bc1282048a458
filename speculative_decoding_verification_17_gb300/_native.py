"""Build and load ``libspecverify.so``, the C-ABI library of the verify step.

The library is compiled in-tree from ``csrc/`` for sm_103a only (one ``-gencode``), one
nvcc process per translation unit in parallel, and linked against the static CUDA runtime
so loading it needs no CUDA library path. Loading never falls back to anything: a missing
or stale library is an error.
"""
from __future__ import annotations

import ctypes
import glob
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
SO = os.path.join(BUILD, "libspecverify.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
              "-I", CSRC] + os.environ.get("SV_NVCC_EXTRA", "").split()


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale() -> bool:
    if not os.path.exists(SO):
        return True
    t = os.path.getmtime(SO)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(
        os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every ``csrc/*.cu`` and link ``_build/libspecverify.so``."""
    if not force and not _stale():
        return SO
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = SO + f".tmp{os.getpid()}"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs],
                       capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, SO)
    return SO


_lock = threading.Lock()
_lib = None


def lib():
    """The loaded library (built first if absent or older than its sources)."""
    global _lib
    with _lock:
        if _lib is None:
            path = SO
            if _stale():
                build()
            if not os.path.exists(path):
                raise RuntimeError("libspecverify.so is missing and could not be built")
            L = ctypes.CDLL(path)
            _declare(L)
            _lib = L
    return _lib


def _declare(L):
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.sv_version.restype = I
    L.sv_version.argtypes = []
    L.sv_status_string.restype = ctypes.c_char_p
    L.sv_status_string.argtypes = [I]
    L.sv_last_cuda_error.restype = I
    L.sv_last_cuda_error.argtypes = []
    L.spec_verify_sample_workspace.restype = Z
    L.spec_verify_sample_workspace.argtypes = [I, I, I, I]
    L.spec_verify_sample_launches.restype = I
    L.spec_verify_sample_launches.argtypes = [I, I, I, I]
    L.spec_verify_sample.restype = I
    L.spec_verify_sample.argtypes = [P, P, I, P, P, P, I, I, I, F, P, P, P, P, P, P, Z, P]
    L.spec_verify_greedy_workspace.restype = Z
    L.spec_verify_greedy_workspace.argtypes = [I, I, I, I]
    L.spec_verify_greedy.restype = I
    L.spec_verify_greedy.argtypes = [P, I, P, P, I, I, I, P, P, P, Z, P]
    L.spec_verify_greedy_noalloc.restype = I
    L.spec_verify_greedy_noalloc.argtypes = [P, I, P, P, I, I, I, P, P, P]
    L.logit_gap_gate_workspace.restype = Z
    L.logit_gap_gate_workspace.argtypes = [I, I, I]
    L.logit_gap_gate.restype = I
    L.logit_gap_gate.argtypes = [P, I, I, I, F, P, I, P, P, P, P, Z, P]
    L.ngram_propose.restype = I
    L.ngram_propose.argtypes = [P, P, I, I, I, I, I, P, P, P]
    L.draft_confidence_workspace.restype = Z
    L.draft_confidence_workspace.argtypes = [I, I, I, I]
    L.draft_confidence_stop.restype = I
    L.draft_confidence_stop.argtypes = [P, I, P, I, I, I, F, I, F, P, P, P, Z, P]
    D = ctypes.c_double
    L.gate_risk_coverage_workspace.restype = Z
    L.gate_risk_coverage_workspace.argtypes = [I, I]
    L.gate_risk_coverage.restype = I
    L.gate_risk_coverage.argtypes = [P, P, P, I, P, I, P, I, D, D, P, P, P, Z, P]
    L.conformal_residual.restype = I
    L.conformal_residual.argtypes = [P, P, I, I, I, P, P]
    L.conformal_quantile_workspace.restype = Z
    L.conformal_quantile_workspace.argtypes = [I]
    L.conformal_quantile.restype = I
    L.conformal_quantile.argtypes = [P, I, D, P, P, Z, P]
    L.conformal_quantile_barrier_selftest.restype = I
    L.conformal_quantile_barrier_selftest.argtypes = [P, I, P, P, Z, ctypes.c_uint, P]
    L.conformal_admit_workspace.restype = Z
    L.conformal_admit_workspace.argtypes = [I, I, I, I]
    L.conformal_admit.restype = I
    L.conformal_admit.argtypes = [P, I, I, I, I, P, P, P, P, P, Z, P]
    L.ready_cache_record_workspace.restype = Z
    L.ready_cache_record_workspace.argtypes = [I, I, I]
    L.ready_cache_record.restype = I
    L.ready_cache_record.argtypes = [P, P, I, I, P, P, P, P, P, P, I, P, I, I, P, P, P, Z, P]
    L.ready_cache_serve.restype = I
    L.ready_cache_serve.argtypes = [P, P, I, I, P, P, P, P, P, I, F, P, I, I, P, P, P]
    L.ready_cache_invalidate.restype = I
    L.ready_cache_invalidate.argtypes = [P, I, P, P, I, P]

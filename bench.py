"""Benchmark of the speculative-decoding verify step on GB300.

One step = one spec_verify_sample call (the fused verify kernel: tempered softmax of the
k+1 target rows and k draft rows, accept tests, accepted prefix, residual or bonus draw)
over one batch of the B=512, k=8, V=128256 bf16, T=0.7 workload, inputs resident in HBM.
The metric is verified draft positions per second (sum of n_r per step / step time), with
the logit bandwidth (each needed logit read once) against the measured HBM peak.

Secondary rows time the other calls of the hot path on their own workloads (greedy verify,
logit-gap gate, n-gram proposal + greedy verify, the fp32 sampled verify, the draft
confidence stop, the gate calibration sweep, the conformal residual, quantile and gate, and
the ready-distribution cache's record and serve)
with the same event timing; workloads that fit in L2 get an L2 flush before every timed
launch.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
Under torchrun every rank runs its own replica of the batch (request sharding, no
collective on the data path): value = positions of all ranks / max rank time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "verified draft positions/sec and logit GB/s (fraction of GB300 HBM peak)"
HEAD = 3  # index of the headline workload in synth.WORKLOADS
# The sampled-verify workloads whose inputs exceed L2 (timed back to back without a flush):
# the headline (B=512, k=8, V=128256 bf16) and the fp32 one (B=256, k=4, V=151936).
TIMED_WORKLOADS = {
    3: "z_p~N(0,2.5^2), z_q=0.6 z_p+N(0,1.5^2)",
    2: "z_p~N(0,3^2) plus one planted peak +U(2,10) per row, z_q=z_p+N(0,0.7^2)",
}
L2_BYTES = 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------------------ helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def _code_only(text: str) -> str:
    """C/C++/CUDA source with its comments and blank lines removed (string and character
    literals kept), so that a digest of it changes with the code and not with the
    comments."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = (line.rstrip() for line in "".join(out).splitlines())
    return "\n".join(line for line in lines if line)


def source_digest(unit: str = "sv_verify.cu") -> str:
    """sha256 prefix of what the profiled kernel is built from: the code (comments removed)
    of its translation unit and of every header it includes from the package or `include/`
    (recursively), and the statements of the build script that set the compiler flags (ARCH,
    NVCC_FLAGS)."""
    pkg = os.path.join(ROOT, "speculative_decoding_verification_17_gb300")
    dirs = [os.path.join(pkg, "csrc"), os.path.join(ROOT, "include")]
    seen, todo = [], [unit]
    while todo:
        name = todo.pop(0)
        if name in seen:
            continue
        path = next((os.path.join(d, name) for d in dirs
                     if os.path.exists(os.path.join(d, name))), None)
        if path is None:
            continue
        seen.append(name)
        todo += re.findall(r'^#include "([^"]+)"', open(path).read(), re.M)
    h = hashlib.sha256()
    for name in sorted(seen):
        path = next(os.path.join(d, name) for d in dirs if os.path.exists(os.path.join(d, name)))
        with open(path, encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + _code_only(f.read()).encode())
    with open(os.path.join(pkg, "_native.py")) as f:
        build = f.read()
    flags = re.findall(r"^(?:ARCH|NVCC_FLAGS) = .*?\n(?=\S|\n|\Z)", build, re.M | re.S)
    h.update(b"_native.py\0" + "".join(flags).encode())
    return h.hexdigest()[:16]


def profiled_traffic(kernel: str, workload: str, unit: str = "sv_verify.cu"):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on this source
    (the translation unit `unit` and what it includes)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    s = re.search(r"source_digest:\s*([0-9a-f]+)", text)
    if not m or not s or s.group(1) != source_digest(unit):
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, each stamped with the host time
    it arrived; summary(t0, t1) keeps the samples taken inside the timed window [t0, t1]
    (or, for a window shorter than the sampling period, the nearest sample on each side)."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 2):
        self.gpu = gpu_index
        self.period = period_ms
        self.proc = None
        self.samples = []  # (host time, line)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.period)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            deadline = time.time() + 5.0  # wait for the first sample, so the window is covered
            while not self.samples and time.time() < deadline:
                time.sleep(0.01)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            time.sleep(2 * self.period / 1000.0)  # one more sample past the window
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self, t0: float, t1: float):
        inside = [l for t, l in self.samples if t0 <= t <= t1]
        mode = "inside"
        if not inside:
            before = [l for t, l in self.samples if t < t0][-1:]
            after = [l for t, l in self.samples if t > t1][:1]
            inside = before + after
            mode = "bracketing"
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in inside:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm), "window": mode,
                "period_ms": self.period}


def sample_bytes(n_total: int, B: int, k: int, V: int, elem: int) -> int:
    """Algorithmic bytes of one sampled verify: every needed logit once (sum(n_r + 1) target
    rows, sum(n_r) draft rows) plus the small per-request I/O (draft tokens, uniforms,
    emitted tokens, accept length, 4 bytes each)."""
    return (2 * n_total + B) * V * elem + 4 * B * (k + (k + 1) + (k + 1) + 1)


# ------------------------------------------------------------------------------ timing
def time_launches(fn, steps, warmup, stream, flush=None):
    """Per-launch CUDA-event times (ms) of fn() on `stream`, after `warmup` calls. With
    `flush`, an L2 flush runs before every launch, outside the timed events."""
    import torch

    for _ in range(warmup):
        if flush is not None:
            flush()
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    with torch.cuda.stream(stream):
        for a, b in ev:
            if flush is not None:
                flush()
            a.record(stream)
            fn()
            b.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev]


def make_flush(device):
    """L2 flush before a timed launch: write a buffer twice the size of L2, then read another
    one, so the written lines are back in HBM (their write-back is not charged to the timed
    launch) and L2 holds only clean lines of no use to it."""
    import torch

    buf = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=device)
    clean = torch.zeros(2 * L2_BYTES // 8, dtype=torch.int64, device=device)

    def flush():
        buf.fill_(1)
        clean.max()

    return flush


# ------------------------------------------------------------------------------ ranks
def init_ranks(world: int, device):
    """The process group of a multi-rank run (None for one rank): NCCL between GPUs, gloo when
    the ranks run on host cores. It carries only the barriers and the max-over-ranks timing;
    the data path has no collective."""
    if world <= 1:
        return None
    import torch.distributed as dist

    if device.type == "cuda":
        dist.init_process_group("nccl", device_id=device)
    else:
        dist.init_process_group("gloo")
    return dist


def rank_seed(rank: int, workload: int = HEAD) -> int:
    """Seed of a rank's shard of requests: every rank verifies its own batch."""
    import synth

    return synth.SEED_BASE + workload + 7919 * rank


def max_over_ranks(dist, x: float, device) -> float:
    """The largest value of x over all ranks (x itself for one rank)."""
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, units_per_rank: int, steps: int, max_total_ms: float) -> float:
    """Units of all ranks per second of the slowest rank (weak scaling: each rank does the
    same work)."""
    return world * units_per_rank * steps / (max_total_ms * 1e-3)


# ------------------------------------------------------------------------------ GPU arm
def gb300_arm(args, rank, world, local_rank):
    import numpy as np
    import torch

    import speculative_decoding_verification_17_gb300 as sv
    import synth

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = init_ranks(world, dev)

    w = synth.WORKLOADS[args.workload]
    d = synth.workload_inputs(w, device=dev, seed=rank_seed(rank, args.workload), B=args.requests)
    B, k, V = d["B"], d["k"], d["V"]
    n_total = B * k  # every request drafts k tokens in this workload
    elem = w.elem_bytes
    stream = torch.cuda.Stream(device=dev)
    code = sv.SV_F32 if w.dtype == "f32" else sv.SV_BF16
    args.launches_per_step = sv.spec_verify_sample_launches(B, k, V, code)
    ws = torch.zeros(sv.spec_verify_sample_workspace(B, k, V, code), dtype=torch.uint8,
                     device=dev)
    outs = dict(out_tokens=torch.empty((B, k + 1), dtype=torch.int32, device=dev),
                out_accept_len=torch.empty((B,), dtype=torch.int32, device=dev),
                out_p_draft=torch.empty((B, k), dtype=torch.float32, device=dev),
                out_q_draft=torch.empty((B, k), dtype=torch.float32, device=dev),
                out_resid_mass=torch.empty((B,), dtype=torch.float32, device=dev))

    def step():
        sv.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], d["T"],
                              d["num_draft"], workspace=ws, stream=stream, **outs)

    # ---- timed region: K steps, barrier + synchronize on both sides ----
    clk = ClockSampler(torch.cuda.current_device()).start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    t0 = time.time()
    with torch.cuda.stream(stream):
        for a, b in ev:
            a.record(stream)
            step()
            b.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    wall = t1 - t0
    clk.stop()
    clk.window = (t0, t1)
    if dist:
        dist.barrier()
    per = [a.elapsed_time(b) for a, b in ev]
    total_ms = sum(per)
    mean_ms = total_ms / len(per)
    args.median_ms = statistics.median(per)
    total_ms = max_over_ranks(dist, total_ms, dev)
    acc = outs["out_accept_len"].float().mean().item()

    # ---- end to end through the public call: pinned host inputs in, results out ----
    if args.no_e2e:
        return finish_line(args, rank, world, dev, dist, d, w, stream, total_ms, mean_ms, acc,
                           clk, wall, None)
    h_t = d["target"].cpu().pin_memory()
    h_d = d["draft"].cpu().pin_memory()
    h_x = d["draft_tokens"].cpu().pin_memory()
    h_u = d["uniforms"].cpu().pin_memory()
    d_t, d_d = torch.empty_like(d["target"]), torch.empty_like(d["draft"])
    d_x, d_u = torch.empty_like(d["draft_tokens"]), torch.empty_like(d["uniforms"])
    h_out = {kk: torch.empty(v.shape, dtype=v.dtype).pin_memory() for kk, v in outs.items()}
    h2d = sum(t.numel() * t.element_size() for t in (h_t, h_d, h_x, h_u))
    d2h = sum(t.numel() * t.element_size() for t in h_out.values())

    def e2e_step():
        with torch.cuda.stream(stream):
            d_t.copy_(h_t, non_blocking=True)
            d_d.copy_(h_d, non_blocking=True)
            d_x.copy_(h_x, non_blocking=True)
            d_u.copy_(h_u, non_blocking=True)
            sv.spec_verify_sample(d_t, d_d, d_x, d_u, d["T"], None, workspace=ws, stream=stream,
                                  **outs)
            for kk, v in outs.items():
                h_out[kk].copy_(v, non_blocking=True)

    e2e_steps = max(3, min(args.steps, 10))
    e2e_ms = time_launches(e2e_step, e2e_steps, 2, stream)
    e2e_total = max_over_ranks(dist, sum(e2e_ms), dev)
    del h_t, h_d, d_t, d_d

    e2e = {"value": whole_job_rate(world, n_total, e2e_steps, e2e_total), "unit": "positions/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "ms_per_step": e2e_total / e2e_steps}
    return finish_line(args, rank, world, dev, dist, d, w, stream, total_ms, mean_ms, acc, clk,
                       wall, e2e)


def finish_line(args, rank, world, dev, dist, d, w, stream, total_ms, mean_ms, acc, clk, wall,
                e2e):
    B, k, V = d["B"], d["k"], d["V"]
    n_total = B * k
    elem = w.elem_bytes
    peak, peak_kind = measured_peaks()
    abytes = sample_bytes(n_total, B, k, V, elem)
    achieved = abytes / (mean_ms * 1e-3) / 1e9
    value = whole_job_rate(world, n_total, args.steps, total_ms)
    rows = {}
    if rank == 0 and not args.no_rows:
        rows = secondary_rows(args, dev, stream, peak, head=d)
        # the secondary rows on a line of their own, ahead of the headline line
        print(json.dumps({"rows": rows}), flush=True)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(d, w, budget_s=args.cpu_seconds)

    if rank == 0:
        ename = "F32" if w.dtype == "f32" else "BF16"
        clocks = clk.summary(*clk.window)
        med = getattr(args, "median_ms", None)
        line = {
            "metric": METRIC,
            "value": value,
            "unit": "positions/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": total_ms / args.steps,
            "ms_per_step_median": med,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": w.dtype,
            "data": "synthetic (seeded)",
            "config": {
                "workload": f"sampled verify B={B} k={k} V={V} {w.dtype} T={w.T}: "
                            f"{TIMED_WORKLOADS[w.index]}",
                "global_batch": B * world,
                "draft_positions_per_step": n_total * world,
                "l2": f"inputs {abytes / 1e9:.2f} GB > 129 MB L2: no flush",
                "parallelism": f"request-sharded replicas x{world}" if world > 1 else "single GPU",
            },
            "mean_accept_len": acc,
            "roofline": {
                "bound": "hbm",
                "kernel": f"segment_kernel<SampleOp<{ename}>>" + (
                    f" + draw_kernel<{ename}>" if args.launches_per_step > 1 else ""),
                "achieved": achieved,
                "peak": peak,
                "unit": "GB/s",
                "frac": achieved / peak,
                "peak_source": "measured hbm_gbs" if peak_kind == "measured" else "fallback",
                "traffic": profiled_traffic("segment_kernel_sample", f"b{B}_k{k}_v{V}_{w.dtype}"),
                "bytes_per_launch": abytes,
                "launch_ms": mean_ms,
            },
            "e2e": e2e,
            "gpu_launches": args.steps * args.launches_per_step,
            "clocks": clocks,
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        if rows:
            line["configs_2_3"] = target_configs(rows, line)
        line = _rounded(line, 4)
        print(json.dumps(line))
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def _rounded(x, digits: int = 5):
    """x with every float rounded to `digits` significant digits (the headline line stays
    short)."""
    if isinstance(x, float):
        return float(f"{x:.{digits}g}")
    if isinstance(x, dict):
        return {k: _rounded(v, digits) for k, v in x.items()}
    if isinstance(x, list):
        return [_rounded(v, digits) for v in x]
    return x


def target_configs(rows, line):
    """The two configurations the >= 70 % bandwidth target names, in brief: the fp32 sampled
    verify (B=256, k=4, V=151936) with its 1280-row gate, and the bf16 sampled verify (B=512,
    k=8, V=128256; the headline, or its row when another workload was timed). Each gives ms
    per launch (median), GB/s, the fraction of the peak and, where a committed ncu summary
    was taken on the current source, the DRAM traffic per launch."""
    out = {}
    for key, src, kern, unit in (
            ("sample_b256_k4_v151936_f32", "sample_b256_k4_v151936_f32", "segment_kernel",
             "sv_verify.cu"),
            ("gate_n1280_v151936_f32", "gate_n1280_v151936_f32", "segment_kernel", "sv_gate.cu")):
        r = rows.get(src)
        if r:
            out[key] = {"ms": r["ms"], "gbs": r["gbs"], "frac": r["frac"],
                        "traffic": profiled_traffic(kern, key, unit)}
    rf = line["roofline"]
    if line["config"]["workload"].startswith("sampled verify B=512 k=8 V=128256 bf16"):
        out["sample_b512_k8_v128256_bf16"] = {
            "ms": line["ms_per_step_median"], "gbs": rf["achieved"], "frac": rf["frac"],
            "traffic": rf["traffic"]}
    return out


def secondary_rows(args, dev, stream, peak, head=None):
    """Event-timed launches of the other calls of the path on their own workloads (and the
    greedy verify on the headline batch's target rows, `head`)."""
    import torch

    import speculative_decoding_verification_17_gb300 as sv
    import synth

    steps = max(5, min(args.steps, 20))
    flush = make_flush(dev)
    rows = {}

    def gbs(nbytes, ms):
        return nbytes / (ms * 1e-3) / 1e9

    # fp32 sampled verify + gate (B=256, k=4, V=151936)
    w = synth.WORKLOADS[2]
    d = synth.workload_inputs(w, device=dev)
    B, k, V = d["B"], d["k"], d["V"]
    ws = torch.zeros(sv.spec_verify_sample_workspace(B, k, V, sv.SV_F32), dtype=torch.uint8,
                     device=dev)
    ms = statistics.median(time_launches(
        lambda: sv.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                                      d["T"], None, workspace=ws, stream=stream),
        steps, 3, stream))
    nb = sample_bytes(B * k, B, k, V, 4)
    rows["sample_b256_k4_v151936_f32"] = dict(
        ms=ms, positions_per_s=B * k / (ms * 1e-3), gbs=gbs(nb, ms), frac=gbs(nb, ms) / peak,
        bytes=nb)
    rows_t = d["target"].reshape(-1, V)
    gws = torch.zeros(sv.logit_gap_gate_workspace(rows_t.shape[0], V, sv.SV_F32),
                      dtype=torch.uint8, device=dev)
    ms = statistics.median(time_launches(
        lambda: sv.logit_gap_gate(rows_t, d["tau"], d["answer_set"], workspace=gws, stream=stream),
        steps, 3, stream))
    nb = rows_t.numel() * 4
    rows["gate_n1280_v151936_f32"] = dict(ms=ms, rows_per_s=rows_t.shape[0] / (ms * 1e-3),
                                          gbs=gbs(nb, ms), frac=gbs(nb, ms) / peak, bytes=nb)
    del d, rows_t, ws, gws

    # greedy verify on the headline batch's target rows (B=512, k=8, V=128256 bf16, 1.18 GB)
    if head is not None:
        B, k, V = head["B"], head["k"], head["V"]
        gws = torch.zeros(sv.spec_verify_greedy_workspace(B, k, V, sv.SV_BF16),
                          dtype=torch.uint8, device=dev)
        ms = statistics.median(time_launches(
            lambda: sv.spec_verify_greedy(head["target"], head["draft_tokens"], None,
                                          workspace=gws, stream=stream),
            steps, 3, stream))
        nb = B * (k + 1) * V * 2
        rows[f"greedy_b{B}_k{k}_v{V}_bf16"] = dict(
            ms=ms, positions_per_s=B * k / (ms * 1e-3), gbs=gbs(nb, ms),
            frac=gbs(nb, ms) / peak, bytes=nb)
        del gws
        # draft-side confidence stop on the same batch's draft rows (k rows per request)
        nb = B * k * V * 2
        cws = torch.zeros(sv.draft_confidence_workspace(B, k, V, sv.SV_BF16), dtype=torch.uint8,
                          device=dev)
        cnd = torch.empty((B,), dtype=torch.int32, device=dev)
        cc = torch.empty((B, k), dtype=torch.float32, device=dev)
        for mode, name, floor in ((sv.SV_CONF_TOP_PROB, "top", 0.05),
                                  (sv.SV_CONF_INV_ENTROPY, "inv_entropy", 0.2)):
            ms = statistics.median(time_launches(
                lambda: sv.draft_confidence_stop(head["draft"], head["T"], mode, floor,
                                                 out_num_draft=cnd, out_conf=cc,
                                                 workspace=cws, stream=stream),
                steps, 3, stream))
            rows[f"confidence_{name}_b{B}_k{k}_v{V}_bf16"] = dict(
                ms=ms, positions_per_s=B * k / (ms * 1e-3), gbs=gbs(nb, ms),
                frac=gbs(nb, ms) / peak, bytes=nb)
        del cws, cnd, cc
        # conformal residual of the draft rows against the target rows at the same positions
        tgt = head["target"][:, :k].contiguous()
        rr = torch.empty((B * k,), dtype=torch.float32, device=dev)
        ms = statistics.median(time_launches(
            lambda: sv.conformal_residual(head["draft"], tgt, out_resid=rr, stream=stream),
            steps, 3, stream))
        nb = 2 * B * k * V * 2
        rows[f"conformal_residual_b{B}_k{k}_v{V}_bf16"] = dict(
            ms=ms, rows_per_s=B * k / (ms * 1e-3), gbs=gbs(nb, ms), frac=gbs(nb, ms) / peak,
            bytes=nb)
        del tgt, rr
        # conformal gate over K = 4 layers: the batch's B*(k+1) target rows seen as
        # [B*(k+1)/4, 4, V] (1.18 GB)
        ns = B * (k + 1) // 4
        z4 = head["target"].reshape(-1, V)[: ns * 4].reshape(ns, 4, V)
        Q4 = torch.tensor([3.0, 2.0, 1.5, 1.0], dtype=torch.float32, device=dev)
        aws = torch.zeros(sv.conformal_admit_workspace(ns, 4, V, sv.SV_BF16), dtype=torch.uint8,
                          device=dev)
        ms = statistics.median(time_launches(
            lambda: sv.conformal_admit(z4, Q4, want_gap=False, workspace=aws, stream=stream),
            steps, 3, stream))
        nb = ns * 4 * V * 2
        rows[f"conformal_admit_n{ns}_k4_v{V}_bf16"] = dict(
            ms=ms, steps_per_s=ns / (ms * 1e-3), gbs=gbs(nb, ms), frac=gbs(nb, ms) / peak,
            bytes=nb)
        del z4, aws

    # ready-distribution cache: record 2048 sessions from the headline's target rows (0.53 GB
    # scanned; with the full distributions kept, as much again written), then serve 16384
    # requests against them
    if head is not None:
        V = head["V"]
        S, E = 2048, 16
        zr = head["target"].reshape(-1, V)[:S]
        g = torch.Generator(device=dev).manual_seed(6)
        sid = torch.arange(S, dtype=torch.int32, device=dev)
        ent = torch.randint(0, 1000, (S, E), generator=g, device=dev, dtype=torch.int32)
        n_s = torch.randint(0, 4096, (S,), generator=g, device=dev)
        L = torch.full((S,), E, dtype=torch.int32, device=dev)
        Bh = torch.full((S,), 64, dtype=torch.int64, device=dev)
        st_out = torch.empty((S,), dtype=torch.int32, device=dev)
        rws = torch.zeros(sv.ready_cache_record_workspace(S, V, sv.SV_BF16), dtype=torch.uint8,
                          device=dev)
        for keep, tag in ((False, ""), (True, "_keep_dist")):
            table = sv.ReadyCacheTable(S, E, dev, V=V, dist_dtype=torch.bfloat16,
                                       keep_dist=keep)
            ms = statistics.median(time_launches(
                lambda: table.record(sid, n_s, ent, L, Bh, zr, out_status=st_out,
                                     workspace=rws, stream=stream), steps, 3, stream))
            nb = S * V * 2 * (2 if keep else 1)
            rows[f"ready_cache_record_s{S}_v{V}_bf16{tag}"] = dict(
                ms=ms, sessions_per_s=S / (ms * 1e-3), gbs=gbs(nb, ms), frac=gbs(nb, ms) / peak,
                bytes=nb)
        R = 16384
        rs = torch.randint(0, S, (R,), generator=g, device=dev, dtype=torch.int32)
        rstart, rtok, rlen = n_s[rs.long()], ent[rs.long()], L[rs.long()]
        A = torch.arange(0, V, 3, dtype=torch.int32, device=dev)
        otok = torch.empty((R,), dtype=torch.int32, device=dev)
        orea = torch.empty((R,), dtype=torch.int32, device=dev)
        ms = statistics.median(time_launches(
            lambda: table.serve(rs, rstart, rtok, rlen, 2.0, A, out_token=otok, out_reason=orea,
                                stream=stream), steps, 3, stream, flush))
        rows[f"ready_cache_serve_r{R}"] = dict(ms=ms, requests_per_s=R / (ms * 1e-3),
                                                us=ms * 1e3)
        del table, rws, zr

    # gate calibration: risk-coverage sweep over 16M decision points and 1024 thresholds
    # (201 MB of inputs, past L2), and at the pre-positioning page's 128 points
    g = torch.Generator(device=dev).manual_seed(5)
    for npts, T, tag in ((1 << 24, 1024, "n16m_t1024"), (128, 64, "n128_t64")):
        gp = torch.rand((npts,), generator=g, device=dev) * 8
        tk = torch.randint(0, 64, (npts,), generator=g, device=dev, dtype=torch.int32)
        fl = torch.where(torch.rand((npts,), generator=g, device=dev) < 0.9, tk, tk + 1)
        A = torch.arange(0, 64, 2, dtype=torch.int32, device=dev)
        taus = torch.linspace(0, 8, T, device=dev)
        sws = torch.zeros(sv.gate_risk_coverage_workspace(npts, T), dtype=torch.uint8,
                          device=dev)
        pts = torch.empty((T, 8), dtype=torch.float64, device=dev)
        ti = torch.empty((1,), dtype=torch.int32, device=dev)
        ms = statistics.median(time_launches(
            lambda: sv.gate_risk_coverage(gp, tk, fl, A, taus, 1.959964, 0.1, out_points=pts,
                                          out_tau_index=ti, workspace=sws, stream=stream),
            steps, 3, stream, flush if npts < (1 << 20) else None))
        nb = npts * 12
        rows[f"gate_risk_coverage_{tag}"] = dict(
            ms=ms, points_per_s=npts / (ms * 1e-3), gbs=gbs(nb, ms), frac=gbs(nb, ms) / peak,
            bytes=nb)
        del gp, tk, fl, sws, pts, ti
    # split-conformal quantile of 16M scores (64 MB, three radix passes) and of 4096
    for n, tag in ((1 << 24, "n16m"), (4096, "n4096")):
        rs = torch.rand((n,), generator=g, device=dev)
        qws = torch.zeros(sv.conformal_quantile_workspace(n), dtype=torch.uint8, device=dev)
        qo = torch.empty((1,), dtype=torch.float32, device=dev)
        ms = statistics.median(time_launches(
            lambda: sv.conformal_quantile(rs, 0.9, out_q=qo, workspace=qws, stream=stream),
            steps, 3, stream, flush))
        rows[f"conformal_quantile_{tag}"] = dict(ms=ms, scores_per_s=n / (ms * 1e-3),
                                                 gbs=gbs(3 * n * 4, ms), bytes=3 * n * 4)
        del rs, qws, qo

    # bf16 Zipf workload: sampled + greedy (fits in L2: flushed before every launch)
    w = synth.WORKLOADS[1]
    d = synth.workload_inputs(w, device=dev)
    B, k, V = d["B"], d["k"], d["V"]
    ws = torch.zeros(sv.spec_verify_sample_workspace(B, k, V, sv.SV_BF16), dtype=torch.uint8,
                     device=dev)
    ms = statistics.median(time_launches(
        lambda: sv.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                                      d["T"], None, workspace=ws, stream=stream),
        steps, 3, stream, flush))
    nb = sample_bytes(B * k, B, k, V, 2)
    rows["sample_b64_k5_v32000_bf16_l2flushed"] = dict(
        ms=ms, positions_per_s=B * k / (ms * 1e-3), gbs=gbs(nb, ms), frac=gbs(nb, ms) / peak,
        bytes=nb)
    gws = torch.zeros(sv.spec_verify_greedy_workspace(B, k, V, sv.SV_BF16), dtype=torch.uint8,
                      device=dev)
    ms = statistics.median(time_launches(
        lambda: sv.spec_verify_greedy(d["target"], d["draft_tokens"], None, workspace=gws,
                                      stream=stream),
        steps, 3, stream, flush))
    nb = B * (k + 1) * V * 2
    rows["greedy_b64_k5_v32000_bf16_l2flushed"] = dict(
        ms=ms, positions_per_s=B * k / (ms * 1e-3), gbs=gbs(nb, ms), frac=gbs(nb, ms) / peak,
        bytes=nb)
    del d, ws, gws

    # tiny fp32 case: latency
    d = synth.workload_inputs(0, device=dev)
    ms = statistics.median(time_launches(
        lambda: sv.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                                      d["T"], None, stream=stream), steps, 3, stream, flush))
    rows["sample_b1_k4_v1000_f32_latency"] = dict(ms=ms, us=ms * 1e3)

    # the two small workloads replayed from a CUDA graph, as a serving loop runs them: no host
    # launch overhead, inputs warm in L2 (per call: the replay of 20 captured calls / 20)
    for wi, tag in ((0, "sample_b1_k4_v1000_f32_graph"), (1, "sample_b64_k5_v32000_bf16_graph")):
        d = synth.workload_inputs(wi, device=dev)
        B, k, V = d["B"], d["k"], d["V"]
        code = sv.SV_F32 if d["dtype"] == "f32" else sv.SV_BF16
        ws = torch.zeros(sv.spec_verify_sample_workspace(B, k, V, code), dtype=torch.uint8,
                         device=dev)
        per_graph = 20

        def call():
            sv.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                                  d["T"], None, workspace=ws)

        side = torch.cuda.Stream(device=dev)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(3):
                call()
        torch.cuda.current_stream().wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(per_graph):
                call()
        ms = statistics.median(time_launches(graph.replay, steps, 3, stream)) / per_graph
        rows[tag] = dict(ms=ms, us=ms * 1e3, positions_per_s=B * k / (ms * 1e-3))
        del d, ws, graph

    # n-gram proposal feeding the greedy verify (B=128, L=8192, V=32000)
    w4 = synth.workload_inputs(4, device=dev)
    dr, nd = sv.ngram_propose(w4["history"], w4["hist_len"], w4["n_max"], w4["n_min"], w4["k"])
    torch.cuda.synchronize()
    tgt = synth.greedy_targets(dr, nd, w4["V"], k=w4["k"], seed=w4["seed"])
    gws = torch.zeros(sv.spec_verify_greedy_workspace(w4["B"], w4["k"], w4["V"], sv.SV_BF16),
                      dtype=torch.uint8, device=dev)
    od, on = torch.empty_like(dr), torch.empty_like(nd)

    def chain():
        sv.ngram_propose(w4["history"], w4["hist_len"], w4["n_max"], w4["n_min"], w4["k"],
                         out_draft=od, out_num_draft=on, stream=stream)
        sv.spec_verify_greedy(tgt, od, on, workspace=gws, stream=stream)

    ms = statistics.median(time_launches(chain, steps, 3, stream, flush))
    npos = int(nd.sum().item())
    nb = w4["history"].numel() * 4 + int((nd.clamp(min=0) + 1).sum().item()) * w4["V"] * 2
    rows["ngram_greedy_b128_l8192_v32000_bf16_l2flushed"] = dict(
        ms=ms, proposed_positions=npos, requests_with_proposal=int((nd > 0).sum().item()),
        positions_per_s=npos / (ms * 1e-3), gbs=gbs(nb, ms), bytes=nb)
    ms = statistics.median(time_launches(
        lambda: sv.ngram_propose(w4["history"], w4["hist_len"], w4["n_max"], w4["n_min"],
                                 w4["k"], out_draft=od, out_num_draft=on, stream=stream),
        steps, 3, stream, flush))
    rows["ngram_b128_l8192"] = dict(ms=ms, us=ms * 1e3)
    return rows


# ------------------------------------------------------------------------------ CPU oracle
def _oracle_sample_rate(target, draft, tokens, uniforms, T, threads):
    import oracle

    t0 = time.perf_counter()
    oracle.spec_verify_sample(target, draft, tokens, None, uniforms, T, threads=threads)
    return time.perf_counter() - t0


def _one_thread(target, draft, tokens, uniforms, T, budget_s):
    """The oracle on one host thread, over the first requests of the sample that fit in
    about budget_s seconds: (positions per second, requests, seconds)."""
    k = tokens.shape[1]
    t1 = _oracle_sample_rate(target[:1], draft[:1], tokens[:1], uniforms[:1], T, 1)
    n1 = int(min(target.shape[0], max(1, budget_s / max(t1, 1e-6))))
    t = _oracle_sample_rate(target[:n1], draft[:n1], tokens[:n1], uniforms[:n1], T, 1)
    return n1 * k / t, n1, t


def cpu_baseline(d, w, budget_s=15.0):
    """The oracle, as it stands, on the host cores, over a bounded sample of the requests
    of the same workload (inputs copied from the device): the rate on every core, and the
    rate of one thread on a smaller sample."""
    threads = os.cpu_count() or 1
    k = d["k"]
    # calibrate on a few requests, then size the sample for ~budget_s of CPU time
    n0 = min(d["B"], threads)
    sl = slice(0, n0)
    t = _oracle_sample_rate(d["target"][sl].cpu(), d["draft"][sl].cpu(),
                            d["draft_tokens"][sl].cpu(), d["uniforms"][sl].cpu(), d["T"], threads)
    cpu_per_req = t * threads / n0
    n = int(min(d["B"], max(n0, budget_s / max(cpu_per_req, 1e-6))))
    sl = slice(0, n)
    tgt, dft = d["target"][sl].cpu(), d["draft"][sl].cpu()
    tok, uni = d["draft_tokens"][sl].cpu(), d["uniforms"][sl].cpu()
    t = _oracle_sample_rate(tgt, dft, tok, uni, d["T"], threads)
    v1, n1, t1 = _one_thread(tgt, dft, tok, uni, d["T"], budget_s / 3)
    return {"value": n * k / t, "unit": "positions/s", "cores": threads, "kind": "oracle",
            "sample": f"first {n} of {d['B']} requests ({n * k} positions), {t:.2f} s on "
                      f"{threads} threads",
            "one_thread": {"value": v1, "unit": "positions/s",
                           "sample": f"first {n1} requests on 1 thread, {t1:.2f} s"}}


def reference_arm(args, rank, world):
    """The oracle timed on the host cores on the same workload, metric and unit."""
    if rank != 0:
        return
    import synth

    w = synth.WORKLOADS[args.workload]
    e = w.extra
    threads = os.cpu_count() or 1
    per_step = max(threads, 16)
    d = synth.sample_inputs(per_step, w.k, w.V, w.dtype, w.T, device="cpu",
                            seed=synth.SEED_BASE + w.index, target_std=e["target_std"],
                            draft_noise=e["draft_noise"], draft_scale=e["draft_scale"],
                            peak=e.get("peak"))
    for _ in range(args.warmup):
        _oracle_sample_rate(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], w.T,
                            threads)
    times = [_oracle_sample_rate(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], w.T,
                                 threads) for _ in range(args.steps)]
    total = sum(times)
    value = per_step * w.k * args.steps / total
    # one thread, on the step's sample (after the timed steps)
    v1, n1, t1 = _one_thread(d["target"], d["draft"], d["draft_tokens"], d["uniforms"], w.T,
                             args.cpu_seconds / 3)
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "positions/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded; shapes and value distributions of the workload)",
        "config": {"workload": f"sampled verify {w.name}: B={w.B}, k={w.k}, V={w.V}, "
                               f"{w.dtype} logits, T={w.T}, {TIMED_WORKLOADS[w.index]}; each step "
                               f"a bounded sample of {per_step} requests",
                   "global_batch": per_step, "parallelism": f"{threads} host threads"},
        "cpu_baseline": {"value": value, "unit": "positions/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{per_step} requests per step ({per_step * w.k} positions)",
                         "one_thread": {"value": v1, "unit": "positions/s",
                                        "sample": f"{n1} requests on 1 thread, {t1:.2f} s"}},
        "e2e": {"value": value, "unit": "positions/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def kernels_once():
    """Two passes of one launch of each secondary call, on workloads past L2, and nothing
    timed: the command line for an ncu capture of those kernels. Order in each pass: logit_gap_gate
    (1280 fp32 rows of V=151936), spec_verify_greedy, draft_confidence_stop (top probability,
    then inverse entropy) and conformal_admit (K=4) on the B=256 k=8 V=128256 bf16 batch,
    conformal_residual (its draft rows against target rows 0..k-1), gate_risk_coverage (16M
    points, 1024 thresholds), conformal_quantile (16M scores), ready_cache_record (2048
    sessions from that batch's target rows) and ready_cache_serve (16384 requests), and
    ngram_propose (128 histories of 8192 tokens)."""
    import torch

    import speculative_decoding_verification_17_gb300 as sv
    import synth

    dev = torch.device("cuda")
    d = synth.workload_inputs(HEAD, device=dev, B=256)
    B, k, V = d["B"], d["k"], d["V"]
    w2 = synth.workload_inputs(2, device=dev)
    rows2 = w2["target"].reshape(-1, w2["V"])
    tgt = d["target"][:, :k].contiguous()
    ns = B * (k + 1) // 4
    z4 = d["target"].reshape(-1, V)[: ns * 4].reshape(ns, 4, V)
    Q4 = torch.tensor([3.0, 2.0, 1.5, 1.0], device=dev)
    g = torch.Generator(device=dev).manual_seed(5)
    npts = 1 << 24
    gp = torch.rand((npts,), generator=g, device=dev) * 8
    tk = torch.randint(0, 64, (npts,), generator=g, device=dev, dtype=torch.int32)
    fl = torch.where(torch.rand((npts,), generator=g, device=dev) < 0.9, tk, tk + 1)
    A = torch.arange(0, 64, 2, dtype=torch.int32, device=dev)
    taus = torch.linspace(0, 8, 1024, device=dev)
    rs = torch.rand((npts,), generator=g, device=dev)
    S, E, R = 2048, 16, 16384
    zr = d["target"].reshape(-1, V)[:S]
    sid = torch.arange(S, dtype=torch.int32, device=dev)
    ent = torch.randint(0, 1000, (S, E), generator=g, device=dev, dtype=torch.int32)
    n_s = torch.randint(0, 4096, (S,), generator=g, device=dev)
    L = torch.full((S,), E, dtype=torch.int32, device=dev)
    Bh = torch.full((S,), 64, dtype=torch.int64, device=dev)
    table = sv.ReadyCacheTable(S, E, dev, V=V, dist_dtype=torch.bfloat16, keep_dist=False)
    rq = torch.randint(0, S, (R,), generator=g, device=dev, dtype=torch.int32)
    rstart, rtok, rlen = n_s[rq.long()], ent[rq.long()], L[rq.long()]
    Av = torch.arange(0, V, 3, dtype=torch.int32, device=dev)
    w4 = synth.workload_inputs(4, device=dev)
    for _ in range(2):
        sv.logit_gap_gate(rows2, w2["tau"], w2["answer_set"])
        sv.spec_verify_greedy(d["target"], d["draft_tokens"])
        sv.draft_confidence_stop(d["draft"], d["T"], sv.SV_CONF_TOP_PROB, 0.05)
        sv.draft_confidence_stop(d["draft"], d["T"], sv.SV_CONF_INV_ENTROPY, 0.2)
        sv.conformal_admit(z4, Q4, want_gap=False)
        sv.conformal_residual(d["draft"], tgt)
        sv.gate_risk_coverage(gp, tk, fl, A, taus, 1.959964, 0.1)
        sv.conformal_quantile(rs, 0.9)
        table.record(sid, n_s, ent, L, Bh, zr)
        table.serve(rq, rstart, rtok, rlen, 2.0, Av)
        sv.ngram_propose(w4["history"], w4["hist_len"], w4["n_max"], w4["n_min"], w4["k"])
    torch.cuda.synchronize()
    print("kernels-once ok")


def small_once():
    """Three calls each of the two small sampled-verify workloads (B=1, k=4, V=1000 fp32, then
    B=64, k=5, V=32000 bf16), each after an L2 flush, and nothing timed: the command line for
    an ncu capture of the small batches' kernels."""
    import torch

    import speculative_decoding_verification_17_gb300 as sv
    import synth

    dev = torch.device("cuda")
    flush = make_flush(dev)
    for wi in (0, 1):
        d = synth.workload_inputs(wi, device=dev)
        B, k, V = d["B"], d["k"], d["V"]
        code = sv.SV_F32 if d["dtype"] == "f32" else sv.SV_BF16
        ws = torch.zeros(sv.spec_verify_sample_workspace(B, k, V, code), dtype=torch.uint8,
                         device=dev)
        for _ in range(3):
            flush()
            sv.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], d["uniforms"],
                                  d["T"], None, workspace=ws)
    torch.cuda.synchronize()
    print("small-once ok")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-rows", action="store_true", help="skip the secondary rows")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--workload", type=int, choices=sorted(TIMED_WORKLOADS), default=HEAD,
                    help="the sampled-verify workload to time (default: the headline, 3)")
    ap.add_argument("--requests", type=int, default=None,
                    help="batch size of the timed workload (default: its own)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end leg")
    ap.add_argument("--kernels-once", action="store_true",
                    help="one untimed launch of each secondary call (for an ncu capture)")
    ap.add_argument("--small-once", action="store_true",
                    help="three untimed calls of each small sampled workload (for an ncu capture)")
    args = ap.parse_args()
    if args.kernels_once:
        kernels_once()
        return
    if args.small_once:
        small_once()
        return
    args.warmup = max(3, args.warmup)  # at least three untimed warm-up steps
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        reference_arm(args, rank, world)
    else:
        gb300_arm(args, rank, world, local_rank)


if __name__ == "__main__":
    main()

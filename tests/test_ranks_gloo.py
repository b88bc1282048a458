"""The multi-rank path of the benchmark, on host cores with gloo and two ranks.

Under torchrun every rank verifies its own shard of requests (no collective on the data path)
and the ranks meet only for barriers and for the max-over-ranks timing. These tests run that
host logic with world size 2 on the CPU: the process group, the per-rank seeds, the maximum of
the step times, the whole-job rate, that each rank's shard is independent of the others, and
that the reference arm prints one line from rank 0 only.
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    import synth

    dist = bench.init_ranks(world, torch.device("cpu"))
    # this rank's shard: a small sampled-verify batch from its own seed, verified locally
    d = synth.sample_inputs(3, 4, 1000, "f32", 0.8, device="cpu",
                            seed=bench.rank_seed(rank))
    o = oracle.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], None,
                                  d["uniforms"], 0.8)
    step_ms = 3.0 + 2.0 * rank  # rank 1 is the slow one
    dist.barrier()
    slowest = bench.max_over_ranks(dist, step_ms, torch.device("cpu"))
    rate = bench.whole_job_rate(world, 3 * 4, 10, slowest * 10)
    dist.barrier()
    dist.destroy_process_group()
    np.savez(os.path.join(out_dir, f"rank{rank}.npz"), tok=o["tokens"], acc=o["accept_len"],
             target=d["target"].numpy(), slowest=slowest, rate=rate, seed=bench.rank_seed(rank))


def test_two_gloo_ranks_share_timing_not_data(tmp_path):
    import oracle
    import synth

    world, port = 2, _free_port()
    mp.start_processes(_rank_main, args=(world, port, str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    r = [np.load(tmp_path / f"rank{i}.npz") for i in range(world)]
    # both ranks see the slowest rank's time, and the rate counts every rank's positions
    for x in r:
        assert float(x["slowest"]) == 5.0
        assert float(x["rate"]) == pytest.approx(world * 3 * 4 / 5e-3)
    # distinct seeds, distinct shards
    assert int(r[0]["seed"]) != int(r[1]["seed"])
    assert not np.array_equal(r[0]["target"], r[1]["target"])
    # each rank's result is what one process gets from that rank's seed: no cross-rank data
    import bench

    for i, x in enumerate(r):
        d = synth.sample_inputs(3, 4, 1000, "f32", 0.8, device="cpu",
                                seed=bench.rank_seed(i))
        o = oracle.spec_verify_sample(d["target"], d["draft"], d["draft_tokens"], None,
                                      d["uniforms"], 0.8)
        assert np.array_equal(o["tokens"], x["tok"])
        assert np.array_equal(o["accept_len"], x["acc"])
        assert (o["accept_len"] >= 0).all()


def test_single_rank_needs_no_process_group():
    import bench

    assert bench.init_ranks(1, torch.device("cpu")) is None
    assert bench.max_over_ranks(None, 2.5, torch.device("cpu")) == 2.5
    assert bench.whole_job_rate(1, 4096, 50, 25.0) == pytest.approx(4096 * 50 / 0.025)


def test_reference_arm_under_torchrun_prints_one_line_from_rank_zero():
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(port),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3"]
    env = dict(os.environ, OMP_NUM_THREADS="1")
    p = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    assert line["n_gpus"] == 2
    assert line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle"

"""The N > 1 path on CPU: world-size-2 gloo process groups.

The attention path shards with no exchange (every (batch, head) problem is
independent), so the multi-rank logic is only timing aggregation (max over
ranks), the whole-job throughput arithmetic, per-rank input seeds, and
"rank 0 prints one line".  These run here without a GPU.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    sys.path.insert(0, ROOT)
    import bench
    from io_aware_attention_flash_gb300 import workloads as wl

    got = bench.max_over_ranks([10.0 + rank, 5.0 - rank, float(rank)], torch.device("cpu"))
    # each rank draws its own batch: seed + rank
    q0 = wl.make_inputs(1, 8, 1, 64, seed=100 + rank)[0]
    digests = [None] * world
    dist.all_gather_object(digests, float(q0.float().sum()))
    out[rank] = {"max": got, "distinct_inputs": len(set(digests)) == world}
    dist.destroy_process_group()


def test_timing_aggregation_over_two_gloo_ranks():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        assert res[rank]["max"] == [11.0, 5.0, 1.0]
        assert res[rank]["distinct_inputs"]


def test_whole_job_throughput_is_weak_scaling():
    sys.path.insert(0, ROOT)
    import bench
    # two ranks each did 1e12 FLOPs; the slower took 2 ms -> 1000 TFLOP/s job-wide
    assert bench.whole_job_tflops(2, 1e12, 2.0) == pytest.approx(1000.0)
    assert bench.max_over_ranks([1.0, 2.0], torch.device("cpu")) == [1.0, 2.0]  # no process group


def test_reference_arm_under_torchrun_prints_once():
    """`bench.py --impl reference` launched like the multi-GPU driver (two
    ranks): rank 0 alone times the oracle and prints one JSON line; the other
    rank exits 0 without work."""
    port = _free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3", "--workload", "small"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["value"] > 0 and rec["n_gpus"] == 2
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["e2e"]["h2d_bytes_per_step"] == 0

"""The N>1 path of bench.py on CPU with the gloo backend (world size 2).

The attention path needs no collective: each rank runs its own replica of the
workload.  What crosses ranks is only the timing: a barrier around the timed
region and the slowest rank's time (max over ranks), from which rank 0 reports
whole-job throughput.  These tests run that logic with gloo on CPU, and the
reference arm under torchrun, where rank 0 alone works and prints."""
import json
import os
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

from conftest import ROOT


def _worker(rank, world, port, times, out_q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    slowest = bench.max_over_ranks(times[rank], dist, device="cpu")
    value = bench.weak_scaling_value(1e9, slowest, world)
    out_q.put((rank, slowest, value))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_weak_scaling_with_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [1.25, 2.5]
    port = 29531
    procs = [ctx.Process(target=_worker, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [2.5, 2.5]                 # both ranks agree on the slowest time
    assert res[0][2] == pytest.approx(2 * 1e9 / 2.5e-3 / 1e9)  # 2 replicas of 1 GB in 2.5 ms


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.0, None) == 3.0
    assert bench.weak_scaling_value(2e9, 1.0, 1) == pytest.approx(2000.0)


def test_reference_arm_under_torchrun_prints_once(tmp_path):
    """--impl reference at N=2: rank 0 times the CPU oracle and prints one line; rank 1 exits 0."""
    env = dict(os.environ, OMP_NUM_THREADS="1", PYTHONPATH=ROOT)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", "--master-port=29533", os.path.join(ROOT, "bench.py"),
           "--impl", "reference", "--gpus", "2", "--steps", "2", "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env, cwd=tmp_path, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["unit"] == "GB/s" and rec["cpu_baseline"]["kind"] == "oracle"

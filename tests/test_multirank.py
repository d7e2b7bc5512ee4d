"""The benchmark's multi-rank path on the CPU with two gloo ranks.

The product shards by rows with no exchange, so several GPUs run independent
replicas: the timed regions meet at a barrier and each time is the largest
over the ranks (bench.barrier, bench.max_over_ranks); the reference arm runs
on rank 0 alone, the other ranks leaving without work.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import time

    import torch.distributed as tdist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        time.sleep(0.05 * rank)          # ranks arrive at different times
        bench.barrier()
        v = bench.max_over_ranks(1.5 + rank)
        w = bench.max_over_ranks(-3.0 * (rank + 1))
        bench.barrier()
        q.put((rank, v, w))
    finally:
        tdist.destroy_process_group()


def test_max_over_ranks_and_barrier_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 2.5, -3.0), (1, 2.5, -3.0)]


def test_single_process_helpers():
    sys.path.insert(0, ROOT)
    import bench
    bench.barrier()                      # no process group: nothing to do
    assert bench.max_over_ranks(4.25) == 4.25


@pytest.mark.parametrize("rank", [1])
def test_reference_arm_other_ranks_exit_quietly(rank):
    """Under torchrun the reference arm's rank 0 alone runs and prints; rank 1
    exits 0 at once with no output."""
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""


def test_reference_arm_ffn_block():
    """The reference arm on the Q6_K-like FFN block (gate and up from one
    activation, down at K = 14336): one JSON line timing the oracle over
    sampled rows of all three matrices."""
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "q6k_ffn_14336x4096", "--steps", "1", "--warmup", "1"], capture_output=True, text=True,
                       env=env, timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["config"]["down"] == [4096, 14336] and d["config"]["gate_up_rows"] == [14336, 14336]


def _all_workloads():
    sys.path.insert(0, ROOT)
    import bench
    return (sorted(bench.WORKLOADS) + sorted(bench.GROUPED) + sorted(bench.FFN) + sorted(bench.KV) +
            sorted(bench.FP8) + sorted(bench.STACK) + sorted(bench.W2))


@pytest.mark.parametrize("workload", _all_workloads())
def test_reference_arm_every_workload(workload):
    """Every workload's reference arm (the oracle on the host cores) prints one
    line with the metric, unit and direction the GPU arm reports, so the two
    lines compare."""
    sys.path.insert(0, ROOT)
    import bench
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        workload, "--steps", "1", "--warmup", "1"], capture_output=True, text=True, env=env,
                       timeout=900)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["metric"] == bench.metric_for(workload)
    assert d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1

"""The benchmark's multi-rank path on CPU (gloo, world size 2): every rank runs
its own rows with no data-path collective; the job's time is the slowest
rank's and its throughput counts all ranks' tokens."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    slowest = bench.max_over_ranks(1.0 + rank, world)
    value = bench.job_throughput(65536, world, slowest)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, slowest, value))


def test_two_rank_aggregation_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in res:
        assert slowest == pytest.approx(2.0)
        assert value == pytest.approx(2 * 65536 / 2e-3)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(1000, 1, 1.0) == pytest.approx(1e6)


def test_reference_arm_prints_on_rank_zero_only():
    """Under torchrun the reference arm (the oracle on the host cores) runs and
    prints on rank 0; the other ranks exit 0 without work."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "1"]
    env1 = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    r1 = subprocess.run(cmd, env=env1, capture_output=True, text=True, timeout=300)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    env0 = dict(os.environ, RANK="0", LOCAL_RANK="0", WORLD_SIZE="2")
    r0 = subprocess.run(cmd, env=env0, capture_output=True, text=True, timeout=300)
    assert r0.returncode == 0, r0.stderr
    lines = [l for l in r0.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["config"]["workload"] == "fixed256_B8H12N8192"

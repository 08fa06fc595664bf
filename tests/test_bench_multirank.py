"""The benchmark's multi-rank host logic on CPU: two gloo ranks (the N>1 path
launched by torchrun runs N independent replicas, one per GPU, and reports the
slowest rank's time and the whole job's throughput).  No GPU is used."""
import os
import socket
import subprocess
import sys
from pathlib import Path

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = Path(__file__).resolve().parent.parent


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, str(ROOT))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank's own step time; the job takes as long as the slowest
        local_ms = [3.0, 5.0][rank]
        slowest = bench.max_over_ranks(local_ms)
        value = bench.job_throughput(1e12, world, slowest)
        out.put((rank, slowest, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time_and_job_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see the slower rank's 5 ms; 2 ranks x 1 TFLOP each in 5 ms = 400 TFLOP/s
    assert [r[1] for r in results] == [5.0, 5.0]
    assert all(abs(r[2] - 400.0) < 1e-9 for r in results)


def test_single_process_helpers():
    sys.path.insert(0, str(ROOT))
    import bench
    assert bench.max_over_ranks(7.5) == 7.5
    assert bench.job_throughput(2e12, 1, 4.0) == pytest.approx(500.0)


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun every rank but 0 exits 0 at once, printing nothing."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""

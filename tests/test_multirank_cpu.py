"""The benchmark's multi-rank host logic with world_size 2 on gloo (CPU, no GPU): ranks run
independent replicas, the job time is the slowest rank's, the value counts every rank's work,
and the reference arm prints from rank 0 only."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        my_ms = 1.0 + rank  # rank 1 is the slow one
        ms = bench.max_over_ranks(my_ms, world)
        out[rank] = (ms, bench.job_throughput(100.0, world, ms))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_slowest_rank_sets_the_time():
    world = 2
    out = mp.Manager().dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    for r in range(world):
        ms, value = out[r]
        assert ms == 2.0
        assert value == pytest.approx(100.0 * 2 / 2.0e-3)


def test_reference_arm_prints_on_rank0_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""

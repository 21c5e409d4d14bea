"""The N > 1 bench path on CPU: replicas with max-over-ranks timing (gloo, world size 2)."""
import os
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.reduce_max(1.0 + rank * 0.5, world, "cpu")
        out[rank] = t
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_reduce_max_over_two_gloo_ranks():
    world = 2
    port = 29500 + (os.getpid() % 1000)
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, start_method="spawn")
    assert dict(out) == {0: 1.5, 1: 1.5}


def test_whole_job_value_is_replica_sum():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.whole_job_gbs(1e9, 1, 1.0)
    assert one == pytest.approx(1000.0)
    assert bench.whole_job_gbs(1e9, 4, 1.0) == pytest.approx(4 * one)


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0 and r.stdout.strip() == ""

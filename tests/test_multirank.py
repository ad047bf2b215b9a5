"""The benchmark's multi-rank logic on CPU with the gloo backend
(world_size 2): max over ranks, the whole-job rate of replicas, and the
reference arm's non-zero ranks exiting without work."""
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    got = bench.max_over_ranks(ms, world, "cpu")
    out[rank] = (got, bench.job_rate(1e9, got, world))
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_with_gloo():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn")
    for r in range(world):
        got, rate = out[r]
        assert got == 15.0  # every rank sees the slowest rank's time
        assert rate == pytest.approx(2 * 1e9 / 15e-3 / 1e9)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert p.returncode == 0
    assert p.stdout.strip() == ""

"""Host logic of bench.py for more than one rank, on the CPU.

With N ranks the bench runs N independent replicas of the step (one per
GPU; the path has no exchange step) and reports the whole job: the slowest
rank's time and the work of all ranks.  The aggregation is checked here
with two gloo ranks; the reference arm prints from rank 0 only, and the
other ranks exit 0 without work.
"""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        value, total = bench.job_rate(2.0e12, 10, times[rank], world, torch.device("cpu"))
        out[rank] = (value, total)
    finally:
        dist.destroy_process_group()


def test_job_rate_takes_the_slowest_rank_and_all_work():
    world, times = 2, [100.0, 150.0]
    out = mp.Manager().dict()
    mp.start_processes(_worker, args=(world, _free_port(), times, out), nprocs=world,
                       start_method="spawn")
    want_total = max(times)
    want_value = 2.0e12 * 10 * world / (want_total * 1e-3) / 1e12
    for rank in range(world):
        value, total = out[rank]
        assert total == want_total
        assert value == pytest.approx(want_value, rel=1e-12)


def test_job_rate_one_rank():
    sys.path.insert(0, ROOT)
    import bench
    value, total = bench.job_rate(3.0e12, 4, 20.0, 1, torch.device("cpu"))
    assert total == 20.0
    assert value == pytest.approx(3.0e12 * 4 / 0.02 / 1e12)


def test_reference_arm_other_ranks_exit_quietly():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "1"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""

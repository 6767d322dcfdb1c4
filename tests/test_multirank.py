"""The replica (weak-scaling) accounting of bench.py across two gloo ranks on
the CPU: every rank times its own replica, the job takes the slowest rank's
time, and the job rate is the units of all ranks over that time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                     # rank 1 is the slower replica
        slowest = bench.max_over_ranks(ms, world)  # CPU tensors: gloo
        out[rank] = (slowest, bench.job_rate(1e9, slowest, world))
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time_and_add_their_units():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        slowest, rate = out[rank]
        assert slowest == 15.0
        assert rate == pytest.approx(2 * 1e9 / 15e-3)


def test_one_rank_is_the_identity():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_rate(2e9, 4.0, 1) == pytest.approx(5e11)


def test_gpus_flag_must_match_the_launch():
    """--gpus N is honoured only as the world size of the launch: N ranks
    started by torchrun.  A mismatch is refused (non-zero exit), never run
    as a different number of replicas."""
    assert bench.check_world(1, 1) is None
    assert bench.check_world(8, 8) is None
    assert "WORLD_SIZE=1" in bench.check_world(8, 1)
    assert bench.check_world(2, 4) is not None
    assert bench.check_world(0, 1) is not None


def test_bench_exits_non_zero_when_gpus_exceeds_the_world():
    import subprocess
    import sys
    env = dict(os.environ, WORLD_SIZE="1", RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, bench.__file__, "--gpus", "2", "--steps", "1"],
                       capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 2 and "WORLD_SIZE=1" in r.stderr

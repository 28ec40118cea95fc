"""Multi-rank host logic of bench.py on CPU (gloo, world size 2).

With --gpus N every rank steps its own copy of the workload (weak scaling, no
data-path collective); the only exchange is the max over ranks of the timed
region, and rank 0 alone prints.  These tests run that logic on two gloo
ranks without a GPU.
"""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        mine = 10.0 + 5.0 * rank                       # rank 1 is the slow one
        out[rank] = bench.max_over_ranks(mine, world, torch.device("cpu"))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_two_gloo_ranks():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    assert out[0] == 15.0 and out[1] == 15.0


def test_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.job_throughput_gbs(87e9, 40.0, 1)
    two = bench.job_throughput_gbs(87e9, 40.0, 2)
    assert two == pytest.approx(2 * one)
    assert bench.max_over_ranks(3.5, 1, None) == 3.5


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the reference arm (the oracle on the host cores) runs on rank 0;
    every other rank exits 0 at once, without work or output."""
    import subprocess
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
               MASTER_PORT=str(_free_port()))
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                          "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=300, env=env,
                         cwd=ROOT)
    assert res.returncode == 0, res.stderr[-2000:]
    assert res.stdout.strip() == ""

"""The N > 1 path of bench.py on CPU: two gloo ranks run independent replicas, and the
whole-job rate is the units of both ranks over the slowest rank's time."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = [2.0, 3.0][rank]  # rank 1 is the slower replica
        value, t = bench.whole_job_rate(dist, torch, elapsed, 6.0)
        dist.barrier()
        out[rank] = (value, t)
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_whole_job_over_the_slowest_rank():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    for r in (0, 1):
        value, t = res[r]
        assert t == pytest.approx(3.0)
        assert value == pytest.approx(2 * 6.0 / 3.0)


def test_one_process_is_its_own_whole_job():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.whole_job_rate(None, torch, 2.0, 6.0) == (3.0, 2.0)

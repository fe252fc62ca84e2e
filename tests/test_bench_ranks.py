"""The benchmark's multi-rank aggregation on CPU: two gloo ranks with different times and unit
counts.  The job value is the units of all ranks over the slowest rank's time (max over ranks);
no data-path collective exists, only this reduction of the measurements."""
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


def _rank(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slowest
        local_units = 16 * (rank + 1)
        out[rank] = bench.job_throughput(local_ms, local_units)
    finally:
        dist.destroy_process_group()


def test_two_rank_job_throughput_uses_total_units_and_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank, args=(world, _free_port(), out), nprocs=world, join=True,
                           start_method="spawn")
        res = dict(out)
    for r in range(world):
        value, ms, units = res[r]
        assert units == 16 + 32
        assert ms == pytest.approx(15.0)
        assert value == pytest.approx(48 / 15e-3)


def test_single_process_job_throughput():
    sys.path.insert(0, ROOT)
    import bench
    value, ms, units = bench.job_throughput(4.0, 16)
    assert (units, ms) == (16, 4.0) and value == pytest.approx(4000.0)

"""The bench's multi-rank aggregation on CPU: two gloo ranks (replicas) report
different work and times; the whole-job value is the work of both over the
slower rank's time, and every rank gets the same figures."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    units = [3.0e9, 5.0e9][rank]
    ms = [12.0, 20.0][rank]
    out[rank] = bench.job_throughput(units, ms, world, "cpu")
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_sum_work_over_slowest_time():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    for r in range(world):
        value, slowest = res[r]
        assert slowest == 20.0
        assert value == pytest.approx(8.0e9 / 0.020)


def test_single_rank_is_local_throughput():
    import bench
    value, ms = bench.job_throughput(1.0e9, 4.0, 1)
    assert ms == 4.0 and value == pytest.approx(2.5e11)

"""The benchmark's multi-rank bookkeeping (replicas, no data-path collective)
on two gloo ranks on the CPU: the job time is the slowest rank's and the job
value counts every rank's replica."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist

    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, dist, "cpu")
    val = bench.job_tflops(1e12, 4, world, ms)
    dist.barrier()
    out[rank] = (ms, val)
    dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_rank_max_time_and_job_value():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert out[0] == out[1]
    ms, val = out[0]
    assert ms == 15.0
    assert abs(val - 1e12 * 4 * 2 / 15e-3 / 1e12) < 1e-9


def test_single_process_defaults():
    import bench

    assert bench.max_over_ranks(3.5) == 3.5
    assert bench.job_tflops(2e12, 10, 1, 20.0) == pytest.approx(1000.0)

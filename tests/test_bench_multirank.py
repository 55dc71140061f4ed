"""Host logic of bench.py's multi-process path on CPU: two gloo ranks.

bench.py runs one replica per GPU (the decode path needs no exchange between
GPUs).  Its only cross-rank logic is the barrier around the timed region and
the whole-job figure: units of all ranks over the slowest rank's time.  These
run here as two gloo processes on 127.0.0.1.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench.barrier(world)
    elapsed = bench.max_over_ranks(0.5 + rank * 0.25, "cpu")  # rank 1 is the slow one
    value = bench.job_throughput(100.0, 4, world, elapsed)
    bench.barrier(world)
    out[rank] = (elapsed, value)
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_slowest_time():
    world, port = 2, _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    assert out[0] == out[1]
    elapsed, value = out[0]
    assert elapsed == pytest.approx(0.75)
    assert value == pytest.approx(100.0 * 4 * 2 / 0.75)


def test_single_process_is_identity():
    import bench
    assert not dist.is_initialized()
    assert bench.max_over_ranks(1.25, "cpu") == 1.25
    assert bench.job_throughput(10.0, 3, 1, 2.0) == 15.0

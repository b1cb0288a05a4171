"""Host logic of the N > 1 benchmark path, on CPU with a world_size-2 gloo
group: the job's time is the slowest rank's, and the job's throughput counts
the work of every replica."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [0.75, 1.25][rank]
        t = bench.max_over_ranks(local, dist, torch.device("cpu"))
        out[rank] = t
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()  # no fork of a threaded test process
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == pytest.approx(1.25) and out[1] == pytest.approx(1.25)


def test_single_process_is_identity():
    assert bench.max_over_ranks(0.5) == 0.5


def test_job_throughput_counts_every_replica():
    one = bench.job_throughput(1, 30_000_000_000, 10, 2.0)
    two = bench.job_throughput(2, 30_000_000_000, 10, 2.0)
    assert one == pytest.approx(0.15) and two == pytest.approx(0.30)

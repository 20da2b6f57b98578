"""The multi-rank (replica) measurement path on CPU: world size 2 over gloo.

Decode at batch 1 does not shard, so N GPUs run N independent replicas with
no data-path collective; the only collective is the benchmark's max-over-ranks
of the timed region.  This checks that reduction and the whole-job rate."""
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
        secs = [1.5, 2.5][rank]                       # rank 1 is the slow one
        t = bench.max_over_ranks(secs, dist, "cpu")
        rate = bench.job_throughput(10, world, t)
        out[rank] = (t, rate)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_rate_world2():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, start_method="spawn")
        res = dict(out)
    assert res[0] == res[1] == (2.5, 2 * 10 / 2.5)


def test_single_rank_identity():
    assert bench.max_over_ranks(3.0) == 3.0
    assert bench.job_throughput(7, 1, 0.5) == 14.0

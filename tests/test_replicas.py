"""Multi-GPU use of the block is replicas only (independent token batches per
GPU, no collective on the data path).  The benchmark's only cross-rank steps
-- a barrier and the max over ranks of the timed region -- are checked here on
CPU with two gloo ranks."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, _ = bench.dist_env()
        assert (r, w) == (rank, world)
        bench.barrier(world)
        my_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
        worst = bench.max_over_ranks(my_ms, world)
        out[rank] = (worst, bench.job_throughput(64, 20, world, worst))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_and_whole_job_throughput():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0  # every rank sees the slowest replica
    assert res[0][1] == pytest.approx(64 * 20 * 2 / 0.015)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(64, 10, 1, 1000.0) == pytest.approx(640.0)

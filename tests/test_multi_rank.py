"""The multi-GPU path of bench.py on CPU: two gloo ranks.

Ranks shard the work by (batch, head) with no exchange on the data path;
they only meet at a barrier and reduce their elapsed times with a max.  This
checks that logic (and that each rank draws its own batch) without a GPU.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import workloads
        w = workloads.get("tiny")
        bench.rank_barrier(world)
        slowest = bench.max_over_ranks_of(10.0 + rank, world, torch.device("cpu"))
        seed = bench.rank_seed(w, rank)
        q, _, _, _ = workloads.make_inputs(w, seed=seed)
        seeds = [None] * world
        dist.all_gather_object(seeds, (seed, float(q.float().sum())))
        out[rank] = (slowest, seeds)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, join=True,
                       start_method="spawn")
    assert sorted(out.keys()) == [0, 1]
    for rank in range(world):
        slowest, seeds = out[rank]
        assert slowest == 11.0                       # max over ranks of 10 + rank
        assert seeds[0][0] != seeds[1][0]            # each rank its own batch
        assert seeds[0][1] != seeds[1][1]


def test_whole_job_aggregation():
    import bench
    # 2 ranks, each 7.037e13 FLOP per step in 28 ms (the slowest rank)
    v = bench.whole_job_tflops(2, 7.037e13, 28.0)
    assert v == pytest.approx(2 * 7.037e13 / 0.028 / 1e12)
    assert bench.whole_job_tflops(1, 1e12, 1.0) == pytest.approx(1000.0)

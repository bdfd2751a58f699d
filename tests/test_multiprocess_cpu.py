"""bench.py's multi-process path on CPU: two gloo ranks (world size 2), as
torchrun would start them with --nproc-per-node 2 on one node.

The path runs one independent replica per rank (there is no data exchange
in the method); what is shared is the job's timing: the step time reported
is the largest over the ranks, and each rank draws its own inputs.
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        ms = 10.0 + 5.0 * rank                      # the slower replica decides
        got = bench.max_over_ranks(ms, dist, "cpu")
        seeds = [None] * world
        dist.all_gather_object(seeds, bench.replica_seed(rank))
        out[rank] = (got, seeds)
    finally:
        dist.destroy_process_group()


def test_two_ranks_report_the_slowest_step_and_distinct_replicas():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    assert len(set(res[0][1])) == world


def test_single_process_needs_no_group():
    import bench

    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5

"""The bench's multi-rank host logic on CPU: two gloo ranks on 127.0.0.1.

With N GPUs the bench runs one replica per rank (attention over independent
heads needs no exchange), meets at a barrier around the timed region and
takes the slowest rank's time.  This checks that aggregation without GPUs.
"""

import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port),
                      RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    bench._barrier(dist)
    elapsed = 10.0 + 5.0 * rank                      # rank 1 is the slow one
    got = bench._max_over_ranks(dist, elapsed, torch.device("cpu"))
    out[rank] = got
    bench._barrier(dist)
    dist.destroy_process_group()


def test_two_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    with mp.get_context("spawn").Manager() as mgr:   # no fork of a threaded process
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        assert dict(out) == {0: 15.0, 1: 15.0}

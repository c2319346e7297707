"""The benchmark's multi-rank logic (one independent replica per rank,
barrier and max-over-ranks timing on a gloo group), run as two CPU
processes. No GPU: the data path has no collective to test."""
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


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    r, ws, local = bench.world()
    assert (r, ws, local) == (rank, world, rank)
    bench.init_group(ws)
    bench.barrier(ws)
    elapsed = 10.0 + 5.0 * rank          # each rank's own timed region, ms
    out[rank] = bench.reduce_max(elapsed, ws)
    bench.barrier(ws)
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_ranks_take_the_max_elapsed_time():
    world = 2
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_rank_needs_no_group():
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    bench.barrier(1)

"""The benchmark's multi-rank path (replicas only) on CPU with gloo: the
slowest rank's time decides, and the value counts every rank's units."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        elapsed = 1.0 + rank          # rank 1 is the slower one
        t = bench.max_over_ranks(elapsed, ws)
        v = bench.aggregate_value(10.0, elapsed, ws)
        bench.barrier(ws)
        out[rank] = (t, v)
    finally:
        dist.destroy_process_group()


def test_replica_aggregation_two_ranks():
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    for rank in range(world):
        t, v = out[rank]
        assert t == 2.0                       # max over ranks
        assert v == pytest.approx(10.0 * 2 / 2.0)  # all ranks' units / slowest time

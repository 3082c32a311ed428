"""Replica logic of bench.py on CPU: world-size-2 gloo ranks, barrier and the max of
the timed region over ranks (the multi-GPU run is N independent replicas)."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist
    import bench
    r, w, local = bench.dist_init(None)
    assert (r, w, local) == (rank, world, rank)
    bench.barrier(w)
    out[rank] = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_over_ranks():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world,
                       start_method="spawn", join=True)
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(3.0, 1) == 3.0
    bench.barrier(1)

"""The benchmark's N-replica host logic (barrier + max over ranks) on two CPU ranks
with the gloo backend.  The decode path itself has no exchange step: every rank runs
an independent replica, so only the timing aggregation crosses ranks."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, l = bench.dist_env()
    assert (w, r, l) == (world, rank, rank)
    bench.barrier(world)
    got = bench.aggregate_max(10.0 * (rank + 1), world, device="cpu")
    out[rank] = got
    dist.destroy_process_group()


def test_two_rank_max_aggregation():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert dict(out) == {0: 20.0, 1: 20.0}


def test_single_process_is_identity():
    import bench
    assert bench.aggregate_max(3.5, 1) == 3.5

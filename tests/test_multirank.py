"""Replica timing across ranks (bench.py under torchrun): barrier and the max
over ranks, exercised with the gloo backend at world size 2 on the CPU."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench

    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank)
    bench.barrier(w)
    out[rank] = bench.max_over_ranks(1.5 + rank, w)
    bench.barrier(w)
    torch.distributed.destroy_process_group()


@pytest.mark.skipif(torch.cuda.is_available(), reason="CPU (gloo) test")
def test_max_over_ranks_gloo_world2():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert dict(out) == {0: 2.5, 1: 2.5}

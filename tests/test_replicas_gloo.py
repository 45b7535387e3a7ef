"""The bench's multi-GPU path is replicas only: each rank sorts its own input
and the ranks meet only for a barrier and the max-over-ranks time.  That host
logic runs here as two gloo processes on the CPU."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    ws, r, local, pg = bench.dist_setup(None)
    assert (ws, r, local) == (world, rank, rank)
    bench.barrier(pg)
    t = bench.max_over_ranks(pg, 10.0 + rank, "cpu")   # each rank's own timing
    out[rank] = t
    pg.destroy_process_group()


@pytest.mark.skipif(torch.cuda.is_available(), reason="CPU (gloo) test of the host logic")
def test_two_replicas_agree_on_the_max_time():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert dict(out) == {0: 11.0, 1: 11.0}

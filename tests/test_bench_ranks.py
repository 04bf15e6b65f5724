"""bench.py's multi-rank reduction on CPU (gloo, world size 2): every rank gets the slowest rank's time.

On GPUs the path shards by independent heads with no collective; the only cross-rank step of the bench is
this max of the per-rank step times (and a barrier)."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    out[rank] = bench.max_over_ranks(1.5 + rank * 2.25)
    dist.barrier()
    dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, join=True, start_method="spawn")
        assert dict(out) == {0: 3.75, 1: 3.75}


def test_max_over_ranks_without_a_process_group():
    import bench
    assert bench.max_over_ranks(2.5) == 2.5

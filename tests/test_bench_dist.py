"""The bench's multi-rank plumbing on CPU (gloo, world size 2): every rank
ends with the max of the per-rank step times, and the whole-job value
counts every rank's tokens (weak scaling, no collective on the data path)."""
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
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    bench.barrier(world)
    total_ms = 10.0 * (rank + 1)          # rank 1 is the slow one
    mx = bench.max_over_ranks(total_ms, world)
    out[rank] = mx
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, start_method="spawn", join=True)
    assert out[0] == out[1] == 20.0


def test_single_rank_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    bench.barrier(1)

"""The benchmark's multi-rank logic on CPU: two gloo ranks, max over ranks
of the timed region, whole-job weak-scaling throughput."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, lr, w = bench.dist_env()
        assert (r, lr, w) == (rank, rank, world)
        t = 1.5 + rank  # rank 1 is the slower one
        m = bench.max_over_ranks(t, world)
        out[rank] = m
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    world = 2
    port = _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        assert dict(out) == {0: 2.5, 1: 2.5}


def test_weak_scaling_value():
    # 2 ranks, 10 steps of 1e12 FLOPs each, slowest rank 4 s -> 5 TFLOP/s
    assert bench.weak_scaling_value(1e12, 10, 2, 4.0) == pytest.approx(5.0)
    assert bench.max_over_ranks(3.0, 1) == 3.0

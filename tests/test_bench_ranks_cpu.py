"""The bench's multi-replica path on CPU: two gloo ranks (one process each,
rendezvous on 127.0.0.1) run the same barrier / max-over-ranks / whole-job
throughput code the GPU run uses under torchrun with NCCL.  No GPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        r = bench.Ranks(world, rank, dist, device="cpu")
        r.barrier()
        ms = 1.0 + rank            # rank 1 is the slow replica
        slowest = r.max(ms)
        rate = r.throughput(1.0e9, slowest)
        out[rank] = (slowest, rate)
        r.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    port = _free_port()
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
    for rank in range(world):
        slowest, rate = out[rank]
        assert slowest == 2.0
        assert rate == pytest.approx(2 * 1.0e9 / 2.0e-3)


def test_single_process_needs_no_collective():
    sys.path.insert(0, ROOT)
    import bench
    r = bench.Ranks(1, 0, None, device="cpu")
    r.barrier()
    assert r.max(3.5) == 3.5
    assert r.throughput(10.0, 2.0) == pytest.approx(5000.0)

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


def test_reference_arm_prints_the_contract_line():
    """`bench.py --impl reference` (the fp64 oracle on the host cores, one
    process, no GPU) prints one JSON line with every key of the bench
    contract, marked as the reference arm."""
    import json
    import subprocess
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "0"], cwd=ROOT, capture_output=True, text=True, timeout=600, check=True)
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    j = json.loads(lines[0])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in j, key
    assert j["impl"] == "reference" and j["value"] > 0 and j["higher_is_better"] is True
    assert j["n_gpus"] == 1 and j["steps"] == 1 and j["warmup"] == 0
    assert j["cpu_baseline"]["kind"] == "oracle" and j["cpu_baseline"]["cores"] >= 1
    assert j["e2e"]["h2d_bytes_per_step"] == 0 and j["e2e"]["d2h_bytes_per_step"] == 0
    assert j["e2e"]["value"] == j["value"] and j["cpu_baseline"]["value"] == j["value"]
    assert "workload" in j["config"]

"""The N > 1 path of bench.py on the CPU: replicas report the slowest rank's
time and the whole-job aggregate (gloo, world size 2, no GPU)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank  # rank 1 is the slow replica
        got = bench.max_over_ranks(ms, world, "cpu")
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    assert dict(out) == {0: 15.0, 1: 15.0}


def test_aggregate_is_whole_job():
    b = bench.config_block()["bytes_per_step"]
    # 7 projections x 28 layers, [q; k; v] and [gate; up] one launch each (x read once)
    assert b == 3369046016
    one = bench.aggregate_gbps(b, 0.5, 1)
    assert bench.aggregate_gbps(b, 0.5, 2) == pytest.approx(2 * one)
    assert one == pytest.approx(b / 0.5e-3 / 1e9)
    assert bench.max_over_ranks(3.0, 1, "cpu") == 3.0


def test_workload_matches_the_decode_step():
    g = bench.workload_gemvs()
    assert len(g) == 28 * 4
    names = [n for n, *_ in g[:4]]
    assert names == ["qkv", "o", "gate_up", "down"]
    # per-GEMV byte counts of the shapes
    assert bench.gemv_bytes(512, 1024, 1) == 273408
    assert bench.gemv_bytes(3584, 3584, 1) == 6637568
    assert bench.gemv_bytes(37888, 3584, 1) == 70099968
    assert bench.gemv_bytes(3584, 18944, 1) == 35053568

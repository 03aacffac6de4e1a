"""The multi-rank host logic of bench.py on CPU (gloo, world size 2).

On N GPUs the benchmark runs one independent replica per rank: the decode
path has no exchange. What crosses ranks is host logic only, checked here:
the barrier around the timed region, the max of the per-rank times (the
slowest rank sets the whole-job time), the weak-scaling aggregate (every
rank's KV bytes over that time), and the reference arm, which only rank 0
runs.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, local = bench._dist()
        bench._barrier(w)
        mx = bench._barrier_max(times[rank], w, "cpu")
        # the reference arm: ranks other than 0 return at once, without work
        ref = bench.run_reference(None) if r != 0 else None
        bench._barrier(w)
        q.put((r, w, local, mx, ref))
    finally:
        dist.destroy_process_group()


def test_two_ranks_barrier_and_max_over_ranks():
    world, port = 2, _free_port()
    times = [1.25, 3.5]  # ms: rank 1 is the slower one
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == world and r[2] == r[0] for r in res)
    assert all(r[3] == max(times) for r in res)  # every rank sees the slowest rank's time
    assert res[1][4] == 0  # rank 1's reference arm did nothing


def test_single_rank_needs_no_process_group():
    assert bench._barrier_max(2.5, 1, "cpu") == 2.5
    bench._barrier(1)  # no-op without a process group


def test_weak_scaling_aggregate():
    # every rank streams the same bytes per step; the job time is the slowest rank's
    kvb, K, ms = 1207959552, 10, 4.5
    one = bench.aggregate_gbs(kvb, K, 1, ms)
    assert one == pytest.approx(kvb * K / 4.5e-3 / 1e9)
    assert bench.aggregate_gbs(kvb, K, 2, ms) == pytest.approx(2 * one)
    assert bench.aggregate_gbs(kvb, K, 2, 2 * ms) == pytest.approx(one)

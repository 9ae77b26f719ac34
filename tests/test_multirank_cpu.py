"""The multi-rank bench logic on CPU: two ``gloo`` ranks.

The path shards into independent replicas (one per GPU, no exchange step),
so the only cross-rank work is the timing reduction: every rank must end
with the slowest rank's times, and the whole-job rate is world size times
one replica's work over that slowest time.  Each rank also draws its own
seeded inputs.  No GPU and no kernel is involved.
"""

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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import workloads

        # rank r pretends its steps took (r + 1) times as long
        mine = [10.0 * (rank + 1), 6.0 * (rank + 1), 4.0 * (rank + 1), 20.0 * (rank + 1)]
        got = bench.max_over_ranks(mine, dist, torch.device("cpu"))
        c = workloads.PREFILL_CONFIGS["tiny"]
        q, _, _ = workloads.prefill_inputs(c["B"], c["Hq"], c["Hkv"], c["N"], c["d"],
                                           c["seed"] + 1000 * rank)
        out[rank] = (got, float(q.float().sum()))
        # the reference arm: rank 0 alone runs (not here: it would time the
        # oracle), every other rank returns at once without work
        if rank != 0:
            class A:
                steps, warmup = 1, 3
            assert bench.run_reference(A, rank, world) is None
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_draw_their_own_inputs():
    world = 2
    with mp.get_context("spawn").Manager() as m:       # no fork of this threaded process
        out = m.dict()
        mp.spawn(_rank_main, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    slowest = [20.0, 12.0, 8.0, 40.0]
    for r in range(world):
        assert res[r][0] == pytest.approx(slowest)
    assert res[0][1] != res[1][1]          # per-rank seeds give different inputs


def test_job_rates_are_world_times_one_replica():
    import bench

    flops, dbytes, K = 2.0e11, 1.3e8, 10
    one = bench.job_rates(1, K, flops, dbytes, fwd_sum_ms=2.0, dec_sum_ms=0.5)
    two = bench.job_rates(2, K, flops, dbytes, fwd_sum_ms=2.0, dec_sum_ms=0.5)
    assert one[0] == pytest.approx(flops / 2.0e-4 / 1e12)   # 0.2 ms per step
    assert one[1] == pytest.approx(dbytes / 5.0e-5 / 1e9)
    assert two[0] == pytest.approx(2 * one[0]) and two[1] == pytest.approx(2 * one[1])
    assert two[2] == pytest.approx(one[2]) and two[3] == pytest.approx(one[3])

"""Host logic of bench.py's multi-rank path (one process per GPU, replicas:
each rank runs its own request, no data-path collective): the job's step time
is the slowest rank's, and the value is the work of all ranks over that time.
Run with two gloo ranks on the CPU, plus the per-step launch count claimed in
the JSON line."""
import os
import socket

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
import workloads as W


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank: int, world: int, port: int, q) -> None:
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [3.0, 5.0][rank]                   # rank 1 is the slow one
        dist.barrier()
        m = bench.max_over_ranks(ms, dist, "cpu")
        q.put((rank, m, bench.whole_job_rate(1e12, m, world)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, rate in got:
        assert m == 5.0
        # two ranks of 1e12 flops per 5 ms step: 400 TFLOP/s for the job
        assert rate == pytest.approx(400.0)


def test_one_rank_is_its_own_time():
    assert bench.max_over_ranks(3.5, None, "cpu") == 3.5
    assert bench.whole_job_rate(4e12, 2.0, 1) == pytest.approx(2000.0)


def test_launches_per_step_match_the_planner():
    """count, [logical count,] schedule, emit, attention; key lists: count,
    schedule, emit (+ a validation pass above 196,608 tokens), attention; no
    permutation kernels (SVG temporal heads are permuted inside the loads)."""
    assert bench.launches_per_step(W.tiny_block_mask(), {}) == 5
    assert bench.launches_per_step(W.segment_mask(1, 1, 1, 2048), {}) == 5
    assert bench.launches_per_step(W.svg_mask(1, 4, 4, 64), {"n_temporal_heads": 2}) == 4
    kl = W.random_keylist(1, 1, 1, 1024, hi=10)
    assert bench.launches_per_step(kl, {}) == 4
    kl.N = 200000
    assert bench.launches_per_step(kl, {}) == 5

"""The benchmark's multi-rank host logic on the CPU with two gloo ranks:
torchrun-style environment set-up, the barrier, the max-over-ranks timing and
the whole-job throughput. Replicas only: no data-path collective exists."""

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    r, w = bench.dist_setup()
    assert (r, w) == (rank, world)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    # rank r "took" 10*(r+1) ms for the same per-rank work
    elapsed = 10.0 * (rank + 1)
    m = bench.max_over_ranks(elapsed, w)
    units = 1000.0
    rate = bench.job_throughput(units, m / 1e3, w)
    q.put((rank, m, rate))
    dist.destroy_process_group()


def test_two_gloo_ranks_max_and_throughput():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, m, rate in got:
        assert m == 20.0                       # the slowest rank sets the time
        assert rate == pytest.approx(2 * 1000.0 / 0.020)  # both ranks' units


def test_single_rank_needs_no_process_group(monkeypatch):
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.delenv("RANK", raising=False)
    assert bench.dist_setup() == (0, 1)
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(10.0, 2.0, 1) == 5.0


def _ref_worker(rank, world, q):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world))
    # only rank 0 does the work; other ranks return None at once
    class A:
        workload, tokens, steps, warmup = "pr1_t128_h4096_n2", 0, 1, 3
    out = bench.reference_arm(A, rank, world)
    q.put((rank, out is None))


def test_reference_arm_runs_on_rank_zero_only():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_ref_worker, args=(r, 2, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=600)
        assert p.exitcode == 0
    got = dict(q.get(timeout=10) for _ in range(2))
    assert got == {0: False, 1: True}

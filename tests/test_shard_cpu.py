"""The token-shard form of the step across ranks, on the CPU.

* tw_shard_rows (libtw, host code) equals the oracle's row-by-row owner rule
  for every T <= 300 and world <= 8, and for large batches.
* TokenShardStep's collectives, with 2 and 3 gloo ranks: each rank must
  receive its shard of every rank's partial in rank order, and the gathered
  output and residual must equal the whole-batch result bit for bit. The
  fused step itself needs a GPU; here the test hands TokenShardStep a stand-in
  for it that applies the oracle to the received slices (the product path
  never imports the oracle).

[W] "TokenWeave: Why Hiding Tensor-Parallel Communication Needs Wave
Arithmetic, Not Finer Tiles", "Fix two": reduce-scatter and all-gather at
token boundaries."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import reduce_rmsnorm_gb300 as tw
import synth
from oracle import bf16, fused, shards


@pytest.fixture(scope="module")
def L():
    from reduce_rmsnorm_gb300 import build
    build.build()
    return tw.lib()


def test_shard_rows_equals_the_oracle(L):
    for T in range(0, 301):
        for world in range(1, 9):
            for rank in range(world):
                assert tw.tw_shard_rows(T, world, rank) == shards.shard_rows(T, world, rank)
    # large batches: the closed form of the same rule (the brute-force oracle
    # is pinned above on every small case)
    for T, world in ((1024, 8), (8192, 8), (16384, 3), (70001, 7), (2 ** 40 + 5, 16)):
        s = -(-T // world)
        for rank in range(world):
            a = min(rank * s, T)
            assert tw.tw_shard_rows(T, world, rank) == (a, min(a + s, T) - a)


def test_shard_rows_rejects_bad_args(L):
    for args in ((-1, 2, 0), (8, 0, 0), (8, 2, 2), (8, 2, -1)):
        with pytest.raises(tw.TwError):
            tw.tw_shard_rows(*args)
    import ctypes
    x = ctypes.c_int64()
    assert L.tw_shard_rows(8, 2, 0, None, ctypes.byref(x)) == tw.TW_ERR_INVALID_ARG
    assert L.tw_shard_rows(8, 2, 0, ctypes.byref(x), None) == tw.TW_ERR_INVALID_ARG


def _oracle_step(seen):
    """Stand-in for the fused step on one rank's shard: the oracle applied to
    the received slices (test code only). Records what it received."""

    def step(partials, residual, gamma, eps, out):
        seen.append(partials.clone())
        pb, rb, gb = synth.bits(partials), synth.bits(residual), synth.bits(gamma)
        res = fused.residual_fp32_rank_order(pb, rb)
        _, y64 = fused.reduce_residual_rmsnorm(pb, rb, gb, eps)
        residual.copy_(torch.from_numpy(res.view(np.int16)).view(torch.bfloat16))
        out.copy_(torch.from_numpy(bf16.encode_rne(y64).view(np.int16)).view(torch.bfloat16))

    return step


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, T, H, q):
    try:
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        import torch.distributed as dist
        from reduce_rmsnorm_gb300.shard import TokenShardStep
        dist.init_process_group("gloo", rank=rank, world_size=world)
        p, r, g = synth.make_inputs(T, H, world, 0.02, seed=T + world)
        seen = []
        step = TokenShardStep(T, H, local_step=_oracle_step(seen))
        residual, out = r.clone(), torch.zeros_like(r)
        step(p[rank].contiguous(), residual, g, synth.EPS, out)
        # what this rank received: its shard of every rank's partial, in rank order
        row0, rows = tw.tw_shard_rows(T, world, rank)
        if rows:
            assert len(seen) == 1
            assert torch.equal(seen[0].view(torch.int16), p[:, row0:row0 + rows].view(torch.int16))
        else:
            assert not seen
        # the gathered results equal the whole-batch step
        pb, rb, gb = synth.bits(p), synth.bits(r), synth.bits(g)
        want_res = fused.residual_fp32_rank_order(pb, rb)
        _, y64 = fused.reduce_residual_rmsnorm(pb, rb, gb, synth.EPS)
        assert np.array_equal(synth.bits(residual), want_res)
        assert np.array_equal(synth.bits(out), bf16.encode_rne(y64))
        dist.destroy_process_group()
        q.put((rank, "ok"))
    except Exception as e:  # reported by the parent
        q.put((rank, repr(e)))


@pytest.mark.parametrize("world,T", [(2, 64), (2, 37), (3, 10), (3, 2)])
def test_token_shard_step_gloo(L, world, T):
    """T = 64 over 2 ranks tiles exactly (gathered straight into the outputs);
    37 over 2 and 10 over 3 leave a short last shard; 2 over 3 leaves rank 2
    with no rows."""
    H = 16
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, T, H, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    got = dict(q.get(timeout=180) for _ in range(world))
    for pr in procs:
        pr.join(timeout=60)
    assert got == {r: "ok" for r in range(world)}

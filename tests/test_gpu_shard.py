"""The token-shard step's product path on one GPU: a one-rank NCCL group, so
the collectives are real NCCL calls on the device and the local step is
libtw's fused kernel. With one rank the shard is the whole batch, so the
result must equal the plain fused call bit for bit, and the oracle on
sampled rows. (Two or more ranks need as many GPUs; their collective plumbing
is tested with gloo ranks on the CPU.) Needs a GPU."""

import os
import socket

import numpy as np
import pytest
import torch

import reduce_rmsnorm_gb300 as tw
import synth
from parity import check_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from reduce_rmsnorm_gb300 import build
    build.build()
    tw.lib()
    tw.tw_device_status(reset=True)
    yield
    assert tw.tw_device_status(reset=True) == 0


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_token_shard_step_one_nccl_rank():
    import torch.distributed as dist
    from reduce_rmsnorm_gb300.shard import TokenShardStep
    os.environ.setdefault("NCCL_NVLS_ENABLE", "0")
    dist.init_process_group("nccl", init_method="tcp://127.0.0.1:%d" % _free_port(), rank=0,
                            world_size=1, device_id=torch.device("cuda", 0))
    try:
        T, H = 1024, 8192
        p, r, g = synth.make_inputs(T, H, 1, 0.02, seed=21)
        P, R, G = p.cuda(), r.cuda(), g.cuda()
        R2 = R.clone()
        out, out2 = torch.empty_like(R), torch.empty_like(R)
        step = TokenShardStep(T, H, device=P.device)
        step(P[0], R, G, synth.EPS, out)
        tw.tw_fused_reduce_residual_rmsnorm(P, R2, G, synth.EPS, out2)
        torch.cuda.synchronize()
        assert torch.equal(R.view(torch.int16), R2.view(torch.int16))
        assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
        rows = sorted(set(np.random.default_rng(4).choice(T, 64, replace=False).tolist()) | {0, T - 1})
        check_rows(p, r, g, synth.EPS, R.cpu(), out.cpu(), rows=rows)
    finally:
        dist.destroy_process_group()

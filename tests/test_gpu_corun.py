"""The split pipelined against a GEMM that produces partial 0 on another
stream (tw_run_split_after): each fused half must start only after its GEMM
half has finished. Checked two ways: against the oracle, on the final
partials (partial 0 as the GEMM wrote it), the residual before the call and
gamma, at the rows around the split and 64 seeded rows; and bit for bit
against the unsplit fused step recomputed on the same partials. Needs a GPU.

Pages: [G] "TokenWeave Guide: Compute-Communication Overlap for LLMs",
"Architectural Foundations of TokenWeave"."""

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


@pytest.mark.parametrize("T,budget", [(4096, 4), (2048, 0), (1024, 8), (4864, 2), (4096, 0),
                                      (1024, 2)])
def test_split_after_gemm_matches_unsplit(T, budget):
    H, N, eps = 8192, 8, synth.EPS
    K = 4 * H // N
    dev = torch.device("cuda")
    p, r, g = synth.make_inputs(T, H, N, 0.02, seed=11)
    P, R, G = p.to(dev), r.to(dev), g.to(dev)
    R0 = R.clone()
    gen = torch.Generator(device=dev).manual_seed(5)
    x = torch.randn((T, K), generator=gen, device=dev).to(torch.bfloat16)
    w = (torch.randn((K, H), generator=gen, device=dev) * K ** -0.5).to(torch.bfloat16)
    out = torch.empty_like(R)
    torch.cuda.synchronize()
    C = (T + 127) // 128 * (H // 128) // 8
    prefix = tw.tw_wave_split(T, C, 148)[0]
    if prefix == T:
        prefix = T // 2 + 64  # exercise both halves
    sa = torch.cuda.Stream()
    sb = torch.cuda.Stream(priority=-1)
    e1, e2 = torch.cuda.Event(), torch.cuda.Event()
    with torch.cuda.stream(sa):
        torch.matmul(x[:prefix], w, out=P[0, :prefix])
        e1.record(sa)
        torch.matmul(x[prefix:], w, out=P[0, prefix:])
        e2.record(sa)
    tw.tw_run_split_after(prefix, P, R, G, eps, out, sb, e1, e2, sm_budget=budget)
    sa.wait_stream(sb)
    torch.cuda.synchronize()
    out_ref = torch.empty_like(R)
    tw.tw_fused_reduce_residual_rmsnorm(P, R0, G, eps, out_ref)
    torch.cuda.synchronize()
    # against the oracle: the partials as the GEMM left them, the residual and
    # gamma as they were before the call
    rows = sorted({0, prefix - 1, prefix, T - 1} |
                  set(np.random.default_rng(T + budget).choice(T, 64, replace=False).tolist()))
    check_rows(P.cpu(), r, g, eps, R.cpu(), out.cpu(), rows=rows)
    assert torch.equal(R.view(torch.int16), R0.view(torch.int16))
    assert torch.equal(out.view(torch.int16), out_ref.view(torch.int16))

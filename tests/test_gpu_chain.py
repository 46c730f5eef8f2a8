"""A chain of fused steps on one stream, each consuming the previous step's
outputs as a decoder stack does: step l reads Y of step l-1 as its partial 0
and the residual that step l-1 wrote in place. Launched back to back
(programmatic dependent launch lets a step's CTAs become resident while the
previous step drains), the chain must equal, bit for bit, the same chain run
with a full device synchronisation between steps; every synchronised step is
also checked against the oracle.

Pages cited: [W] "TokenWeave: Why Hiding Tensor-Parallel Communication Needs
Wave Arithmetic, Not Finer Tiles", "Fix two" (the fused step between layers)."""

import numpy as np
import pytest
import torch

import reduce_rmsnorm_gb300 as tw
import synth
from parity import check_rows

pytestmark = pytest.mark.gpu

EPS = synth.EPS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from reduce_rmsnorm_gb300 import build
    build.build()
    tw.lib()
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    tw.tw_device_status(reset=True)
    yield
    assert tw.tw_device_status(reset=True) == 0, "a kernel gave up on a bounded wait"


def _inputs(T, H, N, L, seed):
    """Layer 0's partials, the other layers' partials 1..N-1, R, gamma."""
    p, r, g = synth.make_inputs(T, H, N, 0.02, seed=seed)
    extra = [synth.make_inputs(T, H, N, 0.02, seed=seed + 1 + l)[0][1:] for l in range(1, L)]
    return p, extra, r, g


def _chain(p, extra, r, g, L, sm_budget, sync, split=False):
    """Runs the chain on a created stream; returns (final R, [Y_l], snapshots).
    With sync, every step's inputs and results are copied to the host. With
    split, each step is the planned split step (tw_run_wave_split: plan on the
    host, halves on two streams, joined on the first)."""
    dev = torch.device("cuda", 0)
    P0 = p.to(dev)
    E = [e.to(dev) for e in extra]
    R = r.to(dev).contiguous()
    G = g.to(dev)
    outs = [torch.empty_like(R) for _ in range(L)]
    torch.cuda.synchronize()
    s = torch.cuda.Stream(dev)
    s2 = torch.cuda.Stream(dev)
    T, H = R.shape
    ctas = -(-T // 128) * (H // 128) // 8
    snaps = []
    with torch.cuda.stream(s):
        for l in range(L):
            plist = [P0[i] for i in range(P0.shape[0])] if l == 0 else [outs[l - 1]] + list(E[l - 1])
            if sync:
                before = (torch.stack([x.cpu() for x in plist]), R.cpu())
            if split:
                tw.tw_run_wave_split(ctas, 148, plist, R, G, EPS, outs[l], s, s2,
                                     sm_budget=sm_budget)
            else:
                tw.tw_fused_reduce_residual_rmsnorm(plist, R, G, EPS, outs[l], stream=s,
                                                    sm_budget=sm_budget)
            if sync:
                torch.cuda.synchronize()
                snaps.append((before[0], before[1], R.cpu(), outs[l].cpu()))
    torch.cuda.synchronize()
    return R, outs, snaps, g


CASES = [
    # T, H, N, layers, sm_budget, planned split step
    (512, 8192, 8, 6, 0, False),     # 3-4 rows per CTA: CTAs of the next step start early
    (1024, 8192, 8, 6, 0, False),    # the Llama-3.3-70B layer shape
    (333, 4104, 3, 5, 0, False),     # ragged rows and chunks, runtime N
    (128, 4096, 2, 8, 0, False),     # the PR1 shape: one row per CTA, the direct form
    (152, 4096, 8, 6, 0, False),     # one row per CTA on every SM, the direct form
    (150, 16384, 8, 4, 0, False),    # one row per CTA, the direct form at KMAX = 8
    (100, 12296, 8, 4, 0, False),    # one row per CTA, ragged KMAX = 8 at N = 8: the ring
    (304, 4096, 8, 5, 0, False),     # one direct CTA per row, two per SM
    (600, 3080, 2, 4, 0, False),     # one direct CTA per row, ragged, four per SM
    (520, 8192, 2, 4, 0, False),     # two-pipeline chunk ring from 3 rows per CTA (N <= 2)
    (256, 8192, 8, 4, 8, False),     # under an SM budget of 8
    (4096, 8192, 8, 3, 0, True),     # planned 2048/2048 split on two streams, per step
    (4864, 8192, 2, 3, 16, True),    # uneven planned split under a budget
    (1024, 8192, 2, 5, 8, False),    # two-pipeline chunk ring (N <= 4, >= 4 rows per CTA)
    (2048, 8192, 4, 4, 0, False),    # two-pipeline chunk ring on the whole GPU
    (512, 6152, 3, 4, 8, False),     # two-pipeline chunk ring, ragged rows
    (512, 8192, 12, 4, 8, False),    # two-pipeline row ring (N >= 9 under a budget)
    (256, 8192, 16, 3, 4, False),    # two-pipeline row ring, compile-time N = 16
]


@pytest.mark.parametrize("T,H,N,L,budget,split", CASES)
def test_chain_back_to_back_equals_synchronised(T, H, N, L, budget, split):
    p, extra, r, g = _inputs(T, H, N, L, seed=T + 31 * N)
    R_a, outs_a, _, _ = _chain(p, extra, r, g, L, budget, sync=False, split=split)
    R_b, outs_b, snaps, g_cpu = _chain(p, extra, r, g, L, budget, sync=True, split=split)
    for l in range(L):
        assert torch.equal(outs_a[l].view(torch.int16), outs_b[l].view(torch.int16)), \
            "step %d differs back to back" % l
    assert torch.equal(R_a.view(torch.int16), R_b.view(torch.int16))
    rng = np.random.default_rng(T)
    rows = np.unique(np.concatenate([[0, T - 1], rng.integers(0, T, size=min(T, 48))]))
    for l, (pin, rin, rout, yout) in enumerate(snaps):
        if l > 0:  # the step really read the previous step's output
            assert torch.equal(pin[0].view(torch.int16), snaps[l - 1][3].view(torch.int16))
            assert torch.equal(rin.view(torch.int16), snaps[l - 1][2].view(torch.int16))
        check_rows(pin, rin, g_cpu, EPS, rout, yout, rows=rows)

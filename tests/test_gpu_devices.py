"""The binding refuses tensors and streams that are not on the current
device, before any launch. The C ABI launches on the current device and takes
raw pointers, so another GPU's buffer would otherwise reach the kernel. Runs
on one GPU: the binding's view of the current device is made to differ from
the tensors' device, which is what a caller with another device current would
present. Needs a GPU."""

import pytest
import torch

import reduce_rmsnorm_gb300 as tw
import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from reduce_rmsnorm_gb300 import build
    build.build()
    tw.lib()
    tw.tw_device_status(reset=True)
    yield
    assert tw.tw_device_status(reset=True) == 0


def test_mismatched_device_is_refused_before_any_launch(monkeypatch):
    T, H, N = 64, 4096, 2
    p, r, g = synth.make_inputs(T, H, N, 0.05, seed=3)
    P, R, G = p.cuda(), r.cuda(), g.cuda()
    out = torch.zeros_like(R)
    R0 = R.clone()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    here = torch.cuda.current_device()
    monkeypatch.setattr(tw, "_current_device", lambda: here + 1)
    for call in (lambda: tw.tw_fused_reduce_residual_rmsnorm(P, R, G, synth.EPS, out),
                 lambda: tw.tw_run_split(32, P, R, G, synth.EPS, out, sa, sb),
                 lambda: tw.tw_run_wave_split(8, 148, P, R, G, synth.EPS, out, sa, sb),
                 lambda: tw.tw_run_split_after(32, P, R, G, synth.EPS, out, sa),
                 lambda: tw.FusedCall(P, R, G, synth.EPS, out),
                 lambda: tw.PlannedSplitCall(8, 148, P, R, G, synth.EPS, out, sa, sb),
                 lambda: tw.tw_reduce_partials(P, out),
                 lambda: tw.tw_add_rmsnorm(out, R, G, synth.EPS, out)):
        with pytest.raises(ValueError, match="current device"):
            call()
    torch.cuda.synchronize()
    assert torch.equal(R.view(torch.int16), R0.view(torch.int16))
    assert not out.view(torch.int16).any()
    # with the real current device the same call runs
    monkeypatch.setattr(tw, "_current_device", lambda: here)
    tw.tw_fused_reduce_residual_rmsnorm(P, R, G, synth.EPS, out, stream=sa)
    torch.cuda.synchronize()
    assert out.view(torch.int16).any()

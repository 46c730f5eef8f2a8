"""Failure path of the kernels' bounded waits, on a GPU, without a fault: a
diagnostic kernel waits on a barrier phase that nothing completes; the wait
must give up, raise the device error word, leave the context usable, and the
word must clear on reset."""

import pytest
import torch

import reduce_rmsnorm_gb300 as tw
import synth
from parity import check_rows, to_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from reduce_rmsnorm_gb300 import build
    build.build()
    tw.lib()
    tw.tw_device_status(reset=True)
    yield
    tw.tw_device_status(reset=True)


def test_bounded_wait_gives_up_and_reports():
    assert tw.tw_device_status(reset=True) == 0
    tw.tw_debug_wait_timeout(20_000_000)          # 20 ms
    code = tw.tw_device_status(reset=False)
    assert code & 1, "the bounded wait did not report"
    assert tw.tw_device_status(reset=True) == code
    assert tw.tw_device_status(reset=True) == 0   # cleared
    # the context is still usable: a normal fused call afterwards is correct
    p, r, g = synth.make_inputs(16, 4096, 2, 0.05, seed=1)
    P, R, G = to_gpu(p, r, g)
    out = torch.empty_like(R)
    tw.tw_fused_reduce_residual_rmsnorm(P, R, G, synth.EPS, out)
    torch.cuda.synchronize()
    check_rows(p, r, g, synth.EPS, R, out)
    assert tw.tw_device_status(reset=True) == 0


def test_wait_probe_rejects_bad_limits():
    for bad in (0, 999, 3_000_000_000):
        with pytest.raises(tw.TwError) as e:
            tw.tw_debug_wait_timeout(bad)
        assert e.value.status == tw.TW_ERR_INVALID_ARG

"""Several host threads calling the library at once, each on its own streams
(the library keeps per-device attributes behind lock-free flags and per-thread
split events). ctypes releases the GIL during the foreign call, so the calls
really overlap. Every thread's results must equal a single-thread reference
bit for bit. Needs a GPU."""

import threading

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


def test_concurrent_host_threads_bitwise():
    T, H, N = 2048, 8192, 8
    p, r, g = synth.make_inputs(T, H, N, 0.02, seed=77)
    dev = torch.device("cuda", 0)
    P, G = p.to(dev), g.to(dev)
    ref_R = r.to(dev)
    ref_out = torch.empty_like(ref_R)
    tw.tw_fused_reduce_residual_rmsnorm(P, ref_R, G, synth.EPS, ref_out)
    torch.cuda.synchronize()

    n_threads, iters = 6, 20
    results, errors = [None] * n_threads, []
    barrier = threading.Barrier(n_threads, timeout=120)

    def worker(i):
        try:
            torch.cuda.set_device(0)
            sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
            R = r.to(dev)
            R0 = R.clone()
            out = torch.empty_like(R)
            torch.cuda.synchronize()
            barrier.wait()
            for k in range(iters):
                R.copy_(R0)          # default stream; joined below
                sa.wait_stream(torch.cuda.current_stream())
                if k % 2:
                    tw.tw_run_split(T // 2 + 64 * (i % 3), P, R, G, synth.EPS, out, sa, sb,
                                    sm_budget=(0 if i % 2 else 16))
                else:
                    tw.tw_fused_reduce_residual_rmsnorm(P, R, G, synth.EPS, out, stream=sa,
                                                        sm_budget=i * 5)
                torch.cuda.current_stream().wait_stream(sa)
            torch.cuda.synchronize()
            results[i] = (R.clone(), out.clone())
        except Exception as e:  # reported below
            errors.append(repr(e))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(n_threads)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=300)
    assert not errors, errors
    for R, out in results:
        assert torch.equal(R.view(torch.int16), ref_R.view(torch.int16))
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16))


def test_many_tiny_calls():
    """10,000 one-row calls back to back: no error accumulates."""
    p, r, g = synth.make_inputs(1, 8, 1, 0.05, seed=3)
    P, R, G = p.cuda(), r.cuda(), g.cuda()
    out = torch.empty_like(R)
    call = tw.FusedCall(P, R, G, synth.EPS, out)
    for _ in range(10_000):
        call()
    torch.cuda.synchronize()
    assert tw.tw_device_status(reset=True) == 0

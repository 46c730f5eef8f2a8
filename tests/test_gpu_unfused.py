"""The unfused baseline (reduce, then standalone residual add + RMSNorm)
against its oracle, and against the fused step within tolerance. Needs a GPU.

Pages: [W] "TokenWeave: Why Hiding Tensor-Parallel Communication Needs Wave
Arithmetic, Not Finer Tiles", "Fix two"; [G] "TokenWeave Guide: Compute-
Communication Overlap for LLMs", "The Standard RMSNorm Memory Round-Trip"."""

import numpy as np
import pytest
import torch

import reduce_rmsnorm_gb300 as tw
import synth
from oracle import bf16, fused, unfused
from parity import check_rows, to_gpu

pytestmark = pytest.mark.gpu
EPS = synth.EPS


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from reduce_rmsnorm_gb300 import build
    build.build()
    tw.lib()
    tw.tw_device_status(reset=True)
    yield
    assert tw.tw_device_status(reset=True) == 0


def _check_unfused(p, r, g, S, R, Y):
    pb, rb, gb = synth.bits(p), synth.bits(r), synth.bits(g)
    s_want, r_want, y64 = unfused.reduce_then_rmsnorm(pb, rb, gb, EPS)
    assert np.array_equal(synth.bits(S.cpu()), s_want), "reduced sum not bit-exact"
    assert np.array_equal(synth.bits(R.cpu()), r_want), "updated residual not bit-exact"
    y = bf16.decode(synth.bits(Y.cpu()))
    # inputs to the norm are exact bf16 values; beyond the output rounding only
    # the fp32 sum of squares, rsqrtf and two products err (well under 2^-16
    # relative)
    ms = np.mean(bf16.decode(r_want) ** 2, axis=1, keepdims=True)
    delta = np.abs(bf16.decode(gb))[None, :] * 2.0 ** -16 * np.abs(bf16.decode(r_want)) / np.sqrt(ms + EPS)
    assert np.all(np.abs(y - y64) <= 2 * bf16.ulp(y64) + delta)


@pytest.mark.parametrize("T,H,N", [(1, 8, 1), (5, 4104, 3), (64, 8192, 8), (33, 16384, 8),
                                   (3, 32768, 2), (200, 4096, 16),
                                   (5000, 1024, 4)])   # more rows than the capped grid
def test_unfused_parity(T, H, N):
    p, r, g = synth.make_inputs(T, H, N, 0.02, seed=T + N)
    P, R, G = to_gpu(p, r, g)
    S = torch.empty_like(R)
    Y = torch.empty_like(R)
    tw.tw_reduce_partials(P, S)
    tw.tw_add_rmsnorm(S, R, G, EPS, Y)
    torch.cuda.synchronize()
    _check_unfused(p, r, g, S, R, Y)


def test_unfused_in_place_sum_is_output():
    """sum and out may be the same buffer: the reduce writes S into out, the
    norm reads each row before writing it."""
    p, r, g = synth.make_workload("llama70b_t1024_h8192_n8")
    P, R, G = to_gpu(p, r, g)
    Y = torch.empty_like(R)
    tw.tw_reduce_partials(P, Y)
    S_copy = Y.clone()
    tw.tw_add_rmsnorm(Y, R, G, EPS, Y)
    torch.cuda.synchronize()
    _check_unfused(p, r, g, S_copy, R, Y)


def test_unfused_close_to_exact_step():
    """Both pipelines compute the same step. The unfused one also rounds the
    partial sum S to bf16 before adding the residual, an error relative to |S|
    (not to |z|, so it dominates where S and R cancel), and normalises the
    rounded residual: |Y - y64| <= 2 ulp(y64) + r |gamma| ulp(S64), with
    r = 1/sqrt(mean z^2 + eps) and S64 the exact partial sum."""
    p, r, g = synth.make_workload("pr1_t128_h4096_n2")
    P, R, G = to_gpu(p, r, g)
    Y = torch.empty_like(R)
    tw.tw_reduce_partials(P, Y)
    tw.tw_add_rmsnorm(Y, R, G, EPS, Y)
    torch.cuda.synchronize()
    pb, rb, gb = synth.bits(p), synth.bits(r), synth.bits(g)
    z64, y64 = fused.reduce_residual_rmsnorm(pb, rb, gb, EPS)
    s64 = sum(bf16.decode(pb[i]) for i in range(pb.shape[0]))
    rscale = 1.0 / np.sqrt(np.mean(z64 * z64, axis=1, keepdims=True) + EPS)
    bound = 2 * bf16.ulp(y64) + rscale * np.abs(bf16.decode(gb))[None, :] * bf16.ulp(s64)
    y = bf16.decode(synth.bits(Y.cpu()))
    assert np.all(np.abs(y - y64) <= bound)


def test_unfused_validation():
    p, r, g = synth.make_inputs(4, 4096, 2, 0.02)
    P, R, G = to_gpu(p, r, g)
    with pytest.raises(tw.TwError) as e:
        tw.tw_reduce_partials(P, P[0])          # sum_out overlaps a partial
    assert e.value.status == tw.TW_ERR_INVALID_ARG
    with pytest.raises(tw.TwError) as e:
        tw.tw_add_rmsnorm(R, R, G, EPS, torch.empty_like(R))   # residual overlaps sum
    assert e.value.status == tw.TW_ERR_INVALID_ARG

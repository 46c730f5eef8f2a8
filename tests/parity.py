"""Parity helpers: compare the CUDA path's outputs with the oracle's.

Tolerances (floating point; the pages fix no precision beyond bf16 storage):
  * updated residual: bit-exact to the oracle's fp32 rank-order emulation
    (only IEEE additions are involved, so no rounding freedom), and within
    1 bf16 ulp of the exact fp64 sum plus the fp32 summation bound
    N * 2^-24 * (sum_r |P_r| + |R|); the bound matters only where the terms
    cancel to a result much smaller than themselves.
  * output Y: |Y - y64| <= 2 * ulp_bf16(y64) + delta, with
    delta = r * |gamma_j| * N * 2^-24 * (sum_r |P_r| + |R|), the fp32
    summation error bound of the N additions carried through the scale
    r = 1/sqrt(mean z^2 + eps). The final bf16 rounding is 0.5 ulp; the rest
    covers fp32 accumulation of the sum of squares and rsqrtf.
"""

import numpy as np
import torch

from oracle import bf16, fused
import synth


def to_gpu(partials, residual, gamma):
    out = (partials.cuda().contiguous(), residual.cuda().contiguous(), gamma.cuda().contiguous())
    torch.cuda.synchronize()  # later launches may use other streams
    return out


def check_rows(partials_cpu, residual_cpu, gamma_cpu, eps, res_gpu, out_gpu, rows=None):
    """Check GPU results for the given rows (None = all). Inputs are the CPU
    bf16 tensors BEFORE the call; res_gpu / out_gpu are the results (any device).
    Returns a dict of error statistics; raises AssertionError on a violation."""
    pb = synth.bits(partials_cpu)
    rb = synth.bits(residual_cpu)
    gb = synth.bits(gamma_cpu)
    res_bits = synth.bits(res_gpu.cpu())
    out_bits = synth.bits(out_gpu.cpu())
    if rows is not None:
        rows = np.asarray(rows)
        pb, rb, res_bits, out_bits = pb[:, rows], rb[rows], res_bits[rows], out_bits[rows]
    n = pb.shape[0]
    z64, y64 = fused.reduce_residual_rmsnorm(pb, rb, gb, eps)
    # residual: bit-exact to the fp32 emulation, and <= 1 ulp of the exact sum
    emu = fused.residual_fp32_rank_order(pb, rb)
    mism = np.count_nonzero(emu != res_bits)
    assert mism == 0, "updated residual differs from fp32 rank-order emulation in %d places" % mism
    absum = np.abs(bf16.decode(rb))
    for r in range(n):
        absum = absum + np.abs(bf16.decode(pb[r]))
    r_dec = bf16.decode(res_bits)
    assert np.all(np.abs(r_dec - z64) <= bf16.ulp(z64) + n * 2.0 ** -24 * absum), \
        "residual beyond 1 ulp of exact plus the fp32 summation bound"
    # output: 2 ulp + fp32 summation floor
    ms = np.mean(z64 * z64, axis=1, keepdims=True)
    rscale = 1.0 / np.sqrt(ms + eps)
    g64 = np.abs(bf16.decode(gb))[None, :]
    delta = rscale * g64 * n * 2.0 ** -24 * absum
    y = bf16.decode(out_bits)
    err = np.abs(y - y64)
    tol = 2.0 * bf16.ulp(y64) + delta
    bad = err > tol
    assert not np.isnan(y).any() or np.isnan(y64).any(), "NaN in output"
    assert not bad.any(), "output beyond tolerance at %d places, e.g. %s" % (
        np.count_nonzero(bad), list(zip(*np.nonzero(bad)))[:5])
    ulps = err / bf16.ulp(y64)
    rel = err / np.maximum(np.abs(y64), 1e-30)
    return dict(max_ulp=float(ulps.max(initial=0.0)), max_rel=float(rel[np.abs(y64) > 1e-3].max(initial=0.0)),
                rows=int(y.shape[0]))

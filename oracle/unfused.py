"""Oracle of the unfused baseline: a reduce that writes its sum to HBM, then a
standalone residual-add + RMSNorm that reads it back.

TEST INFRASTRUCTURE (see the package docstring).

This is the one-GPU analogue of the pipeline the pages compare against, an
all-reduce followed by a separate RMSNorm ([W] "Fix two": the serving engine
normalises after the all-reduce, and a standalone RMSNorm reads its input
twice and writes once; [G] "The Standard RMSNorm Memory Round-Trip": the
reduced tensor goes to HBM and a second kernel reads it back). Its arithmetic
differs from the fused step only by two extra bf16 roundings that the HBM
round trip forces:

    S   = bf16( ((P_0 + P_1) + ...) + P_{N-1} )      fp32 adds, rank order
    x   = fp32(S) + fp32(R)                           fp32 add
    R'  = bf16(x)
    Y   = RMSNorm(R') * gamma                         (on the stored bf16 R')

The first two are emulated bit for bit (fp32 adds are IEEE operations);
the norm is the fp64 formula applied to the bf16 values the second kernel
reads.
"""

import numpy as np

from . import bf16
from .fused import rms_norm


def reduce_sum_bits(partials):
    """S: fp32 rank-order sum of the partials, rounded once to bf16 bits."""
    p = np.asarray(partials)
    if p.ndim == 2:
        p = p[None]
    acc = bf16.decode(p[0]).astype(np.float32)
    for r in range(1, p.shape[0]):
        acc = (acc + bf16.decode(p[r]).astype(np.float32)).astype(np.float32)
    return bf16.encode_rne(acc)


def add_residual_bits(sum_bits, residual_bits):
    """R': bf16(fp32(S) + fp32(R)) as bits."""
    x = (bf16.decode(sum_bits).astype(np.float32)
         + bf16.decode(residual_bits).astype(np.float32)).astype(np.float32)
    return bf16.encode_rne(x)


def reduce_then_rmsnorm(partials, residual, gamma, eps):
    """(S bits, R' bits, y64): the unfused pipeline's intermediate, updated
    residual and exact fp64 norm of the stored residual."""
    s = reduce_sum_bits(partials)
    r_new = add_residual_bits(s, residual)
    y = rms_norm(bf16.decode(r_new), bf16.decode(gamma), eps)
    return s, r_new, y

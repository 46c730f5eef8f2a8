"""fp64 oracle of the fused reduce + residual + RMSNorm step.

TEST INFRASTRUCTURE (see the package docstring).

What the step computes ([W] "Fix two: RMSNorm was never insignificant", the
per-CTA sketch and the four numbered steps; [G] "Fused AllReduce-RMSNorm:
Bypassing Global Memory"), recast for one GPU whose HBM holds the N ranks'
partial outputs:

    z      = sum_{r=0}^{N-1} P_r + R            (the reduced vector plus residual)
    R'     = bf16(z)                             (updated residual, written back)
    y_i    = z_i / sqrt( (1/H) sum_j z_j^2 + eps ) * gamma_i
    Y      = bf16(y)

The RMSNorm formula is the one of [G] "The Standard RMSNorm Memory
Round-Trip"; [W]'s sketch computes the same scale as rsqrt(variance /
hidden_size + eps) with variance = dot(vec, vec). The normalised vector is the
unrounded sum held in registers ([W] step 2: the sum of squares is taken on
the register-resident result), so z, not bf16(z), feeds the norm.

This module is the plain definition in fp64 on the exact bf16 input values;
the method reaches the same result (up to rounding order) with a faster
dataflow, so no algorithmic steps are restated here. Rows are processed in
blocks of ``block_rows`` only to bound memory; every row is independent.
"""

import numpy as np

from . import bf16


def _as_partials(partials):
    p = np.asarray(partials)
    if p.ndim == 2:
        p = p[None]
    return p


def rms_norm(z, gamma, eps):
    """RMSNorm of each row of the float64 matrix z, by the formula.

    y[t, i] = z[t, i] / sqrt(mean_j z[t, j]^2 + eps) * gamma[i]
    ([G] "The Standard RMSNorm Memory Round-Trip"; mean divisor is the hidden
    size H, [W] "Fix two" sketch).
    """
    z = np.asarray(z, dtype=np.float64)
    gamma = np.asarray(gamma, dtype=np.float64)
    h = z.shape[-1]
    ms = np.sum(z * z, axis=-1, keepdims=True) / h
    return z / np.sqrt(ms + float(eps)) * gamma


def reduce_residual(partials, residual):
    """z = sum_r P_r + R in float64 on the decoded bf16 values.

    partials: uint16 bf16 bits, shape [N, T, H] (or [T, H] for N = 1);
    residual: uint16 bits [T, H]. Returns float64 [T, H].
    """
    p = _as_partials(partials)
    z = bf16.decode(residual).astype(np.float64)
    for r in range(p.shape[0]):
        z = z + bf16.decode(p[r])
    return z


def reduce_residual_rmsnorm(partials, residual, gamma, eps, block_rows=64):
    """The fused step's exact result: (z64, y64), both float64 [T, H].

    z64 is the reduced sum plus residual; the updated residual is bf16(z64)
    up to rounding order. y64 is RMSNorm(z64) * gamma.
    """
    p = _as_partials(partials)
    residual = np.asarray(residual)
    g = bf16.decode(gamma)
    t_rows, h = residual.shape
    z_out = np.empty((t_rows, h), dtype=np.float64)
    y_out = np.empty((t_rows, h), dtype=np.float64)
    for r0 in range(0, t_rows, block_rows):
        r1 = min(t_rows, r0 + block_rows)
        z = reduce_residual(p[:, r0:r1], residual[r0:r1])
        z_out[r0:r1] = z
        y_out[r0:r1] = rms_norm(z, g, eps)
    return z_out, y_out


def normalize_shards(z, gamma_bits, eps, shard_rows):
    """RMSNorm applied to token-contiguous shards of ``shard_rows`` rows each
    (the last shard may be shorter), concatenated.

    [W] "Fix two": the reduce-scatter splits only at token boundaries, so each
    shard holds complete token embeddings and is normalised on its own.
    """
    g = bf16.decode(gamma_bits)
    parts = [rms_norm(z[s:s + shard_rows], g, eps) for s in range(0, z.shape[0], shard_rows)]
    return np.concatenate(parts, axis=0) if parts else np.empty_like(z)


def residual_fp32_rank_order(partials, residual):
    """The updated residual as an fp32 machine computes it in fixed rank order.

    acc = P_0; acc = acc + P_1; ...; acc = acc + P_{N-1}; acc = acc + R, each
    addition an IEEE binary32 add (round to nearest even), then one bf16 RNE
    rounding. Ranks are summed in order 0..N-1 and the residual last, as in
    [W] "Fix two" (reduce, then "vec += residual"). Returns uint16 bits.
    """
    p = _as_partials(partials)
    acc = bf16.decode(p[0]).astype(np.float32)
    for r in range(1, p.shape[0]):
        acc = (acc + bf16.decode(p[r]).astype(np.float32)).astype(np.float32)
    acc = (acc + bf16.decode(residual).astype(np.float32)).astype(np.float32)
    return bf16.encode_rne(acc)

"""Seeded synthetic inputs for the fused reduce + residual + RMSNorm step.

Shared by the tests, the benchmark and the smoke check, and by both sides of
every parity comparison (the CUDA path and the CPU oracle). It holds none of
the method's arithmetic: it draws random numbers with NumPy's PCG64 generator
(platform independent, so the same seed gives the same bits on x86 and Arm)
and casts them to bf16 with PyTorch's round-to-nearest-even cast.

Recipe (one generator per call, seeded with ``seed``; draws in this order):
  for r in 0..N-1:
      P_r = standard_normal([T, H], fp32) * p_sigma
      if outlier_frac > 0:
          mask = uniform([T, H], fp32) < outlier_frac ; P_r[mask] *= outlier_scale
      P_r = bf16(P_r)
  R     = bf16(standard_normal([T, H], fp32) * r_sigma)
  gamma = bf16(standard_normal([H], fp32) * g_sigma + g_mu)

The workloads are the layer shapes of the models the pages evaluate (Llama
3.3 70B: hidden 8192; Llama 3.1 405B: hidden 16384) with N = 8 tensor-parallel
ranks' partial outputs standing in for the all-reduce inputs. The pages'
serving datasets are not needed for this step: its cost depends only on
T, H and N.
"""

import numpy as np
import torch

# name -> (T, H, N, p_sigma, outlier_frac)
WORKLOADS = {
    "pr1_t128_h4096_n2": dict(T=128, H=4096, N=2, p_sigma=0.05),
    "llama70b_t1024_h8192_n8": dict(T=1024, H=8192, N=8, p_sigma=0.02),
    "split_t2048_h8192_n8": dict(T=2048, H=8192, N=8, p_sigma=0.02),
    "split_t4096_h8192_n8": dict(T=4096, H=8192, N=8, p_sigma=0.02),
    "split_t8192_h8192_n8": dict(T=8192, H=8192, N=8, p_sigma=0.02),
    "llama405b_t8192_h16384_n8": dict(T=8192, H=16384, N=8, p_sigma=0.01,
                                      outlier_frac=0.01, outlier_scale=50.0),
}

EPS = 1e-5


def _bf16(x_np):
    return torch.from_numpy(np.ascontiguousarray(x_np)).to(torch.bfloat16)


def make_inputs(T, H, N, p_sigma, r_sigma=1.0, g_mu=1.0, g_sigma=0.1,
                outlier_frac=0.0, outlier_scale=50.0, seed=0):
    """Return (partials [N,T,H], residual [T,H], gamma [H]) as CPU bf16 tensors."""
    rng = np.random.Generator(np.random.PCG64(seed))
    partials = torch.empty((N, T, H), dtype=torch.bfloat16)
    for r in range(N):
        x = rng.standard_normal((T, H), dtype=np.float32) * np.float32(p_sigma)
        if outlier_frac > 0:
            mask = rng.random((T, H), dtype=np.float32) < np.float32(outlier_frac)
            x[mask] *= np.float32(outlier_scale)
        partials[r] = _bf16(x)
    residual = _bf16(rng.standard_normal((T, H), dtype=np.float32) * np.float32(r_sigma))
    gamma = _bf16(rng.standard_normal((H,), dtype=np.float32) * np.float32(g_sigma)
                  + np.float32(g_mu))
    return partials, residual, gamma


def make_workload(name, seed=0, T=None):
    """Inputs of a named workload (optionally with a different token count)."""
    w = dict(WORKLOADS[name])
    if T is not None:
        w["T"] = T
    return make_inputs(seed=seed, **w)


def bits(t):
    """A bf16 tensor's raw bits as a NumPy uint16 array (for the oracle)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)

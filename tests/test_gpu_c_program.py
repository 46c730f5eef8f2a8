"""The C ABI used from C alone, on the GPU: a C99 program that includes only
include/tw.h and the CUDA runtime header allocates device buffers, runs the
fused step and the planned split step through libtw, and checks the results
against closed forms. No Python, torch or binding is involved in the call.

Inputs: every partial is 1, the residual 0 and gamma a ramp of small
integers, so z = N exactly in every element, the updated residual must be
bf16(N) exactly, and Y_j = bf16(gamma_j * N / sqrt(N^2 + eps)) within 2 bf16
ulp ([W] "TokenWeave: Why Hiding Tensor-Parallel Communication Needs Wave
Arithmetic, Not Finer Tiles", "Fix two": z = sum of the partials plus the
residual, y = z * rsqrt(mean z^2 + eps) * w)."""

import os
import shutil
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_PROGRAM = r"""
#include <math.h>
#include <stdio.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <cuda_runtime.h>
#include "tw.h"

static uint16_t to_bf16(float f) {           /* exact for the values used here */
  uint32_t u; memcpy(&u, &f, 4); return (uint16_t)(u >> 16);
}
static double from_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16; float f; memcpy(&f, &u, 4); return f;
}
static double ulp_bf16(double v) {
  int e; frexp(fabs(v), &e);                  /* |v| in [2^(e-1), 2^e) */
  if (e - 1 < -126) e = -125;
  return ldexp(1.0, e - 1 - 7);
}

int main(void) {
  const int N = 8; const int64_t T = 300, H = 4096; const float eps = 1e-5f;
  const size_t bytes = (size_t)T * H * 2;
  uint16_t* h = malloc(bytes); uint16_t* g = malloc(H * 2); uint16_t* y = malloc(bytes);
  void* part[8]; void *res, *gam, *out;
  for (int64_t i = 0; i < T * H; ++i) h[i] = to_bf16(1.0f);
  for (int64_t j = 0; j < H; ++j) g[j] = to_bf16((float)(1 + j % 7));
  for (int r = 0; r < N; ++r) {
    if (cudaMalloc(&part[r], bytes) != cudaSuccess) return 10;
    cudaMemcpy(part[r], h, bytes, cudaMemcpyHostToDevice);
  }
  if (cudaMalloc(&res, bytes) || cudaMalloc(&gam, H * 2) || cudaMalloc(&out, bytes)) return 11;
  cudaMemcpy(gam, g, H * 2, cudaMemcpyHostToDevice);
  const double want_scale = N / sqrt((double)N * N + eps);
  for (int pass = 0; pass < 2; ++pass) {
    cudaMemset(res, 0, bytes);
    int st;
    if (pass == 0) {
      st = tw_fused_reduce_residual_rmsnorm((const void* const*)part, N, res, gam, eps, T, H,
                                            out, NULL, 0);
    } else {
      cudaStream_t a, b; cudaStreamCreate(&a); cudaStreamCreate(&b);
      int64_t p = -1, s = -1;
      tw_split_opts every = {NULL, 0, 0};        /* every offset, no threshold */
      st = tw_run_wave_split(300, 132, &every, (const void* const*)part, N, res, gam, eps, T, H,
                             out, a, b, 0, &p, &s);
      if (st == TW_OK && (p != 132 || s != 168)) return 12;   /* the worked example */
      cudaStreamSynchronize(a); cudaStreamDestroy(a); cudaStreamDestroy(b);
    }
    if (st != TW_OK) { fprintf(stderr, "%s\n", tw_strerror(st)); return 13; }
    if (cudaDeviceSynchronize() != cudaSuccess) return 14;
    cudaMemcpy(h, res, bytes, cudaMemcpyDeviceToHost);
    cudaMemcpy(y, out, bytes, cudaMemcpyDeviceToHost);
    for (int64_t i = 0; i < T * H; ++i) {
      if (from_bf16(h[i]) != (double)N) return 15;                       /* bit-exact */
      const double want = from_bf16(g[i % H]) * want_scale;
      if (fabs(from_bf16(y[i]) - want) > 2 * ulp_bf16(want)) return 16;   /* 2 ulp */
    }
  }
  int code = -1;
  if (tw_device_status(1, &code) != TW_OK || code != 0) return 17;
  puts("c gpu ok");
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_runs_the_step_on_the_gpu(tmp_path):
    from reduce_rmsnorm_gb300 import build
    lib = build.build()
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    src = tmp_path / "prog.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "prog"
    libdir = next(d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"))
                  if os.path.isdir(d))
    cmd = ["gcc", "-std=c99", "-O1", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(cuda, "include"), str(src), lib, "-L", libdir, "-lcudart", "-lm",
           "-Wl,-rpath," + os.path.dirname(lib) + ":" + libdir, "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "c gpu ok" in r.stdout, (r.returncode, r.stdout, r.stderr)

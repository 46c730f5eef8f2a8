"""The boundary is a C ABI: a C99 program that includes only include/tw.h
compiles with gcc (no C++ or CUDA headers needed), links against libtw.so,
and calls the host-only entry points. Runs on the CPU."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "tw.h"

int main(void) {
  int64_t p = -1, s = -1;
  /* the wave-arithmetic blog's worked example: 300 CTAs on 132 SMs -> 132 / 168 */
  tw_split_opts every = {NULL, 0, 0};
  if (tw_wave_split(300, 300, 132, &every, &p, &s) != TW_OK || p != 132 || s != 168) return 1;
  /* default offsets and threshold (NULL options): single wave keeps the batch whole */
  if (tw_wave_split(1024, 64, 148, NULL, &p, &s) != TW_OK || p != 1024 || s != 0) return 2;
  if (tw_wave_split(-1, 64, 148, NULL, &p, &s) != TW_ERR_INVALID_ARG) return 3;
  int64_t toks[1] = {4096}, pref[1] = {2112};
  if (tw_split_lookup(toks, pref, 1, 4096, 256, 148, NULL, &p, &s) != TW_OK || p != 2112) return 4;
  if (strncmp(tw_strerror(TW_ERR_ALIGN), "TW_ERR_ALIGN", 12) != 0) return 5;
  /* validation before any CUDA call: N = 0 is rejected without a GPU */
  const void* parts[1] = {NULL};
  if (tw_fused_reduce_residual_rmsnorm(parts, 0, NULL, NULL, 1e-5f, 4, 16, NULL, NULL, 0) !=
      TW_ERR_INVALID_ARG) return 6;
  /* plan + run in one call: an empty batch plans (0, 0) and launches nothing */
  p = s = -1;
  if (tw_run_wave_split(0, 148, NULL, parts, 1, NULL, NULL, 1e-5f, 0, 16, NULL, NULL, NULL, 0,
                        &p, &s) != TW_OK || p != 0 || s != 0) return 7;
  puts("c abi ok");
  return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c_program_against_header_and_library(tmp_path):
    from reduce_rmsnorm_gb300 import build
    lib = build.build()
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    cmd = ["gcc", "-std=c99", "-Wall", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           str(src), lib, "-Wl,-rpath," + os.path.dirname(lib), "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and "c abi ok" in r.stdout, (r.returncode, r.stdout, r.stderr)

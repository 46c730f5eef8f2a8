"""Build libtw.so in-tree with nvcc for sm_103a.

    python -m reduce_rmsnorm_gb300.build            # build if sources changed
    python -m reduce_rmsnorm_gb300.build --force    # rebuild

Translation units compile in parallel into ``_build/`` (git-ignored), then
link into ``reduce_rmsnorm_gb300/libtw.so``. The CUDA runtime is linked
statically, so the library needs only the driver at run time. Processes that
build at once (the ranks of a torchrun job) take an exclusive file lock in
turn; whoever gets it second finds the library up to date.
"""

import argparse
import concurrent.futures
import fcntl
import hashlib
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build", "libtw")
LIB = os.path.join(PKG, "libtw.so")

SOURCES = ["fused_kernel.cu", "unfused_kernels.cu", "abi.cpp", "planner.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2,-fvisibility=hidden",
              "-I", INCLUDE, "-I", CSRC] + ARCH


def _nvcc():
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cuda, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def _digest():
    h = hashlib.sha256()
    for name in sorted(os.listdir(CSRC)) + ["../../include/tw.h"]:
        p = os.path.normpath(os.path.join(CSRC, name))
        if os.path.isfile(p):
            h.update(name.encode())
            with open(p, "rb") as f:
                h.update(f.read())
    h.update(" ".join(NVCC_FLAGS).encode())
    h.update(os.uname().machine.encode())
    return h.hexdigest()


def _up_to_date(stamp, digest):
    if not (os.path.exists(LIB) and os.path.exists(stamp)):
        return False
    with open(stamp) as f:
        return f.read().strip() == digest


def build(force=False, verbose=False, ptxas_verbose=False):
    """Compile and link libtw.so; returns its path."""
    os.makedirs(BUILD, exist_ok=True)
    stamp = os.path.join(BUILD, "stamp")
    digest = _digest()
    if not force and _up_to_date(stamp, digest):
        return LIB
    with open(os.path.join(BUILD, "lock"), "w") as lock:
        fcntl.flock(lock, fcntl.LOCK_EX)  # released when the file closes
        if not force and _up_to_date(stamp, digest):
            return LIB  # another process built it meanwhile
        return _build_locked(stamp, digest, verbose, ptxas_verbose)


def _build_locked(stamp, digest, verbose, ptxas_verbose):
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, src + ".o")
        cmd = [nvcc] + NVCC_FLAGS + ["-c", os.path.join(CSRC, src), "-o", obj]
        if ptxas_verbose and src.endswith(".cu"):
            cmd += ["-Xptxas", "-v"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
        return obj, r.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_verbose:
        for _, err in results:
            if err:
                sys.stderr.write(err)
    objs = [o for o, _ in results]
    tmp = "%s.tmp%d" % (LIB, os.getpid())
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, LIB)
    with open(stamp, "w") as f:
        f.write(digest)
    return LIB


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    a = ap.parse_args()
    print(build(force=a.force, verbose=True, ptxas_verbose=a.ptxas_verbose))


if __name__ == "__main__":
    main()

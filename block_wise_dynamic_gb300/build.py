"""Builds the C-ABI shared library ``libbwd.so`` in-tree for sm_103a.

Four translation units (the host codebook builder, the host shard planner,
the optimizer kernels and the stable-embedding kernels) are compiled in parallel and linked with the
static CUDA runtime, so the library depends only on the driver.  No
fast-math: every code decision must be IEEE.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_PATH = os.path.join(PKG, "libbwd.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
HOST_FLAGS = ["-O2", "-fPIC", "-std=c++17", "-ffp-contract=off", "-Wall"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--fmad=false", "-Xcompiler", "-fPIC,-ffp-contract=off"]

SOURCES = {
    "codebook.o": os.path.join(CSRC, "codebook.cpp"),
    "shard.o": os.path.join(CSRC, "shard.cpp"),
    "kernels.o": os.path.join(CSRC, "kernels.cu"),
    "embedding.o": os.path.join(CSRC, "embedding.cu"),
}
HEADERS = [os.path.join(CSRC, h) for h in ("tables.h", "exact_div.cuh", "host_util.h")] + [os.path.join(INCLUDE, "bwd.h")]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libbwd.so")


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = list(SOURCES.values()) + HEADERS + [os.path.abspath(__file__)]
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link ``libbwd.so`` if a source is newer; return its path."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    nvcc = _nvcc()
    procs = []
    for obj, src in SOURCES.items():
        out = os.path.join(BUILD_DIR, obj)
        if src.endswith(".cu"):
            cmd = [nvcc, *NVCC_FLAGS, *ARCH, "-I", INCLUDE, "-c", src, "-o", out]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
        else:
            cuda_inc = os.path.join(os.path.dirname(os.path.dirname(nvcc)), "include")
            cmd = ["g++", *HOST_FLAGS, "-I", INCLUDE, "-I", cuda_inc, "-c", src, "-o", out]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    for cmd, pr in procs:
        log, _ = pr.communicate()
        if verbose and log:
            sys.stdout.write(log)
        if pr.returncode != 0:
            raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{log}")
    tmp = LIB_PATH + ".tmp"
    link = [nvcc, "-shared", *ARCH, "-o", tmp] + [os.path.join(BUILD_DIR, o) for o in SOURCES]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(link)}\n{r.stdout}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))

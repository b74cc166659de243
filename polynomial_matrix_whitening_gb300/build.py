"""Builds libanvil.so in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each .cu under csrc/ compiles to its own object in parallel; the objects link into
``polynomial_matrix_whitening_gb300/libanvil.so`` with the CUDA runtime linked
statically, so the library loads (and exports its symbols) on a machine without a
GPU driver as well.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libanvil.so")
# The timeline build (-DANVIL_TIMELINE): the same library with the cascade kernel's
# per-item timestamps, for performance work only (anvil_timeline_read).
BUILD_TL = os.path.join(PKG, "_build_timeline")
LIB_TL = os.path.join(PKG, "libanvil_timeline.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I" + os.path.join(ROOT, "include")] + ARCH


def nvcc():
    path = shutil.which("nvcc")
    if path:
        return path
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libanvil")


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), timeline: bool = False) -> str:
    """Compiles and links libanvil.so (or, with timeline=True, libanvil_timeline.so);
    returns the library's path."""
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
                     + glob.glob(os.path.join(ROOT, "include", "*.h")))
    build_dir, lib = (BUILD_TL, LIB_TL) if timeline else (BUILD, LIB)
    if timeline:
        extra_flags = list(extra_flags) + ["-DANVIL_TIMELINE"]
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    jobs = []
    for src in sources:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        if force or _stale(obj, [src] + headers):
            jobs.append([cc, "-c", src, "-o", obj] + NVCC_FLAGS + list(extra_flags))
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
            results = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs))
        for cmd, r in zip(jobs, results):
            if verbose or r.returncode != 0:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed on {cmd[2]}")
    objs = [os.path.join(build_dir, os.path.basename(s)[:-3] + ".o") for s in sources]
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [cc, "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            raise RuntimeError(f"nvcc link of {os.path.basename(lib)} failed")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, timeline="--timeline" in sys.argv))

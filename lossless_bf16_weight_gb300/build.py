"""Build the shared library libuw.so in-tree with nvcc for sm_103a.

Translation units are compiled in parallel into _build/ and linked against
the shared CUDA runtime.  Host C++ (the compressor) is plain -O3 with OpenMP,
no architecture-specific flags, so the same source builds on x86-64 and
aarch64 hosts.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libuw.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["compress.cpp", "api.cu", "autotune.cu", "gemv.cu", "gemv_kg.cu", "gemm_tc.cu", "decompress.cu", "transcode.cu", "swiglu.cu",
           "noalloc.cu", "schedule.cu", "diag.cu"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(src: str, verbose: bool) -> list[str]:
    common = ["-O3", "-std=c++17", "-I", INCLUDE, "-I", CSRC, "-Xcompiler", "-fPIC,-fopenmp,-Wall"]
    if src.endswith(".cu"):
        f = common + ARCH + ["-lineinfo", "--expt-relaxed-constexpr"]
        if verbose:
            f += ["-Xptxas", "-v"]
        return f
    return common


def _deps_newer(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    watched = [src, os.path.join(INCLUDE, "uw.h")] + [
        os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".h", ".cuh"))]
    return any(os.path.getmtime(p) > t for p in watched)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    jobs = []
    objs = []
    for s in SOURCES:
        src = os.path.join(CSRC, s)
        obj = os.path.join(BUILD, s + ".o")
        objs.append(obj)
        if force or _deps_newer(obj, src):
            jobs.append([nvcc, *_flags(s, verbose), "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    failed = []
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 4))) as ex:
        for cmd, r in ex.map(run, jobs):
            if r.returncode != 0 or (verbose and r.stderr):
                sys.stderr.write(r.stderr)
            if r.returncode != 0:
                failed.append(cmd[-3])
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(failed))
    if jobs or force or not os.path.exists(LIB):
        tmp = LIB + ".tmp%d" % os.getpid()
        subprocess.check_call([nvcc, "-shared", *ARCH, "-cudart", "shared", "-o", tmp, *objs,
                               "-Xcompiler", "-fopenmp"])
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

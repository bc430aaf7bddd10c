"""Builds libqsa.so in-tree with nvcc for sm_103a (no CMake).

Each translation unit compiles in parallel; the objects link into
``top_block_selection_gb300/lib/libqsa.so`` with the CUDA runtime linked
statically, so the library needs only the NVIDIA driver at run time.
Run ``python -m top_block_selection_gb300._build`` or call ``build()``.
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
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(HERE, "lib")
OBJDIR = os.path.join(LIBDIR, "obj")
LIBPATH = os.path.join(LIBDIR, "libqsa.so")

SOURCES = ["qsa_runtime.cu", "score_tc.cu", "select.cu", "convert.cu", "fused.cu", "fused_h1.cu",
           "fused_h2.cu", "fused_h4.cu", "fused_h8.cu", "fused_h16.cu", "fused_h32.cu",
           "split_reduce.cu", "split_reduce_static.cu", "qsa_api.cpp"]
HEADERS = ["qsa_device.cuh", "qsa_internal.h", "select_row.cuh", "select_warp.cuh", "fused_kernel.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libqsa.so")


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, extra_flags=()) -> str:
    """Compile (if stale) and return the path of libqsa.so."""
    nvcc = _nvcc()
    os.makedirs(OBJDIR, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "qsa.h")]
    jobs = []
    objs = []
    for src in SOURCES:
        sp = os.path.join(CSRC, src)
        op = os.path.join(OBJDIR, src + ".o")
        objs.append(op)
        if _stale(op, [sp, __file__] + hdrs):
            jobs.append([nvcc, *ARCH, *COMMON, *extra_flags, "-c", sp, "-o", op])
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for cmd, res in zip(jobs, ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs)):
                if verbose and (res.stdout or res.stderr):
                    sys.stderr.write(res.stdout + res.stderr)
                if res.returncode != 0:
                    raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    if jobs or _stale(LIBPATH, objs):
        cmd = [nvcc, *ARCH, "-shared", "-o", LIBPATH, *objs, "-lrt", "-ldl", "-lpthread"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("link failed:\n" + " ".join(cmd) + "\n" + res.stdout + res.stderr)
    return LIBPATH


if __name__ == "__main__":
    print(build(verbose=True))

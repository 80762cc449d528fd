"""Compile the engine's C-ABI shared library for sm_103a (in-tree).

One nvcc invocation per translation unit, run in parallel, then one link:
``paged_kv_cache_step_gb300/_build/libgrowpage.so``.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libgrowpage.so")

SOURCES = ["growpage.cpp", "k_summaries.cu", "k_demand.cu", "k_demand_tc.cu", "k_compress.cu", "k_attention.cu",
           "k_attention_tc.cu", "k_entropy.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                   "-I", INCLUDE, "-I", CSRC] + list(extra)


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    deps = [src, os.path.join(CSRC, "gp_kernels.h"), os.path.join(CSRC, "gp_internal.h"),
            os.path.join(CSRC, "demand_common.cuh"), os.path.join(INCLUDE, "growpage.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    """Build (if stale) and return the path of libgrowpage.so."""
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    jobs = []
    objs = []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        objs.append(obj)
        if _stale(obj, path) or ptxas_info:
            extra = ["-Xptxas", "-v"] if (ptxas_info and src.endswith(".cu")) else []
            jobs.append([nvcc] + _flags(extra) + ["-c", path, "-o", obj])

    def run(cmd):
        res = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, res

    rebuilt = False
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            for cmd, res in ex.map(run, jobs):
                if verbose or ptxas_info or res.returncode != 0:
                    print(" ".join(cmd))
                    print(res.stdout + res.stderr)
                if res.returncode != 0:
                    raise RuntimeError(f"nvcc failed on {cmd[-3]}")
        rebuilt = True
    if rebuilt or not os.path.exists(LIB):
        cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", LIB] + objs + [
            "-Xlinker", "-rpath=/usr/local/cuda/lib64"]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            print(" ".join(cmd))
            print(res.stdout + res.stderr)
            raise RuntimeError("link failed")
    return LIB


if __name__ == "__main__":
    import sys
    print(build(verbose=True, ptxas_info="--ptxas" in sys.argv))

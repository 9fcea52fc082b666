"""Builds libmsa.so (the CUDA kernels + C ABI) in-tree with nvcc for sm_103a.

Every .cu file under csrc/ is compiled in parallel into an object, then linked
into block_sparse_gqa_topk_gb300/libmsa.so.  No torch, no cmake.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "libmsa.so")
BUILD = os.path.join(ROOT, "_build")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC",
    "--expt-relaxed-constexpr", "-I" + INCLUDE, "-I" + CSRC,
]


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(out, deps):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdrs = sorted(glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    objs = []
    jobs = []
    for src in srcs:
        obj = os.path.join(BUILD, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + hdrs):
            cmd = [nvcc, *NVCC_FLAGS, "-c", src, "-o", obj]
            if verbose:
                cmd.insert(1, "-Xptxas=-v")
            jobs.append(cmd)

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
        return r.stdout + r.stderr

    if jobs:
        with ThreadPoolExecutor(max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
            for log in ex.map(run, jobs):
                if verbose and log:
                    sys.stdout.write(log)
    if force or jobs or _stale(OUT, objs):
        tmp = OUT + f".tmp{os.getpid()}"
        subprocess.check_call([nvcc, "-shared", "-gencode", "arch=compute_103a,code=sm_103a",
                               "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lpthread", "-lrt"])
        os.replace(tmp, OUT)
    return OUT


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

"""Builds libgs_gb300.so (the C-ABI CUDA library) in-tree for sm_103a, and its
bounds-checked twin libgs_gb300_checked.so (the same sources with -DGS_CHECKED:
every index read from memory is tested before use, failures are counted and
the access skipped, gs_check_report returns the count).

Each translation unit of both libraries is compiled by nvcc in parallel, then
each library is linked with the shared CUDA runtime.  Forward-decision code
relies on IEEE rounding of every operation, so both libraries are compiled
without fma contraction (-fmad=false), with IEEE division and square root and
without flush-to-zero; fused multiply-adds appear only where the source spells
__fmaf_rn.

    python -m differentiable_rasterizer_gb300.build [--verbose]
"""
from __future__ import annotations

import concurrent.futures
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libgs_gb300.so")
CHECKED_LIB = os.path.join(OUT_DIR, "libgs_gb300_checked.so")
# (library, object directory, extra flags)
VARIANTS = ((LIB, OUT_DIR, []), (CHECKED_LIB, os.path.join(OUT_DIR, "checked"), ["-DGS_CHECKED"]))
SOURCES = ["abi.cu", "project.cu", "binsort.cu", "prune.cu", "raster.cu", "dssim.cu", "compose.cu", "compact.cu", "adam.cu"]
HEADERS = ["gs_common.cuh", "project_math.cuh", "scan.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-fmad=false", "-prec-div=true", "-prec-sqrt=true", "-ftz=false",
              "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden", "-I", os.path.join(ROOT, "include")]


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, force: bool = False) -> str:
    """Build both libraries (only what is stale); returns the plain library's path."""
    nvcc = _nvcc()
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "gs.h")]
    jobs, links = [], []
    for lib, obj_dir, extra in VARIANTS:
        os.makedirs(obj_dir, exist_ok=True)
        objs, fresh = [], False
        for src in SOURCES:
            s = os.path.join(CSRC, src)
            o = os.path.join(obj_dir, src.replace(".cu", ".o"))
            objs.append(o)
            if force or _stale(o, [s] + hdrs):
                cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", s, "-o", o]
                if verbose:
                    cmd += ["-Xptxas", "-v"]
                jobs.append(cmd)
                fresh = True
        links.append((lib, objs, fresh))

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    workers = min(16, max(1, os.cpu_count() or 1), max(1, len(jobs)))
    with concurrent.futures.ThreadPoolExecutor(max_workers=workers) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or r.returncode != 0:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed: " + " ".join(cmd))
    for lib, objs, fresh in links:
        if force or fresh or _stale(lib, objs):
            tmp = lib + ".tmp%d" % os.getpid()
            subprocess.check_call([nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs])
            os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(verbose="--verbose" in sys.argv, force="--force" in sys.argv))

"""Build libgbq.so in-tree: every csrc/*.cu compiled for sm_103a in parallel, then linked.

Usage: python -m ffn_rotate_quantize_gb300.build [--force] [--debug]   (or call build_lib()).

--debug builds libgbq_debug.so instead: the same sources with -DGBQ_DEBUG_BOUNDS, so every kernel
checks its computed global-memory accesses against the tensors' extents, records GBQ_DEV_BOUNDS in
the device status word on a violation and skips the access (no trap).  Select it at run time with
GBQ_LIB=<path to libgbq_debug.so>.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(os.path.dirname(HERE), "_build")
LIB = os.path.join(HERE, "libgbq.so")
BUILD_DEBUG = os.path.join(os.path.dirname(HERE), "_build_debug")
LIB_DEBUG = os.path.join(HERE, "libgbq_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(obj: str, deps: list[str]) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    return any(os.path.getmtime(d) > t for d in deps)


def build_lib(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    nvcc = _nvcc()
    build_dir, lib_path = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    flags = FLAGS + (["-DGBQ_DEBUG_BOUNDS"] if debug else [])
    os.makedirs(build_dir, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(os.path.dirname(HERE), "include", "*.h"))
    jobs = []
    objs = []
    for src in sources:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or _stale(obj, [src] + headers):
            jobs.append([nvcc, *ARCH, *flags, "-c", src, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        list(ex.map(run, jobs))
    if jobs or not os.path.exists(lib_path):
        tmp = lib_path + ".tmp"
        run([nvcc, *ARCH, "-shared", *objs, "-o", tmp])
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build_lib(force="--force" in sys.argv, verbose=True, debug="--debug" in sys.argv))

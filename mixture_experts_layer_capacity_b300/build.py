"""Build ``libmoe.so`` in-tree with nvcc for sm_103a.

    python -m mixture_experts_layer_capacity_b300.build [--force] [--debug-bounds | --timeline]

Each ``csrc/*.cu`` compiles to an object under ``_build/`` (rebuilt when the
source or any header is newer), then the objects link into
``mixture_experts_layer_capacity_b300/libmoe.so`` against the shared CUDA
runtime.  The driver API (tensor-map encoding) is reached through the
runtime's entry-point query, so libcuda is not linked.

``--debug-bounds`` builds the same sources with ``-DMOE_DEBUG_BOUNDS`` into
``libmoe_debug_bounds.so``: the routing and combine kernels then check every
expert and row index against its range and record
MOE_DEVICE_INDEX_OUT_OF_RANGE instead of making the access.  Load it by
setting ``MOE_LIBRARY`` to its path before the binding is first used.

``--timeline`` builds them with ``-DMOE_TIMELINE`` into
``libmoe_timeline.so``: CTA 0 of every routed CTA-pair GEMM launch then
stamps each unit's MMA and epilogue phases with the global timer, read back
with ``moe_timeline_read`` (``timeline.py`` prints them).  The stamps cost a
few stores per unit, so this library is for profiling, not for timing.
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
BUILD = os.path.join(ROOT, "_build", "libmoe")
LIB = os.path.join(PKG, "libmoe.so")
BUILD_DEBUG = os.path.join(ROOT, "_build", "libmoe_debug_bounds")
LIB_DEBUG = os.path.join(PKG, "libmoe_debug_bounds.so")
BUILD_TIMELINE = os.path.join(ROOT, "_build", "libmoe_timeline")
LIB_TIMELINE = os.path.join(PKG, "libmoe_timeline.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
         "-Xcompiler", "-fPIC,-fvisibility=hidden", "-I", os.path.join(ROOT, "include")]


def _headers():
    return (glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
            + glob.glob(os.path.join(ROOT, "include", "*.h")))


def _newest(paths):
    return max((os.path.getmtime(p) for p in paths), default=0.0)


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False,
          timeline: bool = False) -> str:
    if debug_bounds and timeline:
        raise ValueError("debug_bounds and timeline are separate builds")
    if debug_bounds:
        build_dir, lib, flags = BUILD_DEBUG, LIB_DEBUG, FLAGS + ["-DMOE_DEBUG_BOUNDS"]
    elif timeline:
        build_dir, lib, flags = BUILD_TIMELINE, LIB_TIMELINE, FLAGS + ["-DMOE_TIMELINE"]
    else:
        build_dir, lib, flags = BUILD, LIB, FLAGS
    os.makedirs(build_dir, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    hdr_time = _newest(_headers())
    jobs = []
    objs = []
    for src in sources:
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or not os.path.exists(obj) or os.path.getmtime(obj) < max(
                os.path.getmtime(src), hdr_time):
            jobs.append([NVCC, *ARCH, *flags, "-c", src, "-o", obj])

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)

    with ThreadPoolExecutor(max_workers=min(8, max(1, len(jobs)))) as ex:
        list(ex.map(run, jobs))
    if jobs or not os.path.exists(lib) or os.path.getmtime(lib) < _newest(objs):
        tmp = lib + f".tmp{os.getpid()}"
        run([NVCC, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
             "-Xlinker", "-rpath,/usr/local/cuda/lib64"])
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True,
                debug_bounds="--debug-bounds" in sys.argv, timeline="--timeline" in sys.argv))

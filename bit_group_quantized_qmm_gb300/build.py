"""Build libqmm_gb300.so in-tree with nvcc for sm_103a.

Each CUDA translation unit is compiled in parallel into ``_build/``, then
linked (static CUDA runtime) into ``libqmm_gb300.so`` beside this file.
Rebuilds only what is older than its sources.

``build(checked=True)`` makes the test-only checked variant,
``libqmm_gb300_checked.so`` (objects in ``_build_checked/``): the same sources
with ``QMM_CHECKS=1``, whose kernels test their internal index ranges (weight
chunks inside the blob, tensor-memory columns inside the allocation, scale
stages inside their slots) and record a failure in the device error word
instead of making the access. The binding loads it instead of the product
library when the environment sets ``QMM_CHECKED_LIBRARY=1``.
"""

from __future__ import annotations

import glob
import os
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libqmm_gb300.so")
BUILD_CHECKED = os.path.join(HERE, "_build_checked")
LIB_CHECKED = os.path.join(HERE, "libqmm_gb300_checked.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC",
    "-I", INCLUDE, "-I", CSRC,
]


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _newest(paths):
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile and link the library (or its checked variant); returns its path."""
    build_dir, lib = (BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD, LIB)
    flags = NVCC_FLAGS + (["-DQMM_CHECKS=1"] if checked else [])
    os.makedirs(build_dir, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    hdr_time = _newest(headers) if headers else 0.0
    nvcc = _nvcc()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        if (not force and os.path.exists(obj)
                and os.path.getmtime(obj) >= max(os.path.getmtime(src), hdr_time)):
            return obj
        cmd = [nvcc, *flags, "-c", src, "-o", obj + ".tmp"]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        os.replace(obj + ".tmp", obj)
        return obj

    with ThreadPoolExecutor(max_workers=min(8, len(sources))) as ex:
        objs = list(ex.map(compile_one, sources))
    if force or not os.path.exists(lib) or os.path.getmtime(lib) < _newest(objs):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-cudart", "static",
               "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


def build_all(force: bool = False) -> None:
    """The product library and its checked variant."""
    build(force=force)
    build(force=force, checked=True)


if __name__ == "__main__":
    print(build(verbose=True))

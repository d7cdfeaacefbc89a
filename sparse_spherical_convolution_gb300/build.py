"""Compiles the CUDA library (sm_103a) into an in-tree shared object.

    python -m sparse_spherical_convolution_gb300.build [--force] [-v] [--debug-bounds]

Each translation unit is compiled in parallel with
``nvcc -gencode arch=compute_103a,code=sm_103a -O3 -lineinfo`` and linked
with ``nvcc -shared``.  The result lives in ``_build/`` next to this file.

``--debug-bounds`` builds the bounds-checked variant of the same sources
(``-DDISCO_DEBUG_BOUNDS``, ``LIB_BOUNDS``): every kernel range-checks its
gather indices and TMA / bulk-copy coordinates and reports a failed check
through ``disco_device_status`` instead of touching memory outside a tensor.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import platform
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, f"libdisco_gb300_{platform.machine()}.so")
LIB_BOUNDS = os.path.join(BUILD, f"libdisco_gb300_{platform.machine()}_bounds.so")
SOURCES = ["disco_capi.cu", "disco_psi.cu", "disco_contract.cu", "disco_fused.cu",
           "disco_fwd_tc.cu", "disco_bwd_tc.cu", "disco_gemm_tc.cu", "disco_host.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _compile(src: str, verbose: bool, debug_bounds: bool = False) -> str:
    tag = "_bounds" if debug_bounds else ""
    obj = os.path.join(BUILD, os.path.splitext(src)[0] + f"_{platform.machine()}{tag}.o")
    cmd = [_nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr",
           "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
    if debug_bounds:
        cmd.insert(1, "-DDISCO_DEBUG_BOUNDS")
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose:
        sys.stderr.write(r.stderr)
    return obj


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "disco.h")]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    lib = LIB_BOUNDS if debug_bounds else LIB
    os.makedirs(BUILD, exist_ok=True)
    if not force and not _stale(lib):
        return lib
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, debug_bounds), SOURCES))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug_bounds="--debug-bounds" in sys.argv))

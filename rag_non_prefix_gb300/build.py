"""Builds the sm_103a shared libraries in-tree (nvcc only; no cmake).

* ``rag_non_prefix_gb300/libcacheblend.so``: the blended-prefill kernels and runtime
  behind include/cacheblend.h.
* ``harness/libsynth.so``: the harness's device-side input generator.
* ``harness/libsynth_host.so``: the same generator on the host (gcc, OpenMP), so that
  CPU-side inputs of billion-parameter shapes take seconds instead of minutes.

Objects are compiled in parallel into ``_build/`` and relinked only when a source or
header is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fno-strict-aliasing"]

LIBS = {
    os.path.join(PKG, "libcacheblend.so"): {
        "srcs": [os.path.join(PKG, "csrc", f) for f in ("kernels_bw.cu", "select.cu", "gemm.cu", "gemm_pair.cu", "gemm_noalloc.cu", "attention.cu",
                                                               "codec.cu", "decode.cu", "gemv.cu", "engine.cu",
                                                               "controller.cpp")],
        "deps": [os.path.join(PKG, "csrc", f) for f in ("common.cuh", "internal.h")] + [os.path.join(INCLUDE, "cacheblend.h")],
        "build": os.path.join(PKG, "_build"),
    },
    os.path.join(ROOT, "harness", "libsynth.so"): {
        "srcs": [os.path.join(ROOT, "harness", "csrc", "synth.cu")],
        "deps": [],
        "build": os.path.join(ROOT, "harness", "_build"),
    },
}


# plain C libraries (gcc; they run on the host of whichever machine builds them)
HOST_LIBS = {
    os.path.join(ROOT, "harness", "libsynth_host.so"): [os.path.join(ROOT, "harness", "csrc", "synth_host.c")],
}


def gcc() -> str:
    p = shutil.which("gcc") or shutil.which("cc")
    if not p:
        raise RuntimeError("gcc not found: needed for the host-side libraries")
    return p


def _build_host(lib: str, srcs) -> None:
    if not _stale(lib, srcs):
        return
    base = [gcc(), "-O2", "-shared", "-fPIC", "-ffp-contract=off", "-o", lib, *srcs]
    r = subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, text=True)
    if r.returncode != 0:  # no OpenMP runtime: single-threaded build of the same code
        r = subprocess.run(base, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"gcc failed for {lib}:\n{r.stdout}\n{r.stderr}")


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return p


def _stale(target: str, inputs) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(f) > t for f in inputs)


def _compile(src: str, obj: str, deps) -> None:
    if not _stale(obj, [src] + list(deps)):
        return
    cmd = [nvcc(), *ARCH, *FLAGS, "-I", INCLUDE, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")


def build(verbose: bool = False) -> list:
    """Compile every library; returns the library paths."""
    out = []
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        for lib, spec in LIBS.items():
            os.makedirs(spec["build"], exist_ok=True)
            objs = [os.path.join(spec["build"], os.path.splitext(os.path.basename(s))[0] + ".o") for s in spec["srcs"]]
            list(ex.map(lambda so: _compile(so[0], so[1], spec["deps"]), zip(spec["srcs"], objs)))
            if _stale(lib, objs):
                cmd = [nvcc(), *ARCH, "-shared", "-o", lib, *objs]
                r = subprocess.run(cmd, capture_output=True, text=True)
                if r.returncode != 0:
                    raise RuntimeError(f"link failed for {lib}:\n{r.stdout}\n{r.stderr}")
            if verbose:
                print("built", lib, file=sys.stderr)
            out.append(lib)
    for lib, srcs in HOST_LIBS.items():
        _build_host(lib, srcs)
        if verbose:
            print("built", lib, file=sys.stderr)
        out.append(lib)
    return out


if __name__ == "__main__":
    build(verbose=True)

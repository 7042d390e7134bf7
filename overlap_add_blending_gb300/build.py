"""Build libtdp.so in-tree with nvcc for sm_103a.

    python -m overlap_add_blending_gb300.build [-v] [-f] [--debug]

Three translation units (host planner, channel-first kernels, token-major
kernels) compiled in parallel and
linked into overlap_add_blending_gb300/libtdp.so.  The CUDA runtime is
linked statically, so the library needs only the CUDA driver at run time.
--debug builds libtdp_debug.so instead, with TDP_DEBUG_CHECKS=1: the hot
kernels check their global and shared indices and report a failed check in
the device error word (bit 8) instead of making the access; the binding
loads it when TDP_DEBUG_CHECKS=1 is set in the environment.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtdp.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libtdp_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["tdp_plan.cpp", "tdp_kernels.cu", "tdp_token_major.cu"]
HEADERS = ["tdp_geometry.h", "tdp_stream.cuh"]


def _nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "bin", "nvcc")):
            return os.path.join(cand, "bin", "nvcc")
    found = shutil.which("nvcc")
    if not found:
        raise RuntimeError("nvcc not found")
    return found


def _flags(verbose: bool, debug: bool = False):
    f = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC] + ARCH
    if debug:
        f += ["-DTDP_DEBUG_CHECKS=1"]
    if verbose:
        f += ["-Xptxas", "-v"]
    return f


def build(verbose: bool = False, force: bool = False, debug: bool = False) -> str:
    """Compile (if any source is newer than the library) and return its path."""
    lib, bdir = (LIB_DEBUG, BUILD_DEBUG) if debug else (LIB, BUILD)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    deps = srcs + [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "tdp.h")]
    if not force and os.path.exists(lib):
        mtime = os.path.getmtime(lib)
        if all(os.path.getmtime(d) <= mtime for d in deps):
            return lib
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()
    objs = [os.path.join(bdir, os.path.splitext(s)[0] + ".o") for s in SOURCES]

    def compile_one(pair):
        src, obj = pair
        cmd = [nvcc, "-c", src, "-o", obj] + _flags(verbose, debug)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        return r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        logs = list(ex.map(compile_one, zip(srcs, objs)))
    tmp = lib + ".tmp"
    cmd = [nvcc, "-shared", "-o", tmp] + objs + ARCH + ["-Xcompiler", "-fPIC"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        sys.stdout.write("".join(logs))
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, debug="--debug" in sys.argv))

"""Build libmxfp8norm.so in-tree with nvcc for sm_103a (GB300).

Each CUDA translation unit is compiled in parallel, then linked into one shared
library next to this file. The CUDA runtime is linked statically, so the library
only needs the NVIDIA driver at run time. No fast-math flags: float32 keeps
IEEE sub-normals, divides and square roots.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libmxfp8norm.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
# The bounds-checking build: the same library with the quantize kernels
# compiled with -DMXFP8_DEBUG_BOUNDS (every global access checked against the
# extents the C ABI states; violations recorded in mxfp8_device_status).
BOUNDS_LIB_PATH = os.path.join(PKG, "libmxfp8norm_bounds.so")
BOUNDS_SOURCE = "mxfp8_kernels.cu"

SOURCES = ["mxfp8_kernels.cu", "mxfp8_update.cu", "mxfp8_gemm.cu", "mxfp8_mm.cu",
           "mxfp8_api.cu"]
HEADERS = [os.path.join(CSRC, h) for h in ("mx_table.h", "mx_update.h", "mx_trace.h",
                                           "mx_gemm.h", "mx_umma.h")] + [
    os.path.join(INCLUDE, "mxfp8norm.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I" + INCLUDE, "-I" + CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link the library (and its bounds-checking twin) if any source
    or header is newer; return the library's path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    objs, procs = [], []
    jobs = [(src, os.path.join(BUILD_DIR, src.replace(".cu", ".o")), []) for src in SOURCES]
    bounds_obj = os.path.join(BUILD_DIR, BOUNDS_SOURCE.replace(".cu", "_bounds.o"))
    jobs.append((BOUNDS_SOURCE, bounds_obj, ["-DMXFP8_DEBUG_BOUNDS"]))
    for src, obj, extra in jobs:
        path = os.path.join(CSRC, src)
        if not extra:
            objs.append(obj)
        if force or _stale(obj, [path, *HEADERS]):
            cmd = [nvcc(), *NVCC_FLAGS, *extra, "-c", path, "-o", obj]
            if ptxas_info:
                cmd.insert(1, "-Xptxas=-v")
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT, text=True)))
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append((cmd, out))
        elif out and (verbose or ptxas_info):
            print(out, file=sys.stderr)
    if failed:
        msg = "\n".join(" ".join(c) + "\n" + o for c, o in failed)
        raise RuntimeError("nvcc failed:\n" + msg)
    kernels_obj = os.path.join(BUILD_DIR, BOUNDS_SOURCE.replace(".cu", ".o"))
    bounds_objs = [bounds_obj if o == kernels_obj else o for o in objs]
    for lib, lib_objs in ((LIB_PATH, objs), (BOUNDS_LIB_PATH, bounds_objs)):
        if force or procs or _stale(lib, lib_objs):
            tmp = lib + f".tmp{os.getpid()}"
            cmd = [nvcc(), *ARCH, "-shared", *lib_objs, "-o", tmp]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            subprocess.run(cmd, check=True)
            os.replace(tmp, lib)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))

"""Build the CUDA library ``libmoe_w8a8.so`` in-tree with nvcc (sm_103a only).

Each translation unit compiles in parallel into ``_build/``; the shared
library lands next to this file, where the binding loads it.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoe_w8a8.so")
# the checked build (-DMOE_CHECKED=1): every data-derived index range-checked
# in the kernels, an index out of range reported through the device error
# word instead of read or written (see internal.h)
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "libmoe_w8a8_checked.so")
SOURCES = ["api.cu", "route.cu", "router.cu", "pointwise.cu", "gemm.cu", "gemm_pair.cu", "gemm_skinny.cu",
           "static_linear.cu", "fp8.cu", "gemm_fp8_pair.cu", "fused.cu"]
HEADERS = ["internal.h", "ptx.cuh", "gemm_common.cuh", "gemm_skinny.cuh", "router_small.cuh"]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    # every binary32 multiply/add of the method rounds on its own
    "-fmad=false",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-I", os.path.join(ROOT, "include"),
]


def nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cuda, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=(), checked: bool = False) -> str:
    """Compile the library (the checked build with checked=True) and return its path."""
    build_dir, lib_path = (BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD, LIB)
    if checked:
        extra_flags = (*extra_flags, "-DMOE_CHECKED=1")
    os.makedirs(build_dir, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "moe_w8a8.h")]
    procs, objs = [], []
    for src in SOURCES:
        src_path = os.path.join(CSRC, src)
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(obj)
        if force or _stale(obj, [src_path, *headers]):
            cmd = [nvcc(), *NVCC_FLAGS, *extra_flags, "-c", src_path, "-o", obj]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode != 0:
            sys.stderr.write(out.decode(errors="replace"))
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    if force or _stale(lib_path, objs):
        tmp = lib_path + f".tmp{os.getpid()}"
        cmd = [nvcc(), "-shared", "-gencode", "arch=compute_103a,code=sm_103a", *objs, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, checked="--checked" in sys.argv))

"""Builds libmageflow.so in-tree for sm_103a with nvcc (no JIT cache, no torch extension).

    python packed_rectified_flow_packer_b300/build.py [--force]

Objects go to packed_rectified_flow_packer_b300/_build/ and the library to
packed_rectified_flow_packer_b300/libmageflow.so.  Rebuilds only what changed.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmageflow.so")
# the bounds-checked variant (-DMF_CHECKED): same sources and ABI, kernels check every
# plan-derived index they read
BUILD_CHECKED = os.path.join(PKG, "_build_checked")
LIB_CHECKED = os.path.join(PKG, "libmageflow_checked.so")
CUDA_HOME = os.environ.get("CUDA_HOME", "/usr/local/cuda")
NVCC = os.path.join(CUDA_HOME, "bin", "nvcc")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC]
SOURCES = ["plan.cpp", "api.cu", "gemm.cu", "attention.cu", "attention_bwd.cu", "block_bwd.cu", "pointwise.cu", "noalloc.cu"]


def _deps(src):
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return [os.path.join(CSRC, src), os.path.join(INCLUDE, "mageflow.h"), __file__] + headers


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, force, checked=False):
    obj = os.path.join(BUILD_CHECKED if checked else BUILD, src + ".o")
    if not force and not _stale(obj, _deps(src)):
        return obj, None
    flags = COMMON + (["-DMF_CHECKED"] if checked else [])
    cmd = [NVCC] + ARCH + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
    if src.endswith(".cpp"):
        cmd = [NVCC] + flags + ["-x", "c++", "-c", os.path.join(CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        return obj, f"{' '.join(cmd)}\n{r.stdout}\n{r.stderr}"
    return obj, None


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    lib = LIB_CHECKED if checked else LIB
    os.makedirs(BUILD_CHECKED if checked else BUILD, exist_ok=True)
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda s: _compile(s, force, checked), SOURCES))
    errors = [e for _, e in results if e]
    if errors:
        raise RuntimeError("libmageflow build failed:\n" + "\n".join(errors))
    objs = [o for o, _ in results]
    if force or _stale(lib, objs):
        cmd = [NVCC] + ARCH + ["-shared", "-cudart", "shared", "-o", lib] + objs + [
            "-Xlinker", "-rpath=" + os.path.join(CUDA_HOME, "lib64")]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"libmageflow link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose:
        print(lib)
    return lib


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, checked="--checked" in sys.argv)

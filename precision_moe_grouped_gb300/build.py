"""Builds libmoe.so (the C-ABI library) from csrc/ with nvcc for sm_103a.

Each .cu file compiles in parallel to an object in _build/, then one link
step writes libmoe.so next to this file.  build(checks=True) makes the
bounds-checked debug build instead: the same sources with -DMOE_CHECKS,
objects in _build_checks/, library libmoe_checked.so (the binding loads it
when MOE_CHECKED=1).  Usage: python -m precision_moe_grouped_gb300.build
[--force] [--checks]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoe.so")
BUILD_CHECKS = os.path.join(PKG, "_build_checks")
LIB_CHECKS = os.path.join(PKG, "libmoe_checked.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    p = os.path.join(cuda, "bin", "nvcc")
    return p if os.path.exists(p) else "nvcc"


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [
        os.path.join(os.path.dirname(PKG), "include", "moe.h")]


def _compile(src: str, extra, build_dir: str) -> str:
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [_nvcc(), *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
    return obj


def build(force: bool = False, extra=(), checks: bool = False) -> str:
    """Compile (if any source is newer than the library) and return its path."""
    lib, build_dir = (LIB_CHECKS, BUILD_CHECKS) if checks else (LIB, BUILD)
    extra = list(extra) + (["-DMOE_CHECKS"] if checks else [])
    if not force and os.path.exists(lib):
        lib_t = os.path.getmtime(lib)
        if all(os.path.getmtime(d) <= lib_t for d in _deps()):
            return lib
    os.makedirs(build_dir, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, build_dir), _sources()))
    tmp = lib + ".tmp"
    cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, checks="--checks" in sys.argv))

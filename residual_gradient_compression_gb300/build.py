"""Builds libadacomp.so in-tree for GB300 (sm_103a) with nvcc.

One nvcc invocation compiles the three translation units in parallel; the result is
placed next to this file and loaded by the package's ctypes binding. With
ADACOMP_DEBUG_CHECKS=1 in the environment, the build and the binding use the debug
library instead, libadacomp_debug.so beside it, built with -DADACOMP_DEBUG_CHECKS:
every compress, decode and materialise call then waits for its stream (unless the
stream is being captured) and returns ADACOMP_ERR_CUDA for an error raised by its own
kernels.
"""
from __future__ import annotations

import glob
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
LIB = os.path.join(HERE, "libadacomp.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources():
    return sorted(glob.glob(os.path.join(HERE, "csrc", "*.cu")))


def _inputs():
    return sources() + glob.glob(os.path.join(HERE, "csrc", "*.cuh")) + [
        os.path.join(ROOT, "include", "adacomp.h")]


LIB_DEBUG = os.path.join(HERE, "libadacomp_debug.so")


def debug_requested() -> bool:
    return os.environ.get("ADACOMP_DEBUG_CHECKS") == "1"


def lib_path(debug: bool | None = None) -> str:
    """The library the environment selects (the debug build with ADACOMP_DEBUG_CHECKS=1)."""
    return LIB_DEBUG if (debug_requested() if debug is None else debug) else LIB


def up_to_date(debug: bool | None = None) -> bool:
    path = lib_path(debug)
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(p) <= t for p in _inputs())


def command(out: str, debug: bool = False, verbose: bool = False) -> list:
    nvcc = os.environ.get("NVCC", "nvcc")
    cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-shared", "-Xcompiler", "-fPIC",
           "--threads", "4", *(["-DADACOMP_DEBUG_CHECKS"] if debug else []),
           "-I", os.path.join(ROOT, "include"), "-o", out, *sources()]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def build(force: bool = False, verbose: bool = False, debug: bool | None = None) -> str:
    debug = debug_requested() if debug is None else debug
    path = lib_path(debug)
    if not force and up_to_date(debug):
        return path
    tmp = path + f".tmp{os.getpid()}"
    subprocess.check_call(command(tmp, debug, verbose))
    os.replace(tmp, path)
    return path


if __name__ == "__main__":
    print(build(force=True, verbose=True))

"""Builds libgqa.so in-tree with nvcc for sm_103a (B300), and its checking
twin libgqa_debug.so (the same sources compiled with GQA_DEBUG: device
bounds checks that flag GQA_DEVERR_BOUNDS and skip the access, never trap).
The two compile in parallel."""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB = os.path.join(PKG, "libgqa.so")
DEBUG_LIB = os.path.join(PKG, "libgqa_debug.so")
MAIN_SRC = os.path.join(PKG, "csrc", "gqa_lib.cu")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC,-O2", "-shared",
    "-I" + os.path.join(ROOT, "include"),
]


def _sources():
    return [MAIN_SRC] + glob.glob(os.path.join(PKG, "csrc", "*.cuh")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(s) <= t for s in _sources())


def build(force: bool = False, verbose: bool = False, debug: bool = True) -> str:
    jobs = []
    for lib, extra in ((LIB, []), (DEBUG_LIB, ["-DGQA_DEBUG"])):
        if lib == DEBUG_LIB and not debug:
            continue
        if not force and up_to_date(lib):
            continue
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [NVCC] + FLAGS + extra + (["-Xptxas", "-v"] if verbose else []) + ["-o", tmp, MAIN_SRC]
        jobs.append((subprocess.Popen(cmd), tmp, lib))
    failed = [j for j in jobs if j[0].wait() != 0]
    if failed:
        raise subprocess.CalledProcessError(failed[0][0].returncode, "nvcc")
    for _, tmp, lib in jobs:
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

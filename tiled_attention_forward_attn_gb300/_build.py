"""Builds the CUDA library ``libfa.so`` in-tree for sm_103a with nvcc, and
its guarded twin ``libfa_guarded.so`` (the same sources compiled with
``-DFA_GUARDED=1``: every TMA tile origin, TMEM column range and global
store is bounds-checked, a failure sets FA_DEVICE_STATUS_BOUNDS; a debug
build for tests, not for timing).  Both are compiled in parallel.

The libraries are plain C ABI (``include/fa.h``) with the CUDA runtime
linked statically, so they depend on nothing but the NVIDIA driver at run
time.
"""
from __future__ import annotations

import os
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG_DIR, "libfa.so")
GUARDED_LIB_PATH = os.path.join(PKG_DIR, "libfa_guarded.so")
SOURCES = ("fa_api.cu",)
HEADERS = ("fa_bwd_kernel.cuh", "fa_fwd_d256.cuh", "fa_fwd_kernel.cuh", "fa_order_ablation.cuh",
           "fa_splitkv.cuh", "ptx.cuh")

NVCC_FLAGS = (
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-shared",
)


def _inputs():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "fa.h"))
    return files


def up_to_date(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _command(out: str, guarded: bool, verbose: bool):
    cmd = [nvcc(), *NVCC_FLAGS, "-I", INCLUDE, "-I", CSRC, "-o", out,
           *[os.path.join(CSRC, s) for s in SOURCES]]
    if guarded:
        cmd.insert(1, "-DFA_GUARDED=1")
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    return cmd


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libfa.so and libfa_guarded.so (each skipped when it is newer
    than every source); returns the path of libfa.so."""
    jobs = []
    for path, guarded in ((LIB_PATH, False), (GUARDED_LIB_PATH, True)):
        if force or not up_to_date(path):
            tmp = path + f".tmp{os.getpid()}"
            jobs.append((subprocess.Popen(_command(tmp, guarded, verbose)), tmp, path))
    failed = None
    for proc, tmp, path in jobs:
        if proc.wait() != 0:
            failed = path
        elif failed is None:
            os.replace(tmp, path)
    if failed is not None:
        raise subprocess.CalledProcessError(1, f"nvcc ({os.path.basename(failed)})")
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))

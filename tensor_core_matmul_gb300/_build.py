"""In-tree build of libtcgemm.so (nvcc, sm_103a only).

One translation unit, one -gencode, no cmake: the library builds in seconds
both on an x86 build host (cross-compiling) and on an aarch64 GPU host.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(PKG, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libtcgemm.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
_lock = threading.Lock()


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (CUDA toolkit required to build libtcgemm)")


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))


def is_stale(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(s) > t for s in sources())


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None) -> str:
    """Compile csrc/tcgemm.cu into _lib/libtcgemm.so unless it is up to date."""
    with _lock:
        if not force and not extra_flags and not is_stale():
            return LIB_PATH
        os.makedirs(LIB_DIR, exist_ok=True)
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = [nvcc(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "--shared", "-Xcompiler", "-fPIC",
               "-I", INCLUDE, os.path.join(CSRC, "tcgemm.cu"), "-o", tmp]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        if extra_flags:
            cmd[1:1] = list(extra_flags)
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + res.stdout + res.stderr)
        if verbose:
            print(res.stdout + res.stderr)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH

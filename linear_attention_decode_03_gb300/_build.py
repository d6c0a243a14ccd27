"""In-tree build of libkda.so for sm_103a with nvcc (no torch extension machinery).

The library links the CUDA runtime statically, so it loads without any
library-path setup; it contains only the CUDA kernels and the C ABI declared
in include/kda.h.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
SOURCES = [os.path.join(PKG_DIR, "csrc", "kda_step.cu"), os.path.join(PKG_DIR, "csrc", "kda_linear.cu")]
HEADERS = [os.path.join(ROOT, "include", "kda.h")]
LIB_PATH = os.path.join(PKG_DIR, "libkda.so")
# KDA_DEBUG build: adds the device check for duplicate slots in a step (KDA_ERR_DUPLICATE)
DEBUG_LIB_PATH = os.path.join(PKG_DIR, "libkda_debug.so")
ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkda.so")


def up_to_date(path: str = LIB_PATH) -> bool:
    if not os.path.exists(path):
        return False
    t = os.path.getmtime(path)
    return all(os.path.getmtime(p) <= t for p in SOURCES + HEADERS)


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile libkda.so (or, with debug, libkda_debug.so: -DKDA_DEBUG) in place,
    skipped when it is newer than its sources."""
    out = DEBUG_LIB_PATH if debug else LIB_PATH
    if not force and up_to_date(out):
        return out
    tmp = out + f".tmp{os.getpid()}"
    # --threads: the translation units compile in parallel (--split-compile, which also
    # splits a unit's kernels across processes, gives slower step kernels)
    cmd = [nvcc_path(), *ARCH_FLAGS, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           "-cudart", "static", "--threads", "0", "-I", os.path.join(ROOT, "include"),
           *(["-DKDA_DEBUG"] if debug else []), "-o", tmp, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed ({res.returncode}):\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, out)
    if verbose:
        print(res.stderr)
    return out


if __name__ == "__main__":
    print(build(force=True, verbose=True))

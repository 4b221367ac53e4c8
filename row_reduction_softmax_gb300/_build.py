"""Build librrs.so in-tree from the CUDA sources, for sm_103a only.

Each translation unit is compiled by its own ``nvcc`` process (in parallel),
then linked into one shared library with the CUDA runtime linked statically,
so the library needs nothing but the driver at run time.  No cmake, no torch
extension machinery: plain ``nvcc``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_DIR = os.path.join(PKG_DIR, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "librrs.so")

SOURCES = ["capi.cu", "softmax_row.cu", "softmax_split.cu", "softmax_staged.cu", "row_sum.cu",
           "softmax_noalloc.cu", "softmax_cols.cu", "softmax_rows_two_pass.cu",
           "gelu.cu", "attention.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    exe = shutil.which("nvcc")
    if exe is None:
        cand = "/usr/local/cuda/bin/nvcc"
        if os.path.exists(cand):
            return cand
        raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build librrs")
    return exe


def compile_flags(ptxas_verbose: bool = False) -> list[str]:
    flags = ARCH + [
        "-O3", "-lineinfo", "-std=c++17",
        "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
        "-I", INCLUDE, "-I", CSRC,
    ]
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]
    return flags


def _compile(src: str, verbose: bool, ptxas_verbose: bool) -> str:
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), "-c", os.path.join(CSRC, src), "-o", obj] + compile_flags(ptxas_verbose)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or ptxas_verbose or r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src} (exit {r.returncode})")
    return obj


def build(verbose: bool = False, ptxas_verbose: bool = False) -> str:
    """Compile every CUDA source and link ``_lib/librrs.so``; returns its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, ptxas_verbose), SOURCES))
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if verbose or r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
    if r.returncode != 0:
        raise RuntimeError(f"link of librrs.so failed (exit {r.returncode})")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, ptxas_verbose="--ptxas" in sys.argv))

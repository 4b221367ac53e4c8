"""The C ABI used from a plain C program (no Python, no PyTorch).

``tests/c/abi_example.c`` includes only ``rrs.h`` and the CUDA runtime, makes
device buffers with cudaMalloc, runs softmax_rows and row_sum on a stream and
checks the header's promised argument errors.  On the CPU the program is
compiled and linked against librrs.so (the header is valid C); on a GPU it
runs and its results are compared with the float64 oracle.
"""
from __future__ import annotations

import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from gpu_helpers import check_row_sum, check_softmax

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(tmp_path) -> str:
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    from row_reduction_softmax_gb300 import _build
    if not os.path.exists(_build.LIB_PATH):
        _build.build()
    exe = str(tmp_path / "abi_example")
    lib_dir = os.path.dirname(_build.LIB_PATH)
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-O1",
           os.path.join(ROOT, "tests", "c", "abi_example.c"), "-o", exe,
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", lib_dir, "-lrrs", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{lib_dir}", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return exe


def test_c_program_compiles_and_links(tmp_path):
    assert os.path.exists(_compile(tmp_path))


def _lcg_uniform(n: int) -> np.ndarray:
    """The program's generator: 64-bit LCG, top 24 bits, uniform in [-8, 8)."""
    out = np.empty(n, dtype=np.float32)
    state = 12345
    mask = (1 << 64) - 1
    for i in range(n):
        state = (state * 6364136223846793005 + 1442695040888963407) & mask
        out[i] = np.float32((state >> 40) / float(1 << 24) * 16.0 - 8.0)
    return out


@pytest.mark.gpu
@pytest.mark.parametrize("M,N", [(37, 1000), (6, 40000), (3, 300001)])
def test_c_program_results_match_the_oracle(tmp_path, M, N):
    exe = _compile(tmp_path)
    out = str(tmp_path / "out.bin")
    r = subprocess.run([exe, out, str(M), str(N)], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    data = np.fromfile(out, dtype=np.float32)
    x = data[:M * N].reshape(M, N)
    y = data[M * N:2 * M * N].reshape(M, N)
    s = data[2 * M * N:]
    if M * N <= 40000:                      # the generator, retraced in Python, on the small case
        assert np.array_equal(x.ravel(), _lcg_uniform(M * N))
    check_softmax(y, x, f"C program {M}x{N}")
    check_row_sum(s, x, f"C program {M}x{N}")
    assert np.allclose(oracle.softmax_rows(x).sum(axis=1), 1.0)

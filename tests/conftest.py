"""Shared test setup: the ``gpu`` marker and the library build.

Tests marked ``gpu`` need a CUDA device and call the kernels through the
C ABI; everything else runs on a CPU-only machine.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_addoption(parser):
    parser.addoption("--cuda-blocking", action="store_true",
                     help="debug mode: every launch synchronous (CUDA_LAUNCH_BLOCKING=1), so a "
                          "failing kernel is reported at its own launch")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the kernels through the C ABI)")
    if config.getoption("--cuda-blocking"):
        os.environ["CUDA_LAUNCH_BLOCKING"] = "1"   # before the first CUDA call of the session


def _cuda_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _cuda_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def lib():
    """The built C-ABI library (built here from source if it is missing)."""
    from row_reduction_softmax_gb300 import _build
    if not os.path.exists(_build.LIB_PATH):
        _build.build()
    import row_reduction_softmax_gb300 as rrs
    return rrs.load_library()

"""Shared pytest configuration: the ``gpu`` marker and common helpers."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a); run with -m gpu")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="session")
def libsdv():
    """libsdv.so built in-tree (nvcc cross-compiles without a GPU) and loaded."""
    from speculative_decode_verify_sdv_gb300 import build, sdv
    build.build()
    return sdv.load()

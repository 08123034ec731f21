"""Shared pytest setup.

Markers: ``gpu`` -- needs a CUDA device and the built ``libcr.so``.
Everything else runs on the CPU (oracle pins, host logic, the C-ABI symbol
table, gloo multi-process tests).
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: test needs a CUDA GPU and libcr.so")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


@pytest.fixture(autouse=True)
def _device_check_word(request):
    """Under the checked build (CR_LIBRARY pointing at it and
    CR_ASSERT_CHECK_WORD=1), every GPU test must leave the device error
    word at zero: no index check failed in any kernel it launched."""
    yield
    if os.environ.get("CR_ASSERT_CHECK_WORD") != "1" or "gpu" not in request.keywords:
        return
    from fsdp_emulated_ranks_gb300 import cr
    word = cr.cr_check_word(True)
    assert word != -1, "CR_ASSERT_CHECK_WORD is set but the loaded library has no device checks"
    assert word == 0, f"device index check failed: error word {word:#x}"

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

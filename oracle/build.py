"""Compile the C++ oracle into ``oracle/_build/liboracle.so`` with g++.

Test infrastructure only: the oracle is the CPU reference the tests, the
smoke check and the benchmark's CPU-baseline leg compare against; nothing in
the product library links it.  ``-ffp-contract=off`` keeps every fp32
operation individually rounded (no fused multiply-add), on x86-64 and on
aarch64 alike.  The sources keep to plain scalar loops, so they are also
valid C; every exported function has C linkage (``oracle.h``) for ctypes.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liboracle.so")
SOURCES = ["collectives.cpp", "adamw_fsdp.cpp", "buckets.cpp"]
CFLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math",
          "-fPIC", "-Wall", "-Wextra", "-Wno-unused-parameter"]


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = SOURCES + ["oracle.h", "build.py"]
    return any(os.path.getmtime(os.path.join(HERE, s)) > t for s in deps)


def build(force: bool = False) -> str:
    """Build the oracle library if missing or out of date; return its path."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    tmp = LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = (["g++"] + CFLAGS + ["-shared", "-o", tmp]
           + [os.path.join(HERE, s) for s in SOURCES] + ["-lm"])
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))

"""The kernels' chunk-index division (csrc/fastdiv.h) is exact: compiled
for the host and checked against plain division on edge, workload and
random divisors and dividends."""
import os
import subprocess
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_fastdiv_matches_division():
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "fastdiv_check")
        subprocess.run(["g++", "-O2", "-std=c++17", "-I",
                        os.path.join(ROOT, "fsdp_emulated_ranks_gb300", "csrc"),
                        os.path.join(ROOT, "tests", "fastdiv_check.cpp"), "-o", exe], check=True)
        res = subprocess.run([exe], capture_output=True, text=True)
        assert res.returncode == 0, res.stdout
        assert "mismatches=0" in res.stdout

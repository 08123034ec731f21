"""Error contract of the launching entry points, from a C++ caller.

tests/cuda_error_check.cu links libcr.so directly (no Python binding) and
makes CUDA refuse every kind of launch the library issues -- plain and
chained kernel launches, event records, copies, the reducer's and the
communicator's launches -- by enqueueing them on a stream whose capture has
been invalidated.  No GPU work is involved in the refusals.  Each call must
return CR_ERR_CUDA naming the CUDA error, leave every buffer unchanged, and
the calls that follow on a healthy stream must succeed with the right
results (a refused chained launch must not leave a stale error behind for
the next call).
"""
import os
import subprocess

import pytest
import torch

from fsdp_emulated_ranks_gb300 import build, cr

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module")
def error_check_bin(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    cr.lib()  # fails loudly if the library is missing
    libdir = os.path.dirname(os.path.abspath(cr.LIB_PATH))
    exe = str(tmp_path_factory.mktemp("cuda_error") / "cuda_error_check")
    subprocess.run([build.nvcc()] + build.ARCH +
                   ["-O2", "-std=c++17", "-I", build.INCLUDE,
                    os.path.join(HERE, "cuda_error_check.cu"), "-o", exe,
                    os.path.abspath(cr.LIB_PATH), "-Xlinker", "-rpath", "-Xlinker", libdir],
                   check=True, capture_output=True, text=True, timeout=300)
    return exe


def test_refused_launches_report_cuda_error_and_leave_the_library_usable(error_check_bin):
    res = subprocess.run([error_check_bin], capture_output=True, text=True, timeout=300)
    out = res.stdout + res.stderr
    assert res.returncode == 0, out[-4000:]
    assert "ALL OK" in out, out[-4000:]
    refused = [l for l in out.splitlines() if l.startswith("refused")]
    # 24 launching entry points (the range forms, the FSDP2 table upload and
    # the planned step included), the reducer on two streams, two
    # communicator ranks
    assert len(refused) == 28, out
    assert "buffers changed by refused calls: 0" in out

"""The GPU suites once more against the checked build of the library, whose
kernels verify on the device the index arithmetic behind every access (the
chunk of an element, its offset inside a shard, the tile of a tensor, the
multiply-shift division against plain division).  A failed check sets a
bit of a device error word and skips the access -- it does not trap -- and
the shared fixture in conftest.py asserts the word is zero after each GPU
test.  This is the stand-in for compute-sanitizer, which this pool closes."""
import os
import subprocess
import sys

import pytest
import torch

from fsdp_emulated_ranks_gb300 import build as libbuild

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SUITES = ["tests/test_parity_gpu.py", "tests/test_parity_wire_hsdp_gpu.py",
          "tests/test_fuzz_gpu.py", "tests/test_pdl_gpu.py", "tests/test_reducer_gpu.py",
          "tests/test_graph_gpu.py", "tests/test_comm_gpu.py", "tests/test_cuda_error_gpu.py",
          "tests/test_fullsize_gpu.py", "tests/test_fullsize_more_gpu.py",
          "tests/test_threads_gpu.py", "tests/test_zero_stages_gpu.py", "tests/test_range_gpu.py"]


@pytest.fixture(scope="module")
def checked_lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    return libbuild.build(checked=True)


def _env(lib):
    env = dict(os.environ)
    env.update(CR_LIBRARY=lib, CR_ASSERT_CHECK_WORD="1")
    return env


def test_error_word_reports_a_failed_check(checked_lib):
    """The channel works: the self-test kernel fails a check on purpose
    (no memory access), the host reads that bit, clearing resets it."""
    code = ("import torch; from fsdp_emulated_ranks_gb300 import cr; cr.lib();"
            "assert cr.cr_check_word(True) == 0;"
            "cr.cr_check_selftest(); torch.cuda.synchronize();"
            "w = cr.cr_check_word(True); assert w == 1 << 31, hex(w);"
            "assert cr.cr_check_word(False) == 0; print('ok')")
    res = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=_env(checked_lib),
                         capture_output=True, text=True, timeout=600)
    assert res.returncode == 0 and "ok" in res.stdout, res.stdout + res.stderr


def test_gpu_suites_pass_with_device_checks(checked_lib):
    # the suites include the full-size cases: leave them this process's cached memory
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    res = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu",
                          "-p", "no:cacheprovider"] + SUITES,
                         cwd=ROOT, env=_env(checked_lib), capture_output=True, text=True,
                         timeout=3000)
    tail = "\n".join(res.stdout.splitlines()[-15:])
    assert res.returncode == 0, tail + res.stderr[-2000:]
    assert " passed" in tail

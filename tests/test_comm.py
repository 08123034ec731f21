"""Failure detection of the thread-per-rank communicator, on the host only.

Each emulated rank is a Python thread calling cr_comm_* (ctypes releases
the GIL while a call blocks).  The failures are those real ranks meet: a
rank that never joins (every waiting rank must return CR_ERR_TIMEOUT within
the timeout, and the communicator stays broken), calls that disagree
(CR_ERR_INVALID_ARG on every rank), a rank id used twice.  None of these
cases reaches a launch -- the pointers are never dereferenced -- so no GPU
is involved, and none would be on a machine that has one."""
import threading
import time

import pytest

from fsdp_emulated_ranks_gb300 import build as libbuild
from fsdp_emulated_ranks_gb300 import cr

FAKE = 1 << 40
TIMEOUT, INVALID = 5, 1


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()
    cr.lib()


def run_ranks(calls):
    """calls: {rank_thread_id: callable}.  Returns {id: (status, seconds)}."""
    out = {}

    def body(k, fn):
        t0 = time.monotonic()
        try:
            fn()
            out[k] = (0, time.monotonic() - t0)
        except cr.CRError as e:
            out[k] = (e.status, time.monotonic() - t0)

    threads = [threading.Thread(target=body, args=(k, fn)) for k, fn in calls.items()]
    for t in threads:
        t.start()
    for t in threads:
        t.join(30)
        assert not t.is_alive(), "a rank thread is still blocked"
    return out


def test_missing_rank_times_out_every_waiting_rank():
    comm = cr.cr_comm_create(4, 300, 0)
    res = run_ranks({r: (lambda r=r: cr.cr_comm_all_reduce(comm, r, FAKE + r * 4096, 100,
                                                           "f32", "sum"))
                     for r in range(3)})   # rank 3 never joins
    for r in range(3):
        status, secs = res[r]
        assert status == TIMEOUT, res
        assert 0.25 <= secs < 5.0, res
    assert cr.cr_comm_broken(comm) == 1
    # a broken communicator refuses every later call at once
    t0 = time.monotonic()
    with pytest.raises(cr.CRError) as e:
        cr.cr_comm_all_reduce(comm, 3, FAKE, 100, "f32", "sum")
    assert e.value.status == TIMEOUT and time.monotonic() - t0 < 0.1
    assert "broken" in str(e.value)
    cr.cr_comm_destroy(comm)


def test_mismatched_calls_fail_on_every_rank_and_launch_nothing():
    comm = cr.cr_comm_create(3, 5000, 0)
    counts = [100, 100, 101]
    res = run_ranks({r: (lambda r=r: cr.cr_comm_all_reduce(comm, r, FAKE + r * 4096, counts[r],
                                                           "bf16", "avg"))
                     for r in range(3)})
    assert all(res[r][0] == INVALID for r in range(3)), res
    assert cr.cr_comm_broken(comm) == 0
    # the next collective can be joined: a different collective on one rank
    calls = {0: lambda: cr.cr_comm_all_gather(comm, 0, FAKE, FAKE + 8192, 64, "f32")}
    for r in (1, 2):
        calls[r] = (lambda r=r: cr.cr_comm_all_reduce(comm, r, FAKE + r * 4096, 64, "f32", "sum"))
    res = run_ranks(calls)
    assert all(res[r][0] == INVALID for r in range(3)), res
    # dtype disagreement in a reduce-scatter
    dts = ["f32", "f32", "bf16"]
    res = run_ranks({r: (lambda r=r: cr.cr_comm_reduce_scatter(
        comm, r, FAKE + r * 4096, FAKE + (1 << 30) + r * 4096, 96, dts[r], "sum", dts[r]))
        for r in range(3)})
    assert all(res[r][0] == INVALID for r in range(3)), res
    assert cr.cr_comm_broken(comm) == 0
    cr.cr_comm_destroy(comm)


def test_rank_joining_twice_is_rejected():
    comm = cr.cr_comm_create(2, 300, 0)
    res = run_ranks({k: (lambda: cr.cr_comm_all_reduce(comm, 0, FAKE, 16, "f32", "sum"))
                     for k in range(2)})
    assert sorted(s for s, _ in res.values()) == [INVALID, TIMEOUT], res
    cr.cr_comm_destroy(comm)


def test_argument_errors():
    for n, t in ((0, 100), (65, 100), (2, 0)):
        with pytest.raises(cr.CRError) as e:
            cr.cr_comm_create(n, t, 0)
        assert e.value.status == INVALID
    comm = cr.cr_comm_create(2, 100, 0)
    for rank in (-1, 2):
        with pytest.raises(cr.CRError) as e:
            cr.cr_comm_all_reduce(comm, rank, FAKE, 16, "f32", "sum")
        assert e.value.status == INVALID
    assert cr.cr_comm_broken(comm) == 0
    cr.cr_comm_destroy(comm)
    assert cr.lib().cr_comm_broken(None) == -1

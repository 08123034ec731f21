"""The thread-per-rank communicator on the GPU: each of N host threads is a
rank that calls the collectives on its own tensors, in the same order, for
several rounds; results must equal the oracle's ring collectives exactly
as the single-call entry points do (bitwise, every dtype)."""
import threading

import numpy as np
import pytest
import torch

import oracle as O
from fsdp_emulated_ranks_gb300 import build as libbuild
from fsdp_emulated_ranks_gb300 import cr
from fsdp_emulated_ranks_gb300 import inputs as I
from gpu_util import assert_match, to_dev, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    libbuild.build()
    cr.lib()


def per_rank(n, fn):
    errors = []

    def body(r):
        try:
            fn(r)
        except Exception as e:  # surfaced in the main thread
            errors.append((r, e))

    ts = [threading.Thread(target=body, args=(r,)) for r in range(n)]
    for t in ts:
        t.start()
    for t in ts:
        t.join(60)
    assert not errors, errors


@pytest.mark.parametrize("n", [2, 5, 8])
def test_threads_as_ranks(n):
    count = 16 * n * 100 + 7
    stream = torch.cuda.Stream()
    comm = cr.cr_comm_create(n, 20000, stream)
    L = cr.cr_chunk_len(count, n)
    for rnd in range(3):
        host = I.host_rank_buffers(n, count, "bf16", std=0.02, seed0=100 * rnd + n)
        bufs = [to_dev(x, "bf16") for x in host]
        shards = [torch.empty(max(0, min(count, (j + 1) * L) - min(count, j * L)),
                              dtype=torch.float32, device="cuda") for j in range(n)]
        gathered = [torch.empty(count, dtype=torch.float32, device="cuda") for _ in range(n)]
        torch.cuda.synchronize()

        def rank(r):
            # every rank: reduce-scatter to fp32, all-gather the shards,
            # then an in-place all-reduce of its bf16 buffer
            cr.cr_comm_reduce_scatter(comm, r, bufs[r], shards[r], count, "bf16", "avg", "f32")
            cr.cr_comm_all_gather(comm, r, shards[r], gathered[r], count, "f32")
            cr.cr_comm_all_reduce(comm, r, bufs[r], count, "bf16", "avg")

        per_rank(n, rank)
        stream.synchronize()
        want_rs, _ = O.ring_reduce_scatter(host, "bf16", "avg", "f32")
        want_ar, _ = O.ring_all_reduce(host, "bf16", "avg")
        full = np.concatenate(want_rs)
        for r in range(n):
            assert_match(to_host(shards[r], "f32"), want_rs[r], "f32", f"round {rnd} shard {r}")
            assert_match(to_host(gathered[r], "f32"), full, "f32", f"round {rnd} gather {r}")
            assert_match(to_host(bufs[r], "bf16"), want_ar[r], "bf16", f"round {rnd} rank {r}")
    assert cr.cr_comm_broken(comm) == 0
    cr.cr_comm_destroy(comm)


def test_launch_error_reaches_every_rank():
    """An argument error found at launch (a misaligned buffer on one rank)
    is returned to every rank, and the communicator stays usable."""
    n, count = 3, 1000
    comm = cr.cr_comm_create(n, 20000, torch.cuda.current_stream())
    base = [torch.zeros(count + 1, dtype=torch.float32, device="cuda") for _ in range(n)]
    ptrs = [b.data_ptr() for b in base]
    ptrs[1] += 2   # not 4-byte aligned: rejected before any launch
    status = {}

    def rank(r):
        try:
            cr.cr_comm_all_reduce(comm, r, ptrs[r], count, "f32", "sum")
            status[r] = 0
        except cr.CRError as e:
            status[r] = e.status

    per_rank(n, rank)
    assert status == {0: 3, 1: 3, 2: 3}
    assert cr.cr_comm_broken(comm) == 0
    cr.cr_comm_destroy(comm)

"""The slab split of one workload across GPUs, on the CPU.

cr_slab_range (a host function of libcr) must partition [0, count) for any
slab count, into whole chunks while there are no more slabs than ranks.
Under a world-size-2 gloo run, each rank takes its slab as bench.py's
--split slab does and reduces it with the oracle's per-element ring fold;
the slabs put side by side must be the oracle's whole-buffer all-reduce,
bit for bit: the split needs no exchange and changes no fold order.
"""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from fsdp_emulated_ranks_gb300 import build as libbuild
from fsdp_emulated_ranks_gb300 import cr


@pytest.fixture(scope="module")
def L():
    libbuild.build()
    return cr.lib()


@pytest.mark.parametrize("n", [1, 2, 3, 4, 8, 13, 64])
@pytest.mark.parametrize("count", [0, 1, 7, 8 * 1000, 8 * 1000 + 5, 12345, 1 << 25])
def test_slabs_partition_the_range(L, n, count):
    Lc = cr.cr_chunk_len(count, n)
    for G in (1, 2, 3, 4, 5, 8, 16, 64, 70):
        b = [cr.cr_slab_range(count, n, G, g) for g in range(G)]
        assert b[0][0] == 0 and b[-1][1] == count
        for (lo, hi), (lo2, _) in zip(b, b[1:]):
            assert lo <= hi == lo2
        for lo, hi in b:
            if lo == count:
                continue
            if G <= n:
                assert lo % Lc == 0   # whole chunks
            else:
                assert lo % 16 == 0


def test_slab_range_rejects_bad_arguments(L):
    for args in ((100, 0, 2, 0), (100, 8, 0, 0), (100, 8, 2, 2), (100, 8, 2, -1)):
        with pytest.raises(cr.CRError) as ei:
            cr.cr_slab_range(*args)
        assert ei.value.status == 1


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out, n, count):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import bench
    import oracle as O
    import torch.distributed as dist
    from fsdp_emulated_ranks_gb300 import inputs as I
    bench.init_dist(world, "gloo")
    lo, hi = bench.slab_bounds(count, n, world, rank)
    host = I.host_rank_buffers(n, count, "bf16", std=0.02, seed0=0)
    idx = np.arange(lo, hi)
    Lc = O.chunk_len(count, n)
    vals = np.stack([b[idx] for b in host], axis=1) if hi > lo else np.zeros((0, n), np.uint16)
    mine = O.fold_columns(vals, (idx // Lc).astype(np.int32), "bf16", "avg", "bf16")
    got = [None] * world
    dist.all_gather_object(got, (lo, hi, mine.tobytes()))
    if rank == 0:
        want, _ = O.ring_all_reduce(host, "bf16", "avg")
        out["bounds"] = [(a, b) for a, b, _ in got]
        out["equal"] = b"".join(x for _, _, x in got) == want[0].tobytes()
    dist.destroy_process_group()


@pytest.mark.parametrize("n,count", [(8, 8 * 1000 + 5), (3, 1001)])
def test_two_ranks_split_one_all_reduce(n, count):
    world = 2
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, _free_port(), out, n, count), nprocs=world, join=True)
    (a0, b0), (a1, b1) = out["bounds"]
    assert a0 == 0 and b0 == a1 and b1 == count
    assert out["equal"]

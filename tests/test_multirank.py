"""World-size-2 gloo run of the benchmark's multi-rank host logic on CPU:
barrier, max-over-ranks timing and whole-job throughput.  Each GPU runs its
own independent instance of the workload, so these are the only places the
ranks interact."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist
    bench.init_dist(world, "gloo")
    assert bench.dist_env() == (world, rank, rank)
    bench.barrier(world)
    # rank r took (r + 1) * 10 ms for 5 steps of 1 GB each
    total_ms = (rank + 1) * 10.0
    gbs, ms = bench.job_throughput(1e9, total_ms, 5, world, device="cpu")
    out[rank] = (gbs, ms, bench.max_over_ranks(float(rank), world, "cpu"))
    dist.destroy_process_group()


def test_two_rank_timing_uses_slowest_rank():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    slowest_ms = world * 10.0 / 5
    for rank in range(world):
        gbs, ms, mx = out[rank]
        assert ms == pytest.approx(slowest_ms)
        assert gbs == pytest.approx(world * 1e9 / (slowest_ms * 1e-3) / 1e9)
        assert mx == world - 1


def _worker_one_dies(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import time
    import bench
    bench.init_dist(world, "gloo", timeout_s=5)
    if rank == 1:
        os._exit(0)          # the rank dies between steps, without a word
    t0 = time.monotonic()
    try:
        bench.barrier(world)
        out[rank] = ("no error", time.monotonic() - t0)
    except Exception as e:   # the survivor learns of it from the process group
        out[rank] = (type(e).__name__, time.monotonic() - t0)


def test_dead_rank_fails_the_barrier_instead_of_hanging():
    """A rank that exits between steps: the other rank's next barrier fails
    with an error within the process-group timeout (5 s here), so an N > 1
    benchmark run ends instead of waiting forever."""
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.spawn(_worker_one_dies, args=(world, port, out), nprocs=world, join=True)
    kind, secs = out[0]
    assert kind != "no error"
    assert secs < 20.0

"""GPU tests of the DDP reducer through the C ABI: gradients written on a
compute stream and marked ready one by one (in backward order and in random
orders), bucket all-reduces run on a separate communication stream with and
without a CTA cap.  After finalize every tensor must hold, bit for bit,
what cr_bucket_all_reduce_fused gives on the same inputs, and the oracle's
bucketed all-reduce (bitwise)."""
import numpy as np
import pytest
import torch

import oracle as O
from fsdp_emulated_ranks_gb300 import build as libbuild
from fsdp_emulated_ranks_gb300 import cr
from fsdp_emulated_ranks_gb300 import inputs as I
from gpu_util import assert_match, to_dev, to_host

pytestmark = pytest.mark.gpu

TORCH = {"bf16": torch.bfloat16, "f32": torch.float32}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    libbuild.build()
    cr.lib()


def case(n, dt, seed, T=40):
    rng = np.random.default_rng(seed)
    numels = [int(x) for x in rng.integers(1, 60000, T)]
    numels[3] = 0  # an empty tensor is still marked
    es = 2 if dt == "bf16" else 4
    plan = cr.cr_bucket_plan(numels, es, 256 * 1024)
    host = [[I.host_rank_buffers(1, k, dt, std=0.02 if dt == "bf16" else 1.0,
                                 seed0=seed * 1000 + r * T + t)[0]
             for t, k in enumerate(numels)] for r in range(n)]
    return plan, numels, host


def dev_tensors(host, dt):
    return [to_dev(x, dt) if x.size else torch.empty(0, dtype=TORCH[dt], device="cuda")
            for row in host for x in row]


def run_reducer(plan, n, host, dt, op, order, comm_ctas, iterations=1):
    """Backward emulation: zeroed gradients, each written on the compute
    stream just before it is marked ready."""
    T = plan.ntensors
    src = dev_tensors(host, dt)
    grads = [torch.zeros_like(x) for x in src]
    compute, comm = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    red = cr.cr_reducer_create(plan, n, grads, dt, op, comm_ctas, comm)
    launched = []
    for it in range(iterations):
        with torch.cuda.stream(compute):
            for g in grads:
                g.zero_()
            for t in order:
                for r in range(n):
                    grads[r * T + t].copy_(src[r * T + t])
                cr.cr_reducer_mark_ready(red, t, compute)
                launched.append(cr.cr_reducer_launched(red))
            assert cr.cr_reducer_launched(red) == plan.nbuckets
            cr.cr_reducer_finalize(red, compute)
            assert cr.cr_reducer_launched(red) == 0
    torch.cuda.synchronize()
    cr.cr_reducer_destroy(red)
    return grads, launched


@pytest.mark.parametrize("n", [2, 5, 8])
@pytest.mark.parametrize("dt,op", [("bf16", "avg"), ("f32", "sum")])
@pytest.mark.parametrize("order", ["backward", "random"])
@pytest.mark.parametrize("comm_ctas", [0, 1, 19])
def test_reducer_matches_fused_all_reduce(n, dt, op, order, comm_ctas):
    plan, numels, host = case(n, dt, seed=n * 7 + len(dt))
    T = plan.ntensors
    rng = np.random.default_rng(n)
    idx = list(range(T - 1, -1, -1)) if order == "backward" else [int(x) for x in rng.permutation(T)]
    got, launched = run_reducer(plan, n, host, dt, op, idx, comm_ctas)
    ref = dev_tensors(host, dt)
    cr.cr_bucket_all_reduce_fused(plan, n, ref, dt, op)
    torch.cuda.synchronize()
    for k in range(n * T):
        assert torch.equal(got[k].view(torch.int16 if dt == "bf16" else torch.int32),
                           ref[k].view(torch.int16 if dt == "bf16" else torch.int32)), k
    # launches never go backwards and end with every bucket
    assert launched == sorted(launched) and launched[-1] == plan.nbuckets
    if order == "backward":
        oplan = O.bucket_plan(numels, 2 if dt == "bf16" else 4, 256 * 1024)
        want = O.bucketed_all_reduce(oplan, host, dt, op)
        for r in range(n):
            for t in range(T):
                assert_match(to_host(got[r * T + t], dt), want[r][t], dt, f"rank {r} tensor {t}")


def test_reducer_two_iterations():
    n, dt = 4, "bf16"
    plan, numels, host = case(n, dt, seed=99)
    T = plan.ntensors
    got, _ = run_reducer(plan, n, host, dt, "avg", list(range(T - 1, -1, -1)), 8, iterations=2)
    ref = dev_tensors(host, dt)
    cr.cr_bucket_all_reduce_fused(plan, n, ref, dt, "avg")
    torch.cuda.synchronize()
    for k in range(n * T):
        assert torch.equal(got[k].view(torch.int16), ref[k].view(torch.int16)), k


def test_reducer_errors_leave_state():
    n, dt = 2, "f32"
    plan, numels, host = case(n, dt, seed=5, T=12)
    T = plan.ntensors
    grads = dev_tensors(host, dt)
    red = cr.cr_reducer_create(plan, n, grads, dt, "sum", 0, None)
    with pytest.raises(cr.CRError) as e:
        cr.cr_reducer_finalize(red)
    assert e.value.status == 1
    cr.cr_reducer_mark_ready(red, T - 1)
    with pytest.raises(cr.CRError) as e:
        cr.cr_reducer_mark_ready(red, T - 1)
    assert e.value.status == 1
    with pytest.raises(cr.CRError) as e:
        cr.cr_reducer_mark_ready(red, T)
    assert e.value.status == 1
    for t in range(T - 2, -1, -1):
        cr.cr_reducer_mark_ready(red, t)
    cr.cr_reducer_finalize(red)
    torch.cuda.synchronize()
    ref = dev_tensors(host, dt)
    cr.cr_bucket_all_reduce_fused(plan, n, ref, dt, "sum")
    torch.cuda.synchronize()
    for k in range(n * T):
        assert torch.equal(grads[k], ref[k]), k
    cr.cr_reducer_destroy(red)

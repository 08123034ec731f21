"""GPU parity for the low-precision wire and the HSDP two-level reduction,
through the C ABI, against the oracle's literal ring simulations on the same
seeded inputs.

The bf16 wire rounds each forwarded partial exactly where the oracle's ring
rounds its message, and HSDP folds the S ranks of a group and then the R
groups in the two rings' orders, so every result is bitwise equal to the
oracle's (the bar of the other collectives).  Sizes
span several vectors and CTAs plus ragged tails; offsets 1 and "16B" force
the element-wise and 16-byte kernels.
"""
import numpy as np
import pytest
import torch

import oracle as O
from fsdp_emulated_ranks_gb300 import build as libbuild
from fsdp_emulated_ranks_gb300 import cr
from fsdp_emulated_ranks_gb300 import inputs as I
from gpu_util import Guarded, assert_match, to_dev, to_host

pytestmark = pytest.mark.gpu

FLOAT_PAIRS = [("f32", "sum", "f32"), ("bf16", "avg", "bf16"), ("bf16", "avg", "f32"),
               ("f32", "avg", "f32"), ("bf16", "sum", "bf16")]
PAIRS = FLOAT_PAIRS + [("i32", "sum", "i32")]
ESIZE = {"f32": 4, "bf16": 2, "i32": 4}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    libbuild.build()
    cr.lib()


def eoff(offset, dt):
    return 16 // ESIZE[dt] if offset == "16B" else offset


def host_inputs(n, count, dt, seed):
    return I.host_rank_buffers(n, count, dt, std=0.02 if dt == "bf16" else 1.0, seed0=seed)


def sizes(n):
    return [0, 1, 7, 8 * n * 3, 8 * n * 37 + 5, 1000, 4099]


# ---- bf16 wire -------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 7, 8, 13, 64])
@pytest.mark.parametrize("pair", FLOAT_PAIRS)
@pytest.mark.parametrize("offset", [0, 1, "16B"])
@pytest.mark.parametrize("wire", ["bf16", "f32"])
def test_reduce_scatter_wire(n, pair, offset, wire):
    dt, op, out = pair
    for count in sizes(n):
        host = host_inputs(n, count, dt, seed=n * 500 + count)
        want = O.ring_reduce_scatter_wire(host, dt, op, wire, out)
        bufs = [to_dev(x, dt, eoff(offset, dt)) for x in host]
        shards = [Guarded(w.size, out, eoff(offset, out)) for w in want]
        cr.cr_reduce_scatter_wire(bufs, count, dt, op, wire, [s.ptr() for s in shards], out)
        torch.cuda.synchronize()
        for j in range(n):
            shards[j].check()
            assert_match(shards[j].host(), want[j], out, f"n={n} count={count} shard {j}")


@pytest.mark.parametrize("n", [1, 2, 3, 4, 8, 13, 64])
@pytest.mark.parametrize("pair", FLOAT_PAIRS)
@pytest.mark.parametrize("offset", [0, 1, "16B"])
def test_all_reduce_wire(n, pair, offset):
    dt, op, out = pair
    for count in sizes(n):
        host = host_inputs(n, count, dt, seed=n * 700 + count)
        want = O.ring_all_reduce_wire(host, dt, op, "bf16", out)
        bufs = [to_dev(x, dt, eoff(offset, dt)) for x in host]
        outs = [Guarded(count, out, eoff(offset, out)) for _ in range(n)]
        cr.cr_all_reduce_wire(bufs, count, dt, op, "bf16", [o.ptr() for o in outs], out)
        torch.cuda.synchronize()
        for r in range(n):
            outs[r].check()
            assert_match(outs[r].host(), want[r], out, f"n={n} count={count} rank {r}")


@pytest.mark.parametrize("n", [4, 8])
def test_bf16_wire_differs_from_f32_wire(n):
    """The wire rounding is really applied: with fp32 inputs the bf16-wire
    result differs from the ordinary all-reduce, on the GPU as in the
    oracle, and the GPU matches the oracle bit for bit."""
    count = 8 * n * 64
    host = host_inputs(n, count, "f32", seed=11)
    bufs = [to_dev(x, "f32") for x in host]
    plain = [torch.empty(count, dtype=torch.float32, device="cuda") for _ in range(n)]
    wired = [torch.empty(count, dtype=torch.float32, device="cuda") for _ in range(n)]
    cr.cr_all_reduce(bufs, count, "f32", "sum", plain, "f32")
    cr.cr_all_reduce_wire(bufs, count, "f32", "sum", "bf16", wired, "f32")
    torch.cuda.synchronize()
    p, w = to_host(plain[0], "f32"), to_host(wired[0], "f32")
    assert np.mean(p != w) > 0.5
    want = O.ring_all_reduce_wire(host, "f32", "sum", "bf16", "f32")
    assert w.tobytes() == want[0].tobytes()


@pytest.mark.parametrize("n", [2, 4, 8, 5])
def test_all_reduce_wire_in_place(n):
    count = 8 * n * 50 + 3
    host = host_inputs(n, count, "bf16", seed=3)
    want = O.ring_all_reduce_wire(host, "bf16", "avg", "bf16", "bf16")
    bufs = [to_dev(x, "bf16") for x in host]
    cr.cr_all_reduce_wire(bufs, count, "bf16", "avg", "bf16", bufs, "bf16")
    torch.cuda.synchronize()
    for r in range(n):
        assert_match(to_host(bufs[r], "bf16"), want[r], "bf16", f"rank {r}")


# ---- HSDP ------------------------------------------------------------------------

MESHES = [(1, 1), (1, 4), (4, 1), (2, 2), (2, 4), (4, 2), (2, 3), (3, 5), (8, 8)]


@pytest.mark.parametrize("R,S", MESHES)
@pytest.mark.parametrize("pair", PAIRS)
@pytest.mark.parametrize("offset", [0, 1, "16B"])
def test_hsdp_reduce_scatter(R, S, pair, offset):
    dt, op, out = pair
    n = R * S
    for count in sizes(n) + [8 * S * R * 5 + 8 * S]:
        host = host_inputs(n, count, dt, seed=n * 900 + count)
        want = O.hsdp_reduce_scatter(host, R, S, dt, op, out)
        bufs = [to_dev(x, dt, eoff(offset, dt)) for x in host]
        shards = [Guarded(w.size, out, eoff(offset, out)) for w in want]
        cr.cr_hsdp_reduce_scatter(bufs, R, S, count, dt, op, [s.ptr() for s in shards], out)
        torch.cuda.synchronize()
        for q in range(n):
            shards[q].check()
            assert_match(shards[q].host(), want[q], out,
                         f"{R}x{S} count={count} group {q // S} shard {q % S}")
        for r in range(n):
            assert to_host(bufs[r], dt).tobytes() == host[r].tobytes()


@pytest.mark.parametrize("R,S", [(2, 4), (4, 2), (3, 2)])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_hsdp_in_place(R, S, dt):
    n = R * S
    count = 8 * S * 40 + 5
    host = host_inputs(n, count, dt, seed=21)
    want = O.hsdp_reduce_scatter(host, R, S, dt, "avg", dt)
    bufs = [to_dev(x, dt) for x in host]
    L = cr.cr_chunk_len(count, S)
    shards = [bufs[g * S + j][j * L:(j + 1) * L] for g in range(R) for j in range(S)]
    cr.cr_hsdp_reduce_scatter(bufs, R, S, count, dt, "avg", shards, dt)
    torch.cuda.synchronize()
    for q in range(n):
        assert_match(to_host(shards[q], dt), want[q], dt, f"group {q // S} shard {q % S}")


@pytest.mark.parametrize("R,S", [(1, 4), (4, 1)])
def test_hsdp_degenerate_meshes(R, S):
    """R = 1 is the reduce-scatter over S ranks; S = 1 the all-reduce over R
    ranks: the GPU result equals the one-level collectives bit for bit."""
    n = R * S
    count = 8 * n * 33 + 7
    host = host_inputs(n, count, "bf16", seed=5)
    bufs = [to_dev(x, "bf16") for x in host]
    L = cr.cr_chunk_len(count, S)
    lens = [min(count, (j + 1) * L) - min(count, j * L) for j in range(S)]
    hs = [torch.empty(lens[q % S], dtype=torch.float32, device="cuda") for q in range(n)]
    cr.cr_hsdp_reduce_scatter(bufs, R, S, count, "bf16", "avg", hs, "f32")
    if R == 1:
        ref = [torch.empty(lens[j], dtype=torch.float32, device="cuda") for j in range(S)]
        cr.cr_reduce_scatter(bufs, count, "bf16", "avg", ref, "f32")
    else:
        ref = [torch.empty(count, dtype=torch.float32, device="cuda") for _ in range(R)]
        cr.cr_all_reduce(bufs, count, "bf16", "avg", ref, "f32")
    torch.cuda.synchronize()
    for q in range(n):
        assert torch.equal(hs[q], ref[q])

"""Calls that need several launches (fused bucket all-reduce, bucket pack,
FSDP2 step) chain them with programmatic dependent launch.  The chain must
still look like one stream-ordered operation to the caller: work the caller
enqueues next on the same stream sees every launch's results, the first
launch's included; and a captured CUDA graph of a chained call replays
the same results."""
import numpy as np
import pytest
import torch

from fsdp_emulated_ranks_gb300 import build as libbuild
from fsdp_emulated_ranks_gb300 import cr
from fsdp_emulated_ranks_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    libbuild.build()
    cr.lib()


def tensors(n, numels, seed):
    out = []
    for r in range(n):
        for t, k in enumerate(numels):
            x = torch.empty(k, dtype=torch.bfloat16, device="cuda")
            I.torch_fill_normal_(x, 0.02, seed + 1000 * r + t)
            out.append(x)
    return out


def big_case(seed, T=300):
    rng = np.random.default_rng(seed)
    # large first tensors: the first launch runs long, so a broken chain
    # would let the caller's next kernel read its tensors too early
    numels = [int(x) for x in rng.integers(1 << 10, 1 << 20, T)]
    numels[:20] = [1 << 22] * 20
    return numels


def test_fused_chain_is_stream_ordered():
    n = 8
    numels = big_case(1)
    plan = cr.cr_bucket_plan(numels, 2, 25 << 20)
    t = tensors(n, numels, 0)
    ref = [x.clone() for x in t]
    cr.cr_bucket_all_reduce_fused(plan, n, ref, "bf16", "avg")
    torch.cuda.synchronize()
    cr.cr_bucket_all_reduce_fused(plan, n, t, "bf16", "avg")
    snap = [x.clone() for x in t]          # same stream, right behind the chain
    torch.cuda.synchronize()
    for k in range(len(t)):
        assert torch.equal(snap[k].view(torch.int16), ref[k].view(torch.int16)), k


def test_pack_chain_is_stream_ordered():
    n = 8
    numels = big_case(2)
    plan = cr.cr_bucket_plan(numels, 2, 25 << 20)
    t = tensors(n, numels, 10)
    B = plan.nbuckets
    buckets = [torch.empty(int(plan.bucket_numel[b]), dtype=torch.bfloat16, device="cuda")
               for _ in range(n) for b in range(B)]
    torch.cuda.synchronize()
    cr.cr_bucket_pack(plan, n, t, buckets)
    snap = [x.clone() for x in buckets]
    torch.cuda.synchronize()
    T = plan.ntensors
    for r in range(n):
        for k in range(T):
            b, off = plan.tensor_bucket[k], plan.tensor_offset[k]
            got = snap[r * B + b][off:off + numels[k]]
            assert torch.equal(got.view(torch.int16), t[r * T + k].view(torch.int16)), (r, k)


def test_fsdp2_chain_is_stream_ordered():
    n = 8
    shapes = [(4096, 1024)] * 10 + [(257, 33)] * 150   # more than one launch of 64
    cfg = cr.adamw_cfg()

    def state(seed):
        g, m_, mm, v, p = [], [], [], [], []
        for i, (d0, row) in enumerate(shapes):
            for r in range(n):
                x = torch.empty(d0 * row, dtype=torch.bfloat16, device="cuda")
                I.torch_fill_normal_(x, 1e-3, seed + 100 * i + r)
                g.append(x)
                p.append(torch.empty(d0 * row, dtype=torch.bfloat16, device="cuda"))
            Lr = -(-d0 // n)
            for j in range(n):
                k = max(0, min(d0, (j + 1) * Lr) - min(d0, j * Lr)) * row
                x = torch.empty(k, dtype=torch.float32, device="cuda")
                I.torch_fill_normal_(x, 0.02, seed + 7 * i + j + 5000)
                m_.append(x if k else 0)
                mm.append(torch.zeros(k, dtype=torch.float32, device="cuda") if k else 0)
                v.append(torch.zeros(k, dtype=torch.float32, device="cuda") if k else 0)
        return g, m_, mm, v, p

    a, b = state(3), state(3)
    cr.cr_fsdp2_step(shapes, n, a[0], a[1], a[2], a[3], cfg, a[4])
    torch.cuda.synchronize()
    cr.cr_fsdp2_step(shapes, n, b[0], b[1], b[2], b[3], cfg, b[4])
    snap = [x.clone() for x in b[4]]
    torch.cuda.synchronize()
    for k in range(len(snap)):
        assert torch.equal(snap[k].view(torch.int16), a[4][k].view(torch.int16)), k


def test_chained_call_replays_from_a_graph():
    n = 8
    numels = big_case(4)
    plan = cr.cr_bucket_plan(numels, 2, 25 << 20)
    src = tensors(n, numels, 20)
    ref = [x.clone() for x in src]
    cr.cr_bucket_all_reduce_fused(plan, n, ref, "bf16", "avg")
    work = [torch.empty_like(x) for x in src]
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        cr.cr_bucket_all_reduce_fused(plan, n, work, "bf16", "avg")
    for w, x in zip(work, src):
        w.copy_(x)
    g.replay()
    torch.cuda.synchronize()
    for k in range(len(work)):
        assert torch.equal(work[k].view(torch.int16), ref[k].view(torch.int16)), k


@pytest.mark.parametrize("n", [3, 8])
def test_back_to_back_dependent_calls_overlap_safely(n):
    """Single-launch kernels are dispatched during the previous kernel's last
    wave and wait for it before their first access.  A long chain of calls
    that each read what the one before wrote -- in-place all-reduce, then
    reduce-scatter into shards that are rank j's own chunk, then all-gather
    back in place, 30 times over -- must give exactly what the arithmetic
    says: int32 SUM multiplies every element by n per all-reduce (the
    reduce-scatter + all-gather pair is one more), with wrap modulo 2^32."""
    count = 8 * n * 50000 + 8 * n
    rng = np.random.default_rng(n)
    x = rng.integers(-1000, 1000, size=count, dtype=np.int32)
    bufs = [torch.from_numpy(x.copy()).cuda() for _ in range(n)]
    L = cr.cr_chunk_len(count, n)
    shards = [bufs[j][j * L:min((j + 1) * L, count)] for j in range(n)]
    rounds = 30
    for _ in range(rounds):
        cr.cr_all_reduce(bufs, count, "i32", "sum", bufs, "i32")
        cr.cr_reduce_scatter(bufs, count, "i32", "sum", shards, "i32")
        cr.cr_all_gather(shards, count, "i32", bufs)
    torch.cuda.synchronize()
    factor = pow(n, 2 * rounds, 1 << 32)
    want = ((x.astype(np.int64) % (1 << 32)) * factor % (1 << 32)).astype(np.uint32).view(np.int32)
    for r in range(n):
        assert np.array_equal(bufs[r].cpu().numpy(), want), r


def test_overlapped_calls_interleaved_with_torch_kernels():
    """Library calls launched as programmatic dependents, with ordinary torch
    kernels between them on the same stream: each torch kernel must see the
    finished all-reduce, and the next all-reduce must see what the torch
    kernel wrote (a kernel without the early trigger releases its dependent
    only when it completes).  int32 SUM over 4 ranks, exact closed form."""
    n = 4
    count = 8 * n * 40000 + 12
    rng = np.random.default_rng(11)
    x = rng.integers(-50, 50, size=count).astype(np.int64)
    bufs = [torch.from_numpy(x.astype(np.int32)).cuda() for _ in range(n)]
    want = [x.copy() for _ in range(n)]
    for k in range(12):
        cr.cr_all_reduce(bufs, count, "i32", "sum", bufs, "i32")
        tot = sum(want)
        want = [tot.copy() for _ in range(n)]
        bufs[k % n].add_(k + 1)            # a torch kernel on rank k % n's buffer
        want[k % n] = want[k % n] + (k + 1)
        bufs[(k + 1) % n].mul_(-1)         # and another on the next rank's
        want[(k + 1) % n] = -want[(k + 1) % n]
    torch.cuda.synchronize()
    for r in range(n):
        w = ((want[r] % (1 << 32)).astype(np.uint64) % (1 << 32)).astype(np.uint32).view(np.int32)
        assert np.array_equal(bufs[r].cpu().numpy(), w), r

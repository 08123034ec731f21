"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (same generators, seeds, buffer layout and calls).

The oracle cannot reduce tens of GB in a test, so each check compares a
seeded random sample of output elements, computed one by one by the oracle
from the same elements' inputs, plus properties that hold at any size
(every rank's all-reduce output identical, pack then unpack is the
identity).  The 4-rank fp32 workload is small enough to compare in full.
"""
import numpy as np
import pytest
import torch

import oracle as O
from fsdp_emulated_ranks_gb300 import build as libbuild
from fsdp_emulated_ranks_gb300 import cr
from fsdp_emulated_ranks_gb300 import inputs as I
from gpu_util import assert_match, to_host

pytestmark = pytest.mark.gpu
NSAMP = 1 << 18


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    libbuild.build()
    cr.lib()
    yield
    torch.cuda.empty_cache()


def ranks(n, count, dtype, std, seed0):
    out = []
    for r in range(n):
        t = torch.empty(count, dtype=dtype, device="cuda")
        I.torch_fill_normal_(t, std, seed0 + r)
        out.append(t)
    return out


def sample_idx(count, seed, k=NSAMP):
    g = torch.Generator().manual_seed(seed)
    idx = torch.randint(0, count, (k,), generator=g)
    idx = torch.cat([idx, torch.tensor([0, count - 1])])
    return torch.unique(idx).cuda()


def gather(bufs, idx, dt):
    cols = torch.stack([b[idx] for b in bufs], dim=1).contiguous()
    return to_host(cols.view(-1), dt).reshape(cols.shape)


def test_allreduce_sum_f32_4ranks_full():
    """4 ranks x 2^20 fp32 from one stream seeded 0, compared in full."""
    n, count = 4, 1 << 20
    host = I.host_rank_buffers(n, count, "f32", seed0=0, one_stream=True)
    want_ar, _ = O.ring_all_reduce(host, "f32", "sum")
    want_rs, _ = O.ring_reduce_scatter(host, "f32", "sum")
    bufs = [torch.from_numpy(x).cuda() for x in host]
    L = count // n
    shards = [torch.empty(L, dtype=torch.float32, device="cuda") for _ in range(n)]
    cr.cr_reduce_scatter(bufs, count, "f32", "sum", shards, "f32")
    cr.cr_all_reduce(bufs, count, "f32", "sum", bufs, "f32")
    torch.cuda.synchronize()
    for r in range(n):
        assert_match(to_host(shards[r], "f32"), want_rs[r], "f32", f"shard {r}")
        assert_match(to_host(bufs[r], "f32"), want_ar[r], "f32", f"rank {r}")


@pytest.mark.parametrize("n,count", [(8, 1 << 25)] + [(k, 1 << 27) for k in (2, 4, 16, 32, 64)]
                         + [(8, 1 << 29)])
def test_allreduce_avg_bf16_sampled(n, count):
    """8 x 64 MiB (the headline), the rank sweep at 256 MiB per rank and the
    1 GiB-per-rank end of the size sweep; in place, as benchmarked."""
    std, seed0 = (0.02, 0) if (n, count) == (8, 1 << 25) else (1.0, 0)
    bufs = ranks(n, count, torch.bfloat16, std, seed0)
    idx = sample_idx(count, seed=n)
    vals = gather(bufs, idx, "bf16")
    L = cr.cr_chunk_len(count, n)
    chunk = (idx.cpu().numpy() // L).astype(np.int32)
    want = O.fold_columns(vals, chunk, "bf16", "avg", "bf16")
    cr.cr_all_reduce(bufs, count, "bf16", "avg", bufs, "bf16")
    torch.cuda.synchronize()
    got = gather(bufs, idx, "bf16")
    for r in range(n):
        assert_match(got[:, r].copy(), want, "bf16", f"rank {r}")
        if r:
            assert torch.equal(bufs[r].view(torch.int16), bufs[0].view(torch.int16))
    del bufs
    torch.cuda.empty_cache()


def test_reduce_scatter_and_all_gather_bf16_sampled():
    n, count = 8, 1 << 25
    bufs = ranks(n, count, torch.bfloat16, 0.02, 0)
    L = count // n
    shards = [torch.empty(L, dtype=torch.float32, device="cuda") for _ in range(n)]
    idx = sample_idx(count, seed=99)
    vals = gather(bufs, idx, "bf16")
    chunk = (idx.cpu().numpy() // L).astype(np.int32)
    want = O.fold_columns(vals, chunk, "bf16", "avg", "f32")
    cr.cr_reduce_scatter(bufs, count, "bf16", "avg", shards, "f32")
    torch.cuda.synchronize()
    flat = torch.cat(shards)
    assert_match(to_host(flat[idx], "f32"), want, "f32", "reduce-scatter")
    # all-gather the bf16 cast of the shards back into the rank buffers
    b16 = [s.to(torch.bfloat16) for s in shards]
    cr.cr_all_gather(b16, count, "bf16", bufs)
    torch.cuda.synchronize()
    full = torch.cat(b16)
    for r in range(n):
        assert torch.equal(bufs[r].view(torch.int16), full.view(torch.int16))
    del bufs, shards, b16, flat, full
    torch.cuda.empty_cache()


def test_ddp_buckets_full_workload_sampled():
    """300 bf16 tensors per rank, 8 ranks, 25 MiB buckets, laid out as the
    benchmark lays them out (256-byte aligned tensors and buckets)."""
    n = 8
    numels = [int(k) for k in I.bucket_numels()]
    P = sum(numels)
    plan = cr.cr_bucket_plan(numels, 2, 25 * 1024 * 1024)
    oplan = O.bucket_plan(numels, 2, 25 * 1024 * 1024)
    assert plan.tensor_offset == [int(x) for x in oplan.tensor_offset]
    tens, flats = [], []
    for r in range(n):
        flat = torch.empty(P + 128 * len(numels), dtype=torch.bfloat16, device="cuda")
        I.torch_fill_normal_(flat, 1e-3, 1000 + r)
        off, row = 0, []
        for k in numels:
            row.append(flat[off:off + k])
            off += (k + 127) // 128 * 128
        tens.append(row)
        flats.append(flat)
    orig = [f.clone() for f in flats]
    bks = []
    for r in range(n):
        sizes = [(int(k) + 127) // 128 * 128 for k in plan.bucket_numel]
        flat = torch.empty(sum(sizes), dtype=torch.bfloat16, device="cuda")
        off, row = 0, []
        for k, s in zip(plan.bucket_numel, sizes):
            row.append(flat[off:off + int(k)])
            off += s
        bks.append(row)
    flat_t = [x for row in tens for x in row]
    flat_b = [x for row in bks for x in row]
    # pack then unpack is the identity, over every byte
    cr.cr_bucket_pack(plan, n, flat_t, flat_b)
    for row in tens:
        for x in row:
            x.zero_()
    cr.cr_bucket_unpack(plan, n, flat_b, flat_t)
    torch.cuda.synchronize()
    off = 0
    for t, k in enumerate(numels):
        for r in range(n):
            assert torch.equal(tens[r][t].view(torch.int16), orig[r][off:off + k].view(torch.int16)), (r, t)
        off += (k + 127) // 128 * 128
    # every bucket holds the packed tensors at the planned offsets
    for b in range(plan.nbuckets):
        members = [t for t in range(len(numels)) if plan.tensor_bucket[t] == b]
        for t in members[:3] + members[-3:]:
            o = plan.tensor_offset[t]
            for r in (0, n - 1):
                assert torch.equal(bks[r][b][o:o + numels[t]].view(torch.int16),
                                   tens[r][t].view(torch.int16))
    # all-reduce AVG per bucket, sampled against the oracle
    want = {}
    for b in range(plan.nbuckets):
        cnt = int(plan.bucket_numel[b])
        idx = sample_idx(cnt, seed=b, k=2048)
        vals = gather([bks[r][b] for r in range(n)], idx, "bf16")
        L = cr.cr_chunk_len(cnt, n)
        want[b] = (idx, O.fold_columns(vals, (idx.cpu().numpy() // L).astype(np.int32),
                                       "bf16", "avg", "bf16"))
    cr.cr_bucket_all_reduce(plan, n, flat_b, "bf16", "avg")
    cr.cr_bucket_unpack(plan, n, flat_b, flat_t)
    torch.cuda.synchronize()
    for b, (idx, w) in want.items():
        got = gather([bks[r][b] for r in range(n)], idx, "bf16")
        for r in range(n):
            assert_match(got[:, r].copy(), w, "bf16", f"bucket {b} rank {r}")
    for t in (0, len(numels) // 2, len(numels) - 1):
        b, o = plan.tensor_bucket[t], plan.tensor_offset[t]
        for r in range(n):
            assert torch.equal(tens[r][t].view(torch.int16),
                               bks[r][b][o:o + numels[t]].view(torch.int16))
    del tens, bks, flats, orig, flat_t, flat_b
    torch.cuda.empty_cache()


def test_fsdp_step_1p3b_sampled():
    """8 ranks, flat 1.3e9 params: bf16 grads N(0, 1e-3^2) seeded 1000 + r,
    fp32 master N(0, 0.02^2) seeded 2000, m = v = 0, AdamW step 1."""
    n, count = 8, 1_300_000_000
    L = count // n
    grads = ranks(n, count, torch.bfloat16, 1e-3, 1000)
    params = [torch.empty(count, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    master_full = torch.empty(count, dtype=torch.float32, device="cuda")
    I.torch_fill_normal_(master_full, 0.02, 2000)
    master = [master_full[j * L:(j + 1) * L] for j in range(n)]
    mv = torch.zeros(2 * count, dtype=torch.float32, device="cuda")
    m = [mv[j * L:(j + 1) * L] for j in range(n)]
    v = [mv[count + j * L:count + (j + 1) * L] for j in range(n)]
    idx = sample_idx(count, seed=4)
    g = gather(grads, idx, "bf16")
    p0 = to_host(master_full[idx], "f32")
    chunk = (idx.cpu().numpy() // L).astype(np.int32)
    gavg = O.fold_columns(g, chunk, "bf16", "avg", "f32")
    pm, mm, vm = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
    cfg = O.AdamWConfig()
    O.adamw(pm, mm, vm, gavg, cfg)
    cr.cr_fsdp_step(grads, count, master, m, v, cr.adamw_cfg(), params)
    torch.cuda.synchronize()
    assert_match(to_host(master_full[idx], "f32"), pm, "f32", "master")
    assert_match(to_host(mv[:count][idx], "f32"), mm, "f32", "m")
    assert_match(to_host(mv[count:][idx], "f32"), vm, "f32", "v")
    want_p = O.f32_to_bf16(pm)
    got_p = gather(params, idx, "bf16")
    for r in range(n):
        assert_match(got_p[:, r].copy(), want_p, "bf16", f"params[{r}]")
    for r in range(1, n):
        assert torch.equal(params[r].view(torch.int16), params[0].view(torch.int16))
    del grads, params, master_full, mv
    torch.cuda.empty_cache()


def embed(vals, keys, nkeys):
    """Place sampled columns (vals [k, n]) into small rank buffers of nkeys
    equal blocks, each sample in the block of its key (its chunk of the
    full-size problem), so that a ring over the small buffers reduces every
    sample in the same order as the full-size ring.  Returns the buffers,
    the block size M and each sample's position."""
    k, n = vals.shape
    counts = np.bincount(keys, minlength=nkeys)
    M = max(1, int(counts.max()))
    pos = np.empty(k, np.int64)
    fill = np.zeros(nkeys, np.int64)
    for s, key in enumerate(keys):
        pos[s] = key * M + fill[key]
        fill[key] += 1
    bufs = [np.zeros(nkeys * M, vals.dtype) for _ in range(n)]
    for r in range(n):
        bufs[r][pos] = vals[:, r]
    return bufs, M, pos


def test_allreduce_bf16_wire_full_sampled():
    """The bf16-wire all-reduce of 8 x 64 MiB, as benchmarked (in place),
    sampled and reduced by the oracle's literal ring with bf16 messages."""
    n, count = 8, 1 << 25
    bufs = ranks(n, count, torch.bfloat16, 0.02, 0)
    idx = sample_idx(count, seed=123, k=1 << 16)
    vals = gather(bufs, idx, "bf16")
    L = cr.cr_chunk_len(count, n)
    chunk = (idx.cpu().numpy() // L).astype(np.int64)
    small, M, pos = embed(vals, chunk, n)
    want = O.ring_all_reduce_wire(small, "bf16", "avg", "bf16", "bf16")[0][pos]
    cr.cr_all_reduce_wire(bufs, count, "bf16", "avg", "bf16", bufs, "bf16")
    torch.cuda.synchronize()
    got = gather(bufs, idx, "bf16")
    for r in range(n):
        assert_match(got[:, r].copy(), want, "bf16", f"rank {r}")
    del bufs
    torch.cuda.empty_cache()


def test_hsdp_2x4_full_sampled():
    """HSDP on the 2 x 4 mesh, 64 MiB bf16 per rank, as benchmarked: each
    sample keeps its shard j and outer chunk i in the embedded problem."""
    R, S, count = 2, 4, 1 << 25
    n = R * S
    bufs = ranks(n, count, torch.bfloat16, 0.02, 0)
    L = -(-count // S)
    shards = [torch.empty(min(L, count - j * L), dtype=torch.bfloat16, device="cuda")
              for _ in range(R) for j in range(S)]
    idx = sample_idx(count, seed=321, k=1 << 16)
    vals = gather(bufs, idx, "bf16")
    e = idx.cpu().numpy().astype(np.int64)
    j = e // L
    k = e - j * L
    L2 = -(-L // R)   # every shard is full: count = S * L
    i = k // L2
    small, M, pos = embed(vals, j * R + i, S * R)
    want = O.hsdp_reduce_scatter(small, R, S, "bf16", "avg", "bf16")
    cr.cr_hsdp_reduce_scatter(bufs, R, S, count, "bf16", "avg", shards, "bf16")
    torch.cuda.synchronize()
    Ls = R * M  # shard length of the embedded problem
    for g in range(R):
        flat = torch.cat(shards[g * S:(g + 1) * S])
        got = to_host(flat[idx], "bf16")
        ref = np.concatenate(want[g * S:(g + 1) * S])[pos]
        assert_match(got, ref, "bf16", f"group {g}")
        assert Ls * S == sum(w.size for w in want[g * S:(g + 1) * S])
    del bufs, shards
    torch.cuda.empty_cache()


# ---- beyond 2^32 elements per buffer ----------------------------------------
# Element indices and chunk divisions switch to 64-bit arithmetic once a
# buffer holds 2^32 elements or more (the multiply-shift division covers
# dividends below 2^32 only).  N = 2 keeps the footprint at tens of GB.

BIG_RAGGED = (1 << 32) + 301            # odd: vector path plus an element tail
BIG_EVEN = 2 * ((1 << 31) + 80)         # shard length a multiple of 16


def edge_idx(count, extra=(), seed=0):
    L = -(-count // 2)
    fixed = [0, 1, L - 1, L, L + 1, (1 << 32) - 1, 1 << 32, (1 << 32) + 1, count - 17,
             count - 16, count - 1, *extra]
    idx = torch.cat([sample_idx(count, seed, k=1 << 14).cpu(),
                     torch.tensor([i for i in fixed if 0 <= i < count])])
    return torch.unique(idx).cuda()


def pick(shards, L, idx):
    """Elements idx of the concatenation of equal-length shards, without
    building the concatenation."""
    out = torch.empty(idx.numel(), dtype=shards[0].dtype, device="cuda")
    which = idx // L
    for j, sh in enumerate(shards):
        m = which == j
        out[m] = sh[idx[m] - j * L]
    return out


def test_allreduce_bf16_beyond_2_32_elements():
    n, count = 2, BIG_RAGGED
    bufs = ranks(n, count, torch.bfloat16, 0.02, 40)
    idx = edge_idx(count, seed=1)
    vals = gather(bufs, idx, "bf16")
    L = cr.cr_chunk_len(count, n)
    chunk = (idx.cpu().numpy() // L).astype(np.int32)
    want = O.fold_columns(vals, chunk, "bf16", "avg", "bf16")
    cr.cr_all_reduce(bufs, count, "bf16", "avg", bufs, "bf16")
    torch.cuda.synchronize()
    got = gather(bufs, idx, "bf16")
    for r in range(n):
        assert_match(got[:, r].copy(), want, "bf16", f"rank {r}")
    assert torch.equal(bufs[0].view(torch.int16), bufs[1].view(torch.int16))
    del bufs
    torch.cuda.empty_cache()


def test_reduce_scatter_and_all_gather_beyond_2_32_elements():
    n, count = 2, BIG_EVEN
    L = count // n
    bufs = ranks(n, count, torch.bfloat16, 0.02, 50)
    idx = edge_idx(count, seed=2)
    vals = gather(bufs, idx, "bf16")
    chunk = (idx.cpu().numpy() // L).astype(np.int32)
    want = O.fold_columns(vals, chunk, "bf16", "avg", "bf16")
    shards = [torch.empty(L, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    cr.cr_reduce_scatter(bufs, count, "bf16", "avg", shards, "bf16")
    torch.cuda.synchronize()
    assert_match(to_host(pick(shards, L, idx), "bf16"), want, "bf16", "reduce-scatter")
    cr.cr_all_gather(shards, count, "bf16", bufs)
    torch.cuda.synchronize()
    for r in range(n):
        for j in range(n):
            assert torch.equal(bufs[r][j * L:(j + 1) * L].view(torch.int16),
                               shards[j].view(torch.int16)), (r, j)
    del bufs, shards
    torch.cuda.empty_cache()


def test_hsdp_2x2_beyond_2_32_elements():
    R, S, count = 2, 2, BIG_EVEN
    n = R * S
    L = count // S
    bufs = ranks(n, count, torch.bfloat16, 0.02, 60)
    shards = [torch.empty(L, dtype=torch.bfloat16, device="cuda") for _ in range(R * S)]
    idx = edge_idx(count, seed=3)
    vals = gather(bufs, idx, "bf16")
    e = idx.cpu().numpy().astype(np.int64)
    j = e // L
    i = (e - j * L) // (-(-L // R))
    small, M, pos = embed(vals, j * R + i, S * R)
    want = O.hsdp_reduce_scatter(small, R, S, "bf16", "avg", "bf16")
    cr.cr_hsdp_reduce_scatter(bufs, R, S, count, "bf16", "avg", shards, "bf16")
    torch.cuda.synchronize()
    for g in range(R):
        got = to_host(pick(shards[g * S:(g + 1) * S], L, idx), "bf16")
        ref = np.concatenate(want[g * S:(g + 1) * S])[pos]
        assert_match(got, ref, "bf16", f"group {g}")
    del bufs, shards
    torch.cuda.empty_cache()


@pytest.mark.parametrize("planned", [True, False], ids=["planned", "chained"])
def test_fsdp2_transformer_full_sampled(planned):
    """The FSDP2 step over the benchmark's transformer (145 parameters,
    1.27e9 elements, 8 ranks), laid out and called as benchmarked: one
    launch over the plan's table, or the pointers in the parameter blocks
    of three chained launches.  Each
    sampled element's result depends only on its 8 gradients, its state and
    the rank that owns its row (the fold order): grouped by owner, the
    samples are embedded into a small parameter of N rows whose row j is
    owned by rank j, and that is stepped by the oracle."""
    import bench
    n = 8
    wl = bench.Fsdp2Step(planned=planned)
    wl.setup(torch.device("cuda"))
    rng = np.random.default_rng(7)
    P, I_, J, K = [], [], [], []
    for p, (d0, row) in enumerate(wl.shapes):
        k = d0 * row
        Lr = -(-d0 // n)
        for i in sorted(set(rng.integers(0, k, 48).tolist()) | {0, k - 1}):
            j = (i // row) // Lr
            P.append(p), I_.append(i), J.append(j), K.append(i - j * Lr * row)
    gidx = torch.tensor([wl.offs[p] + i for p, i in zip(P, I_)], device="cuda")
    sidx = torch.tensor([wl.soffs[p][j] + k for p, j, k in zip(P, J, K)], device="cuda")
    g = np.stack([to_host(wl.t_g[r][gidx], "bf16") for r in range(n)], axis=1)   # [s, n]
    st0 = [wl.t_state[sidx + q * wl.so].cpu().numpy() for q in range(3)]       # master, m, v
    wl.step(torch.cuda.current_stream())
    torch.cuda.synchronize()
    st1 = [wl.t_state[sidx + q * wl.so].cpu().numpy() for q in range(3)]
    par = np.stack([to_host(wl.t_p[r][gidx], "bf16") for r in range(n)], axis=1)
    wl.teardown()
    # embed: owner j's samples at row j of an (n x M) parameter
    J = np.array(J)
    M = max(1, int(np.bincount(J, minlength=n).max()))
    col = np.zeros(len(J), np.int64)
    fill = np.zeros(n, np.int64)
    for s, j in enumerate(J):
        col[s] = fill[j]
        fill[j] += 1
    grads = [np.zeros(n * M, np.uint16) for _ in range(n)]
    for r in range(n):
        grads[r][J * M + col] = g[:, r]
    state = [[np.zeros(M, np.float32) for _ in range(n)] for _ in range(3)]
    for q in range(3):
        for s in range(len(J)):
            state[q][J[s]][col[s]] = st0[q][s]
    want_p = O.fsdp2_step([(n, M)], [grads], [state[0]], [state[1]], [state[2]], O.AdamWConfig())
    for q, name in enumerate(("master", "m", "v")):
        ref = np.array([state[q][J[s]][col[s]] for s in range(len(J))], np.float32)
        assert_match(st1[q], ref, "f32", name)
    for r in range(n):
        ref = want_p[0][r][J * M + col]
        assert_match(par[:, r].copy(), ref, "bf16", f"params rank {r}")

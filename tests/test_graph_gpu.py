"""The entry points are capturable in CUDA graphs: they only enqueue work on
the given stream (no host synchronisation, no allocation), so a captured
step replays exactly what the eager calls compute.  Checked bit for bit
against eager runs for the all-reduce, the FSDP step, the no-alloc clipped
step (its one-time address lookup made before capture), a whole DDP
reducer iteration whose communication stream joins the capture through the
reducer's events, a chain of dependent calls that each start as the
programmatic dependent of the one before, the planned FSDP2 step and a
range all-reduce."""
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


def filled(n, count, dtype, std, seed0):
    out = []
    for r in range(n):
        t = torch.empty(count, dtype=dtype, device="cuda")
        I.torch_fill_normal_(t, std, seed0 + r)
        out.append(t)
    return out


def capture(fn):
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        fn()
    torch.cuda.synchronize()
    return g


def test_all_reduce_graph_replay_matches_eager():
    n, count = 8, 8 * 8 * 1000 + 5
    src = filled(n, count, torch.bfloat16, 0.02, 0)
    eager = [x.clone() for x in src]
    cr.cr_all_reduce(eager, count, "bf16", "avg", eager, "bf16")
    work = [torch.empty_like(x) for x in src]
    g = capture(lambda: cr.cr_all_reduce(work, count, "bf16", "avg", work, "bf16"))
    for _ in range(2):  # replay twice on fresh inputs
        for w, x in zip(work, src):
            w.copy_(x)
        g.replay()
        torch.cuda.synchronize()
        for w, e in zip(work, eager):
            assert torch.equal(w.view(torch.int16), e.view(torch.int16))


def fsdp_state(n, count, seed):
    grads = filled(n, count, torch.bfloat16, 1e-3, 1000 + seed)
    L = cr.cr_chunk_len(count, n)
    lens = [max(0, min(count, (j + 1) * L) - min(count, j * L)) for j in range(n)]
    master = []
    for j in range(n):
        t = torch.empty(lens[j], dtype=torch.float32, device="cuda")
        I.torch_fill_normal_(t, 0.02, 2000 + j)
        master.append(t)
    m = [torch.zeros(k, dtype=torch.float32, device="cuda") for k in lens]
    v = [torch.zeros(k, dtype=torch.float32, device="cuda") for k in lens]
    params = [torch.empty(count, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    return grads, master, m, v, params


@pytest.mark.parametrize("clipped", [False, True])
def test_fsdp_step_graph_replay_matches_eager(clipped):
    n, count = 8, 8 * 8 * 3000 + 11
    cfg = cr.adamw_cfg()
    a = fsdp_state(n, count, 1)
    b = fsdp_state(n, count, 1)
    norm_a = torch.zeros(1, dtype=torch.float32, device="cuda")
    norm_b = torch.zeros(1, dtype=torch.float32, device="cuda")

    def step(st, norm):
        g, ms, m, v, p = st
        if clipped:
            cr.cr_fsdp_step_clipped_noalloc(g, count, ms, m, v, cfg, 1e-3, p, norm)
        else:
            cr.cr_fsdp_step(g, count, ms, m, v, cfg, p)

    step(a, norm_a)           # eager (and, for the no-alloc form, its address lookup)
    torch.cuda.synchronize()
    graph = capture(lambda: step(b, norm_b))
    graph.replay()
    torch.cuda.synchronize()
    for xa, xb in zip(a[1] + a[2] + a[3], b[1] + b[2] + b[3]):
        assert torch.equal(xa, xb)
    for pa, pb in zip(a[4], b[4]):
        assert torch.equal(pa.view(torch.int16), pb.view(torch.int16))
    if clipped:
        assert torch.equal(norm_a, norm_b)


def test_reducer_iteration_graph_replay_matches_fused():
    n = 4
    rng = np.random.default_rng(3)
    numels = [int(x) for x in rng.integers(1, 40000, 30)]
    plan = cr.cr_bucket_plan(numels, 2, 128 * 1024)
    T = plan.ntensors
    src = []
    for r in range(n):
        for t, k in enumerate(numels):
            x = torch.empty(k, dtype=torch.bfloat16, device="cuda")
            I.torch_fill_normal_(x, 0.02, 100 * r + t)
            src.append(x)
    grads = [torch.zeros_like(x) for x in src]
    comm = torch.cuda.Stream()
    red = cr.cr_reducer_create(plan, n, grads, "bf16", "avg", 16, comm)

    def iteration():
        # emulated backward: each tensor's gradient written, then marked ready
        for t in range(T - 1, -1, -1):
            for r in range(n):
                grads[r * T + t].copy_(src[r * T + t])
            cr.cr_reducer_mark_ready(red, t)
        cr.cr_reducer_finalize(red)

    g = capture(iteration)
    for g_ in grads:
        g_.zero_()
    g.replay()
    torch.cuda.synchronize()
    ref = [x.clone() for x in src]
    cr.cr_bucket_all_reduce_fused(plan, n, ref, "bf16", "avg")
    torch.cuda.synchronize()
    for k in range(n * T):
        assert torch.equal(grads[k].view(torch.int16), ref[k].view(torch.int16)), k
    cr.cr_reducer_destroy(red)


def test_dependent_chain_graph_replay_matches_eager():
    """Four dependent calls captured in one graph -- in-place all-reduce,
    reduce-scatter into the ranks' own chunks, all-gather back in place,
    all-reduce again -- each launched as the programmatic dependent of the
    one before: the graph keeps their order, bit for bit the eager chain."""
    n, count = 8, 8 * 8 * 2000 + 40
    L = cr.cr_chunk_len(count, n)
    src = filled(n, count, torch.bfloat16, 0.02, 50)

    def chain(bufs):
        shards = [bufs[j][j * L:min((j + 1) * L, count)] for j in range(n)]
        cr.cr_all_reduce(bufs, count, "bf16", "avg", bufs, "bf16")
        cr.cr_reduce_scatter(bufs, count, "bf16", "sum", shards, "bf16")
        cr.cr_all_gather(shards, count, "bf16", bufs)
        cr.cr_all_reduce(bufs, count, "bf16", "avg", bufs, "bf16")

    eager = [x.clone() for x in src]
    chain(eager)
    work = [torch.empty_like(x) for x in src]
    g = capture(lambda: chain(work))
    for _ in range(2):
        for w, x in zip(work, src):
            w.copy_(x)
        g.replay()
        torch.cuda.synchronize()
        for w, e in zip(work, eager):
            assert torch.equal(w.view(torch.int16), e.view(torch.int16))


def test_planned_fsdp2_and_range_graph_replay_matches_eager():
    """The planned FSDP2 step (table uploaded before capture) and a range
    all-reduce over one slab, captured and replayed, against eager calls."""
    n = 4
    shapes = [(10, 64), (3, 8), (33, 100)]
    cfg = cr.adamw_cfg()

    def state(seed):
        grads, master, m, v, params = [], [], [], [], []
        for p, (d, rn) in enumerate(shapes):
            Lr = -(-d // n)
            for r in range(n):
                t = torch.empty(d * rn, dtype=torch.bfloat16, device="cuda")
                I.torch_fill_normal_(t, 1e-3, seed + 10 * p + r)
                grads.append(t)
                params.append(torch.empty(d * rn, dtype=torch.bfloat16, device="cuda"))
                k = max(0, min(d, (r + 1) * Lr) - min(d, r * Lr)) * rn
                mt = torch.empty(k, dtype=torch.float32, device="cuda")
                I.torch_fill_normal_(mt, 0.02, 500 + 10 * p + r)
                master.append(mt if k else 0)
                m.append(torch.zeros(k, dtype=torch.float32, device="cuda") if k else 0)
                v.append(torch.zeros(k, dtype=torch.float32, device="cuda") if k else 0)
        return grads, master, m, v, params

    a, b = state(7), state(7)
    cr.cr_fsdp2_step(shapes, n, *a[:4], cfg, a[4])
    plan = cr.cr_fsdp2_plan_create(shapes, n, *b)
    table = torch.empty(plan.table_bytes, dtype=torch.uint8, device="cuda")
    cr.cr_fsdp2_plan_upload(plan, table)
    torch.cuda.synchronize()
    g = capture(lambda: cr.cr_fsdp2_step_planned(plan, table, cfg))
    g.replay()
    torch.cuda.synchronize()
    for xa, xb in zip(a[1] + a[2] + a[3] + a[4], b[1] + b[2] + b[3] + b[4]):
        if isinstance(xa, int):
            continue
        assert torch.equal(xa.view(torch.int32) if xa.dtype == torch.float32 else xa.view(torch.int16),
                           xb.view(torch.int32) if xb.dtype == torch.float32 else xb.view(torch.int16))

    count = 8 * 4 * 1000 + 3
    lo, hi = cr.cr_slab_range(count, n, 2, 1)
    src = filled(n, count, torch.bfloat16, 0.02, 90)
    whole = [x.clone() for x in src]
    cr.cr_all_reduce(whole, count, "bf16", "avg", whole, "bf16")
    slab = [x[lo:hi].clone() for x in src]
    g2 = capture(lambda: cr.cr_all_reduce_range(slab, count, lo, hi, "bf16", "avg", slab, "bf16"))
    g2.replay()
    torch.cuda.synchronize()
    for s, w in zip(slab, whole):
        assert torch.equal(s.view(torch.int16), w[lo:hi].view(torch.int16))

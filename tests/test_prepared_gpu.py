"""cr.prepare on the GPU: a prepared call issues exactly the direct call.

Each case runs the same work twice, once through the wrappers and once
through a call prepared in advance, on equal inputs, and compares the
results bit for bit: the all-reduce, the FSDP step over three AdamW steps
(cfg.step advanced between invocations of the one prepared call), the
fused bucket all-reduce with the caller's plan object dropped after
preparation (the prepared call keeps it alive), the FSDP2 step from a
plan's table, and the range forms over slabs of the element range."""
import gc

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


def same(a, b):
    return all(torch.equal(x.view(torch.uint8), y.view(torch.uint8)) for x, y in zip(a, b))


def test_prepared_all_reduce_equals_direct_calls():
    n, count = 8, 8 * 8 * 1000 + 5
    src = filled(n, count, torch.bfloat16, 0.02, 0)
    direct = [x.clone() for x in src]
    work = [x.clone() for x in src]
    p = cr.prepare(cr.cr_all_reduce, work, count, "bf16", "avg", work, "bf16")
    for _ in range(3):  # in place, so each call reduces the previous result
        cr.cr_all_reduce(direct, count, "bf16", "avg", direct, "bf16")
        p()
    torch.cuda.synchronize()
    assert same(direct, work)


def fsdp_state(n, count):
    grads = filled(n, count, torch.bfloat16, 1e-3, 1000)
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


def test_prepared_fsdp_step_follows_the_step_counter():
    n, count = 8, 8 * 8 * 500 + 3
    a = fsdp_state(n, count)
    b = [[x.clone() for x in part] for part in a]
    cfg_a, cfg_b = cr.adamw_cfg(), cr.adamw_cfg()
    p = cr.prepare(cr.cr_fsdp_step, b[0], count, b[1], b[2], b[3], cfg_b, b[4])
    for step in (1, 2, 3):
        cfg_a.step = step
        cr.cr_fsdp_step(a[0], count, a[1], a[2], a[3], cfg_a, a[4])
        cfg_b.step = step
        p()
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert same(x, y)


def test_prepared_fused_buckets_keep_the_plan_alive():
    n = 4
    numels = [1000, 37, 2000, 4096, 5]
    tens = []
    for r in range(n):
        for i, k in enumerate(numels):
            t = torch.empty(k, dtype=torch.bfloat16, device="cuda")
            I.torch_fill_normal_(t, 1e-3, 1000 * r + i)
            tens.append(t)
    direct = [t.clone() for t in tens]
    plan = cr.cr_bucket_plan(numels, 2, 4096)
    cr.cr_bucket_all_reduce_fused(plan, n, direct, "bf16", "avg")
    p = cr.prepare(cr.cr_bucket_all_reduce_fused, cr.cr_bucket_plan(numels, 2, 4096), n, tens,
                   "bf16", "avg")
    gc.collect()  # the plan passed to prepare has no other reference
    p()
    torch.cuda.synchronize()
    assert same(direct, tens)


def fsdp2_state(n, shapes):
    """Flat lists indexed p*n + r: bf16 grads and params per rank, fp32
    master/m/v per owner shard (0 for an empty shard)."""
    grads, params, master, m, v = [], [], [], [], []
    for p, (d, rn) in enumerate(shapes):
        grads += filled(n, d * rn, torch.bfloat16, 1e-3, 3000 + 10 * p)
        params += [torch.empty(d * rn, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
        Lr = -(-d // n)
        for j in range(n):
            k = max(0, min(d, (j + 1) * Lr) - min(d, j * Lr)) * rn
            if k == 0:
                master.append(0), m.append(0), v.append(0)
                continue
            t = torch.empty(k, dtype=torch.float32, device="cuda")
            I.torch_fill_normal_(t, 0.02, 4000 + 10 * p + j)
            master.append(t)
            m.append(torch.zeros(k, dtype=torch.float32, device="cuda"))
            v.append(torch.zeros(k, dtype=torch.float32, device="cuda"))
    return grads, master, m, v, params


def clone_state(state):
    return [[x.clone() if isinstance(x, torch.Tensor) else x for x in part] for part in state]


def test_prepared_planned_fsdp2_step_follows_the_step_counter():
    n, shapes = 4, [(10, 64), (3, 8), (17, 40)]
    a = fsdp2_state(n, shapes)
    b = clone_state(a)
    plans, tables = [], []
    for s in (a, b):
        plan = cr.cr_fsdp2_plan_create(shapes, n, s[0], s[1], s[2], s[3], s[4])
        table = torch.empty(plan.table_bytes, dtype=torch.uint8, device="cuda")
        cr.cr_fsdp2_plan_upload(plan, table)
        plans.append(plan), tables.append(table)
    cfg_a, cfg_b = cr.adamw_cfg(), cr.adamw_cfg()
    p = cr.prepare(cr.cr_fsdp2_step_planned, plans[1], tables[1], cfg_b)
    for step in (1, 2, 3):
        cfg_a.step = cfg_b.step = step
        cr.cr_fsdp2_step_planned(plans[0], tables[0], cfg_a)
        p()
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        x = [t for t in x if isinstance(t, torch.Tensor)]
        y = [t for t in y if isinstance(t, torch.Tensor)]
        assert same(x, y)


def test_prepared_range_calls_equal_direct_calls():
    n, count, G = 8, 8 * 8 * 300 + 5, 3
    src = filled(n, count, torch.bfloat16, 0.02, 50)
    direct = [x.clone() for x in src]
    work = [x.clone() for x in src]
    L = cr.cr_chunk_len(count, n)
    preps = []
    for g in range(G):
        lo, hi = cr.cr_slab_range(count, n, G, g)
        slab = [b[lo:hi] for b in work]
        preps.append(cr.prepare(cr.cr_all_reduce_range, slab, count, lo, hi, "bf16", "avg",
                                slab, "bf16"))
    for _ in range(2):  # in place: the second pass reduces the first's result
        cr.cr_all_reduce(direct, count, "bf16", "avg", direct, "bf16")
        for p in preps:
            p()
    torch.cuda.synchronize()
    assert same(direct, work)
    # reduce-scatter by 11 slabs (cutting chunks), prepared, against the
    # whole call; the last shard is short, so both start from the same fill
    shards = [torch.full((L,), -1.0, dtype=torch.float32, device="cuda") for _ in range(n)]
    cr.cr_reduce_scatter(src, count, "bf16", "avg", shards, "f32")
    parts = [torch.full((L,), -1.0, dtype=torch.float32, device="cuda") for _ in range(n)]
    for g in range(11):
        lo, hi = cr.cr_slab_range(count, n, 11, g)
        outs = []
        for j in range(n):
            a, b = max(lo, j * L), min(hi, min(count, (j + 1) * L))
            outs.append(parts[j][a - j * L:] if b > a else None)
        cr.prepare(cr.cr_reduce_scatter_range, [b[lo:hi] for b in src], count, lo, hi, "bf16",
                   "avg", outs, "f32")()
    torch.cuda.synchronize()
    assert same(shards, parts)

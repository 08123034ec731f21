"""cr.prepare on the GPU: a prepared call issues exactly the direct call.

Each case runs the same work twice, once through the wrappers and once
through a call prepared in advance, on equal inputs, and compares the
results bit for bit: the all-reduce, the FSDP step over three AdamW steps
(cfg.step advanced between invocations of the one prepared call), and the
fused bucket all-reduce with the caller's plan object dropped after
preparation (the prepared call keeps it alive)."""
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

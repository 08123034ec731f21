"""Parity at full size for the remaining benchmarked rows, in the launch
configuration the benchmark times: the fused bucket all-reduce over the 300
seeded tensors (three chained launches), the clipped FSDP step over 1.3e9
parameters with max_norm 1.0 (the norm is about 12.7, so clipping is
active), the no_sync accumulation rows over 8 x 2^25 elements, and the
end-to-end leg: the 8 x 64 MiB all-reduce over rank buffers in pinned host
memory, through both host entry points.

As in test_fullsize_gpu.py, the oracle computes a seeded random sample of
output elements one by one from the same elements' inputs.  The clipped
step's global norm is the one quantity no sample determines; it is checked
against its definition -- the L2 norm of the averaged gradient -- computed
in float64 over every element by torch's own reductions, slab by slab."""
import numpy as np
import pytest
import torch

import oracle as O
from fsdp_emulated_ranks_gb300 import build as libbuild
from fsdp_emulated_ranks_gb300 import cr
from fsdp_emulated_ranks_gb300 import inputs as I
from gpu_util import assert_match, clip_coefficients, to_host

pytestmark = pytest.mark.gpu


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


def sample_idx(count, seed, k):
    g = torch.Generator().manual_seed(seed)
    idx = torch.randint(0, count, (k,), generator=g)
    idx = torch.cat([idx, torch.tensor([0, count - 1])])
    return torch.unique(idx).cuda()


def gather(bufs, idx, dt):
    cols = torch.stack([b[idx] for b in bufs], dim=1).contiguous()
    return to_host(cols.view(-1), dt).reshape(cols.shape)


def test_fused_buckets_full_workload_sampled():
    """300 bf16 tensors per rank, 8 ranks, 25 MiB buckets, tensors at
    256-byte aligned offsets of one slab per rank (the benchmark's layout);
    the fused all-reduce takes three chained launches of 128 tensors."""
    n = 8
    numels = [int(k) for k in I.bucket_numels()]
    plan = cr.cr_bucket_plan(numels, 2, 25 * 1024 * 1024)
    tens = []
    for r in range(n):
        flat = torch.empty(sum(numels) + 128 * len(numels), dtype=torch.bfloat16, device="cuda")
        I.torch_fill_normal_(flat, 1e-3, 1000 + r)
        off, row = 0, []
        for k in numels:
            row.append(flat[off:off + k])
            off += (k + 127) // 128 * 128
        tens.append(row)
    # expected values of sampled elements of every tensor, folded in the
    # ring order of their bucket position
    want = {}
    for t, k in enumerate(numels):
        idx = sample_idx(k, seed=t, k=256)
        vals = gather([tens[r][t] for r in range(n)], idx, "bf16")
        b = plan.tensor_bucket[t]
        L = cr.cr_chunk_len(int(plan.bucket_numel[b]), n)
        pos = idx.cpu().numpy() + plan.tensor_offset[t]
        want[t] = (idx, O.fold_columns(vals, (pos // L).astype(np.int32), "bf16", "avg", "bf16"))
    flat_t = [x for row in tens for x in row]
    cr.cr_bucket_all_reduce_fused(plan, n, flat_t, "bf16", "avg")
    torch.cuda.synchronize()
    for t, (idx, w) in want.items():
        got = gather([tens[r][t] for r in range(n)], idx, "bf16")
        for r in range(n):
            assert_match(got[:, r].copy(), w, "bf16", f"tensor {t} rank {r}")
    for t in (0, 150, len(numels) - 1):  # every rank holds the same result
        for r in range(1, n):
            assert torch.equal(tens[r][t].view(torch.int16), tens[0][t].view(torch.int16))
    del tens, flat_t
    torch.cuda.empty_cache()


def test_fsdp_step_clipped_1p3b_sampled():
    """8 ranks, flat 1.3e9 params as the benchmark's clipped row: bf16 grads
    N(0, 1e-3^2) seeded 1000 + r, fp32 master N(0, 0.02^2) seeded 2000,
    m = v = 0, AdamW step 1, max_norm 1.0."""
    n, count, max_norm = 8, 1_300_000_000, 1.0
    L = count // n
    grads = ranks(n, count, torch.bfloat16, 1e-3, 1000)
    params = [torch.empty(count, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    master_full = torch.empty(count, dtype=torch.float32, device="cuda")
    I.torch_fill_normal_(master_full, 0.02, 2000)
    master = [master_full[j * L:(j + 1) * L] for j in range(n)]
    mv = torch.zeros(2 * count, dtype=torch.float32, device="cuda")
    m = [mv[j * L:(j + 1) * L] for j in range(n)]
    v = [mv[count + j * L:count + (j + 1) * L] for j in range(n)]
    # the definition of the norm: || sum_r g_r / N ||_2, in float64
    sumsq, slab = 0.0, 1 << 27
    for lo in range(0, count, slab):
        acc = torch.zeros(min(slab, count - lo), dtype=torch.float64, device="cuda")
        for g in grads:
            acc += g[lo:lo + slab].double()
        sumsq += float(torch.sum((acc / n) ** 2))
        del acc
    norm_ref = sumsq ** 0.5
    assert norm_ref > max_norm  # the workload does clip
    idx = sample_idx(count, seed=5, k=1 << 18)
    g = gather(grads, idx, "bf16")
    p0 = to_host(master_full[idx], "f32")
    ws_bytes = cr.cr_fsdp_clip_workspace_bytes()
    ws = torch.empty(ws_bytes // 8, dtype=torch.float64, device="cuda")
    norm = torch.empty(1, dtype=torch.float32, device="cuda")
    cr.cr_fsdp_step_clipped(grads, count, master, m, v, cr.adamw_cfg(), max_norm, ws, ws_bytes,
                            params, norm)
    torch.cuda.synchronize()
    assert abs(norm.item() - norm_ref) <= 1e-6 * norm_ref, (norm.item(), norm_ref)
    # sampled elements: the oracle's fold and AdamW on the gradient scaled by
    # the fp32 clip coefficient; the library's state must equal that, bit for
    # bit, at one coefficient of the norm's tolerance window
    gavg = O.fold_columns(g, (idx.cpu().numpy() // L).astype(np.int32), "bf16", "avg", "f32")
    got = [to_host(master_full[idx], "f32"), to_host(mv[:count][idx], "f32"),
           to_host(mv[count:][idx], "f32")]
    for coef in clip_coefficients(max_norm, norm_ref):
        pm, mm, vm = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
        O.adamw(pm, mm, vm, (gavg * coef).astype(np.float32), O.AdamWConfig())
        if all(a.tobytes() == b.tobytes() for a, b in zip(got, (pm, mm, vm))):
            break
    else:
        coef = clip_coefficients(max_norm, norm_ref)[0]
        pm, mm, vm = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
        O.adamw(pm, mm, vm, (gavg * coef).astype(np.float32), O.AdamWConfig())
        for a, b, name in zip(got, (pm, mm, vm), ("master", "m", "v")):
            assert_match(a, b, "f32", f"{name} (no coefficient in the window fits)")
    want_p = O.f32_to_bf16(pm)
    got_p = gather(params, idx, "bf16")
    for r in range(n):
        assert_match(got_p[:, r].copy(), want_p, "bf16", f"params[{r}]")
    del grads, params, master_full, mv, ws
    torch.cuda.empty_cache()


@pytest.mark.parametrize("reduce", [False, True])
def test_accumulate_rows_sampled(reduce):
    """8 ranks x 2^25: fp32 accumulators (here N(0, 1), so that the addition
    is not a copy) plus a bf16 micro-step gradient N(0, 1e-3^2) seeded r;
    with reduce, the same pass all-reduces (AVG) the sums in ring order."""
    n, count = 8, 1 << 25
    acc = ranks(n, count, torch.float32, 1.0, 500)
    grads = ranks(n, count, torch.bfloat16, 1e-3, 0)
    idx = sample_idx(count, seed=6 + reduce, k=1 << 18)
    a0 = gather(acc, idx, "f32")
    g0 = gather(grads, idx, "bf16")
    sums = np.empty_like(a0)
    for r in range(n):
        col = a0[:, r].copy()
        O.accumulate(col, g0[:, r].copy(), "bf16")
        sums[:, r] = col
    if reduce:
        L = count // n
        want = O.fold_columns(sums, (idx.cpu().numpy() // L).astype(np.int32), "f32", "avg", "f32")
        cr.cr_all_reduce_accumulate(acc, count, grads, "bf16", "avg")
    else:
        cr.cr_accumulate(acc, count, grads, "bf16")
    torch.cuda.synchronize()
    got = gather(acc, idx, "f32")
    for r in range(n):
        assert_match(got[:, r].copy(), want if reduce else sums[:, r].copy(), "f32", f"rank {r}")
    del acc, grads
    torch.cuda.empty_cache()


@pytest.mark.parametrize("api", ["host", "staged"])
def test_all_reduce_from_host_memory_full_sampled(api):
    """The benchmark's end-to-end leg: 8 x 64 MiB bf16 rank buffers in
    pinned host memory, all-reduced AVG by cr_all_reduce_host (the kernel
    reads and writes host memory) or cr_all_reduce_staged (copy engines,
    sliced over three streams, 2^22-element slices as benchmarked)."""
    n, count = 8, 1 << 25
    dev_bufs = ranks(n, count, torch.bfloat16, 0.02, 0)
    host_in = [b.cpu().pin_memory() for b in dev_bufs]
    host_out = [torch.empty(count, dtype=torch.bfloat16).pin_memory() for _ in range(n)]
    idx = sample_idx(count, seed=8, k=1 << 18)
    L = count // n
    want = O.fold_columns(gather(dev_bufs, idx, "bf16"), (idx.cpu().numpy() // L).astype(np.int32),
                          "bf16", "avg", "bf16")
    if api == "host":
        cr.cr_all_reduce_host(host_in, host_out, count, "bf16", "avg")
    else:
        up, down = torch.cuda.Stream(), torch.cuda.Stream()
        cr.cr_all_reduce_staged(host_in, host_out, dev_bufs, count, "bf16", "avg", 1 << 22,
                                torch.cuda.current_stream(), up, down)
    torch.cuda.synchronize()
    hidx = idx.cpu()
    for r in range(n):
        got = host_out[r][hidx].view(torch.int16).numpy().view(np.uint16).copy()
        assert_match(got, want, "bf16", f"{api} rank {r}")
    for r in range(1, n):
        assert torch.equal(host_out[r].view(torch.int16), host_out[0].view(torch.int16))
    del dev_bufs, host_in, host_out
    torch.cuda.empty_cache()

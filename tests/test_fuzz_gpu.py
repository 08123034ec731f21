"""Seeded random cases for every collective, through the C ABI, against the
oracle.  Unlike the structured parity tests, each rank's buffer gets its own
element offset inside its allocation (0, 1, 2, 3, 8, 16, 17 ...), so a call
mixes 32-byte, 16-byte and unaligned buffers and must take the widest path
that all of them allow; rank counts, sizes (around vector and chunk
boundaries), dtype pairs, ops and in-place forms are drawn too.  Same bar
as the parity tests: bitwise equality with the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
from fsdp_emulated_ranks_gb300 import build as libbuild
from fsdp_emulated_ranks_gb300 import cr
from fsdp_emulated_ranks_gb300 import inputs as I
from gpu_util import Guarded, assert_clipped_match, assert_match, to_dev, to_host

pytestmark = pytest.mark.gpu

PAIRS = [("f32", "sum", "f32"), ("bf16", "avg", "bf16"), ("bf16", "avg", "f32"),
         ("i32", "sum", "i32"), ("f32", "avg", "f32"), ("bf16", "sum", "bf16")]
OFFSETS = [0, 0, 0, 1, 2, 3, 8, 16, 17]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    libbuild.build()
    cr.lib()


def draw_count(rng, n):
    base = int(rng.choice([0, 1, 7, 16 * n, 32 * n * 5, 1000, 4099, 16 * n * 37]))
    return max(0, base + int(rng.integers(-3, 4)))


def host_inputs(n, count, dt, seed):
    return I.host_rank_buffers(n, count, dt, std=0.02 if dt == "bf16" else 1.0, seed0=seed)


def offs(rng, k, dt):
    """Element offsets of k buffers inside their allocations (element
    alignment always holds; 16- and 32-byte alignment only for some)."""
    return [int(rng.choice(OFFSETS)) for _ in range(k)]


@pytest.mark.parametrize("case", range(200))
def test_fuzz_reduce_scatter_all_reduce(case):
    rng = np.random.default_rng(1000 + case)
    n = int(rng.integers(1, 13))
    dt, op, out = PAIRS[int(rng.integers(len(PAIRS)))]
    count = draw_count(rng, n)
    host = host_inputs(n, count, dt, seed=case)
    oi, oo = offs(rng, n, dt), offs(rng, n, out)
    # reduce-scatter
    want, _ = O.ring_reduce_scatter(host, dt, op, out)
    bufs = [to_dev(x, dt, o) for x, o in zip(host, oi)]
    shards = [Guarded(w.size, out, o) for w, o in zip(want, oo)]
    cr.cr_reduce_scatter(bufs, count, dt, op, [s.ptr() for s in shards], out)
    torch.cuda.synchronize()
    for j in range(n):
        shards[j].check()
        assert_match(shards[j].host(), want[j], out, f"RS n={n} count={count} offs={oi}/{oo} j={j}")
    # all-reduce, in place when the dtypes allow and the draw says so
    want, _ = O.ring_all_reduce(host, dt, op, out)
    if dt == out and rng.random() < 0.5:
        cr.cr_all_reduce(bufs, count, dt, op, bufs, out)
        torch.cuda.synchronize()
        got = [to_host(b, out) for b in bufs]
    else:
        outs = [Guarded(count, out, o) for o in oo]
        cr.cr_all_reduce(bufs, count, dt, op, [x.ptr() for x in outs], out)
        torch.cuda.synchronize()
        for x in outs:
            x.check()
        got = [x.host() for x in outs]
    for r in range(n):
        assert_match(got[r], want[r], out, f"AR n={n} count={count} offs={oi}/{oo} r={r}")


@pytest.mark.parametrize("case", range(120))
def test_fuzz_all_gather_and_wire(case):
    rng = np.random.default_rng(2000 + case)
    n = int(rng.integers(1, 13))
    dt = ["f32", "bf16", "i32"][int(rng.integers(3))]
    count = draw_count(rng, n)
    shards = []
    for j in range(n):
        lo, hi = O.chunk_bounds(count, n, j)
        shards.append(host_inputs(1, hi - lo, dt, seed=case * 31 + j)[0])
    want, _ = O.ring_all_gather(shards, count, dt)
    osh, ob = offs(rng, n, dt), offs(rng, n, dt)
    d_sh = [to_dev(s, dt, o) if s.size else 0 for s, o in zip(shards, osh)]
    outs = [Guarded(count, dt, o) for o in ob]
    cr.cr_all_gather(d_sh, count, dt, [o.ptr() for o in outs])
    torch.cuda.synchronize()
    for r in range(n):
        outs[r].check()
        assert_match(outs[r].host(), want[r], dt, f"AG n={n} count={count} offs={osh}/{ob}")
    # bf16-wire all-reduce on float inputs
    fdt, op, fout = PAIRS[int(rng.choice([0, 1, 2, 4, 5]))]
    host = host_inputs(n, count, fdt, seed=case + 77)
    want = O.ring_all_reduce_wire(host, fdt, op, "bf16", fout)
    oi, oo = offs(rng, n, fdt), offs(rng, n, fout)
    bufs = [to_dev(x, fdt, o) for x, o in zip(host, oi)]
    outs = [Guarded(count, fout, o) for o in oo]
    cr.cr_all_reduce_wire(bufs, count, fdt, op, "bf16", [o.ptr() for o in outs], fout)
    torch.cuda.synchronize()
    for r in range(n):
        outs[r].check()
        assert_match(outs[r].host(), want[r], fout, f"wire n={n} count={count} offs={oi}/{oo}")


@pytest.mark.parametrize("case", range(120))
def test_fuzz_hsdp(case):
    rng = np.random.default_rng(3000 + case)
    R, S = int(rng.integers(1, 5)), int(rng.integers(1, 6))
    n = R * S
    dt, op, out = PAIRS[int(rng.integers(len(PAIRS)))]
    count = draw_count(rng, S)
    host = host_inputs(n, count, dt, seed=case * 7)
    want = O.hsdp_reduce_scatter(host, R, S, dt, op, out)
    oi, oo = offs(rng, n, dt), offs(rng, n, out)
    bufs = [to_dev(x, dt, o) for x, o in zip(host, oi)]
    shards = [Guarded(w.size, out, o) for w, o in zip(want, oo)]
    cr.cr_hsdp_reduce_scatter(bufs, R, S, count, dt, op, [s.ptr() for s in shards], out)
    torch.cuda.synchronize()
    for q in range(n):
        shards[q].check()
        assert_match(shards[q].host(), want[q], out, f"{R}x{S} count={count} offs={oi}/{oo} q={q}")


@pytest.mark.parametrize("case", range(100))
def test_fuzz_fused_buckets_and_accumulate(case):
    rng = np.random.default_rng(4000 + case)
    n = int(rng.integers(1, 9))
    dt = ["bf16", "f32"][int(rng.integers(2))]
    es = 2 if dt == "bf16" else 4
    T = int(rng.integers(1, 25))
    numels = [int(x) for x in rng.integers(0, 3000, T)]
    cap = int(rng.integers(64, 20000))
    plan = cr.cr_bucket_plan(numels, es, cap)
    oplan = O.bucket_plan(numels, es, cap)
    host = [[host_inputs(1, k, dt, seed=case * 1000 + r * 50 + t)[0] for t, k in enumerate(numels)]
            for r in range(n)]
    want = O.bucketed_all_reduce(oplan, host, dt, "avg")
    ot = offs(rng, n * T, dt)
    dev_t = [to_dev(host[r][t], dt, ot[r * T + t]) if numels[t] else 0
             for r in range(n) for t in range(T)]
    cr.cr_bucket_all_reduce_fused(plan, n, dev_t, dt, "avg")
    torch.cuda.synchronize()
    for r in range(n):
        for t in range(T):
            if numels[t]:
                assert_match(to_host(dev_t[r * T + t], dt), want[r][t], dt,
                             f"fused n={n} T={T} cap={cap} r={r} t={t}")
    # fused accumulate + all-reduce: fp32 accumulators, grads of dt
    count = draw_count(rng, n)
    acc = host_inputs(n, count, "f32", seed=case + 5)
    g = host_inputs(n, count, dt, seed=case + 9)
    sums = [a.copy() for a in acc]
    for a, x in zip(sums, g):
        O.accumulate(a, x, dt)
    want, _ = O.ring_all_reduce(sums, "f32", "sum")
    oa, og = offs(rng, n, "f32"), offs(rng, n, dt)
    d_acc = [to_dev(x, "f32", o) for x, o in zip(acc, oa)]
    d_g = [to_dev(x, dt, o) for x, o in zip(g, og)]
    cr.cr_all_reduce_accumulate(d_acc, count, d_g, dt, "sum")
    torch.cuda.synchronize()
    for r in range(n):
        assert_match(to_host(d_acc[r], "f32"), want[r], "f32", f"acc n={n} count={count} offs={oa}/{og}")


@pytest.mark.parametrize("case", range(100))
def test_fuzz_fsdp_step(case):
    """FSDP step, plain or clipped, with every grad, param and state buffer
    at its own offset; two consecutive steps (t = 1, 2)."""
    rng = np.random.default_rng(5000 + case)
    n = int(rng.integers(1, 11))
    count = draw_count(rng, n)
    clipped = bool(rng.random() < 0.5)
    grads0 = I.host_rank_buffers(n, count, "bf16", std=1e-3, seed0=case)
    master_full = I.np_normal_f32(count, 0.02, 77 + case)
    bounds = [O.chunk_bounds(count, n, j) for j in range(n)]
    master = [master_full[a:b].copy() for a, b in bounds]
    m = [np.zeros(b - a, np.float32) for a, b in bounds]
    v = [np.zeros(b - a, np.float32) for a, b in bounds]
    ostate = offs(rng, 3 * n, "f32")
    d_state = [Guarded(x.size, "f32", o) for x, o in zip(master + m + v, ostate)]
    for gg, x in zip(d_state, master + m + v):
        if x.size:
            gg.view.copy_(to_dev(x, "f32"))
    d_master, d_m, d_v = d_state[:n], d_state[n:2 * n], d_state[2 * n:]
    d_p = [Guarded(count, "bf16", o) for o in offs(rng, n, "bf16")]
    ws = torch.empty(cr.cr_fsdp_clip_workspace_bytes() // 8, dtype=torch.float64, device="cuda")
    max_norm = 1e-3
    for step in (1, 2):
        grads = grads0 if step == 1 else I.host_rank_buffers(n, count, "bf16", std=1e-3,
                                                             seed0=case + 500)
        d_g = [to_dev(x, "bf16", o) for x, o in zip(grads, offs(rng, n, "bf16"))]
        cfg = O.AdamWConfig(step=step)
        if clipped:
            _, want_norm = O.fsdp_step_clipped(grads, [x.copy() for x in master],
                                               [x.copy() for x in m], [x.copy() for x in v], cfg,
                                               max_norm)
            cr.cr_fsdp_step_clipped(d_g, count, [x.ptr() for x in d_master], [x.ptr() for x in d_m],
                                    [x.ptr() for x in d_v], cr.adamw_cfg(step=step), max_norm, ws,
                                    ws.numel() * 8, [x.ptr() for x in d_p], None)
        else:
            want_p = O.fsdp_step(grads, master, m, v, cfg)
            cr.cr_fsdp_step(d_g, count, [x.ptr() for x in d_master], [x.ptr() for x in d_m],
                            [x.ptr() for x in d_v], cr.adamw_cfg(step=step), [x.ptr() for x in d_p])
        torch.cuda.synchronize()
        for gg in d_state + d_p:
            gg.check()
        if clipped:
            got_state = [[x.host() for x in t] for t in (d_master, d_m, d_v)]
            assert_clipped_match(got_state, [x.host() for x in d_p], grads, master, m, v, cfg,
                                 max_norm, want_norm, f"n={n} count={count} step {step}")
            continue
        for j in range(n):
            for gg, ref, name in ((d_master, master, "master"), (d_m, m, "m"), (d_v, v, "v")):
                assert_match(gg[j].host(), ref[j], "f32", f"{name}[{j}] step {step}")
        for r in range(n):
            assert_match(d_p[r].host(), want_p[r], "bf16", f"n={n} count={count} params[{r}]")


@pytest.mark.parametrize("case", range(120))
def test_fuzz_range_forms(case):
    """Range all-reduce and reduce-scatter over a random slab [lo, hi) of a
    random workload, every slab buffer and shard part at its own offset:
    the slab's elements of the oracle's whole-buffer results, bit for bit,
    with canaries intact."""
    rng = np.random.default_rng(9000 + case)
    n = int(rng.integers(1, 13))
    dt, op, out = PAIRS[int(rng.integers(len(PAIRS)))]
    count = max(1, draw_count(rng, n))
    lo = int(rng.integers(0, count + 1))
    hi = int(rng.integers(lo, count + 1))
    host = host_inputs(n, count, dt, seed=500 + case)
    L = O.chunk_len(count, n)
    oi, oo = offs(rng, n, dt), offs(rng, n, out)
    ar, _ = O.ring_all_reduce(host, dt, op, out)
    slab = [to_dev(np.ascontiguousarray(x[lo:hi]), dt, o) if hi > lo else 0
            for x, o in zip(host, oi)]
    outs = [Guarded(hi - lo, out, o) for o in oo]
    cr.cr_all_reduce_range(slab, count, lo, hi, dt, op, [g.ptr() for g in outs], out)
    torch.cuda.synchronize()
    for r in range(n):
        outs[r].check()
        assert_match(outs[r].host(), ar[r][lo:hi], out, f"AR range n={n} [{lo},{hi}) of {count}")
    rs, _ = O.ring_reduce_scatter(host, dt, op, out)
    parts = []
    for j in range(n):
        a, b = max(lo, j * L), min(hi, (j + 1) * L, count)
        parts.append((a - j * L, max(0, b - a)))
    sh = [Guarded(k, out, o) for (_, k), o in zip(parts, offs(rng, n, out))]
    cr.cr_reduce_scatter_range(slab, count, lo, hi, dt, op, [g.ptr() for g in sh], out)
    torch.cuda.synchronize()
    for j, ((a, k), g) in enumerate(zip(parts, sh)):
        g.check()
        assert_match(g.host(), rs[j][a:a + k], out, f"RS range n={n} shard {j}")


@pytest.mark.parametrize("case", range(100))
def test_fuzz_fsdp2(case):
    """FSDP2 over a random parameter set -- dim0 from 0 to a few times N
    (uneven, empty and one-row shards), rows of 1 to 200 elements -- with
    every grad, param and state buffer at its own offset, so parameters mix
    the vector and the element-wise paths in one launch.  Half the cases
    step through a plan's table (one plan, two steps), half pass the
    pointers per call; both must equal the oracle bitwise at t = 1 and 2."""
    rng = np.random.default_rng(11000 + case)
    n = int(rng.integers(1, 11))
    P = int(rng.integers(1, 13))
    shapes = []
    for _ in range(P):
        d0 = int(rng.choice([0, 1, max(1, n - 1), n, 2 * n + 1, int(rng.integers(1, 4 * n + 8))]))
        row = int(rng.choice([1, 3, 8, 16, 64, 100, int(rng.integers(1, 201))]))
        shapes.append((d0, row))
    planned = bool(rng.random() < 0.5)
    cfgs = [O.AdamWConfig(step=1), O.AdamWConfig(step=2)]
    master, m, v = [], [], []
    for p, (d0, row) in enumerate(shapes):
        Lr = -(-d0 // n) if d0 else 0
        ks = [max(0, min(d0, (j + 1) * Lr) - min(d0, j * Lr)) * row for j in range(n)]
        master.append([I.np_normal_f32(k, 0.02, 100 * case + 10 * p + j) for j, k in enumerate(ks)])
        m.append([np.zeros(k, np.float32) for k in ks])
        v.append([np.zeros(k, np.float32) for k in ks])
    d_state = [[Guarded(x.size, "f32", o) if x.size else None
                for x, o in zip([x for row in t for x in row], offs(rng, P * n, "f32"))]
               for t in (master, m, v)]
    for dd, t in zip(d_state, (master, m, v)):
        for gg, x in zip(dd, [x for row in t for x in row]):
            if gg is not None:
                gg.view.copy_(to_dev(x, "f32"))
    ptrs = [[gg.ptr() if gg is not None else 0 for gg in dd] for dd in d_state]
    d_p = [Guarded(d0 * row, "bf16", o) if d0 * row else None
           for (d0, row) in shapes for o in offs(rng, n, "bf16")]
    p_ptrs = [gg.ptr() if gg is not None else 0 for gg in d_p]
    # the gradient buffers stay put across the two steps: refilled in place
    g_off = offs(rng, P * n, "bf16")
    d_g = [Guarded(d0 * row, "bf16", o) if d0 * row else None
           for (d0, row), o in zip([s for s in shapes for _ in range(n)], g_off)]
    g_ptrs = [gg.ptr() if gg is not None else 0 for gg in d_g]
    plan = table = None
    if planned:
        plan = cr.cr_fsdp2_plan_create(shapes, n, g_ptrs, *ptrs, p_ptrs)
        table = torch.empty(max(16, plan.table_bytes), dtype=torch.uint8, device="cuda")
        cr.cr_fsdp2_plan_upload(plan, table)
    for step, cfg in ((1, cfgs[0]), (2, cfgs[1])):
        grads = [[I.np_to_bf16_bits(I.np_normal_f32(d0 * row, 1e-3, 7000 * step + 50 * case
                                                    + 7 * p + r)) for r in range(n)]
                 for p, (d0, row) in enumerate(shapes)]
        for gg, x in zip(d_g, [x for row in grads for x in row]):
            if gg is not None:
                gg.view.copy_(to_dev(x, "bf16"))
        want_p = O.fsdp2_step(shapes, grads, master, m, v, cfg)
        if planned:
            cr.cr_fsdp2_step_planned(plan, table, cr.adamw_cfg(step=step))
        else:
            cr.cr_fsdp2_step(shapes, n, g_ptrs, *ptrs, cr.adamw_cfg(step=step), p_ptrs)
        torch.cuda.synchronize()
        what = f"n={n} shapes={shapes} planned={planned} step {step}"
        for dd, t, name in zip(d_state, (master, m, v), ("master", "m", "v")):
            for gg, x in zip(dd, [x for row in t for x in row]):
                if gg is not None:
                    gg.check()
                    assert_match(gg.host(), x, "f32", f"{name}: {what}")
        for q, gg in enumerate(d_p):
            if gg is not None:
                gg.check()
                assert_match(gg.host(), want_p[q // n][q % n], "bf16", f"params[{q}]: {what}")


@pytest.mark.parametrize("case", range(100))
def test_fuzz_fsdp_step_range(case):
    """The FSDP step over a random slab [lo, hi) of a random workload, every
    slab buffer and shard part at its own offset: the slab's elements of
    the oracle's whole step (state and params), bit for bit, with canaries
    intact."""
    rng = np.random.default_rng(13000 + case)
    n = int(rng.integers(1, 11))
    count = max(1, draw_count(rng, n))
    lo = int(rng.integers(0, count + 1))
    hi = int(rng.integers(lo, count + 1))
    L = O.chunk_len(count, n)
    grads = I.host_rank_buffers(n, count, "bf16", std=1e-3, seed0=600 + case)
    bounds = [O.chunk_bounds(count, n, j) for j in range(n)]
    master = [I.np_normal_f32(b - a, 0.02, 700 + case + j) for j, (a, b) in enumerate(bounds)]
    m = [np.zeros(b - a, np.float32) for a, b in bounds]
    v = [np.zeros(b - a, np.float32) for a, b in bounds]
    parts = []  # (first shard element in the slab, elements) per shard
    for j in range(n):
        a, b = max(lo, j * L), min(hi, (j + 1) * L, count)
        parts.append((a - j * L, max(0, b - a)))
    d_state = []
    for t in (master, m, v):
        row = []
        for (a, k), x, o in zip(parts, t, offs(rng, n, "f32")):
            g = Guarded(k, "f32", o) if k else None
            if g is not None:
                g.view.copy_(to_dev(np.ascontiguousarray(x[a:a + k]), "f32"))
            row.append(g)
        d_state.append(row)
    d_g = [to_dev(np.ascontiguousarray(x[lo:hi]), "bf16", o) if hi > lo else 0
           for x, o in zip(grads, offs(rng, n, "bf16"))]
    d_p = [Guarded(hi - lo, "bf16", o) for o in offs(rng, n, "bf16")]
    want_p = O.fsdp_step(grads, master, m, v, O.AdamWConfig())
    cr.cr_fsdp_step_range(d_g, count, lo, hi,
                          *[[g.ptr() if g is not None else 0 for g in row] for row in d_state],
                          cr.adamw_cfg(), [g.ptr() for g in d_p])
    torch.cuda.synchronize()
    what = f"n={n} [{lo},{hi}) of {count}"
    for row, t, name in zip(d_state, (master, m, v), ("master", "m", "v")):
        for j, (g, (a, k)) in enumerate(zip(row, parts)):
            if g is not None:
                g.check()
                assert_match(g.host(), t[j][a:a + k], "f32", f"{name}[{j}] {what}")
    for r in range(n):
        d_p[r].check()
        assert_match(d_p[r].host(), want_p[r][lo:hi], "bf16", f"params[{r}] {what}")


@pytest.mark.parametrize("case", range(100))
def test_fuzz_bucket_pack_all_reduce_unpack(case):
    """The unfused DDP pipeline -- pack, per-bucket all-reduce, unpack --
    over a random plan, with every tensor and every bucket at its own
    offset (the copies then take the funnel-shift and element paths as well
    as the vector one): the buckets after pack equal the oracle's pack bit
    for bit, and the tensors after unpack the oracle's bucketed all-reduce,
    with canaries intact."""
    rng = np.random.default_rng(15000 + case)
    n = int(rng.integers(1, 9))
    dt = ["bf16", "f32", "i32"][int(rng.integers(3))]
    op = "sum" if dt == "i32" else ["sum", "avg"][int(rng.integers(2))]
    es = 2 if dt == "bf16" else 4
    T = int(rng.integers(1, 31))
    numels = [int(x) if rng.random() > 0.1 else 0 for x in rng.integers(1, 3000, T)]
    cap = int(rng.integers(64, 20000))
    plan = cr.cr_bucket_plan(numels, es, cap)
    oplan = O.bucket_plan(numels, es, cap)
    B = plan.nbuckets
    assert list(plan.bucket_numel) == [int(x) for x in oplan.bucket_numel]
    host = [[host_inputs(1, k, dt, seed=case * 1000 + r * 50 + t)[0] for t, k in enumerate(numels)]
            for r in range(n)]
    ot = offs(rng, n * T, dt)
    dev_t = [to_dev(host[r][t], dt, ot[r * T + t]) if numels[t] else 0
             for r in range(n) for t in range(T)]
    d_b = [Guarded(int(k), dt, o) for _ in range(n)
           for k, o in zip(plan.bucket_numel, offs(rng, B, dt))]
    cr.cr_bucket_pack(plan, n, dev_t, [g.ptr() for g in d_b])
    torch.cuda.synchronize()
    want_b = O.bucket_pack(oplan, host)
    what = f"n={n} {dt} T={T} cap={cap}"
    for r in range(n):
        for b in range(B):
            d_b[r * B + b].check()
            assert_match(d_b[r * B + b].host(), want_b[r][b], dt, f"pack r={r} b={b} {what}")
    cr.cr_bucket_all_reduce(plan, n, [g.ptr() for g in d_b], dt, op)
    d_out = [Guarded(k, dt, o) for _ in range(n) for k, o in zip(numels, offs(rng, T, dt))]
    cr.cr_bucket_unpack(plan, n, [g.ptr() for g in d_b], [g.ptr() for g in d_out])
    torch.cuda.synchronize()
    want = O.bucketed_all_reduce(oplan, host, dt, op)
    for r in range(n):
        for t in range(T):
            g = d_out[r * T + t]
            g.check()
            assert_match(g.host(), want[r][t], dt, f"unpack r={r} t={t} {what}")

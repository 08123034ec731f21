"""The range forms of the collectives and of the FSDP step, through the C ABI.

A slab split hands each of G GPUs the elements [begin, end) of every rank
buffer; the range calls reduce them with the whole buffer's chunking, so the
G slab results, put side by side, must be the whole-buffer call's result bit
for bit (and the oracle's).  Here the G slabs run one after another on one
GPU, each in buffers of its own, as each GPU would hold only its slab.
Slabs come from cr_slab_range (whole chunks for G <= N, 16-element
boundaries beyond) and from seeded random cuts that split chunks at odd
elements, so the vector, 16-byte and element-wise paths all run.
"""
import numpy as np
import pytest
import torch

import oracle as O
from fsdp_emulated_ranks_gb300 import build as libbuild
from fsdp_emulated_ranks_gb300 import cr
from fsdp_emulated_ranks_gb300 import inputs as I
from gpu_util import assert_match, to_dev, to_host

pytestmark = pytest.mark.gpu

TDT = {"f32": torch.float32, "bf16": torch.bfloat16, "i32": torch.int32}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    libbuild.build()
    cr.lib()


def cuts(count, n, G, kind, seed):
    """G slabs partitioning [0, count): by cr_slab_range, or random cuts."""
    if kind == "slab":
        return [cr.cr_slab_range(count, n, G, g) for g in range(G)]
    rng = np.random.default_rng(seed)
    inner = sorted(rng.choice(np.arange(1, count), size=min(G - 1, count - 1), replace=False))
    b = [0] + [int(x) for x in inner] + [count]
    while len(b) < G + 1:  # fewer elements than slabs: empty slabs at the end
        b.append(count)
    return list(zip(b[:-1], b[1:]))


def shard_part(count, n, j, lo, hi):
    """Shard j's part inside [lo, hi): (first shard element, length)."""
    L = O.chunk_len(count, n)
    a, b = max(lo, j * L), min(hi, (j + 1) * L, count)
    return (a - j * L, b - a) if b > a else (0, 0)


CASES = [(8, 8 * 4096), (8, 8 * 4096 + 13), (4, 1000), (3, 3 * 40 + 1), (16, 5000), (5, 17)]


@pytest.mark.parametrize("n,count", CASES)
@pytest.mark.parametrize("G", [2, 3, 8])
@pytest.mark.parametrize("kind", ["slab", "random"])
@pytest.mark.parametrize("pair", [("bf16", "avg", "bf16"), ("f32", "sum", "f32"),
                                  ("bf16", "avg", "f32"), ("i32", "sum", "i32")])
def test_all_reduce_slabs_equal_whole_call(n, count, G, kind, pair):
    dt, op, out = pair
    host = I.host_rank_buffers(n, count, dt, std=0.02 if dt == "bf16" else 1.0, seed0=count + G)
    want, _ = O.ring_all_reduce(host, dt, op, out)
    whole = [torch.empty(count, dtype=TDT[out], device="cuda") for _ in range(n)]
    cr.cr_all_reduce([to_dev(x, dt) for x in host], count, dt, op, whole, out)
    got = [np.zeros(count, want[0].dtype) for _ in range(n)]
    for g, (lo, hi) in enumerate(cuts(count, n, G, kind, seed=G * 31 + count)):
        slab_in = [to_dev(np.ascontiguousarray(x[lo:hi]), dt) if hi > lo else 0 for x in host]
        slab_out = [torch.empty(hi - lo, dtype=TDT[out], device="cuda") for _ in range(n)]
        cr.cr_all_reduce_range(slab_in, count, lo, hi, dt, op, slab_out, out)
        torch.cuda.synchronize()
        for r in range(n):
            got[r][lo:hi] = to_host(slab_out[r], out)
    for r in range(n):
        assert_match(got[r], to_host(whole[r], out), out, f"rank {r} vs whole call")
        assert_match(got[r], want[r], out, f"rank {r} vs oracle")


@pytest.mark.parametrize("n,count", CASES)
@pytest.mark.parametrize("G", [2, 3, 8])
@pytest.mark.parametrize("kind", ["slab", "random"])
@pytest.mark.parametrize("pair", [("bf16", "avg", "bf16"), ("f32", "sum", "f32"),
                                  ("bf16", "avg", "f32")])
def test_reduce_scatter_slabs_equal_whole_call(n, count, G, kind, pair):
    dt, op, out = pair
    host = I.host_rank_buffers(n, count, dt, std=0.02 if dt == "bf16" else 1.0, seed0=7 + G)
    want, _ = O.ring_reduce_scatter(host, dt, op, out)
    got = [np.zeros(w.size, w.dtype) for w in want]
    for g, (lo, hi) in enumerate(cuts(count, n, G, kind, seed=G * 17 + count)):
        slab_in = [to_dev(np.ascontiguousarray(x[lo:hi]), dt) if hi > lo else 0 for x in host]
        parts = [shard_part(count, n, j, lo, hi) for j in range(n)]
        outs = [torch.empty(k, dtype=TDT[out], device="cuda") if k else None for _, k in parts]
        cr.cr_reduce_scatter_range(slab_in, count, lo, hi, dt, op,
                                   [o if o is not None else 0 for o in outs], out)
        torch.cuda.synchronize()
        for j, ((a, k), o) in enumerate(zip(parts, outs)):
            if k:
                got[j][a:a + k] = to_host(o, out)
    for j in range(n):
        assert_match(got[j], want[j], out, f"shard {j}")


@pytest.mark.parametrize("n,count", [(8, 8 * 4096), (8, 8 * 4096 + 13), (4, 1000), (16, 5000)])
@pytest.mark.parametrize("G", [2, 3, 8])
def test_in_place_slabs(n, count, G):
    """In place within each slab: the all-reduce overwrites the slab, the
    reduce-scatter writes shard j's part where it sits in rank j's slab."""
    host = I.host_rank_buffers(n, count, "bf16", std=0.02, seed0=3)
    want_ar, _ = O.ring_all_reduce(host, "bf16", "avg")
    want_rs, _ = O.ring_reduce_scatter(host, "bf16", "avg")
    L = O.chunk_len(count, n)
    for lo, hi in cuts(count, n, G, "random", seed=count):
        if hi == lo:
            continue
        slab = [to_dev(np.ascontiguousarray(x[lo:hi]), "bf16") for x in host]
        cr.cr_all_reduce_range(slab, count, lo, hi, "bf16", "avg", slab, "bf16")
        slab2 = [to_dev(np.ascontiguousarray(x[lo:hi]), "bf16") for x in host]
        parts = [shard_part(count, n, j, lo, hi) for j in range(n)]
        shards = [slab2[j][max(lo, j * L) - lo:] if k else 0 for j, (a, k) in enumerate(parts)]
        cr.cr_reduce_scatter_range(slab2, count, lo, hi, "bf16", "avg", shards, "bf16")
        torch.cuda.synchronize()
        for r in range(n):
            assert_match(to_host(slab[r], "bf16"), want_ar[r][lo:hi], "bf16", "AR in place")
        for j, (a, k) in enumerate(parts):
            if k:
                s = max(lo, j * L) - lo
                assert_match(to_host(slab2[j][s:s + k], "bf16"), want_rs[j][a:a + k], "bf16",
                             f"RS in place shard {j}")


@pytest.mark.parametrize("n,count", [(8, 8 * 8 * 300), (8, 8 * 8 * 300 + 5), (3, 3 * 8 * 40 + 7),
                                     (5, 203)])
@pytest.mark.parametrize("G", [2, 3, 8])
@pytest.mark.parametrize("kind", ["slab", "random"])
def test_fsdp_step_slabs_equal_whole_call(n, count, G, kind):
    """The FSDP step over G slabs, two steps in a row, against the oracle's
    whole-buffer step: state parts and parameters bitwise."""
    bounds = [O.chunk_bounds(count, n, j) for j in range(n)]
    master = [I.np_normal_f32(b - a, 0.02, 2000 + j) for j, (a, b) in enumerate(bounds)]
    m = [np.zeros(b - a, np.float32) for a, b in bounds]
    v = [np.zeros(b - a, np.float32) for a, b in bounds]
    slabs = cuts(count, n, G, kind, seed=G + count)
    # each slab's own buffers: grads/params slabs and the state parts it owns
    dev = []
    for lo, hi in slabs:
        parts = [shard_part(count, n, j, lo, hi) for j in range(n)]
        st = [[to_dev(np.ascontiguousarray(x[j][a:a + k]), "f32") if k else 0
               for j, (a, k) in enumerate(parts)] for x in (master, m, v)]
        par = [torch.empty(hi - lo, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
        dev.append((parts, st, par))
    for step in (1, 2):
        grads = I.host_rank_buffers(n, count, "bf16", std=1e-3, seed0=1000 + 50 * step)
        cfg = O.AdamWConfig(step=step)
        want_p = O.fsdp_step(grads, master, m, v, cfg)
        for (lo, hi), (parts, st, par) in zip(slabs, dev):
            g = [to_dev(np.ascontiguousarray(x[lo:hi]), "bf16") if hi > lo else 0 for x in grads]
            cr.cr_fsdp_step_range(g, count, lo, hi, *st, cr.adamw_cfg(step=step), par)
        torch.cuda.synchronize()
        for (lo, hi), (parts, st, par) in zip(slabs, dev):
            for r in range(n):
                assert_match(to_host(par[r], "bf16"), want_p[r][lo:hi], "bf16",
                             f"params rank {r} slab [{lo}, {hi}) step {step}")
            for q, ref in enumerate((master, m, v)):
                for j, (a, k) in enumerate(parts):
                    if k:
                        assert_match(to_host(st[q][j], "f32"), ref[j][a:a + k], "f32",
                                     f"state {q} owner {j} step {step}")


def test_full_range_is_the_whole_call():
    """begin = 0, end = count: the range call is the whole-buffer call."""
    n, count = 8, 8 * 4096 + 5
    host = I.host_rank_buffers(n, count, "bf16", std=0.02, seed0=9)
    a = [to_dev(x, "bf16") for x in host]
    b = [to_dev(x, "bf16") for x in host]
    cr.cr_all_reduce(a, count, "bf16", "avg", a, "bf16")
    cr.cr_all_reduce_range(b, count, 0, count, "bf16", "avg", b, "bf16")
    torch.cuda.synchronize()
    for x, y in zip(a, b):
        assert torch.equal(x.view(torch.int16), y.view(torch.int16))


def test_range_rejects_bad_bounds():
    n, count = 4, 100
    bufs = [torch.empty(count, dtype=torch.float32, device="cuda") for _ in range(n)]
    for lo, hi in ((5, 4), (0, 101), (101, 101)):
        with pytest.raises(cr.CRError) as ei:
            cr.cr_all_reduce_range(bufs, count, lo, hi, "f32", "sum", bufs, "f32")
        assert ei.value.status == 1


@pytest.mark.parametrize("G", [2, 3, 8])
def test_headline_split_into_slabs_full_size(G):
    """The benchmark's --split slab at full size, each slab in buffers of its
    own as on its own GPU: 8 ranks x 2^25 bf16, AVG, in place.  The slabs
    put side by side equal the whole-buffer call on every element of every
    rank, bit for bit (the whole-buffer call is itself checked against the
    oracle at this size in test_fullsize_gpu.py)."""
    n, count = 8, 1 << 25
    bufs = []
    for r in range(n):
        t = torch.empty(count, dtype=torch.bfloat16, device="cuda")
        I.torch_fill_normal_(t, 0.02, r)
        bufs.append(t)
    slabs = [cr.cr_slab_range(count, n, G, g) for g in range(G)]
    parts = [[b[lo:hi].clone() for b in bufs] for lo, hi in slabs]
    cr.cr_all_reduce(bufs, count, "bf16", "avg", bufs, "bf16")
    for (lo, hi), p in zip(slabs, parts):
        cr.cr_all_reduce_range(p, count, lo, hi, "bf16", "avg", p, "bf16")
    torch.cuda.synchronize()
    for r in range(n):
        whole = bufs[r].view(torch.int16)
        for (lo, hi), p in zip(slabs, parts):
            assert torch.equal(p[r].view(torch.int16), whole[lo:hi]), (r, lo, hi)
    del bufs, parts
    torch.cuda.empty_cache()


@pytest.mark.parametrize("G", [2, 8])
def test_fsdp_step_split_into_slabs_large(G):
    """The unclipped FSDP step over 8 x 2^26 parameters split into G slabs,
    each holding its slab of the grads/params and its parts of the owners'
    state: equal, bit for bit, to the whole-buffer step."""
    n, count = 8, 1 << 26
    L = count // n
    grads = []
    for r in range(n):
        t = torch.empty(count, dtype=torch.bfloat16, device="cuda")
        I.torch_fill_normal_(t, 1e-3, 1000 + r)
        grads.append(t)
    master_full = torch.empty(count, dtype=torch.float32, device="cuda")
    I.torch_fill_normal_(master_full, 0.02, 2000)
    state0 = master_full.clone()
    m_full = torch.zeros(count, dtype=torch.float32, device="cuda")
    v_full = torch.zeros(count, dtype=torch.float32, device="cuda")
    params = [torch.empty(count, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    slabs = [cr.cr_slab_range(count, n, G, g) for g in range(G)]
    own = []
    for lo, hi in slabs:
        sg = [g[lo:hi].clone() for g in grads]
        st = []
        for src in (state0, m_full, v_full):
            row = []
            for j in range(n):
                a, b = max(lo, j * L), min(hi, (j + 1) * L)
                row.append(src[a:b].clone() if b > a else 0)
            st.append(row)
        sp = [torch.empty(hi - lo, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
        own.append((sg, st, sp))
    cr.cr_fsdp_step(grads, count, [master_full[j * L:(j + 1) * L] for j in range(n)],
                    [m_full[j * L:(j + 1) * L] for j in range(n)],
                    [v_full[j * L:(j + 1) * L] for j in range(n)], cr.adamw_cfg(), params)
    for (lo, hi), (sg, st, sp) in zip(slabs, own):
        cr.cr_fsdp_step_range(sg, count, lo, hi, *st, cr.adamw_cfg(), sp)
    torch.cuda.synchronize()
    for (lo, hi), (sg, st, sp) in zip(slabs, own):
        for r in range(n):
            assert torch.equal(sp[r].view(torch.int16), params[r][lo:hi].view(torch.int16))
        for q, full in enumerate((master_full, m_full, v_full)):
            for j in range(n):
                a, b = max(lo, j * L), min(hi, (j + 1) * L)
                if b > a:
                    assert torch.equal(st[q][j], full[a:b]), (q, j, lo, hi)
    del grads, params, own
    torch.cuda.empty_cache()


@pytest.mark.parametrize("k", [33, 41, 60])
@pytest.mark.parametrize("n", [3, 8, 64])
def test_range_forms_at_counts_no_buffer_could_hold(k, n):
    """The range calls take slab-local buffers, so a slab of a buffer of
    2^k + 12345 elements per rank (k up to 60) needs only the slab's memory.
    That runs the index arithmetic of the kernels -- the chunk of an element
    (a 64-bit division), its offset inside its shard, the byte offsets from
    the shifted-back pointers -- at element indices far beyond 2^32: a slab
    across the boundary between chunks n/2 - 1 and n/2 and a slab at the
    end of the last chunk.  All-reduce, reduce-scatter (bf16 in, fp32
    shards) and the FSDP step against the oracle, bit for bit."""
    count = (1 << k) + 12345
    L = O.chunk_len(count, n)
    cfg = O.AdamWConfig()
    for lo, hi in ((n // 2 * L - 37, n // 2 * L + 203), (count - 150, count)):
        m = hi - lo
        e = np.arange(m, dtype=object) + lo
        chunk = np.array([int(x // L) for x in e], np.int32)
        host = I.host_rank_buffers(n, m, "bf16", std=0.02, seed0=k * 100 + n)
        vals = np.stack(host, axis=1)
        what = f"count=2^{k}+12345 n={n} [{lo}, {hi})"
        # all-reduce AVG in place
        bufs = [to_dev(x, "bf16") for x in host]
        cr.cr_all_reduce_range(bufs, count, lo, hi, "bf16", "avg", bufs, "bf16")
        torch.cuda.synchronize()
        want = O.fold_columns(vals, chunk, "bf16", "avg", "bf16")
        for r in range(n):
            assert_match(to_host(bufs[r], "bf16"), want, "bf16", f"all-reduce rank {r}, {what}")
        # reduce-scatter to fp32 shard parts
        bufs = [to_dev(x, "bf16") for x in host]
        parts = [shard_part(count, n, j, lo, hi) for j in range(n)]
        outs = [torch.full((max(1, ln),), -1.0, dtype=torch.float32, device="cuda")
                for _, ln in parts]
        cr.cr_reduce_scatter_range(bufs, count, lo, hi, "bf16", "avg",
                                   [o if ln else 0 for o, (_, ln) in zip(outs, parts)], "f32")
        torch.cuda.synchronize()
        gavg = O.fold_columns(vals, chunk, "bf16", "avg", "f32")
        for j, ((a, ln), o) in enumerate(zip(parts, outs)):
            if ln:
                first = j * L + a - lo  # the part's first element, slab-local
                assert_match(to_host(o[:ln], "f32"), gavg[first:first + ln], "f32",
                             f"shard {j}, {what}")
        # the FSDP step: state parts per owner, params slab per rank
        p0 = I.np_normal_f32(m, 0.02, k * 10 + n)
        pm, mm, vm = p0.copy(), np.zeros(m, np.float32), np.zeros(m, np.float32)
        O.adamw(pm, mm, vm, gavg.copy(), cfg)
        st = {name: [] for name in ("master", "m", "v")}
        for j, (a, ln) in enumerate(parts):
            first = j * L + a - lo
            for name, x in (("master", p0), ("m", np.zeros(m, np.float32)),
                            ("v", np.zeros(m, np.float32))):
                st[name].append(to_dev(np.ascontiguousarray(x[first:first + ln]), "f32")
                                if ln else 0)
        grads = [to_dev(x, "bf16") for x in host]
        params = [torch.empty(m, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
        cr.cr_fsdp_step_range(grads, count, lo, hi, st["master"], st["m"], st["v"],
                              cr.adamw_cfg(), params)
        torch.cuda.synchronize()
        for name, ref in (("master", pm), ("m", mm), ("v", vm)):
            got = np.concatenate([to_host(t, "f32") for t in st[name] if isinstance(t, torch.Tensor)])
            assert_match(got, ref, "f32", f"FSDP {name}, {what}")
        for r in range(n):
            assert_match(to_host(params[r], "bf16"), O.f32_to_bf16(pm), "bf16",
                         f"FSDP params rank {r}, {what}")

"""GPU parity: every collective of libcr, called through the C ABI, against
the CPU oracle on the same seeded inputs, element by element.

Every result must be bitwise equal to the oracle's: fp32 / int32 sums and
bucket copies (the kernels fold in the ring's order), bf16 outputs (one
round-to-nearest-even cast of that fp32 value) and the AdamW state
(correctly rounded fp32 operations in the oracle's order).  The clipped
step's norm is summed in another fixed order, so its state is bitwise at a
clip coefficient inside the norm's tolerance window.  Sizes span several 16-byte vectors and CTAs plus a ragged
tail; the unaligned variants start a buffer one element into an allocation
to force the element-wise kernels.  Every output carries canaries that must
survive the call.
"""
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


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    libbuild.build()
    cr.lib()


ESIZE = {"f32": 4, "bf16": 2, "i32": 4}


def eoff(offset, dt):
    """Element offset of a buffer inside its allocation: 0 (32-byte aligned:
    32-byte vector path), "16B" (16- but not 32-byte aligned: 16-byte
    path) or 1 (element-wise path)."""
    return 16 // ESIZE[dt] if offset == "16B" else offset


def sizes(n):
    return [0, 1, 7, 8 * n * 3, 8 * n * 37 + 5, 1000, 4099]


def host_inputs(n, count, dt, seed):
    return I.host_rank_buffers(n, count, dt, std=0.02 if dt == "bf16" else 1.0, seed0=seed)


# ---- reduce-scatter -------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 8, 16, 64])
@pytest.mark.parametrize("pair", PAIRS)
@pytest.mark.parametrize("offset", [0, 1, "16B"])
def test_reduce_scatter(n, pair, offset):
    dt, op, out = pair
    for count in sizes(n):
        host = host_inputs(n, count, dt, seed=n * 100 + count)
        want, _ = O.ring_reduce_scatter(host, dt, op, out)
        bufs = [to_dev(x, dt, eoff(offset, dt)) for x in host]
        shards = [Guarded(w.size, out, eoff(offset, out)) for w in want]
        cr.cr_reduce_scatter(bufs, count, dt, op, [s.ptr() for s in shards], out)
        torch.cuda.synchronize()
        for j in range(n):
            shards[j].check()
            assert_match(shards[j].host(), want[j], out, f"n={n} count={count} shard {j}")
        for r in range(n):  # inputs untouched
            assert to_host(bufs[r], dt).tobytes() == host[r].tobytes()


@pytest.mark.parametrize("n", [2, 4, 8, 5])
@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_reduce_scatter_in_place(n, dt):
    count = 8 * n * 50
    host = host_inputs(n, count, dt, seed=7)
    want, _ = O.ring_reduce_scatter(host, dt, "avg", dt)
    bufs = [to_dev(x, dt) for x in host]
    L = cr.cr_chunk_len(count, n)
    shards = [bufs[j][j * L:(j + 1) * L] for j in range(n)]
    cr.cr_reduce_scatter(bufs, count, dt, "avg", shards, dt)
    torch.cuda.synchronize()
    for j in range(n):
        assert_match(to_host(shards[j], dt), want[j], dt, f"shard {j}")


# ---- all-reduce ----------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 8, 16, 64])
@pytest.mark.parametrize("pair", PAIRS)
@pytest.mark.parametrize("offset", [0, 1, "16B"])
def test_all_reduce(n, pair, offset):
    dt, op, out = pair
    for count in sizes(n):
        host = host_inputs(n, count, dt, seed=n * 300 + count)
        want, _ = O.ring_all_reduce(host, dt, op, out)
        bufs = [to_dev(x, dt, eoff(offset, dt)) for x in host]
        outs = [Guarded(count, out, eoff(offset, out)) for _ in range(n)]
        cr.cr_all_reduce(bufs, count, dt, op, [o.ptr() for o in outs], out)
        torch.cuda.synchronize()
        for r in range(n):
            outs[r].check()
            assert_match(outs[r].host(), want[r], out, f"n={n} count={count} rank {r}")


@pytest.mark.parametrize("n", [2, 3, 4, 8, 13])
@pytest.mark.parametrize("dt,op", [("bf16", "avg"), ("f32", "sum"), ("i32", "sum")])
@pytest.mark.parametrize("count_fn", [lambda n: 8 * n * 64, lambda n: 8 * n * 64 + 3 * n + 1])
def test_all_reduce_in_place(n, dt, op, count_fn):
    """In place, including L not a multiple of the vector width (vectors
    straddling a chunk boundary take the element-wise path)."""
    count = count_fn(n)
    host = host_inputs(n, count, dt, seed=count)
    want, _ = O.ring_all_reduce(host, dt, op, dt)
    bufs = [to_dev(x, dt) for x in host]
    cr.cr_all_reduce(bufs, count, dt, op, bufs, dt)
    torch.cuda.synchronize()
    for r in range(n):
        assert_match(to_host(bufs[r], dt), want[r], dt, f"rank {r}")


# ---- all-gather ----------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 3, 4, 8, 16, 64])
@pytest.mark.parametrize("dt", ["f32", "bf16", "i32"])
@pytest.mark.parametrize("offset", [0, 1, "16B"])
def test_all_gather(n, dt, offset):
    for count in sizes(n):
        shards = []
        for j in range(n):
            lo, hi = O.chunk_bounds(count, n, j)
            shards.append(host_inputs(1, hi - lo, dt, seed=j + count)[0])
        want, _ = O.ring_all_gather(shards, count, dt)
        d_sh = [to_dev(s, dt, eoff(offset, dt)) if s.size else None for s in shards]
        outs = [Guarded(count, dt, eoff(offset, dt)) for _ in range(n)]
        cr.cr_all_gather([s if s is not None else 0 for s in d_sh], count, dt, [o.ptr() for o in outs])
        torch.cuda.synchronize()
        for r in range(n):
            outs[r].check()
            assert_match(outs[r].host(), want[r], dt, f"n={n} count={count} rank {r}")


@pytest.mark.parametrize("n", [2, 4, 8])
def test_all_gather_in_place(n):
    count = 8 * n * 33
    host = host_inputs(n, count, "bf16", seed=3)
    L = count // n
    shards_h = [host[j][j * L:(j + 1) * L].copy() for j in range(n)]
    want, _ = O.ring_all_gather(shards_h, count, "bf16")
    bufs = [to_dev(x, "bf16") for x in host]
    cr.cr_all_gather([bufs[j][j * L:(j + 1) * L] for j in range(n)], count, "bf16", bufs)
    torch.cuda.synchronize()
    for r in range(n):
        assert_match(to_host(bufs[r], "bf16"), want[r], "bf16", f"rank {r}")


def test_all_reduce_equals_gather_of_scatter_on_gpu():
    n, count = 8, 8 * 8 * 1000 + 13
    host = host_inputs(n, count, "bf16", seed=11)
    bufs = [to_dev(x, "bf16") for x in host]
    L = cr.cr_chunk_len(count, n)
    shards = [torch.empty(min(L, max(0, count - j * L)), dtype=torch.bfloat16, device="cuda")
              for j in range(n)]
    outs = [torch.empty(count, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    outs2 = [torch.empty(count, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
    cr.cr_reduce_scatter(bufs, count, "bf16", "avg", shards, "bf16")
    cr.cr_all_gather(shards, count, "bf16", outs)
    cr.cr_all_reduce(bufs, count, "bf16", "avg", outs2, "bf16")
    torch.cuda.synchronize()
    for r in range(n):
        assert torch.equal(outs[r].view(torch.int16), outs2[r].view(torch.int16))


# ---- FSDP step and AdamW ----------------------------------------------------------

def fsdp_case(n, count, seed):
    grads = I.host_rank_buffers(n, count, "bf16", std=1e-3, seed0=1000 + seed)
    master_full = I.np_normal_f32(count, 0.02, 2000 + seed)
    shards = [O.chunk_bounds(count, n, j) for j in range(n)]
    master = [master_full[a:b].copy() for a, b in shards]
    m = [np.zeros(b - a, np.float32) for a, b in shards]
    v = [np.zeros(b - a, np.float32) for a, b in shards]
    return grads, master, m, v


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 8, 16, 33, 64])
@pytest.mark.parametrize("count_fn", [lambda n: 8 * n * 40, lambda n: 8 * n * 40 + 5, lambda n: 1,
                                      lambda n: 100])
@pytest.mark.parametrize("offset", [0, 1, "16B"])
def test_fsdp_step_three_steps(n, count_fn, offset):
    count = count_fn(n)
    grads, master, m, v = fsdp_case(n, count, seed=n)
    d_master = [Guarded(x.size, "f32", eoff(offset, "f32")) for x in master]
    d_m = [Guarded(x.size, "f32", eoff(offset, "f32")) for x in m]
    d_v = [Guarded(x.size, "f32", eoff(offset, "f32")) for x in v]
    for g, src in ((d_master, master), (d_m, m), (d_v, v)):
        for gg, x in zip(g, src):
            if x.size:
                gg.view.copy_(to_dev(x, "f32"))
    d_p = [Guarded(count, "bf16", eoff(offset, "bf16")) for _ in range(n)]
    for step in (1, 2, 3):
        grads = I.host_rank_buffers(n, count, "bf16", std=1e-3, seed0=1000 + 17 * step)
        d_g = [to_dev(x, "bf16", eoff(offset, "bf16")) for x in grads]
        cfg = O.AdamWConfig(step=step)
        want_p = O.fsdp_step(grads, master, m, v, cfg)
        cr.cr_fsdp_step(d_g, count, [x.ptr() for x in d_master], [x.ptr() for x in d_m],
                        [x.ptr() for x in d_v], cr.adamw_cfg(step=step), [x.ptr() for x in d_p])
        torch.cuda.synchronize()
        for j in range(n):
            for gg, ref, name in ((d_master, master, "master"), (d_m, m, "m"), (d_v, v, "v")):
                gg[j].check()
                assert_match(gg[j].host(), ref[j], "f32", f"{name}[{j}] step {step}")
        for r in range(n):
            d_p[r].check()
            assert_match(d_p[r].host(), want_p[r], "bf16", f"params[{r}] step {step}")


@pytest.mark.parametrize("n_elems", [1, 3, 4, 1000, 4096 * 9 + 3])
@pytest.mark.parametrize("with_param", [True, False])
def test_adamw_step(n_elems, with_param):
    rng = np.random.default_rng(n_elems)
    p = (rng.standard_normal(n_elems) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n_elems) * 1e-4).astype(np.float32)
    v = np.abs(rng.standard_normal(n_elems) * 1e-7).astype(np.float32)
    g = (rng.standard_normal(n_elems) * 1e-3).astype(np.float32)
    d = [to_dev(x, "f32") for x in (p, m, v, g)]
    out = Guarded(n_elems, "bf16") if with_param else None
    cfg = O.AdamWConfig(step=4)
    O.adamw(p, m, v, g, cfg)
    cr.cr_adamw_step(n_elems, d[0], d[1], d[2], d[3], cr.adamw_cfg(step=4),
                     out.ptr() if out else None)
    torch.cuda.synchronize()
    for t, ref, name in zip(d[:3], (p, m, v), ("p", "m", "v")):
        assert_match(to_host(t, "f32"), ref, "f32", name)
    if out:
        out.check()
        assert_match(out.host(), O.f32_to_bf16(p), "bf16")


# ---- buckets ------------------------------------------------------------------------

def bucket_case(n, numels, esize, cap, seed, bucket_offset):
    plan = cr.cr_bucket_plan(numels, esize, cap)
    oplan = O.bucket_plan(numels, esize, cap)
    assert plan.tensor_bucket == [int(x) for x in oplan.tensor_bucket]
    assert plan.tensor_offset == [int(x) for x in oplan.tensor_offset]
    dt = "bf16" if esize == 2 else "f32"
    host_t = [[host_inputs(1, int(k), dt, seed=seed + 1000 * r + t)[0] for t, k in enumerate(numels)]
              for r in range(n)]
    return plan, oplan, dt, host_t


@pytest.mark.parametrize("n", [1, 2, 8, 64])
@pytest.mark.parametrize("esize", [2, 4])
@pytest.mark.parametrize("tensor_offset,bucket_offset", [(0, 0), (1, 0), (0, 1), (1, 3)])
def test_bucket_pack_unpack_all_reduce(n, esize, tensor_offset, bucket_offset):
    rng = np.random.default_rng(n * 10 + esize)
    numels = [int(k) for k in rng.integers(0, 20000, size=40)] + [1, 0, 3, 70001]
    cap = 60000 * esize
    plan, oplan, dt, host_t = bucket_case(n, numels, esize, cap, seed=5, bucket_offset=bucket_offset)
    want_b = O.bucket_pack(oplan, host_t)
    d_t = [[to_dev(x, dt, tensor_offset) if x.size else None for x in row] for row in host_t]
    g_b = [[Guarded(int(k), dt, bucket_offset) for k in plan.bucket_numel] for _ in range(n)]
    flat_t = [x if x is not None else 0 for row in d_t for x in row]
    flat_b = [g.ptr() for row in g_b for g in row]
    cr.cr_bucket_pack(plan, n, flat_t, flat_b)
    torch.cuda.synchronize()
    for r in range(n):
        for b in range(plan.nbuckets):
            g_b[r][b].check()
            assert g_b[r][b].host().tobytes() == want_b[r][b].tobytes(), f"pack r={r} b={b}"
    # all-reduce AVG per bucket, then unpack into fresh guarded tensors
    cr.cr_bucket_all_reduce(plan, n, flat_b, dt, "avg")
    want_t = O.bucketed_all_reduce(oplan, host_t, dt, "avg")
    g_t = [[Guarded(int(k), dt, tensor_offset) for k in numels] for _ in range(n)]
    cr.cr_bucket_unpack(plan, n, flat_b, [g.ptr() for row in g_t for g in row])
    torch.cuda.synchronize()
    for r in range(n):
        for t in range(len(numels)):
            g_t[r][t].check()
            assert_match(g_t[r][t].host(), want_t[r][t], dt, f"unpack r={r} t={t}")


@pytest.mark.parametrize("src_shift", range(16))
@pytest.mark.parametrize("dst_shift", [0, 1, 6, 15])
def test_bucket_copy_every_byte_alignment(src_shift, dst_shift):
    """1-byte elements: source and destination misaligned by every amount
    0..15 bytes (tensor offsets inside the bucket shift the destination
    further), ranges shorter than, equal to and longer than one vector."""
    numels = [1, 7, 8, 9, 15, 16, 17, 31, 33, 1000, 20000, 3]
    plan = cr.cr_bucket_plan(numels, 1, 1 << 30)
    oplan = O.bucket_plan(numels, 1, 1 << 30)
    rng = np.random.default_rng(src_shift * 16 + dst_shift)
    host = [rng.integers(0, 256, k).astype(np.uint8) for k in numels]
    want = O.bucket_pack(oplan, [host])[0][0]
    dev_t = []
    for x in host:
        base = torch.empty(x.size + src_shift, dtype=torch.uint8, device="cuda")
        base[src_shift:].copy_(torch.from_numpy(x).cuda())
        dev_t.append(base[src_shift:])
    total = int(plan.bucket_numel[0])
    G = 64
    bbase = torch.full((total + 2 * G + dst_shift,), 0xA5, dtype=torch.uint8, device="cuda")
    lo = G + dst_shift
    cr.cr_bucket_pack(plan, 1, dev_t, [bbase[lo:lo + total]])
    torch.cuda.synchronize()
    h = bbase.cpu().numpy()
    assert np.all(h[:lo] == 0xA5) and np.all(h[lo + total:] == 0xA5), "canary"
    assert h[lo:lo + total].tobytes() == want.tobytes()
    # and back out into fresh tensors shifted the other way
    outs = []
    for x in host:
        base = torch.full((x.size + 2 * G + dst_shift,), 0x5A, dtype=torch.uint8, device="cuda")
        outs.append((base, G + dst_shift, x.size))
    cr.cr_bucket_unpack(plan, 1, [bbase[lo:lo + total]], [b[o:o + k] for b, o, k in outs])
    torch.cuda.synchronize()
    for (b, o, k), x in zip(outs, host):
        hb = b.cpu().numpy()
        assert np.all(hb[:o] == 0x5A) and np.all(hb[o + k:] == 0x5A), "canary"
        assert hb[o:o + k].tobytes() == x.tobytes()


# ---- all-reduce from host memory (pipelined slices) --------------------------------

@pytest.mark.parametrize("n,count", [(8, 8 * 8 * 1000 + 13), (4, 1 << 16), (3, 1000), (1, 77)])
@pytest.mark.parametrize("dt,op", [("bf16", "avg"), ("f32", "sum"), ("i32", "sum")])
@pytest.mark.parametrize("slice_elems", [0, 1, 1000, 4096, 1 << 30])
@pytest.mark.parametrize("streams", ["three", "one"])
def test_all_reduce_staged(n, count, dt, op, slice_elems, streams):
    host = host_inputs(n, count, dt, seed=count + n)
    want, _ = O.ring_all_reduce(host, dt, op, dt)
    tdt = {"bf16": torch.bfloat16, "f32": torch.float32, "i32": torch.int32}[dt]
    h_in = [to_dev(x, dt).cpu().pin_memory() for x in host]
    same = slice_elems == 4096   # host_out == host_in for one variant
    h_out = h_in if same else [torch.empty(count, dtype=tdt).pin_memory() for _ in range(n)]
    d = [torch.empty(count, dtype=tdt, device="cuda") for _ in range(n)]
    sc = torch.cuda.current_stream()
    sh, sd = (torch.cuda.Stream(), torch.cuda.Stream()) if streams == "three" else (sc, sc)
    cr.cr_all_reduce_staged(h_in, h_out, d, count, dt, op, slice_elems, sc, sh, sd)
    sc.synchronize()
    for r in range(n):
        got = h_out[r].view(torch.int16).numpy().view(np.uint16) if dt == "bf16" else h_out[r].numpy()
        assert_match(got, want[r], dt, f"host_out rank {r}")
        assert_match(to_host(d[r], dt), want[r], dt, f"dev rank {r}")


def test_all_reduce_staged_repeated_calls_keep_order():
    """Back-to-back calls on the same buffers: each call's uploads must wait
    for the previous call's downloads (host_out == host_in)."""
    n, count = 8, 1 << 20
    host = host_inputs(n, count, "f32", seed=5)
    h = [torch.from_numpy(x).pin_memory() for x in host]
    d = [torch.empty(count, dtype=torch.float32, device="cuda") for _ in range(n)]
    sh, sd = torch.cuda.Stream(), torch.cuda.Stream()
    cur = [x.copy() for x in host]
    for _ in range(3):
        cr.cr_all_reduce_staged(h, h, d, count, "f32", "sum", 1 << 16, None, sh, sd)
        cur, _ = O.ring_all_reduce(cur, "f32", "sum")
    torch.cuda.synchronize()
    for r in range(n):
        assert_match(h[r].numpy(), cur[r], "f32", f"rank {r}")


# ---- fused bucket all-reduce (no pack) ---------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 3, 8, 16, 64])
@pytest.mark.parametrize("dt,op", [("bf16", "avg"), ("f32", "sum"), ("i32", "sum"), ("f32", "avg")])
@pytest.mark.parametrize("offset", [0, 1, "16B"])
def test_bucket_all_reduce_fused(n, dt, op, offset):
    """Equal, bit for bit, to the oracle's pack -> ring all-reduce per bucket
    -> unpack, including tensors that straddle chunk boundaries of their
    bucket and more tensors than one launch takes."""
    rng = np.random.default_rng(n * 7 + eoff(offset, dt))
    T = 150 if n <= 16 else 40
    numels = [int(k) for k in rng.integers(0, 3000, size=T)] + [1, 0, 7, 20001]
    esize = 2 if dt == "bf16" else 4
    cap = 9000 * esize
    plan = cr.cr_bucket_plan(numels, esize, cap)
    oplan = O.bucket_plan(numels, esize, cap)
    host_t = [[host_inputs(1, k, dt, seed=100 * r + t)[0] for t, k in enumerate(numels)]
              for r in range(n)]
    want = O.bucketed_all_reduce(oplan, host_t, dt, op)
    g = [[Guarded(k, dt, eoff(offset, dt)) for k in numels] for _ in range(n)]
    for r in range(n):
        for t, k in enumerate(numels):
            if k:
                g[r][t].view.copy_(to_dev(host_t[r][t], dt))
    cr.cr_bucket_all_reduce_fused(plan, n, [x.ptr() for row in g for x in row], dt, op)
    torch.cuda.synchronize()
    for r in range(n):
        for t in range(len(numels)):
            g[r][t].check()
            assert_match(g[r][t].host(), want[r][t], dt, f"rank {r} tensor {t}")


# ---- FSDP step with gradient-norm clipping ----------------------------------------

@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 8, 16, 33, 64])
@pytest.mark.parametrize("count_fn", [lambda n: 8 * n * 40, lambda n: 8 * n * 40 + 5,
                                      lambda n: 8 * n * 40 - 3, lambda n: 3])
@pytest.mark.parametrize("clip", ["active", "inactive"])
@pytest.mark.parametrize("ws_parts", [None, 1, 7])
def test_fsdp_step_clipped(n, count_fn, clip, ws_parts):
    count = count_fn(n)
    grads, master, m, v = fsdp_case(n, count, seed=3 * n)
    g_full, _ = O.ring_all_reduce(grads, "bf16", "avg", "f32")
    norm = float(np.linalg.norm(g_full[0].astype(np.float64)))
    max_norm = norm / 3 if clip == "active" else norm * 10 + 1
    cfg = O.AdamWConfig()
    d_master = [to_dev(x, "f32") for x in master]
    d_m = [to_dev(x, "f32") for x in m]
    d_v = [to_dev(x, "f32") for x in v]
    d_g = [to_dev(x, "bf16") for x in grads]
    d_p = [Guarded(count, "bf16") for _ in range(n)]
    # the coefficient's 8 bytes, then room for ws_parts partial sums
    ws_bytes = cr.cr_fsdp_clip_workspace_bytes() if ws_parts is None else 8 * (ws_parts + 1)
    ws = torch.empty(ws_bytes // 8, dtype=torch.float64, device="cuda")
    norm_out = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
    _, want_norm = O.fsdp_step_clipped(grads, [x.copy() for x in master], [x.copy() for x in m],
                                       [x.copy() for x in v], cfg, max_norm)
    cr.cr_fsdp_step_clipped(d_g, count, d_master, d_m, d_v, cr.adamw_cfg(), max_norm, ws,
                            ws_bytes, [x.ptr() for x in d_p], norm_out)
    torch.cuda.synchronize()
    # the norm's summation order differs from the oracle's (fp32 batches,
    # fixed CTA order); the rest is bitwise at a coefficient that norm allows
    assert float(norm_out.item()) == pytest.approx(want_norm, rel=1e-6)
    for r in range(n):
        d_p[r].check()
    got_state = [[to_host(t[j], "f32") for j in range(n)] for t in (d_master, d_m, d_v)]
    coef = assert_clipped_match(got_state, [x.host() for x in d_p], grads, master, m, v, cfg,
                                max_norm, want_norm)
    if clip == "inactive":
        assert coef == np.float32(1.0)


@pytest.mark.parametrize("n", [5, 8, 13])
@pytest.mark.parametrize("aligned", [True, False])
def test_fsdp_step_clipped_ignores_param_contents(n, aligned):
    """For N >= 5 the clipped step parks the averaged gradient in params[0]
    and params[1] between its passes.  The parameters are outputs only:
    whatever they hold on entry (zeros, NaN bit patterns, the previous
    step's values) the results are the same bits, on the vector path
    (aligned) and on the element path (every buffer 2 bytes off)."""
    count = 8 * n * 300 - 5   # L = 2400 (vector path), a short last chunk, a ragged tail
    grads, master, m, v = fsdp_case(n, count, seed=40 + n)
    g_full, _ = O.ring_all_reduce(grads, "bf16", "avg", "f32")
    max_norm = float(np.linalg.norm(g_full[0].astype(np.float64))) / 5
    off = 0 if aligned else 1
    d_g = [to_dev(x, "bf16", off) for x in grads]
    ws = torch.empty(cr.cr_fsdp_clip_workspace_bytes() // 8, dtype=torch.float64, device="cuda")
    results = []
    for fill in (0x0000, 0x7FC1, 0xFFFF):
        d_master = [to_dev(x, "f32") for x in master]
        d_m = [to_dev(x, "f32") for x in m]
        d_v = [to_dev(x, "f32") for x in v]
        d_p = [Guarded(count, "bf16", off) for _ in range(n)]
        for x in d_p:
            x.view.view(torch.int16).fill_(fill - (1 << 16) if fill >= 1 << 15 else fill)
        norm_out = torch.empty(1, dtype=torch.float32, device="cuda")
        cr.cr_fsdp_step_clipped(d_g, count, d_master, d_m, d_v, cr.adamw_cfg(), max_norm, ws,
                                ws.numel() * 8, [x.ptr() for x in d_p], norm_out)
        torch.cuda.synchronize()
        for x in d_p:
            x.check()
        results.append((to_host(norm_out, "f32"),
                        [to_host(x, "f32") for x in d_master + d_m + d_v],
                        [x.host() for x in d_p]))
    for r in results[1:]:
        assert_match(r[0], results[0][0], "f32", "norm")
        for a, b in zip(r[1], results[0][1]):
            assert_match(a, b, "f32", "state")
        for a, b in zip(r[2], results[0][2]):
            assert_match(a, b, "bf16", "params")
    got_state = [results[0][1][q * n:(q + 1) * n] for q in range(3)]
    _, want_norm = O.fsdp_step_clipped(grads, [x.copy() for x in master], [x.copy() for x in m],
                                       [x.copy() for x in v], O.AdamWConfig(), max_norm)
    assert_clipped_match(got_state, results[0][2], grads, master, m, v, O.AdamWConfig(),
                         max_norm, want_norm)


def test_fsdp_step_clipped_is_deterministic():
    n, count = 8, 8 * 8 * 5000 + 3
    grads, master, m, v = fsdp_case(n, count, seed=9)
    d_g = [to_dev(x, "bf16") for x in grads]
    ws = torch.empty(cr.cr_fsdp_clip_workspace_bytes() // 8, dtype=torch.float64, device="cuda")
    outs = []
    for _ in range(3):
        d_master = [to_dev(x, "f32") for x in master]
        d_m = [to_dev(x, "f32") for x in m]
        d_v = [to_dev(x, "f32") for x in v]
        d_p = [torch.empty(count, dtype=torch.bfloat16, device="cuda") for _ in range(n)]
        norm_out = torch.empty(1, dtype=torch.float32, device="cuda")
        cr.cr_fsdp_step_clipped(d_g, count, d_master, d_m, d_v, cr.adamw_cfg(), 1e-3, ws,
                                ws.numel() * 8, d_p, norm_out)
        torch.cuda.synchronize()
        outs.append((norm_out.cpu(), [x.cpu() for x in d_master + d_m + d_v],
                     [x.view(torch.int16).cpu() for x in d_p]))
    for o in outs[1:]:
        assert torch.equal(o[0], outs[0][0])
        assert all(torch.equal(a, b) for a, b in zip(o[1], outs[0][1]))
        assert all(torch.equal(a, b) for a, b in zip(o[2], outs[0][2]))


# ---- all-reduce read and written straight from pinned host memory ------------------

@pytest.mark.parametrize("n,count", [(8, 8 * 8 * 1000 + 13), (4, 1 << 16), (3, 1000), (1, 77), (32, 4099)])
@pytest.mark.parametrize("dt,op", [("bf16", "avg"), ("f32", "sum"), ("i32", "sum")])
@pytest.mark.parametrize("mode", ["out", "in_place", "with_dev"])
def test_all_reduce_host(n, count, dt, op, mode):
    host = host_inputs(n, count, dt, seed=count + 7 * n)
    want, _ = O.ring_all_reduce(host, dt, op, dt)
    tdt = {"bf16": torch.bfloat16, "f32": torch.float32, "i32": torch.int32}[dt]
    h_in = [to_dev(x, dt).cpu().pin_memory() for x in host]
    h_out = h_in if mode == "in_place" else [torch.empty(count, dtype=tdt).pin_memory()
                                             for _ in range(n)]
    d_out = [Guarded(count, dt) for _ in range(n)] if mode == "with_dev" else None
    cr.cr_all_reduce_host(h_in, h_out, count, dt, op,
                          dev_out=[g.ptr() for g in d_out] if d_out else None)
    torch.cuda.synchronize()
    for r in range(n):
        got = h_out[r].view(torch.int16).numpy().view(np.uint16) if dt == "bf16" else h_out[r].numpy()
        assert_match(got, want[r], dt, f"host_out rank {r}")
        if d_out:
            d_out[r].check()
            assert_match(d_out[r].host(), want[r], dt, f"dev_out rank {r}")


def test_all_reduce_host_rejects_pageable_memory():
    n, count = 2, 1024
    pageable = [torch.zeros(count, dtype=torch.float32) for _ in range(n)]
    with pytest.raises(cr.CRError) as ei:
        cr.cr_all_reduce_host(pageable, pageable, count, "f32", "sum")
    assert ei.value.status == 1 and "pinned" in str(ei.value)


# ---- FSDP2 per-parameter step ----------------------------------------------------

FSDP2_SHAPES = [(2, 3), (2, 1), (3, 3), (5, 7), (1, 16), (9, 1), (0, 4), (16, 8), (64, 24),
                (7, 129), (33, 64), (4, 1000)]


def fsdp2_host(shapes, n, seed):
    grads = [I.host_rank_buffers(n, d * rn, "bf16", std=1e-3, seed0=seed + 100 * p)
             for p, (d, rn) in enumerate(shapes)]
    master, m, v = [], [], []
    for p, (d, rn) in enumerate(shapes):
        full = I.np_normal_f32(d * rn, 0.02, seed + 7 * p + 1)
        rows = [O.fsdp2_shard_rows(d, n, j) for j in range(n)]
        master.append([full[lo * rn:hi * rn].copy() for lo, hi in rows])
        m.append([np.zeros((hi - lo) * rn, np.float32) for lo, hi in rows])
        v.append([np.zeros((hi - lo) * rn, np.float32) for lo, hi in rows])
    return grads, master, m, v


@pytest.mark.parametrize("n", [1, 2, 3, 4, 8, 16, 33, 64])
@pytest.mark.parametrize("offset", [0, "16B", 1])
def test_fsdp2_step_two_steps(n, offset):
    shapes = FSDP2_SHAPES
    grads, master, m, v = fsdp2_host(shapes, n, 40 + n)
    gm = [[Guarded(x.size, "f32", eoff(offset, "f32")) for x in row] for row in master]
    gmm = [[Guarded(x.size, "f32", eoff(offset, "f32")) for x in row] for row in m]
    gv = [[Guarded(x.size, "f32", eoff(offset, "f32")) for x in row] for row in v]
    for g, src in ((gm, master), (gmm, m), (gv, v)):
        for grow, srow in zip(g, src):
            for gg, x in zip(grow, srow):
                if x.size:
                    gg.view.copy_(to_dev(x, "f32"))
    gp = [[Guarded(d * rn, "bf16", eoff(offset, "bf16")) for _ in range(n)] for d, rn in shapes]
    for step in (1, 2):
        if step == 2:
            grads = [I.host_rank_buffers(n, d * rn, "bf16", std=1e-3, seed0=500 + 100 * p)
                     for p, (d, rn) in enumerate(shapes)]
        cfg = O.AdamWConfig(step=step)
        want = O.fsdp2_step(shapes, grads, master, m, v, cfg)
        d_g = [to_dev(x, "bf16", eoff(offset, "bf16")) if x.size else None for row in grads for x in row]
        flat = lambda xs: [x.ptr() for row in xs for x in row]
        cr.cr_fsdp2_step(shapes, n, [x if x is not None else 0 for x in d_g], flat(gm), flat(gmm),
                         flat(gv), cr.adamw_cfg(step=step), flat(gp))
        torch.cuda.synchronize()
        for p in range(len(shapes)):
            for j in range(n):
                for g, ref, name in ((gm, master, "master"), (gmm, m, "m"), (gv, v, "v")):
                    g[p][j].check()
                    assert_match(g[p][j].host(), ref[p][j], "f32", f"{name} {p} {j} step {step}")
            for r in range(n):
                gp[p][r].check()
                assert_match(gp[p][r].host(), want[p][r], "bf16", f"param {p} rank {r} step {step}")


@pytest.mark.parametrize("n", [1, 2, 3, 4, 8, 16, 33, 64])
@pytest.mark.parametrize("offset", [0, "16B", 1])
def test_fsdp2_step_planned_two_steps(n, offset):
    """cr_fsdp2_step_planned: the plan made and its table uploaded once,
    then two steps (t = 1, 2) launched from the table, against the oracle."""
    shapes = FSDP2_SHAPES
    grads, master, m, v = fsdp2_host(shapes, n, 80 + n)
    gm = [[Guarded(x.size, "f32", eoff(offset, "f32")) for x in row] for row in master]
    gmm = [[Guarded(x.size, "f32", eoff(offset, "f32")) for x in row] for row in m]
    gv = [[Guarded(x.size, "f32", eoff(offset, "f32")) for x in row] for row in v]
    for g, src in ((gm, master), (gmm, m), (gv, v)):
        for grow, srow in zip(g, src):
            for gg, x in zip(grow, srow):
                if x.size:
                    gg.view.copy_(to_dev(x, "f32"))
    gp = [[Guarded(d * rn, "bf16", eoff(offset, "bf16")) for _ in range(n)] for d, rn in shapes]
    gg_ = [[Guarded(d * rn, "bf16", eoff(offset, "bf16")) for _ in range(n)] for d, rn in shapes]
    flat = lambda xs: [x.ptr() for row in xs for x in row]
    plan = cr.cr_fsdp2_plan_create(shapes, n, flat(gg_), flat(gm), flat(gmm), flat(gv), flat(gp))
    table = Guarded(plan.table_bytes // 4 + 1, "i32")
    cr.cr_fsdp2_plan_upload(plan, table.ptr(), plan.table_bytes)
    del plan  # the uploaded table is all the step needs besides the plan's sizes
    plan = cr.cr_fsdp2_plan_create(shapes, n, flat(gg_), flat(gm), flat(gmm), flat(gv), flat(gp))
    for step in (1, 2):
        if step == 2:
            grads = [I.host_rank_buffers(n, d * rn, "bf16", std=1e-3, seed0=900 + 100 * p)
                     for p, (d, rn) in enumerate(shapes)]
        for grow, srow in zip(gg_, grads):
            for x, h in zip(grow, srow):
                if h.size:
                    x.view.copy_(to_dev(h, "bf16"))
        cfg = O.AdamWConfig(step=step)
        want = O.fsdp2_step(shapes, grads, master, m, v, cfg)
        cr.cr_fsdp2_step_planned(plan, table.ptr(), cr.adamw_cfg(step=step))
        torch.cuda.synchronize()
        table.check()
        for p in range(len(shapes)):
            for j in range(n):
                for g, ref, name in ((gm, master, "master"), (gmm, m, "m"), (gv, v, "v")):
                    g[p][j].check()
                    assert_match(g[p][j].host(), ref[p][j], "f32", f"{name} {p} {j} step {step}")
            for r in range(n):
                gp[p][r].check()
                gg_[p][r].check()
                assert_match(gp[p][r].host(), want[p][r], "bf16", f"param {p} rank {r} step {step}")


@pytest.mark.parametrize("n", [2, 8])
def test_fsdp2_planned_equals_chained_launches(n):
    """300 parameters (more than the 64 one chained launch takes): the single
    planned launch and cr_fsdp2_step's chained launches give the same bits,
    on the same inputs."""
    rng = np.random.default_rng(n)
    shapes = [(int(rng.integers(0, 40)), int(rng.integers(1, 300))) for _ in range(300)]
    grads, master, m, v = fsdp2_host(shapes, n, 7)
    outs = []
    for planned in (False, True):
        d_g = [to_dev(x, "bf16") if x.size else 0 for row in grads for x in row]
        d_st = [[to_dev(x, "f32") if x.size else 0 for row in t for x in row] for t in (master, m, v)]
        d_p = [torch.empty(d * rn, dtype=torch.bfloat16, device="cuda") for d, rn in shapes
               for _ in range(n)]
        if planned:
            plan = cr.cr_fsdp2_plan_create(shapes, n, d_g, *d_st, d_p)
            table = torch.empty(plan.table_bytes, dtype=torch.uint8, device="cuda")
            cr.cr_fsdp2_plan_upload(plan, table)
            cr.cr_fsdp2_step_planned(plan, table, cr.adamw_cfg())
        else:
            cr.cr_fsdp2_step(shapes, n, d_g, *d_st, cr.adamw_cfg(), d_p)
        torch.cuda.synchronize()
        outs.append(([x.cpu() for t in d_st for x in t if not isinstance(x, int)],
                     [x.view(torch.int16).cpu() for x in d_p]))
    for a, b in zip(outs[0][0] + outs[0][1], outs[1][0] + outs[1][1]):
        assert torch.equal(a, b)
    want = O.fsdp2_step(shapes, grads, master, m, v, O.AdamWConfig())
    for p in range(len(shapes)):
        for r in range(n):
            assert_match(to_host(outs[1][1][p * n + r].view(torch.bfloat16), "bf16"), want[p][r],
                         "bf16", f"param {p} rank {r}")


# ---- gradient accumulation (no_sync) ---------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 3, 8, 16, 64])
@pytest.mark.parametrize("gdt", ["bf16", "f32"])
@pytest.mark.parametrize("offset", [0, "16B", 1])
@pytest.mark.parametrize("op", ["avg", "sum"])
def test_accumulate_then_all_reduce(n, gdt, offset, op):
    """Three no_sync micro-steps (cr_accumulate), then the last micro-step
    fused with the all-reduce (cr_all_reduce_accumulate): equal to the
    oracle's accumulations followed by its ring all-reduce."""
    for count in (8 * n * 40, 8 * n * 40 + 5, 7):
        acc_h = [np.zeros(count, np.float32) for _ in range(n)]
        g_acc = [Guarded(count, "f32", eoff(offset, "f32")) for _ in range(n)]
        for x in g_acc:
            x.view.zero_()
        for micro in range(4):
            gh = I.host_rank_buffers(n, count, gdt, std=1e-2, seed0=10 * micro + count)
            for r in range(n):
                O.accumulate(acc_h[r], gh[r], gdt)
            d_g = [to_dev(x, gdt, eoff(offset, gdt)) for x in gh]
            if micro < 3:
                cr.cr_accumulate([x.ptr() for x in g_acc], count, d_g, gdt)
            else:
                cr.cr_all_reduce_accumulate([x.ptr() for x in g_acc], count, d_g, gdt, op)
        want, _ = O.ring_all_reduce(acc_h, "f32", op)
        torch.cuda.synchronize()
        for r in range(n):
            g_acc[r].check()
            assert_match(g_acc[r].host(), want[r], "f32", f"count {count} rank {r}")

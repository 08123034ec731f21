"""C-ABI checks that need no GPU: the library loads, exports every symbol
include/cr.h declares, rejects bad arguments on the host with the documented
status before touching a device, and its host-only parts (bucket plan,
traffic accounting) match the oracle exactly."""
import os
import re

import numpy as np
import pytest

import oracle as O
from fsdp_emulated_ranks_gb300 import build as libbuild
from fsdp_emulated_ranks_gb300 import cr
from fsdp_emulated_ranks_gb300 import inputs as I

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    libbuild.build()
    return cr.lib()


def header_functions():
    text = open(os.path.join(ROOT, "include", "cr.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = set(re.findall(r"\b(cr_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(L):
    declared = header_functions()
    assert set(declared) == set(cr.EXPORTS)
    for name in declared:
        assert hasattr(L, name), name
    assert L.cr_version() == 100


def test_status_strings(L):
    for k, v in cr.STATUS.items():
        assert L.cr_status_string(k).decode() == v


def expect(status, fn, *args, **kw):
    with pytest.raises(cr.CRError) as ei:
        fn(*args, **kw)
    assert ei.value.status == status, str(ei.value)
    return str(ei.value)


# An address never dereferenced: every call below either fails validation or
# has nothing to do (count 0), so no kernel is ever launched on it.
FAKE = 1 << 40


def test_reduce_scatter_validation(L):
    n = 4
    bufs = [FAKE + r * (1 << 20) for r in range(n)]
    outs = [FAKE + (1 << 30) + r * (1 << 20) for r in range(n)]
    expect(1, cr.cr_reduce_scatter, bufs * 17, 8, "f32", "sum", outs * 17, "f32", stream=0)
    expect(1, cr.cr_reduce_scatter, [], 8, "f32", "sum", [], "f32", stream=0)
    expect(2, cr.cr_reduce_scatter, bufs, 8, "i32", "avg", outs, "i32", stream=0)
    expect(2, cr.cr_reduce_scatter, bufs, 8, "f32", "sum", outs, "bf16", stream=0)
    expect(2, cr.cr_reduce_scatter, bufs, 8, "f32", "sum", outs, "i32", stream=0)
    expect(1, cr.cr_reduce_scatter, bufs[:3] + [0], 8, "f32", "sum", outs, "f32", stream=0)
    expect(3, cr.cr_reduce_scatter, [bufs[0] + 2] + bufs[1:], 8, "f32", "sum", outs, "f32", stream=0)
    # overlap: shard 1 inside rank 0's input
    bad = list(outs)
    bad[1] = bufs[0] + 4
    expect(1, cr.cr_reduce_scatter, bufs, 8, "f32", "sum", bad, "f32", stream=0)
    # two outputs overlapping
    bad = list(outs)
    bad[2] = outs[1] + 4
    expect(1, cr.cr_reduce_scatter, bufs, 64, "f32", "sum", bad, "f32", stream=0)
    # in place is legal only with equal dtypes: bf16 -> f32 in place is not
    L_ = cr.cr_chunk_len(64, n)
    inpl = [bufs[j] + j * L_ * 2 for j in range(n)]
    expect(1, cr.cr_reduce_scatter, bufs, 64, "bf16", "sum", inpl, "f32", stream=0)
    # empty count: legal, nothing launched
    cr.cr_reduce_scatter(bufs, 0, "f32", "sum", [0] * n, "f32", stream=0)
    # NULL rank buffers with count > 0 are rejected even when every shard
    # they would feed is empty
    expect(1, cr.cr_reduce_scatter, [0] * n, 2, "f32", "sum", [0] * n, "f32", stream=0)


def test_all_reduce_and_gather_validation(L):
    n = 3
    bufs = [FAKE + r * (1 << 20) for r in range(n)]
    outs = [FAKE + (1 << 30) + r * (1 << 20) for r in range(n)]
    expect(1, cr.cr_all_reduce, bufs, 16, "f32", "sum", [bufs[1]] + outs[1:], "f32", stream=0)
    expect(1, cr.cr_all_reduce, bufs, 16, "bf16", "avg", bufs, "f32", stream=0)
    expect(3, cr.cr_all_reduce, bufs, 16, "bf16", "avg", [outs[0] + 1] + outs[1:], "bf16", stream=0)
    expect(1, cr.cr_all_reduce, bufs, 16, 7, "sum", outs, "f32", stream=0)
    # shard 0 lies inside rank 1's output (only rank 0's chunk 0 is in place)
    expect(1, cr.cr_all_gather, bufs, 16, "f32", [outs[0], bufs[0], outs[2]], stream=0)
    expect(1, cr.cr_all_gather, bufs, 16, "f32", [outs[0], outs[0], outs[2]], stream=0)
    expect(3, cr.cr_all_gather, bufs, 16, "bf16", [outs[0] + 1] + outs[1:], stream=0)
    cr.cr_all_reduce(bufs, 0, "f32", "sum", bufs, "f32", stream=0)
    cr.cr_all_gather([0] * n, 0, "f32", [0] * n, stream=0)


def test_fsdp_and_adamw_validation(L):
    n, count = 2, 16
    g = [FAKE + r * (1 << 20) for r in range(n)]
    p = [FAKE + (1 << 28) + r * (1 << 20) for r in range(n)]
    ms = [FAKE + (2 << 28) + r * (1 << 20) for r in range(n)]
    m = [FAKE + (3 << 28) + r * (1 << 20) for r in range(n)]
    v = [FAKE + (4 << 28) + r * (1 << 20) for r in range(n)]
    expect(1, cr.cr_fsdp_step, g, count, ms, m, v, cr.adamw_cfg(step=0), p, stream=0)
    expect(1, cr.cr_fsdp_step, g, count, ms, m, v, cr.adamw_cfg(beta1=1.0), p, stream=0)
    expect(1, cr.cr_fsdp_step, g, count, ms, m, [m[0], v[1]], cr.adamw_cfg(), p, stream=0)
    expect(1, cr.cr_fsdp_step, g, count, ms, m, v, cr.adamw_cfg(), g, stream=0)
    expect(3, cr.cr_fsdp_step, g, count, [ms[0] + 2, ms[1]], m, v, cr.adamw_cfg(), p, stream=0)
    cr.cr_fsdp_step(g, 0, [0] * n, [0] * n, [0] * n, cr.adamw_cfg(), p, stream=0)
    expect(1, cr.cr_adamw_step, 8, ms[0], ms[0] + 16, m[0], v[0], cr.adamw_cfg(), stream=0)
    expect(1, cr.cr_adamw_step, 8, ms[0], 0, m[0], v[0], cr.adamw_cfg(), stream=0)
    cr.cr_adamw_step(0, 0, 0, 0, 0, cr.adamw_cfg(), stream=0)


def test_bucket_validation(L):
    plan = cr.cr_bucket_plan([4, 8], 2, 64)
    expect(1, cr.cr_bucket_pack, plan, 0, [FAKE] * 2, [FAKE] * 2, stream=0)
    expect(1, cr.cr_bucket_pack, plan, 1, [0, FAKE], [FAKE], stream=0)
    expect(3, cr.cr_bucket_pack, plan, 1, [FAKE + 1, FAKE + 64], [FAKE + 4096], stream=0)
    expect(1, cr.cr_bucket_all_reduce, plan, 1, [FAKE], "f32", "sum", stream=0)
    with pytest.raises(cr.CRError):
        cr.cr_bucket_plan([1, 2], 0, 64)
    with pytest.raises(cr.CRError):
        cr.cr_bucket_plan([1, 2], 2, 0)


@pytest.mark.parametrize("seed", range(6))
def test_bucket_plan_matches_oracle(L, seed):
    rng = np.random.default_rng(seed)
    numels = [int(k) for k in rng.integers(0, 3000, size=rng.integers(0, 80))]
    for esize in (2, 4):
        for cap in (1, 100, 2048, 10000, 1 << 22):
            a = cr.cr_bucket_plan(numels, esize, cap)
            b = O.bucket_plan(numels, esize, cap)
            assert a.nbuckets == b.nbuckets
            assert a.tensor_bucket == [int(x) for x in b.tensor_bucket]
            assert a.tensor_offset == [int(x) for x in b.tensor_offset]
            assert a.bucket_numel == [int(x) for x in b.bucket_numel]


def test_bucket_plan_workload_matches_oracle(L):
    numels = [int(k) for k in I.bucket_numels()]
    cap = 25 * 1024 * 1024
    a = cr.cr_bucket_plan(numels, 2, cap)
    b = O.bucket_plan(numels, 2, cap)
    assert a.tensor_bucket == [int(x) for x in b.tensor_bucket]
    assert a.tensor_offset == [int(x) for x in b.tensor_offset]


@pytest.mark.parametrize("n", [1, 2, 3, 4, 8, 13, 64])
@pytest.mark.parametrize("count", [0, 1, 5, 64, 1000, 4097])
def test_comm_elems_match_oracle_counters(L, n, count):
    bufs = I.integer_valued_f32(n, count, seed=0)
    _, rs = O.ring_reduce_scatter(bufs, "f32", "sum")
    L_ = O.chunk_len(count, n)
    shards = [np.zeros(b - a, np.float32) for a, b in (O.chunk_bounds(count, n, j) for j in range(n))]
    _, ag = O.ring_all_gather(shards, count, "f32")
    _, ar = O.ring_all_reduce(bufs, "f32", "sum")
    _, nv = O.naive_all_reduce(bufs, "f32", "sum")
    assert L_ == cr.cr_chunk_len(count, n)
    for r in range(n):
        assert cr.cr_shard_range(count, n, r) == O.chunk_bounds(count, n, r)
        for coll, t in ((0, rs), (1, ag), (2, ar)):
            assert cr.cr_comm_elems(coll, cr.SCHED_RING, n, count, r) == (t.sent[r], t.recv[r], t.steps)
        assert cr.cr_comm_elems(2, cr.SCHED_NAIVE, n, count, r) == (nv.sent[r], nv.recv[r], nv.steps)
    expect(2, cr.cr_comm_elems, 0, cr.SCHED_NAIVE, n, count, 0)


def test_all_reduce_staged_validation(L):
    n = 2
    h = [FAKE + r * (1 << 20) for r in range(n)]
    o = [FAKE + (1 << 30) + r * (1 << 20) for r in range(n)]
    d = [FAKE + (2 << 30) + r * (1 << 20) for r in range(n)]
    expect(1, cr.cr_all_reduce_staged, h, o, [d[0], d[0]], 16, "f32", "sum", 0, 0, 0, 0)
    expect(1, cr.cr_all_reduce_staged, h, [o[0], o[0]], d, 16, "f32", "sum", 0, 0, 0, 0)
    expect(2, cr.cr_all_reduce_staged, h, o, d, 16, "i32", "avg", 0, 0, 0, 0)
    expect(3, cr.cr_all_reduce_staged, [h[0] + 2, h[1]], o, d, 16, "f32", "sum", 0, 0, 0, 0)
    expect(1, cr.cr_all_reduce_staged, [0, h[1]], o, d, 16, "f32", "sum", 0, 0, 0, 0)
    cr.cr_all_reduce_staged(h, o, d, 0, "f32", "sum", 0, 0, 0, 0)


def test_bucket_all_reduce_fused_validation(L):
    plan = cr.cr_bucket_plan([4, 8, 0], 2, 64)
    t = [FAKE, FAKE + 4096, 0]
    expect(1, cr.cr_bucket_all_reduce_fused, plan, 1, t, "f32", "sum", stream=0)
    expect(1, cr.cr_bucket_all_reduce_fused, plan, 1, [FAKE, FAKE + 4, 0], "bf16", "sum", stream=0)
    expect(1, cr.cr_bucket_all_reduce_fused, plan, 2, t + [FAKE + 8192, FAKE + 4096, 0], "bf16",
           "avg", stream=0)
    expect(3, cr.cr_bucket_all_reduce_fused, plan, 1, [FAKE + 1, FAKE + 4096, 0], "bf16", "sum",
           stream=0)
    expect(2, cr.cr_bucket_all_reduce_fused, cr.cr_bucket_plan([4], 4, 64), 1, [FAKE], "i32",
           "avg", stream=0)


def test_fsdp_step_clipped_validation(L):
    n, count = 2, 16
    g = [FAKE + r * (1 << 20) for r in range(n)]
    p = [FAKE + (1 << 28) + r * (1 << 20) for r in range(n)]
    ms = [FAKE + (2 << 28) + r * (1 << 20) for r in range(n)]
    m = [FAKE + (3 << 28) + r * (1 << 20) for r in range(n)]
    v = [FAKE + (4 << 28) + r * (1 << 20) for r in range(n)]
    ws = FAKE + (5 << 28)
    nb = cr.cr_fsdp_clip_workspace_bytes()
    assert nb >= 16 and nb % 8 == 0
    expect(1, cr.cr_fsdp_step_clipped, g, count, ms, m, v, cr.adamw_cfg(), 0.0, ws, nb, p, stream=0)
    expect(1, cr.cr_fsdp_step_clipped, g, count, ms, m, v, cr.adamw_cfg(), float("inf"), ws, nb, p,
           stream=0)
    expect(1, cr.cr_fsdp_step_clipped, g, count, ms, m, v, cr.adamw_cfg(), 1.0, 0, nb, p, stream=0)
    expect(1, cr.cr_fsdp_step_clipped, g, count, ms, m, v, cr.adamw_cfg(), 1.0, ws, 4, p, stream=0)
    # the coefficient slot alone leaves no room for a partial sum
    expect(1, cr.cr_fsdp_step_clipped, g, count, ms, m, v, cr.adamw_cfg(), 1.0, ws, 8, p, stream=0)
    expect(3, cr.cr_fsdp_step_clipped, g, count, ms, m, v, cr.adamw_cfg(), 1.0, ws + 4, nb, p,
           stream=0)
    expect(1, cr.cr_fsdp_step_clipped, g, count, ms, m, v, cr.adamw_cfg(), 1.0, ms[0], nb, p,
           stream=0)
    expect(1, cr.cr_fsdp_step_clipped, g, count, ms, m, v, cr.adamw_cfg(), 1.0, ws, nb, p,
           norm_out=ws, stream=0)


def test_all_reduce_host_validation(L):
    n = 2
    h = [FAKE + r * (1 << 20) for r in range(n)]
    o = [FAKE + (1 << 30) + r * (1 << 20) for r in range(n)]
    d = [FAKE + (2 << 30) + r * (1 << 20) for r in range(n)]
    expect(1, cr.cr_all_reduce_host, h, [o[0], o[0]], 16, "f32", "sum", stream=0)
    expect(1, cr.cr_all_reduce_host, h, [h[1], o[1]], 16, "f32", "sum", stream=0)
    expect(1, cr.cr_all_reduce_host, h, o, 16, "f32", "sum", dev_out=[d[0], o[1]], stream=0)
    expect(2, cr.cr_all_reduce_host, h, o, 16, "i32", "avg", stream=0)
    expect(3, cr.cr_all_reduce_host, [h[0] + 2, h[1]], o, 16, "f32", "sum", stream=0)
    expect(2, cr.cr_all_reduce_host, h * 17, o * 17, 16, "f32", "sum", dev_out=d * 17, stream=0)
    cr.cr_all_reduce_host(h, o, 0, "f32", "sum", stream=0)


def test_fsdp2_and_accumulate_validation(L):
    n = 2
    g = [FAKE + k * (1 << 20) for k in range(2 * n)]
    p = [FAKE + (1 << 28) + k * (1 << 20) for k in range(2 * n)]
    ms = [FAKE + (2 << 28) + k * (1 << 20) for k in range(2 * n)]
    mm = [FAKE + (3 << 28) + k * (1 << 20) for k in range(2 * n)]
    v = [FAKE + (4 << 28) + k * (1 << 20) for k in range(2 * n)]
    shapes = [(4, 3), (1, 8)]   # second parameter: rank 1's shard is empty
    expect(1, cr.cr_fsdp2_step, shapes, 65, g, ms, mm, v, cr.adamw_cfg(), p, stream=0)
    expect(1, cr.cr_fsdp2_step, shapes, n, g, ms, mm, v, cr.adamw_cfg(step=0), p, stream=0)
    expect(1, cr.cr_fsdp2_step, shapes, n, g, ms, mm, [v[0], ms[0], v[2], v[3]], cr.adamw_cfg(),
           p, stream=0)
    expect(1, cr.cr_fsdp2_step, shapes, n, g[:2] + [0, g[3]], ms, mm, v, cr.adamw_cfg(), p, stream=0)
    expect(3, cr.cr_fsdp2_step, shapes, n, g, [ms[0] + 2] + ms[1:], mm, v, cr.adamw_cfg(), p,
           stream=0)
    a = [FAKE + r * (1 << 20) for r in range(n)]
    gr = [FAKE + (1 << 30) + r * (1 << 20) for r in range(n)]
    expect(2, cr.cr_accumulate, a, 16, gr, "i32", stream=0)
    expect(1, cr.cr_accumulate, a, 16, [a[0], gr[1]], "f32", stream=0)
    expect(3, cr.cr_all_reduce_accumulate, [a[0] + 2, a[1]], 16, gr, "f32", "avg", stream=0)
    expect(1, cr.cr_all_reduce_accumulate, a, 16, gr, "f32", 9, stream=0)
    cr.cr_accumulate(a, 0, gr, "bf16", stream=0)


def test_fsdp2_plan_host_side(L):
    """cr_fsdp2_plan_create checks what cr_fsdp2_step checks and builds the
    table on the host; the table's size follows its layout (tile prefix
    sums padded to 16 bytes, 48 bytes per non-empty parameter, 5N pointers
    each).  Upload and the planned step reject a NULL or misaligned table, a
    short table_bytes and a bad AdamW configuration before any copy or
    launch (every pointer here is fake)."""
    n = 2
    g = [FAKE + k * (1 << 20) for k in range(3 * n)]
    p = [FAKE + (1 << 28) + k * (1 << 20) for k in range(3 * n)]
    ms = [FAKE + (2 << 28) + k * (1 << 20) for k in range(3 * n)]
    mm = [FAKE + (3 << 28) + k * (1 << 20) for k in range(3 * n)]
    v = [FAKE + (4 << 28) + k * (1 << 20) for k in range(3 * n)]
    shapes = [(4, 3), (0, 5), (1, 8)]   # an empty parameter; rank 1's shard of the last is empty
    expect(1, cr.cr_fsdp2_plan_create, shapes, 65, g, ms, mm, v, p)
    expect(1, cr.cr_fsdp2_plan_create, shapes, n, g[:1] + [0] + g[2:], ms, mm, v, p)
    expect(3, cr.cr_fsdp2_plan_create, shapes, n, g, [ms[0] + 2] + ms[1:], mm, v, p)
    expect(1, cr.cr_fsdp2_plan_create, shapes, n, g, ms, mm, [v[0], ms[0]] + v[2:], p)
    plan = cr.cr_fsdp2_plan_create(shapes, n, g, ms, mm, v, p)
    nonempty = 2
    assert plan.table_bytes == 16 + 48 * nonempty + 8 * 5 * n * nonempty
    assert cr.cr_fsdp2_plan_table_bytes(None) == 0
    expect(1, cr.cr_fsdp2_plan_upload, plan, 0, plan.table_bytes, stream=0)
    expect(3, cr.cr_fsdp2_plan_upload, plan, FAKE + 8, plan.table_bytes, stream=0)
    expect(1, cr.cr_fsdp2_plan_upload, plan, FAKE, plan.table_bytes - 1, stream=0)
    expect(1, cr.cr_fsdp2_step_planned, plan, 0, cr.adamw_cfg(), stream=0)
    expect(3, cr.cr_fsdp2_step_planned, plan, FAKE + 8, cr.adamw_cfg(), stream=0)
    expect(1, cr.cr_fsdp2_step_planned, plan, FAKE, cr.adamw_cfg(step=0), stream=0)
    expect(1, cr.cr_fsdp2_step_planned, None, FAKE, cr.adamw_cfg(), stream=0)
    empty = cr.cr_fsdp2_plan_create([], n, [], [], [], [], [])
    assert empty.table_bytes == 16
    del plan, empty


def test_range_forms_validation(L):
    """The range forms check the range, the slab-local buffers and their
    overlaps before anything else, and an empty range has nothing to do
    (every pointer here is fake)."""
    n, count = 4, 1000
    L_ = cr.cr_chunk_len(count, n)
    ins = [FAKE + r * (1 << 20) for r in range(n)]
    outs = [FAKE + (1 << 30) + r * (1 << 20) for r in range(n)]
    for lo, hi in ((5, 4), (0, count + 1), (count + 1, count + 1)):
        expect(1, cr.cr_all_reduce_range, ins, count, lo, hi, "f32", "sum", outs, "f32", stream=0)
        expect(1, cr.cr_reduce_scatter_range, ins, count, lo, hi, "f32", "sum", outs, "f32",
               stream=0)
        expect(1, cr.cr_fsdp_step_range, ins, count, lo, hi, outs, outs, outs, cr.adamw_cfg(),
               ins, stream=0)
    # element alignment of the slab pointers, NULL buffers, overlapping outputs
    expect(3, cr.cr_all_reduce_range, [ins[0] + 2] + ins[1:], count, 0, 10, "f32", "sum", outs,
           "f32", stream=0)
    expect(1, cr.cr_all_reduce_range, [0] + ins[1:], count, 0, 10, "f32", "sum", outs, "f32",
           stream=0)
    expect(1, cr.cr_all_reduce_range, ins, count, 0, 10, "f32", "sum", [outs[0]] * n, "f32",
           stream=0)
    expect(2, cr.cr_all_reduce_range, ins, count, 0, 10, "i32", "avg", outs, "i32", stream=0)
    # reduce-scatter parts: shard 0's part of [0, L + 5) is L elements, shard 1's 5
    expect(1, cr.cr_reduce_scatter_range, ins, count, 0, L_ + 5, "f32", "sum",
           [outs[0], 0, 0, 0], "f32", stream=0)
    # empty ranges: valid, nothing launched
    cr.cr_all_reduce_range(ins, count, 7, 7, "f32", "sum", outs, "f32", stream=0)
    cr.cr_reduce_scatter_range(ins, count, 7, 7, "f32", "sum", [0] * n, "f32", stream=0)
    cr.cr_fsdp_step_range(ins, count, 7, 7, [0] * n, [0] * n, [0] * n, cr.adamw_cfg(), outs,
                          stream=0)


def test_wire_validation(L):
    n = 4
    bufs = [FAKE + r * (1 << 20) for r in range(n)]
    outs = [FAKE + (1 << 30) + r * (1 << 20) for r in range(n)]
    # the wire is f32 or bf16, and a bf16 wire needs floating inputs
    expect(1, cr.cr_all_reduce_wire, bufs, 16, "f32", "sum", "i32", outs, "f32", stream=0)
    expect(1, cr.cr_reduce_scatter_wire, bufs, 16, "f32", "sum", 7, outs, "f32", stream=0)
    expect(2, cr.cr_all_reduce_wire, bufs, 16, "i32", "sum", "bf16", outs, "i32", stream=0)
    expect(2, cr.cr_reduce_scatter_wire, bufs, 16, "i32", "sum", "bf16", outs, "i32", stream=0)
    # everything else is checked as for the f32-wire collectives
    expect(2, cr.cr_all_reduce_wire, bufs, 16, "f32", "sum", "bf16", outs, "bf16", stream=0)
    expect(3, cr.cr_reduce_scatter_wire, [bufs[0] + 1] + bufs[1:], 16, "bf16", "sum", "bf16",
           outs, "bf16", stream=0)
    expect(1, cr.cr_all_reduce_wire, bufs, 16, "f32", "sum", "bf16", [bufs[1]] + outs[1:], "f32",
           stream=0)
    cr.cr_all_reduce_wire(bufs, 0, "f32", "sum", "bf16", outs, "f32", stream=0)
    cr.cr_reduce_scatter_wire(bufs, 0, "bf16", "avg", "bf16", [0] * n, "bf16", stream=0)


def test_hsdp_validation(L):
    R, S = 2, 3
    n = R * S
    bufs = [FAKE + r * (1 << 20) for r in range(n)]
    outs = [FAKE + (1 << 30) + r * (1 << 20) for r in range(n)]
    expect(1, cr.cr_hsdp_reduce_scatter, bufs, 0, S, 16, "f32", "sum", outs, "f32", stream=0)
    expect(1, cr.cr_hsdp_reduce_scatter, bufs, R, 0, 16, "f32", "sum", outs, "f32", stream=0)
    expect(1, cr.cr_hsdp_reduce_scatter, bufs * 11, 9, 8, 16, "f32", "sum", outs * 11, "f32",
           stream=0)
    expect(2, cr.cr_hsdp_reduce_scatter, bufs, R, S, 16, "i32", "avg", outs, "i32", stream=0)
    expect(2, cr.cr_hsdp_reduce_scatter, bufs, R, S, 16, "f32", "sum", outs, "bf16", stream=0)
    expect(3, cr.cr_hsdp_reduce_scatter, [bufs[0] + 2] + bufs[1:], R, S, 16, "f32", "sum", outs,
           "f32", stream=0)
    expect(1, cr.cr_hsdp_reduce_scatter, bufs[:5] + [0], R, S, 16, "f32", "sum", outs, "f32",
           stream=0)
    # shard 0 of group 1 inside rank (0, 0)'s input
    bad = list(outs)
    bad[S] = bufs[0] + 4
    expect(1, cr.cr_hsdp_reduce_scatter, bufs, R, S, 16, "f32", "sum", bad, "f32", stream=0)
    # two groups' copies of shard 1 overlapping
    bad = list(outs)
    bad[S + 1] = outs[1] + 4
    expect(1, cr.cr_hsdp_reduce_scatter, bufs, R, S, 16, "f32", "sum", bad, "f32", stream=0)
    # in place needs equal dtypes
    L_ = cr.cr_chunk_len(48, S)
    inpl = [bufs[g * S + j] + j * L_ * 2 for g in range(R) for j in range(S)]
    expect(1, cr.cr_hsdp_reduce_scatter, bufs, R, S, 48, "bf16", "sum", inpl, "f32", stream=0)
    cr.cr_hsdp_reduce_scatter(bufs, R, S, 0, "f32", "sum", [0] * n, "f32", stream=0)


def test_reducer_validation(L):
    """Argument errors of the DDP reducer, all detected before any CUDA
    call (no reducer is ever created on FAKE pointers)."""
    plan = cr.cr_bucket_plan([8, 16, 4], 2, 40)
    T = plan.ntensors
    t = [FAKE + k * 4096 for k in range(2 * T)]
    expect(1, cr.cr_reducer_create, plan, 2, t, "bf16", "avg", comm_ctas=-1, comm_stream=0)
    expect(1, cr.cr_reducer_create, plan, 0, t, "bf16", "avg", comm_stream=0)
    expect(1, cr.cr_reducer_create, plan, 2, t, "f32", "avg", comm_stream=0)   # elem size 4 != 2
    expect(2, cr.cr_reducer_create, plan, 2, t, "i32", "avg", comm_stream=0)
    expect(3, cr.cr_reducer_create, plan, 2, [t[0] + 1] + t[1:], "bf16", "sum", comm_stream=0)
    expect(1, cr.cr_reducer_create, plan, 2, [t[0], t[0]] + t[2:], "bf16", "sum", comm_stream=0)
    expect(1, cr.cr_reducer_create, plan, 2, t[:-1] + [0], "bf16", "sum", comm_stream=0)
    null = cr.Reducer(0)
    expect(1, cr.cr_reducer_mark_ready, null, 0, compute_stream=0)
    expect(1, cr.cr_reducer_finalize, null, compute_stream=0)
    assert cr.cr_reducer_launched(null) == -1
    cr.cr_reducer_destroy(null)
    L.cr_reducer_destroy(None)

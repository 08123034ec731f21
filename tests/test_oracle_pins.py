"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each test checks the oracle against the pages' worked examples (fixtures in
tests/golden, each with its source), closed forms, exact arithmetic, brute
force on tiny inputs, or an independent library routine.  A plausible slip in
the oracle -- a wrong ring direction, a dropped contribution, an off-by-one
chunk bound, a transposed operand in AdamW -- fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
from fsdp_emulated_ranks_gb300 import inputs as I

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def bitmask_buffers(n, count_per_chunk=1):
    """x_{j,i} = 1 << (n*j + i) as int32: every partial sum names its
    contributors exactly (n*n <= 31 bits)."""
    bufs = []
    for i in range(n):
        b = np.zeros(n * count_per_chunk, np.int32)
        for j in range(n):
            b[j * count_per_chunk:(j + 1) * count_per_chunk] = 1 << (n * j + i)
        bufs.append(b)
    return bufs


def mask_of(contribs, n):
    return sum(1 << (n * j + i) for j, i in contribs)


# ---- a1: chunking ------------------------------------------------------------

def test_uneven_shards_match_pages(golden_dir):
    g = load(golden_dir, "uneven_shards.json")
    for case in g["cases"]:
        got = [list(O.chunk_bounds(case["dim0"], case["world_size"], j))
               for j in range(case["world_size"])]
        assert got == case["rows"], case


def test_flat_parameter_example(golden_dir):
    g = load(golden_dir, "flat_parameter_example.json")
    n = g["world_size"]
    total = g["total_numel"]
    assert [list(O.chunk_bounds(total, n, j)) for j in range(n)] == g["shards"]
    # Contiguous, unpadded offsets in visit order: the planner visits from the
    # last index, so hand it the parameters reversed to get registration order.
    numels = [p["numel"] for p in g["params"]][::-1]
    plan = O.bucket_plan(numels, 4, 1 << 30)
    assert plan.nbuckets == 1
    offs = plan.tensor_offset[::-1]
    for p, off in zip(g["params"], offs):
        assert [int(off), int(off) + p["numel"]] == p["range"]
    # The shard boundary splits the named parameter.
    split = [p for p in g["params"] if p["range"][0] < g["shards"][0][1] < p["range"][1]]
    assert [p["name"] for p in split] == [g["split_param"]]


@pytest.mark.parametrize("count", [0, 1, 7, 8, 13, 64, 1000])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 8, 64])
def test_chunks_partition_buffer(count, n):
    bounds = [O.chunk_bounds(count, n, j) for j in range(n)]
    assert bounds[0][0] == 0 and bounds[-1][1] == count
    for (a, b), (c, d) in zip(bounds, bounds[1:]):
        assert b == c and a <= b
    assert all(b - a <= math.ceil(count / n) for a, b in bounds)


# ---- a2: ring reduce-scatter schedule ---------------------------------------

def test_ring_reduce_scatter_trace_n4(golden_dir):
    g = load(golden_dir, "ring_reduce_scatter_n4.json")
    n = g["n"]
    shards, tr, (chunks, values) = O.ring_reduce_scatter(
        bitmask_buffers(n), "i32", "sum", trace=True)
    for s, step in enumerate(g["steps"]):
        assert list(chunks[s]) == step["sends"], f"step {s + 1}"
        for rank, contribs in step["held_after"].items():
            assert int(values[s][int(rank)]) == mask_of(contribs, n), (s, rank)
    final = g["steps"][-1]["held_after"]
    for j in range(n):
        assert int(shards[j][0]) == mask_of(final[str(j)], n)
    assert tr.steps == n - 1


def test_ring_reduce_scatter_two_rank_example():
    # FSDP1 unit1 with world_size 2: y_0 = x_00 + x_01, y_1 = x_10 + x_11.
    shards, _ = O.ring_reduce_scatter(bitmask_buffers(2, 7), "i32", "sum")
    assert np.all(shards[0] == (1 << 0) + (1 << 1))
    assert np.all(shards[1] == (1 << 2) + (1 << 3))


def order_from_trace(golden):
    """For each chunk j, the order in which ranks' contributions were added,
    read from the page's final partials."""
    final = golden["steps"][-1]["held_after"]
    return {int(r): [i for _, i in contribs] for r, contribs in final.items()}


def test_fold_order_matches_page_schedule(golden_dir):
    """Random fp32 inputs: the oracle's shard j must equal the left fold in
    exactly the page's order of contributions (fp32 addition is not
    associative, so any other order differs somewhere)."""
    g = load(golden_dir, "ring_reduce_scatter_n4.json")
    order = order_from_trace(g)
    n, count = 4, 4 * 257
    bufs = I.host_rank_buffers(n, count, "f32", std=1.0, seed0=11)
    sim, _ = O.ring_reduce_scatter(bufs, "f32", "sum")
    L = count // n
    for j in range(n):
        seg = [b[j * L:(j + 1) * L] for b in bufs]
        acc = seg[order[j][0]].copy()
        for i in order[j][1:]:
            acc = (acc + seg[i]).astype(np.float32)
        assert np.array_equal(sim[j].view(np.uint32), acc.view(np.uint32)), j
    # And a different association does give different bits somewhere.
    naive = [(seg := [b[j * L:(j + 1) * L] for b in bufs])[0] + seg[1] + seg[2] + seg[3]
             for j in range(n)]
    assert any(not np.array_equal(naive[j], sim[j]) for j in range(n))


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 8, 13, 16])
@pytest.mark.parametrize("count", [1, 5, 64, 999])
@pytest.mark.parametrize("dt", ["f32", "bf16", "i32"])
def test_simulation_equals_closed_form_fold(n, count, dt):
    bufs = I.host_rank_buffers(n, count, dt, seed0=100 + n)
    for op, out in [("sum", dt)] + ([("avg", dt), ("avg", "f32")] if dt != "i32" else []):
        sim, _ = O.ring_reduce_scatter(bufs, dt, op, out)
        fold = O.fold_reduce_scatter(bufs, dt, op, out)
        for a, b in zip(sim, fold):
            assert a.tobytes() == b.tobytes(), (op, out)


def _columns(bufs, count, n, L, idx):
    """The sampled elements' values on ranks 0..n-1 and the chunk each
    element belongs to, as the full-size checks gather them."""
    vals = np.stack([b[idx] for b in bufs], axis=1)
    return vals, (idx // L).astype(np.int32)


@pytest.mark.parametrize("n", [2, 3, 4, 8, 13, 64])
@pytest.mark.parametrize("dt,op,out", [("f32", "sum", "f32"), ("f32", "avg", "f32"),
                                       ("bf16", "sum", "bf16"), ("bf16", "avg", "bf16"),
                                       ("bf16", "avg", "f32"), ("bf16", "sum", "f32"),
                                       ("i32", "sum", "i32")])
def test_fold_columns_equals_ring_simulation(n, dt, op, out):
    """The per-element fold used at full size must give, for every
    sampled element, the bytes the literal ring simulation gives for that
    element: same chunk owner, same starting rank, same association, same
    single AVG division and bf16 rounding.  count is chosen so L = ceil(C/N)
    leaves a short last chunk (and empty ones for large N)."""
    count = 5 * n + 3 if n < 64 else 200
    L = math.ceil(count / n)
    bufs = I.host_rank_buffers(n, count, dt, std=1.0, seed0=300 + n)
    sim, _ = O.ring_reduce_scatter(bufs, dt, op, out)
    flat = np.concatenate(sim)
    assert flat.size == count
    idx = np.arange(count)
    vals, chunk = _columns(bufs, count, n, L, idx)
    got = O.fold_columns(vals, chunk, dt, op, out)
    assert got.tobytes() == flat.tobytes()
    # A random subset in shuffled order, as the sampled checks use it.
    rng = np.random.default_rng(n)
    sub = rng.permutation(count)[: max(1, count // 3)]
    vals, chunk = _columns(bufs, count, n, L, sub)
    assert O.fold_columns(vals, chunk, dt, op, out).tobytes() == flat[sub].tobytes()


def test_fold_columns_follows_page_schedule_n4(golden_dir):
    """Against the N=4 ring schedule of the reduce-scatter figure: for each
    chunk, the left fold in the order the trace's final partials list."""
    order = order_from_trace(load(golden_dir, "ring_reduce_scatter_n4.json"))
    n, count = 4, 4 * 301
    L = count // n
    bufs = I.host_rank_buffers(n, count, "f32", std=1.0, seed0=21)
    vals, chunk = _columns(bufs, count, n, L, np.arange(count))
    got = O.fold_columns(vals, chunk, "f32", "sum")
    for e in range(count):
        j = e // L
        acc = np.float32(vals[e, order[j][0]])
        for i in order[j][1:]:
            acc = np.float32(acc + vals[e, i])
        assert got[e].tobytes() == acc.tobytes(), e


@pytest.mark.parametrize("n", [4, 5, 8])
def test_fold_columns_detects_rotated_start(n):
    """Negative check: giving each element the chunk of its neighbour (a
    fold that starts one rank later) changes fp32 bits somewhere, and so do
    a reversed rank order and a divide-by-N applied per addend.  So a slip
    in the per-element fold's (j + k) mod N indexing or in its AVG cannot pass the
    pin above by accident."""
    count = 64 * n
    L = count // n
    bufs = I.host_rank_buffers(n, count, "f32", std=1.0, seed0=700 + n)
    vals, chunk = _columns(bufs, count, n, L, np.arange(count))
    right = O.fold_columns(vals, chunk, "f32", "sum")
    rotated = O.fold_columns(vals, (chunk + 1) % n, "f32", "sum")
    assert np.any(right.view(np.uint32) != rotated.view(np.uint32))
    reversed_order = O.fold_columns(vals[:, ::-1].copy(), (n - 1 - chunk) % n, "f32", "sum")
    assert np.any(right.view(np.uint32) != reversed_order.view(np.uint32))
    avg = O.fold_columns(vals, chunk, "f32", "avg")
    per_addend = O.fold_columns((vals / np.float32(n)).astype(np.float32), chunk, "f32", "sum")
    if n & (n - 1):   # for powers of two both forms are exact scalings
        assert np.any(avg.view(np.uint32) != per_addend.view(np.uint32))
    else:
        assert avg.tobytes() == per_addend.tobytes()


@pytest.mark.parametrize("n", [2, 3, 4, 7, 8, 16, 64])
def test_ring_equals_naive_on_integer_values(n):
    """Integer-valued fp32 with |x| <= 2^10: every partial is exact, so the
    ring must reduce to the textbook sum computed by the naive schedule."""
    count = 3 * n + 5
    bufs = I.integer_valued_f32(n, count, seed=n)
    ring, _ = O.ring_all_reduce(bufs, "f32", "sum")
    naive, _ = O.naive_all_reduce(bufs, "f32", "sum")
    exact = np.sum(np.stack(bufs).astype(np.float64), axis=0)
    for r in range(n):
        assert np.array_equal(ring[r], naive[r])
        assert np.array_equal(ring[r].astype(np.float64), exact)


@pytest.mark.parametrize("n", [2, 3, 4])
@pytest.mark.parametrize("count", [1, 2, 5, 12])
def test_brute_force_tiny(n, count):
    """Exact rational sum, the recursive-summation error bound, and the one
    association the ring fixes, enumerated by hand for N <= 4."""
    rng = np.random.default_rng(1000 * n + count)
    bufs = [(rng.standard_normal(count) * rng.choice([1e-3, 1.0, 1e3], count))
            .astype(np.float32) for _ in range(n)]
    shards, _ = O.ring_reduce_scatter(bufs, "f32", "sum")
    L = math.ceil(count / n)
    u = 2.0 ** -24
    f = np.float32
    for e in range(count):
        j = e // L
        got = float(shards[j][e - j * L])
        xs = [bufs[i][e] for i in range(n)]
        exact = sum(Fraction(float(x)) for x in xs)
        bound = (n - 1) * u * sum(abs(float(x)) for x in xs)
        assert abs(Fraction(got) - exact) <= Fraction(bound) * (1 + 1e-12)
        x = lambda k: xs[(j + k) % n]
        if n == 2:
            want = f(x(1) + x(0))
        elif n == 3:
            want = f(f(x(1) + x(2)) + x(0))
        else:
            want = f(f(f(x(1) + x(2)) + x(3)) + x(0))
        assert np.float32(got).tobytes() == np.float32(want).tobytes()


# ---- a3: average and cast -----------------------------------------------------

@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_avg_is_sum_divided_once(n):
    bufs = I.host_rank_buffers(n, 40 * n, "f32", seed0=5)
    s, _ = O.ring_reduce_scatter(bufs, "f32", "sum")
    a, _ = O.ring_reduce_scatter(bufs, "f32", "avg")
    for x, y in zip(s, a):
        want = np.array([np.float32(v) / np.float32(n) for v in x], np.float32)
        assert np.array_equal(want, y)
        if n & (n - 1) == 0:   # power of two: exact scaling
            assert np.array_equal(x * np.float32(1.0 / n), y)


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(3)
    x = np.concatenate([
        rng.standard_normal(100000).astype(np.float32) * 10.0 ** rng.integers(-30, 30, 100000),
        np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, 3.3895313892515355e38,
                  np.finfo(np.float32).max, np.inf, -np.inf, 1e-40, -1e-45,
                  np.finfo(np.float32).tiny], np.float32)])
    # Exact ties: 1 + 2^-8 (round down to even) and 1 + 3*2^-8 (round up).
    got = O.f32_to_bf16(x)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, want)
    assert O.f32_to_bf16(np.array([1.00390625], np.float32))[0] == 0x3F80
    assert O.f32_to_bf16(np.array([1.01171875], np.float32))[0] == 0x3F82
    nan = O.f32_to_bf16(np.array([np.nan], np.float32))[0]
    assert (nan & 0x7F80) == 0x7F80 and (nan & 0x7F) != 0


def test_bf16_avg_output_rounds_once():
    n = 8
    bufs = I.host_rank_buffers(n, 64 * n, "bf16", std=0.02, seed0=0)
    f32, _ = O.ring_reduce_scatter(bufs, "bf16", "avg", "f32")
    b16, _ = O.ring_reduce_scatter(bufs, "bf16", "avg", "bf16")
    for a, b in zip(f32, b16):
        assert np.array_equal(O.f32_to_bf16(a), b)


# ---- a4 / a5: all-gather and all-reduce -------------------------------------

def test_ring_all_gather_trace_n4(golden_dir):
    g = load(golden_dir, "ring_all_gather_n4.json")
    n = g["n"]
    shards = [np.full(3, 10 + j, np.int32) for j in range(n)]
    bufs, tr, arrival = O.ring_all_gather(shards, 3 * n, "i32", trace=True)
    contents = [list(c) for c in g["initial"]]
    for s, step in enumerate(g["steps"]):
        for r in range(n):
            contents[r].append(int(arrival[s][r]))
            # what r received at step s is what r-1 sent
            assert int(arrival[s][r]) == step["sends"][(r - 1) % n]
        assert contents == step["contents_after"], f"step {s + 1}"
    for r in range(n):
        assert list(bufs[r][::3] - 10) == g["final_by_shard_index"][r]
    assert tr.steps == n - 1


@pytest.mark.parametrize("n,count", [(1, 9), (2, 9), (4, 1 << 12), (5, 23), (8, 8 * 37 + 3), (64, 200)])
@pytest.mark.parametrize("dt,op,out", [("f32", "sum", "f32"), ("bf16", "avg", "bf16"),
                                       ("bf16", "avg", "f32"), ("i32", "sum", "i32")])
def test_all_reduce_is_all_gather_of_reduce_scatter(n, count, dt, op, out):
    bufs = I.host_rank_buffers(n, count, dt, seed0=n + count)
    ar, _ = O.ring_all_reduce(bufs, dt, op, out)
    rs, _ = O.ring_reduce_scatter(bufs, dt, op, out)
    ag, _ = O.ring_all_gather(rs, count, out)
    for r in range(n):
        assert ar[r].tobytes() == ag[r].tobytes()
        assert ar[r].tobytes() == np.concatenate(rs).tobytes()


# ---- a11: traffic counters and the cost model -------------------------------

@pytest.mark.parametrize("n", [2, 4, 8, 16, 64])
def test_traffic_ring_vs_naive(n):
    count = 64 * n
    bufs = I.integer_valued_f32(n, count, seed=1)
    _, ring = O.ring_all_reduce(bufs, "f32", "sum")
    _, naive = O.naive_all_reduce(bufs, "f32", "sum")
    # ring: every rank sends 2(N-1)/N of the buffer, over 2(N-1) steps
    assert ring.sent == [2 * (n - 1) * count // n] * n
    assert ring.recv == ring.sent
    assert ring.steps == 2 * (n - 1)
    # naive: the root receives and sends (N-1) full buffers
    root = naive.sent[0] + naive.recv[0]
    assert root == 2 * (n - 1) * count
    assert all(naive.sent[r] == count and naive.recv[r] == count for r in range(1, n))
    # both move the same total over all links
    assert sum(ring.sent) == sum(naive.sent) == 2 * (n - 1) * count
    assert root == n * ring.sent[0]


def test_traffic_uneven_chunks():
    n, count = 4, 10     # chunks of 3, 3, 3, 1
    bufs = I.integer_valued_f32(n, count, seed=2)
    _, rs = O.ring_reduce_scatter(bufs, "f32", "sum")
    lens = [b - a for a, b in (O.chunk_bounds(count, n, j) for j in range(n))]
    # rank r sends every chunk but its own in reduce-scatter
    assert rs.sent == [count - lens[r] for r in range(n)]


def test_cost_figures(golden_dir):
    g = load(golden_dir, "cost_figures.json")
    ab = g["alpha_beta_64MiB_8ranks"]
    n, S = ab["n"], ab["bytes"]
    for key in ("intra_node", "inter_node"):
        c = ab[key]
        t = O.alpha_beta_ring_allreduce(n, S, c["alpha_s"], c["bw_Bps"])
        alpha_term = O.alpha_beta_ring_allreduce(n, 0.0, c["alpha_s"], c["bw_Bps"])
        assert alpha_term == pytest.approx(c["alpha_term_s"], rel=1e-9)
        assert t - alpha_term == pytest.approx(c["beta_term_s"], rel=0.01)
        assert t == pytest.approx(c["total_s"], rel=0.01)
    rv = g["ring_vs_naive_8ranks"]
    n = rv["n"]
    count = 8 * 1024
    bufs = I.integer_valued_f32(n, count, seed=3)
    _, ring = O.ring_all_reduce(bufs, "f32", "sum")
    _, naive = O.naive_all_reduce(bufs, "f32", "sum")
    assert ring.sent[0] / count == rv["ring_per_rank_in_S"]
    assert (naive.sent[0] + naive.recv[0]) / count == rv["naive_in_S"]
    d7 = g["ddp_7b_8xh100"]
    per_card = 2 * (d7["n"] - 1) / d7["n"] * d7["grad_bytes"]
    assert per_card == pytest.approx(d7["ring_per_card_bytes"], rel=1e-12)
    assert per_card / d7["bw_Bps"] == pytest.approx(d7["t_comm_s"], rel=0.01)
    d70 = g["ddp_70b_64gpus"]
    per_card = 2 * (d70["n"] - 1) / d70["n"] * d70["grad_bytes"]
    assert per_card == pytest.approx(d70["ring_per_card_bytes_approx"], rel=0.01)
    assert per_card / d70["bw_Bps"] == pytest.approx(d70["t_comm_s_approx"], rel=0.01)
    tp = g["tp_allreduce_per_call"]
    n, S = tp["n"], tp["bytes"]
    bufs = I.integer_valued_f32(n, S // 4 // 1024, seed=4)
    _, ring = O.ring_all_reduce(bufs, "f32", "sum")
    assert ring.sent[0] * 4 * 1024 == tp["ring_per_card_bytes"]


# ---- a6 / a7: buckets -----------------------------------------------------------

CAP = 25 * 1024 * 1024


def check_plan_rules(numels, esize, cap, plan):
    t = len(numels)
    tb, to, bn = plan.tensor_bucket, plan.tensor_offset, plan.bucket_numel
    # visit order: from the last tensor to the first, buckets in that order
    order = list(range(t - 1, -1, -1))
    buckets_seen = [int(tb[i]) for i in order]
    assert buckets_seen == sorted(buckets_seen)
    assert (buckets_seen[0] if t else 0) == 0
    for b in range(plan.nbuckets):
        members = [i for i in order if tb[i] == b]
        assert members, "empty bucket"
        # contiguous, unpadded offsets in visit order
        off = 0
        for i in members:
            assert int(to[i]) == off
            off += int(numels[i])
        assert int(bn[b]) == off
        nbytes = off * esize
        assert nbytes <= cap or len(members) == 1
        # greedy: the next bucket's first tensor did not fit here
        if b + 1 < plan.nbuckets:
            first_next = [i for i in order if tb[i] == b + 1][0]
            assert nbytes + int(numels[first_next]) * esize > cap
            assert nbytes > 0


@pytest.mark.parametrize("seed", range(5))
def test_bucket_plan_rules_random(seed):
    rng = np.random.default_rng(seed)
    numels = rng.integers(0, 5000, size=rng.integers(0, 60)).astype(np.uint64)
    for cap in (1, 64, 4000, 10000, 1 << 20):
        plan = O.bucket_plan(numels, 2, cap)
        check_plan_rules(numels, 2, cap, plan)


def test_bucket_plan_workload_sizes():
    numels = I.bucket_numels()
    plan = O.bucket_plan(numels, 2, CAP)
    check_plan_rules(numels, 2, CAP, plan)
    assert int(plan.bucket_numel.sum()) == int(numels.sum())
    # oversize tensors (> 12.5 Mi bf16 elements) sit alone
    for t in np.nonzero(numels * 2 > CAP)[0]:
        assert np.sum(plan.tensor_bucket == plan.tensor_bucket[t]) == 1


def test_bucket_pack_unpack_identity():
    n = 3
    numels = np.array([5, 0, 17, 1, 33, 8], np.uint64)
    plan = O.bucket_plan(numels, 2, 40)
    rng = np.random.default_rng(0)
    tensors = [[rng.integers(0, 65535, int(k)).astype(np.uint16) for k in numels]
               for _ in range(n)]
    buckets = O.bucket_pack(plan, tensors)
    for r in range(n):
        for t, k in enumerate(numels):
            b, off = plan.tensor_bucket[t], int(plan.tensor_offset[t])
            assert np.array_equal(buckets[r][b][off:off + int(k)], tensors[r][t])
    back = O.bucket_unpack(plan, buckets, np.uint16)
    for r in range(n):
        for t in range(len(numels)):
            assert np.array_equal(back[r][t], tensors[r][t])


def test_bucketed_all_reduce_equals_per_tensor_average_on_integers():
    """On integer-valued data (exact sums) and N = 4 (exact /4), the bucket
    pipeline equals the plain per-tensor mean."""
    n = 4
    numels = np.array([7, 100, 3, 64, 1, 250], np.uint64)
    plan = O.bucket_plan(numels, 4, 400)
    rng = np.random.default_rng(1)
    tensors = [[rng.integers(-512, 512, int(k)).astype(np.float32) for k in numels]
               for _ in range(n)]
    out = O.bucketed_all_reduce(plan, tensors, "f32", "avg")
    for t in range(len(numels)):
        want = np.mean(np.stack([tensors[r][t] for r in range(n)]).astype(np.float64), axis=0)
        for r in range(n):
            assert np.array_equal(out[r][t].astype(np.float64), want)


# ---- a9: AdamW ----------------------------------------------------------------

def test_adamw_step1_closed_form():
    """m = v = 0, t = 1: m = (1-b1) g, v = (1-b2) g^2, the bias corrections
    cancel, and p1 = p0 (1 - lr wd) - lr g / (|g| + eps)."""
    cfg = O.AdamWConfig()
    rng = np.random.default_rng(0)
    k = 20000
    g = (rng.standard_normal(k) * 10.0 ** rng.integers(-6, 1, k)).astype(np.float32)
    g[:3] = [0.0, 1e-9, -1e-9]
    p0 = (rng.standard_normal(k) * 0.02).astype(np.float32)
    p, m, v = p0.copy(), np.zeros(k, np.float32), np.zeros(k, np.float32)
    O.adamw(p, m, v, g, cfg)
    gd, pd = g.astype(np.float64), p0.astype(np.float64)
    want_p = pd * (1 - cfg.lr * cfg.weight_decay) - cfg.lr * gd / (np.abs(gd) + cfg.eps)
    u = 2.0 ** -24
    assert np.all(np.abs(p - want_p) <= 8 * u * (np.abs(pd) + cfg.lr))
    assert np.all(np.abs(m - 0.1 * gd) <= 4 * u * np.abs(gd))
    assert np.all(np.abs(v - 0.001 * gd * gd) <= 6 * u * gd * gd + 1e-45)
    # g = 0: pure decoupled decay
    assert p[0] == np.float32(p0[0] * np.float32(1 - cfg.lr * cfg.weight_decay))


def test_adamw_matches_torch_over_steps():
    """Against torch.optim.AdamW in float64, several steps with nonzero
    state; torch orders the operations differently, so agreement is to fp32
    rounding, not bitwise."""
    torch = pytest.importorskip("torch")
    cfgs = [O.AdamWConfig(), O.AdamWConfig(lr=3e-4, beta1=0.9, beta2=0.95, weight_decay=0.1)]
    for cfg in cfgs:
        rng = np.random.default_rng(7)
        k = 4096
        p = (rng.standard_normal(k) * 0.02).astype(np.float32)
        m = np.zeros(k, np.float32)
        v = np.zeros(k, np.float32)
        tp = torch.nn.Parameter(torch.from_numpy(p.astype(np.float64)))
        opt = torch.optim.AdamW([tp], lr=cfg.lr, betas=(cfg.beta1, cfg.beta2),
                                eps=cfg.eps, weight_decay=cfg.weight_decay)
        for step in range(1, 6):
            g = (rng.standard_normal(k) * 1e-3).astype(np.float32)
            cfg.step = step
            O.adamw(p, m, v, g, cfg)
            tp.grad = torch.from_numpy(g.astype(np.float64))
            opt.step()
            ref = tp.detach().numpy()
            st = opt.state[tp]
            assert np.max(np.abs(p - ref)) <= 1e-6 * np.max(np.abs(ref))
            assert np.max(np.abs(m - st["exp_avg"].numpy())) <= 1e-5 * np.max(np.abs(m))
            assert np.max(np.abs(v - st["exp_avg_sq"].numpy())) <= 1e-5 * np.max(np.abs(v))


# ---- a8..a10: FSDP step -----------------------------------------------------------

@pytest.mark.parametrize("n,count", [(2, 14), (4, 4 * 100), (8, 8 * 64 + 5), (3, 2)])
def test_fsdp_step_equals_unsharded_training_step(n, count):
    """The check the pages state for their FSDP simulation: the sharded
    update, re-gathered, equals one unsharded step on the full flat buffer
    (here bit for bit: AdamW is elementwise, so sharding changes no
    operation)."""
    cfg = O.AdamWConfig()
    grads = I.host_rank_buffers(n, count, "bf16", std=1e-3, seed0=1000)
    master_full = I.np_normal_f32(count, 0.02, 2000)
    shards = [slice(*O.chunk_bounds(count, n, j)) for j in range(n)]
    master = [master_full[s].copy() for s in shards]
    m = [np.zeros(s.stop - s.start, np.float32) for s in shards]
    v = [np.zeros(s.stop - s.start, np.float32) for s in shards]
    params = O.fsdp_step(grads, master, m, v, cfg)
    # unsharded: all-reduce AVG into fp32, AdamW on the whole buffer, cast
    g_full, _ = O.ring_all_reduce(grads, "bf16", "avg", "f32")
    p_full = master_full.copy()
    m_full = np.zeros(count, np.float32)
    v_full = np.zeros(count, np.float32)
    O.adamw(p_full, m_full, v_full, g_full[0], cfg)
    assert np.concatenate(master).tobytes() == p_full.tobytes()
    assert np.concatenate(m).tobytes() == m_full.tobytes()
    assert np.concatenate(v).tobytes() == v_full.tobytes()
    want = O.f32_to_bf16(p_full)
    for r in range(n):
        assert params[r].tobytes() == want.tobytes()


def test_fsdp_step_gradient_is_mean_of_ranks():
    """With integer-valued bf16 grads the averaged fp32 gradient is exact;
    step 1 from m = v = 0 then moves each master weight by
    -lr*sign(g) (|g| >> eps) after the decay."""
    n, count = 4, 64
    cfg = O.AdamWConfig()
    rng = np.random.default_rng(5)
    ints = [rng.integers(1, 20, count).astype(np.float32) * rng.choice([-1, 1], count)
            for _ in range(n)]
    grads = [O.f32_to_bf16(x) for x in ints]
    mean = np.mean(np.stack(ints).astype(np.float64), axis=0)
    master = [np.full(count // n, 0.5, np.float32) for _ in range(n)]
    m = [np.zeros(count // n, np.float32) for _ in range(n)]
    v = [np.zeros(count // n, np.float32) for _ in range(n)]
    O.fsdp_step(grads, master, m, v, cfg)
    got_m = np.concatenate(m).astype(np.float64)
    assert np.allclose(got_m, 0.1 * mean, rtol=1e-6, atol=0)
    want = 0.5 * (1 - cfg.lr * cfg.weight_decay) - cfg.lr * np.sign(mean)
    assert np.allclose(np.concatenate(master), want, rtol=0, atol=1e-7)


# ---- FSDP step with gradient-norm clipping ---------------------------------------

def clip_case(n, count, seed):
    grads = I.host_rank_buffers(n, count, "bf16", std=1e-3, seed0=seed)
    master_full = I.np_normal_f32(count, 0.02, seed + 1)
    sl = [slice(*O.chunk_bounds(count, n, j)) for j in range(n)]
    mk = lambda: ([master_full[s].copy() for s in sl],
                  [np.zeros(s.stop - s.start, np.float32) for s in sl],
                  [np.zeros(s.stop - s.start, np.float32) for s in sl])
    return grads, mk


@pytest.mark.parametrize("n,count", [(2, 14), (4, 400), (8, 8 * 64 + 5), (3, 2)])
def test_clip_with_large_max_norm_is_the_plain_step(n, count):
    grads, mk = clip_case(n, count, 50)
    cfg = O.AdamWConfig()
    a_master, a_m, a_v = mk()
    b_master, b_m, b_v = mk()
    pa = O.fsdp_step(grads, a_master, a_m, a_v, cfg)
    pb, norm = O.fsdp_step_clipped(grads, b_master, b_m, b_v, cfg, max_norm=1e30)
    for x, y in zip(pa + a_master + a_m + a_v, pb + b_master + b_m + b_v):
        assert x.tobytes() == y.tobytes()


@pytest.mark.parametrize("n,count", [(4, 4000), (8, 8 * 1000 + 3)])
def test_clip_norm_and_scaled_gradient(n, count):
    """The reported norm is numpy's 2-norm of the averaged fp32 gradient
    (an independent routine); with max_norm = norm / 4 the clipped gradient,
    read back from m = (1 - b1) g at step 1, has norm max_norm."""
    grads, mk = clip_case(n, count, 60)
    cfg = O.AdamWConfig()
    g_full, _ = O.ring_all_reduce(grads, "bf16", "avg", "f32")
    want_norm = float(np.linalg.norm(g_full[0].astype(np.float64)))
    master, m, v = mk()
    _, norm = O.fsdp_step_clipped(grads, master, m, v, cfg, max_norm=1e30)
    assert norm == pytest.approx(want_norm, rel=1e-12)
    master, m, v = mk()
    _, norm2 = O.fsdp_step_clipped(grads, master, m, v, cfg, max_norm=want_norm / 4)
    assert norm2 == norm
    g_clipped = np.concatenate(m).astype(np.float64) / (1 - cfg.beta1)
    # the clipped norm is max_norm * norm / (norm + 1e-6): slightly below max_norm
    want_clipped = (want_norm / 4) * want_norm / (want_norm + 1e-6)
    assert float(np.linalg.norm(g_clipped)) == pytest.approx(want_clipped, rel=1e-6)
    # elementwise: g' = fl(g * c) with c = fl32(max_norm / (norm + 1e-6))
    c = np.float32((want_norm / 4) / (norm + 1e-6))
    gp = (g_full[0] * c).astype(np.float32)
    want_m = np.float32(1 - cfg.beta1) * gp
    assert np.max(np.abs(np.concatenate(m) - want_m)) <= 2 ** -22 * np.max(np.abs(want_m))


@pytest.mark.parametrize("n,count", [(1, 37), (3, 3 * 40 + 2), (8, 8 * 64 + 5)])
@pytest.mark.parametrize("frac", [0.25, 10.0])
def test_clipped_step_at_its_own_coefficient(n, count, frac):
    """The GPU tests check the clipped step at every fp32 coefficient in the
    norm's tolerance window by composing oracle pieces (reduce-scatter,
    g * c, AdamW, cast, all-gather).  At the oracle's own coefficient that
    composition must be orc_fsdp_step_clipped, bit for bit, and the window
    must list that coefficient first."""
    from gpu_util import clip_coefficients, oracle_clipped_at
    grads, mk = clip_case(n, count, 90 + n)
    cfg = O.AdamWConfig()
    g_full, _ = O.ring_all_reduce(grads, "bf16", "avg", "f32")
    max_norm = frac * float(np.linalg.norm(g_full[0].astype(np.float64)))
    master, m, v = mk()
    want_p, norm = O.fsdp_step_clipped(grads, master, m, v, cfg, max_norm)
    coefs = clip_coefficients(max_norm, norm)
    assert coefs[0] == np.float32(min(1.0, max_norm / (norm + 1e-6)))
    assert len(set(float(c) for c in coefs)) == len(coefs)
    if frac > 1:
        assert coefs == [np.float32(1.0)]
    ms, mm, vv = mk()
    params = oracle_clipped_at(grads, ms, mm, vv, cfg, coefs[0])
    for a, b in zip(ms + mm + vv, master + m + v):
        assert a.tobytes() == b.tobytes()
    for a, b in zip(params, want_p):
        assert a.tobytes() == b.tobytes()
    # a neighbouring coefficient gives different state bits
    if frac < 1:
        ms, mm, vv = mk()
        oracle_clipped_at(grads, ms, mm, vv, cfg, np.nextafter(coefs[0], np.float32(2)))
        assert any(a.tobytes() != b.tobytes() for a, b in zip(mm, m))


# ---- FSDP2: per-parameter Shard(0) ----------------------------------------------

def test_fsdp2_unit1_shards_and_reduce_scatter(golden_dir):
    g = load(golden_dir, "fsdp2_unit1.json")
    n = g["world_size"]
    for p in g["params"]:
        for j in range(n):
            assert list(O.fsdp2_shard_rows(p["shape"][0], n, j)) == p["rows"][j], p["name"]
    # reduce-scatter of layer1.weight with bitmask payloads: x_{j,i} = row j
    # of rank i's gradient
    shape = [p for p in g["params"] if p["name"] == g["reduce_scatter"]["param"]][0]["shape"]
    rows, row_numel = shape[0], shape[1]
    bufs = []
    for i in range(n):
        b = np.zeros(rows * row_numel, np.int32)
        for j in range(rows):
            b[j * row_numel:(j + 1) * row_numel] = 1 << (2 * j + i)
        bufs.append(b)
    Lr = -(-rows // n)
    shards = O.ring_reduce_scatter_L(bufs, Lr * row_numel, "i32", "sum")
    rs = g["reduce_scatter"]
    assert np.all(shards[0] == mask_of(rs["rank0_row0"], 2))
    assert np.all(shards[1] == mask_of(rs["rank1_row1"], 2))


def test_fsdp2_uneven_and_empty_shards(golden_dir):
    u = load(golden_dir, "uneven_shards.json")
    for case in u["cases"]:
        got = [list(O.fsdp2_shard_rows(case["dim0"], case["world_size"], j))
               for j in range(case["world_size"])]
        assert got == case["rows"]


def fsdp2_case(shapes, n, seed):
    grads = [I.host_rank_buffers(n, d * rn, "bf16", std=1e-3, seed0=seed + 100 * p)
             for p, (d, rn) in enumerate(shapes)]
    master, m, v = [], [], []
    for p, (d, rn) in enumerate(shapes):
        full = I.np_normal_f32(d * rn, 0.02, seed + 7 * p + 1)
        row_m, row_mm, row_v = [], [], []
        for j in range(n):
            lo, hi = O.fsdp2_shard_rows(d, n, j)
            row_m.append(full[lo * rn:hi * rn].copy())
            row_mm.append(np.zeros((hi - lo) * rn, np.float32))
            row_v.append(np.zeros((hi - lo) * rn, np.float32))
        master.append(row_m); m.append(row_mm); v.append(row_v)
    return grads, master, m, v


SHAPES = [(2, 3), (2, 1), (3, 3), (5, 7), (1, 16), (9, 1), (0, 4), (16, 8)]


@pytest.mark.parametrize("n", [2, 3, 4])
def test_fsdp2_equals_unsharded_step_per_parameter(n):
    """The sharded update, re-gathered, equals one unsharded AdamW step on
    each full parameter after the averaging all-reduce (bit for bit)."""
    cfg = O.AdamWConfig()
    grads, master, m, v = fsdp2_case(SHAPES, n, 70)
    full0 = [np.concatenate(row) if row else np.zeros(0, np.float32) for row in master]
    params = O.fsdp2_step(SHAPES, grads, master, m, v, cfg)
    for p, (d, rn) in enumerate(SHAPES):
        if d * rn == 0:
            continue
        g_full, _ = O.ring_all_reduce(grads[p], "bf16", "avg", "f32")
        pf = full0[p].copy()
        mf = np.zeros_like(pf)
        vf = np.zeros_like(pf)
        O.adamw(pf, mf, vf, g_full[0], cfg)
        assert np.concatenate(master[p]).tobytes() == pf.tobytes(), p
        assert np.concatenate(m[p]).tobytes() == mf.tobytes(), p
        for r in range(n):
            assert params[p][r].tobytes() == O.f32_to_bf16(pf).tobytes(), (p, r)


@pytest.mark.parametrize("n,count", [(2, 14), (4, 64), (3, 10)])
def test_fsdp2_with_scalar_rows_is_the_flat_step(n, count):
    """A 1-D parameter of `count` entries is sharded like the flat buffer of
    the FSDP1 step, so both give identical bits."""
    cfg = O.AdamWConfig()
    grads, master, m, v = fsdp2_case([(count, 1)], n, 90)
    fm = [x.copy() for x in master[0]]
    fmm = [x.copy() for x in m[0]]
    fv = [x.copy() for x in v[0]]
    params2 = O.fsdp2_step([(count, 1)], grads, master, m, v, cfg)
    params1 = O.fsdp_step(grads[0], fm, fmm, fv, cfg)
    for r in range(n):
        assert params2[0][r].tobytes() == params1[r].tobytes()
    for a, b in zip(master[0] + m[0] + v[0], fm + fmm + fv):
        assert a.tobytes() == b.tobytes()


# ---- gradient accumulation (no_sync) ------------------------------------------------

@pytest.mark.parametrize("dt", ["f32", "bf16"])
def test_accumulate_is_fp32_addition(dt):
    rng = np.random.default_rng(3)
    acc = rng.standard_normal(1000).astype(np.float32)
    g = I.host_rank_buffers(1, 1000, dt, std=1e-2, seed0=4)[0]
    want = acc + (O.bf16_to_f32(g) if dt == "bf16" else g)
    O.accumulate(acc, g, dt)
    assert acc.tobytes() == want.astype(np.float32).tobytes()
    # integer-valued micro-steps accumulate exactly
    acc = np.zeros(16, np.float32)
    for k in range(1, 5):
        O.accumulate(acc, np.full(16, float(k), np.float32), "f32")
    assert np.all(acc == 10.0)


# ---- low-precision wire -----------------------------------------------------------

@pytest.mark.parametrize("n", [2, 3, 4, 8])
def test_wire_f32_is_the_plain_ring(n):
    bufs = I.host_rank_buffers(n, 8 * n * 9 + 3, "bf16", std=0.02, seed0=n)
    a = O.ring_all_reduce_wire(bufs, "bf16", "avg", "f32")
    b, _ = O.ring_all_reduce(bufs, "bf16", "avg")
    for x, y in zip(a, b):
        assert x.tobytes() == y.tobytes()


@pytest.mark.parametrize("n", [2, 4, 8])
def test_wire_bf16_exact_when_partials_are_representable(n):
    """Integers with every partial sum below 2^8 in magnitude are exact in
    bf16, so rounding the messages changes nothing."""
    rng = np.random.default_rng(n)
    ints = [rng.integers(-256 // n, 256 // n, size=8 * n * 5).astype(np.float32) for _ in range(n)]
    bufs = [O.f32_to_bf16(x) for x in ints]
    out = O.ring_all_reduce_wire(bufs, "bf16", "sum", "bf16", "f32")
    exact = np.sum(np.stack(ints).astype(np.float64), axis=0)
    for r in range(n):
        assert np.array_equal(out[r].astype(np.float64), exact)


@pytest.mark.parametrize("n", [3, 4, 8])
def test_wire_bf16_rounds_each_hop(n):
    """Against the hand-written hop sequence (torch's bf16 rounding, an
    independent routine): p = x_{j+1}; p = bf16(p) + x_k for the next ranks;
    and within the per-hop rounding bound of the exact sum."""
    torch = pytest.importorskip("torch")
    count = 8 * n * 4
    bufs = I.host_rank_buffers(n, count, "f32", seed0=20 + n)
    shards = O.ring_reduce_scatter_wire(bufs, "f32", "sum", "bf16")
    L = count // n
    rb = lambda x: torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).float().numpy()
    u = 2.0 ** -8
    for j in range(n):
        seg = [b[j * L:(j + 1) * L] for b in bufs]
        p = seg[(j + 1) % n].copy()
        bound = np.zeros(L)
        for k in range(2, n + 1):
            bound += u * np.abs(p.astype(np.float64))
            p = (rb(p) + seg[(j + k) % n]).astype(np.float32)
        assert shards[j].tobytes() == p.tobytes(), j
        exact = np.sum(np.stack(seg).astype(np.float64), axis=0)
        err = np.abs(shards[j].astype(np.float64) - exact)
        assert np.all(err <= bound * 1.01 + n * 2.0 ** -23 * np.abs(np.stack(seg)).sum(0))


# ---- HSDP (shard groups x replicas) ------------------------------------------------

@pytest.mark.parametrize("S", [1, 2, 4])
def test_hsdp_one_replica_is_reduce_scatter(S):
    bufs = I.host_rank_buffers(S, 8 * S * 7 + 1, "bf16", std=0.02, seed0=S)
    h = O.hsdp_reduce_scatter(bufs, 1, S, "bf16", "avg", "f32")
    rs, _ = O.ring_reduce_scatter(bufs, "bf16", "avg", "f32")
    for a, b in zip(h, rs):
        assert a.tobytes() == b.tobytes()


@pytest.mark.parametrize("R", [2, 3, 4])
def test_hsdp_one_rank_per_group_is_all_reduce(R):
    bufs = I.host_rank_buffers(R, 8 * R * 7 + 3, "f32", seed0=R)
    h = O.hsdp_reduce_scatter(bufs, R, 1, "f32", "sum")
    ar, _ = O.ring_all_reduce(bufs, "f32", "sum")
    for g in range(R):
        assert h[g].tobytes() == ar[g].tobytes()


@pytest.mark.parametrize("R,S", [(2, 2), (2, 4), (4, 2), (3, 3)])
def test_hsdp_integer_sum_is_exact_and_replicated(R, S):
    n = R * S
    count = 4 * n + 3
    ints = I.integer_valued_f32(n, count, seed=R * 10 + S)
    h = O.hsdp_reduce_scatter(ints, R, S, "f32", "sum")
    exact = np.sum(np.stack(ints).astype(np.float64), axis=0)
    for g in range(R):
        full = np.concatenate(h[g * S:(g + 1) * S])
        assert np.array_equal(full.astype(np.float64), exact)
    # AVG divides the whole sum by N once
    ha = O.hsdp_reduce_scatter(ints, R, S, "f32", "avg")
    for g in range(R):
        full = np.concatenate(ha[g * S:(g + 1) * S])
        assert np.array_equal(full, (exact.astype(np.float32) / np.float32(n)).astype(np.float32))


def _hsdp_by_hand(x, R, S, count):
    """HSDP's association written out element by element from the two
    rings' conventions (reading of [AIG] 6.3.6 / [DT] section 4): shard
    j = e // L (L = ceil(count/S)); inside group g the ranks are added from
    s = j+1 round to s = j; the R group sums of shard j's offset k are added
    from group i+1 round to group i, where i = k // ceil(len_j / R).  x is
    [R*S][count] float32; returns [count] float32 sums."""
    f = np.float32
    L = -(-count // S)
    out = np.zeros(count, np.float32)
    for e in range(count):
        j, k = e // L, e % L
        len_j = min(L, count - j * L)
        i = k // -(-len_j // R)
        def inner(g):
            acc = f(x[g * S + (j + 1) % S][e])
            for t in range(2, S + 1):
                acc = f(acc + f(x[g * S + (j + t) % S][e]))
            return acc
        acc = inner((i + 1) % R)
        for t in range(2, R + 1):
            acc = f(acc + inner((i + t) % R))
        out[e] = acc
    return out


def _hsdp_slip(x, R, S, count, outer_from_shard, inner_from_zero):
    """_hsdp_by_hand with one plausible slip: the outer ring started at
    group j+1 (the shard index) instead of i+1, or the inner ring started
    at rank 0 instead of j+1."""
    f = np.float32
    L = -(-count // S)
    out = np.zeros(count, np.float32)
    for e in range(count):
        j, k = e // L, e % L
        len_j = min(L, count - j * L)
        i = k // -(-len_j // R)
        s0 = 0 if inner_from_zero else (j + 1) % S
        def inner(g):
            acc = f(x[g * S + s0][e])
            for t in range(1, S):
                acc = f(acc + f(x[g * S + (s0 + t) % S][e]))
            return acc
        g0 = (j + 1) % R if outer_from_shard else (i + 1) % R
        acc = inner(g0)
        for t in range(1, R):
            acc = f(acc + inner((g0 + t) % R))
        out[e] = acc
    return out


@pytest.mark.parametrize("R,S,count", [(2, 2, 4), (2, 3, 7), (3, 2, 11), (2, 2, 9), (3, 3, 13),
                                       (4, 3, 25)])
def test_hsdp_fold_order_by_hand(R, S, count):
    """The oracle's HSDP equals the hand-enumerated parenthesisation on
    random fp32 values, bit for bit.  With three or more operands the order
    matters (two-operand sums are commutative), and there each plausible
    slip -- outer ring started at the shard's index, inner ring started at
    rank 0 -- gives a different answer somewhere: the pin has teeth."""
    rng = np.random.default_rng(R * 100 + S * 10 + count)
    outer_hits = inner_hits = 0
    for trial in range(40):
        x = [(rng.standard_normal(count) * np.exp2(rng.integers(-12, 12, count))).astype(np.float32)
             for _ in range(R * S)]
        got = O.hsdp_reduce_scatter(x, R, S, "f32", "sum")
        want = _hsdp_by_hand(x, R, S, count)
        for g in range(R):
            assert np.concatenate(got[g * S:(g + 1) * S]).tobytes() == want.tobytes()
        outer_hits += _hsdp_slip(x, R, S, count, True, False).tobytes() != want.tobytes()
        inner_hits += _hsdp_slip(x, R, S, count, False, True).tobytes() != want.tobytes()
    if R >= 3:
        assert outer_hits > 0
    if S >= 3:
        assert inner_hits > 0

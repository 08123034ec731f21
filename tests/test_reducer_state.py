"""The DDP reducer's bookkeeping (csrc/reducer_state.h), compiled for the
host: a bucket's all-reduce may start once every gradient in it is ready,
and buckets start strictly in bucket-index order ("AI Infra Guide,
Chapter 6", 6.2.4-6.2.5).  Checked against a model written here from that
rule, on the workload's bucket plan and on random plans, for backward
order, random orders, repeated and out-of-range marks and resets."""
import os
import subprocess
import tempfile

import numpy as np
import pytest

from fsdp_emulated_ranks_gb300 import build as libbuild
from fsdp_emulated_ranks_gb300 import cr
from fsdp_emulated_ranks_gb300 import inputs as I

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    libbuild.build()   # the bucket plans come from libcr's planner


@pytest.fixture(scope="module")
def driver():
    with tempfile.TemporaryDirectory() as d:
        exe = os.path.join(d, "reducer_state_check")
        subprocess.run(["g++", "-O2", "-std=c++17", "-Wall", "-Werror", "-I",
                        os.path.join(ROOT, "fsdp_emulated_ranks_gb300", "csrc"),
                        os.path.join(ROOT, "tests", "reducer_state_check.cpp"), "-o", exe],
                       check=True)
        yield exe


def run(exe, scenarios):
    text = [str(len(scenarios))]
    for tb, nb, marks in scenarios:
        text += [f"{len(tb)} {nb}", " ".join(map(str, tb)) or "", str(len(marks)),
                 " ".join(map(str, marks))]
    res = subprocess.run([exe], input="\n".join(text) + "\n", capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    out, cur = [], None
    for line in res.stdout.splitlines():
        if line.startswith("scenario"):
            cur = {"complete0": line.endswith("=1"), "events": []}
            out.append(cur)
        elif line == "reset":
            cur["events"].append("reset")
        else:
            head, tail = line.split("|")
            rc, launched, complete = map(int, head.split())
            cur["events"].append((rc, launched, bool(complete), [int(x) for x in tail.split()]))
    return out


def model(tb, nb, marks):
    """Bucket b may start once all of its tensors, and all of buckets
    0..b-1, are ready; a tensor marked twice, or outside the plan, is an
    error that changes nothing."""
    members = [set() for _ in range(nb)]
    for t, b in enumerate(tb):
        members[b].add(t)
    ready, launched, events = set(), 0, []
    for t in marks:
        if t == -9:
            ready, launched = set(), 0
            events.append("reset")
            continue
        if not 0 <= t < len(tb):
            events.append((-1, launched, launched == nb, []))
            continue
        if t in ready:
            events.append((-2, launched, launched == nb, []))
            continue
        ready.add(t)
        new = []
        while launched < nb and members[launched] <= ready:
            new.append(launched)
            launched += 1
        events.append((0, launched, launched == nb, new))
    return events


def test_workload_plan_backward_order(driver):
    """The 300-tensor workload: gradients ready last tensor first, as the
    plan was built, so each bucket starts on its last tensor's mark."""
    plan = cr.cr_bucket_plan([int(k) for k in I.bucket_numels()], 2, 25 << 20)
    marks = list(range(plan.ntensors - 1, -1, -1))
    got = run(driver, [(plan.tensor_bucket, plan.nbuckets, marks)])[0]
    assert got["events"] == model(plan.tensor_bucket, plan.nbuckets, marks)
    starts = [e[3] for e in got["events"] if e[3]]
    assert [b for s in starts for b in s] == list(range(plan.nbuckets))
    assert all(len(s) == 1 for s in starts)  # one bucket per completing mark
    assert got["events"][-1][2]


@pytest.mark.parametrize("seed", range(12))
def test_random_plans_and_orders(driver, seed):
    rng = np.random.default_rng(seed)
    scen = []
    for _ in range(6):
        T = int(rng.integers(1, 60))
        numels = [int(x) for x in rng.integers(0, 5000, T)]
        plan = cr.cr_bucket_plan(numels, 4, int(rng.integers(1, 20000)))
        order = [int(x) for x in rng.permutation(T)]
        # errors mixed in: a repeat, an out-of-range index; then a reset and
        # a second iteration in backward order
        extra = [order[0], T, -1] if T > 1 else [T]
        marks = order[:T // 2] + extra + order[T // 2:] + [-9] + list(range(T - 1, -1, -1))
        scen.append((plan.tensor_bucket, plan.nbuckets, marks))
    got = run(driver, scen)
    for (tb, nb, marks), g in zip(scen, got):
        assert not g["complete0"]
        assert g["events"] == model(tb, nb, marks)


def test_empty_plan_is_complete(driver):
    got = run(driver, [([], 0, [0])])[0]
    assert got["complete0"]
    assert got["events"] == [(-1, 0, True, [])]

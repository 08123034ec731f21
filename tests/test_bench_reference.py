"""bench.py's reference arm (the CPU oracle) on every workload, on the CPU.

--impl reference times the oracle on a bounded sample of the workload the
other arm measures: the line names that workload, counts the sample's bytes
by the workload's own formula, and says what the sample was.  --config picks
the benchmark configurations by number and --seed shifts the input values
only.  --iters is another name for --steps.
"""
import argparse
import json

import pytest

import bench

NS = argparse.Namespace(bucket_ntensors=300, fsdp_count=1_300_000_000, fsdp2_layers=24,
                        fsdp2_hidden=2048)
WORKLOADS = ["allreduce", "allreduce_f32", "allreduce_wire", "reduce_scatter", "all_gather",
             "hsdp", "accumulate", "accumulate_allreduce", "fsdp", "fsdp_clipped", "fsdp2",
             "bucket_pack", "bucket_allreduce", "bucket_unpack", "bucket_pipeline",
             "bucket_fused"]


def reference_line(capsys, *extra):
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3",
                       "--ref-sample", "4096", *extra]) == 0
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    return json.loads(lines[0])


@pytest.mark.parametrize("workload", WORKLOADS)
def test_reference_arm_times_the_selected_workload(capsys, workload):
    d = reference_line(capsys, "--workload", workload)
    full = bench.make_workload(workload, NS, plan=False)
    assert d["impl"] == "reference" and d["config"]["workload"] == full.name
    assert d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["higher_is_better"] is True and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["sample"]


def test_sample_bytes_follow_the_workload_formula():
    ns, k = NS, 4096
    assert bench.OracleSample("allreduce", ns, k).nbytes == 2 * 8 * k * 2
    assert bench.OracleSample("reduce_scatter", ns, k).nbytes == 8 * k * 2 + k * 2
    assert bench.OracleSample("all_gather", ns, k).nbytes == k * 2 + 8 * k * 2
    assert bench.OracleSample("hsdp", ns, k).nbytes == 8 * k * 2 + 2 * k * 2
    assert bench.OracleSample("fsdp", ns, k).nbytes == (4 * 8 + 24) * k
    assert bench.OracleSample("fsdp_clipped", ns, k).nbytes == (4 * 8 + 32) * k
    assert bench.OracleSample("accumulate", ns, k).nbytes == 8 * k * 10
    smp = bench.OracleSample("bucket_pipeline", ns, k)
    P = round(smp.nbytes / (3 * 2 * 2 * 8))
    assert smp.nbytes == 3 * 2 * 2 * 8 * P and abs(P - k) <= 300


def test_config_numbers_and_seed(capsys):
    assert bench.CONFIGS[2] == "allreduce" and bench.CONFIGS[5] == "sweep"
    d4 = reference_line(capsys, "--config", "4")
    assert d4["config"]["workload"].startswith("fsdp_step_bf16_8ranks")
    d1 = reference_line(capsys, "--config", "1")
    assert d1["config"]["workload"] == "allreduce_sum_f32_4ranks_4MiB"
    # --seed shifts the values, not the workload or its bytes
    ns = NS
    a = bench.OracleSample("allreduce", ns, 256)
    out_a, _ = a.step()
    bench.SEED_OFFSET = 5
    try:
        b = bench.OracleSample("allreduce", ns, 256)
        out_b, _ = b.step()
    finally:
        bench.SEED_OFFSET = 0
    assert a.nbytes == b.nbytes
    assert any((x != y).any() for x, y in zip(out_a, out_b))


def test_iters_is_steps(capsys):
    d = reference_line(capsys, "--iters", "2")  # the later flag wins, as for --steps twice
    assert d["steps"] == 2
    assert d["cpu_baseline"]["cpu_model"]  # the host CPU is named beside the core count


def test_full_size_reference_has_the_other_arm_config(capsys):
    """At the workload's full size (here the 4 x 2^20 fp32 all-reduce) the
    reference line's config is the workload's own, with no sample key: both
    arms time the same configuration."""
    assert bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3",
                       "--workload", "allreduce_f32", "--ref-sample", str(1 << 20)]) == 0
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    d = json.loads(lines[0])
    full = bench.make_workload("allreduce_f32", NS, plan=False)
    assert d["config"] == bench.workload_config(full, 1)
    assert "sample" not in d["config"]
    assert "4 rank buffers of 1048576 elements" in d["cpu_baseline"]["sample"]


def test_fsdp_row_bytes():
    """(4N + 24) bytes per parameter for the plain step; the clipped step
    parks the averaged gradient for N >= 5, (4N + 32), and reads the
    gradients twice below that, (6N + 24)."""
    assert bench.FsdpStep(8, 100).nbytes == 56 * 100
    assert bench.FsdpStep(8, 100, clip=True).nbytes == 64 * 100
    assert bench.FsdpStep(5, 100, clip=True).nbytes == 52 * 100
    assert bench.FsdpStep(4, 100, clip=True).nbytes == 48 * 100
    assert bench.FsdpStep(2, 100, clip=True).nbytes == 36 * 100


def test_slab_workload_bytes():
    """--split slab: a GPU's share of the bytes is its slab's; the slabs of
    all GPUs add up to the whole workload's bytes."""
    for G in (1, 2, 3, 8):
        ar = [bench.AllReduce(slab=(lo, hi)) for lo, hi in
              (bench.slab_bounds(1 << 25, 8, G, g) for g in range(G))]
        assert sum(w.nbytes for w in ar) == ar[0].full_nbytes == bench.AllReduce().nbytes
        fs = [bench.FsdpStep(8, 1000, slab=(lo, hi)) for lo, hi in
              (bench.slab_bounds(1000, 8, G, g) for g in range(G))]
        assert sum(w.nbytes for w in fs) == fs[0].full_nbytes == 56 * 1000
    with pytest.raises(SystemExit):
        bench.FsdpStep(8, 1000, clip=True, slab=(0, 500))

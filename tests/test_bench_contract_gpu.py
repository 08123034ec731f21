"""bench.py keeps its contract: one JSON line with the metric, the
whole-job value, the roofline of the dominant kernel against the measured
peak, the end-to-end figure with its host<->device bytes, the CPU baseline,
clocks sampled during the timed region and the launch count; the reference
arm prints the same metric and unit with impl=reference.  Runs the real
benchmark briefly on the GPU."""
import json
import os
import subprocess
import sys

import pytest
import torch

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def run(args, timeout=900):
    res = subprocess.run([sys.executable, "bench.py"] + args, cwd=ROOT, capture_output=True,
                         text=True, timeout=timeout)
    assert res.returncode == 0, res.stderr[-3000:]
    lines = [l for l in res.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, res.stdout
    return json.loads(lines[0])


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")


def test_headline_line_has_every_key(tmp_path):
    jsonl = tmp_path / "rows.jsonl"
    d = run(["--steps", "20", "--warmup", "3", "--row-steps", "4", "--cpu-seconds", "1",
             "--cpu-sample", str(1 << 20), "--skip-fsdp", "--jsonl", str(jsonl)])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"):
        assert k in d, k
    assert d["n_gpus"] == 1 and d["steps"] == 20 and d["warmup"] >= 3
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["dtype"] == "f32"
    assert d["value"] > 0 and d["gpu_launches"] == 20
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-3
    e = d["e2e"]
    assert e["h2d_bytes_per_step"] == e["d2h_bytes_per_step"] == 8 * (1 << 25) * 2
    assert 0 < e["value"] < d["value"]
    c = d["cpu_baseline"]
    assert c["kind"] == "oracle" and c["cores"] == 1 and c["value"] > 0
    assert c["cpu_model"]
    assert d["clocks"]["sm_mhz"] > 0 and "reasons" in d["clocks"]
    f = d["l2_flushed"]  # the same step with L2 flushed before each call
    assert f["steps"] >= 20 and f["flush_bytes"] > 2 * (128 << 20) and f["GB/s"] > 0
    assert f["clean"]["ms_median"] > 0   # and with the flush's dirty lines written back first
    assert d["config"]["workload"] == "allreduce_avg_bf16_8ranks_64MiB"
    names = [row["name"] for row in d["rows"]]
    assert "reduce_scatter_avg_bf16_8ranks_64MiB" in names and len(names) >= 10
    for row in d["rows"]:
        assert row["ms_p10"] <= row["ms_median"] <= row["ms_p90"]
    summ = d["rows_summary"]   # every row, compactly, as the line's last key
    assert list(d)[-1] == "rows_summary"
    assert "allreduce" in summ and len(summ) == 1 + len(d["rows"])
    assert summ["allreduce"][2] == r["frac_median"] and summ["allreduce"][3] == r["frac"]
    cfg1 = next(row for row in d["rows"] if row["key"] == "allreduce_f32")
    assert "graph_us" in cfg1 and cfg1["l2_flushed"]["ms_median"] > 0
    assert summ["allreduce_f32"][-2:] == [cfg1["l2_flushed"]["ms_median"],
                                          cfg1["l2_flushed"]["frac"]]
    recs = [json.loads(l) for l in jsonl.read_text().splitlines()]
    assert len(recs) == 1 + len(d["rows"]) and recs[0]["name"] == d["config"]["workload"]
    for k in ("ms_median", "ms_p10", "ms_p90", "algorithmic_bytes", "cpu_baseline"):
        assert k in recs[0], k
    assert all(r["host_cores"] >= 1 and r["peak_GBs"] > 0 for r in recs)


def test_reference_arm_matches_the_metric():
    mine = run(["--steps", "5", "--warmup", "3", "--no-rows", "--no-e2e", "--no-cpu-baseline"])
    ref = run(["--impl", "reference", "--steps", "1", "--warmup", "3",
               "--ref-sample", str(1 << 18)])
    assert ref["impl"] == "reference"
    for k in ("metric", "unit", "higher_is_better", "dtype"):
        assert ref[k] == mine[k], k
    assert ref["config"]["workload"] == mine["config"]["workload"]
    assert ref["e2e"]["h2d_bytes_per_step"] == 0 and ref["cpu_baseline"]["kind"] == "oracle"


@pytest.mark.parametrize("config,workload", [(1, "allreduce_sum_f32_4ranks_4MiB"),
                                             (3, "_bucket_pipeline_bf16_8ranks")])
def test_config_flag_selects_the_same_workload_in_both_arms(config, workload):
    mine = run(["--config", str(config), "--steps", "5", "--warmup", "3", "--no-rows",
                "--no-e2e", "--no-cpu-baseline"])
    ref = run(["--impl", "reference", "--config", str(config), "--steps", "1", "--warmup", "3",
               "--ref-sample", str(1 << 16)])
    assert workload in mine["config"]["workload"]
    assert ref["config"]["workload"] == mine["config"]["workload"]
    assert mine["value"] > 0 and mine["gpu_launches"] >= 5
    assert mine["roofline"]["bound"] == "hbm" and mine["roofline"]["achieved"] > 0
    for k in ("metric", "unit", "higher_is_better", "dtype"):
        assert ref[k] == mine[k], k


@pytest.mark.parametrize("workload", ["allreduce", "fsdp"])
def test_slab_split_on_one_gpu(workload):
    """--split slab on one GPU: the single slab is the whole element range,
    run through the range entry point; same workload and bytes, strong
    scaling."""
    extra = ["--fsdp-count", str(8 * 1000 * 1000)] if workload == "fsdp" else []
    d = run(["--workload", workload, "--split", "slab", "--steps", "5", "--warmup", "3",
             "--no-rows", "--no-e2e", "--no-cpu-baseline"] + extra)
    whole = run(["--workload", workload, "--steps", "5", "--warmup", "3", "--no-rows",
                 "--no-e2e", "--no-cpu-baseline"] + extra)
    assert d["scaling"] == "strong" and whole["scaling"] == "weak"
    assert d["config"]["workload"] == whole["config"]["workload"]
    assert d["roofline"]["algorithmic_bytes_per_launch"] == \
        whole["roofline"]["algorithmic_bytes_per_launch"]
    assert d["value"] > 0

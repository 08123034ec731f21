#!/usr/bin/env python
"""Benchmark of the emulated-rank gradient collectives on one GB300 per rank.

Headline workload: all-reduce AVG of 8 emulated ranks' bf16 gradient
buffers of 33,554,432 elements (64 MiB) each, fp32 accumulation in ring
order, 1/8 fused, bf16 result written back to all 8 buffers (in place, as
DDP does with its gradient buckets).  A step is one cr_all_reduce call.

Metric: effective HBM GB/s per collective call = algorithmic bytes (each
input element read once + each output element written once) / device time,
and its fraction of the measured HBM peak.  Inputs (512 MiB) exceed the
129 MB L2, so no flush is needed between iterations.

Also reported on the same line (N = 1): every other row of the hot path
measured the same way ("rows"), the end-to-end figure through the C ABI
with the inputs copied from pinned host memory and the results copied back
inside the timed region ("e2e"), SM clocks sampled during the timed region
("clocks"), the roofline of the dominant kernel, and the CPU oracle timed on
a bounded sample of the workload on this host ("cpu_baseline").

Multi-GPU (torchrun, one process per GPU): every rank runs its own instance
of the workload (its own 8 emulated ranks); nothing is exchanged on the data
path, so scaling is weak and value = sum of all ranks' bytes / max time.

--impl reference times the CPU oracle (the only reference implementation
this method has) on bounded samples of the same workload.
--sweep runs the message-size / rank-count sweep and fits T = a + bytes/B.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "effective HBM GB/s per collective call and % of GB300 HBM peak (1 GPU)"
UNIT = "GB/s"
HEADLINE = "allreduce_avg_bf16_8ranks_64MiB"
FALLBACK_HBM_GBS = 6800.0


# ---- environment ---------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device=None) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_rank: float, total_ms: float, steps: int, world: int,
                   device=None) -> tuple[float, float]:
    """Whole-job GB/s over all ranks: every rank moved bytes_per_rank per
    step; the job's time is the slowest rank's.  Returns (GB/s, ms/step)."""
    ms = max_over_ranks(total_ms, world, device) / steps
    return world * bytes_per_rank / (ms * 1e-3) / 1e9, ms


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, burst copy)"
    return FALLBACK_HBM_GBS, "fallback"


# ---- clocks during the timed region --------------------------------------------

_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
            0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
            0x2: "applications_clocks_setting", 0x10: "sync_boost"}


class ClockSampler:
    """Polls the SM clock and the clock-event reasons through NVML (read only)
    every ~2 ms on a background thread while the timed region runs."""

    def __init__(self, torch_device):
        self.samples = []
        self.max_mhz = None
        self._h = None
        self._stop = threading.Event()
        try:
            nv = ctypes.CDLL("libnvidia-ml.so.1")
            if nv.nvmlInit_v2() != 0:
                return
            h = ctypes.c_void_p()
            import torch
            uuid = str(getattr(torch.cuda.get_device_properties(torch_device), "uuid", ""))
            ok = False
            if uuid:
                u = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
                ok = nv.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) == 0
            props = torch.cuda.get_device_properties(torch_device)
            if not ok and hasattr(props, "pci_bus_id"):
                bus = "%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0),
                                            props.pci_bus_id, props.pci_device_id)
                ok = nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0
            if not ok:
                ok = nv.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) == 0
            if not ok:
                return
            self._nv, self._h = nv, h
            mx = ctypes.c_uint()
            if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            fn = getattr(nv, "nvmlDeviceGetCurrentClocksEventReasons", None)
            self._reasons_fn = fn or nv.nvmlDeviceGetCurrentClocksThrottleReasons
        except OSError:
            self._h = None

    def _run(self):
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            a = self._nv.nvmlDeviceGetClockInfo(self._h, 1, ctypes.byref(clk))
            b = self._reasons_fn(self._h, ctypes.byref(rs))
            if a == 0 and b == 0:
                self.samples.append((clk.value, rs.value))
            time.sleep(0.002)

    def __enter__(self):
        if self._h is not None:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *exc):
        if self._h is not None:
            self._stop.set()
            self._t.join()

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [],
                    "samples": 0, "source": "unavailable"}
        mhz = [s[0] for s in self.samples]
        bits = 0
        for _, r in self.samples:
            bits |= r
        reasons = sorted(name for bit, name in _REASONS.items() if bits & bit)
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples), "source": "nvml"}


# ---- timing ------------------------------------------------------------------------

def timed(fn, steps, warmup, world, stream, sampler=None):
    """W untimed calls, then exactly `steps` calls between CUDA events on the
    launching stream, bracketed by barrier + synchronize.  Returns
    (total_ms, per_step_ms list)."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ctx = sampler if sampler is not None else _Null()
    with ctx:
        ev[0].record(stream)
        for i in range(steps):
            fn()
            ev[i + 1].record(stream)
        torch.cuda.synchronize()
    barrier(world)
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    return ev[0].elapsed_time(ev[steps]), per


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


# ---- workloads -----------------------------------------------------------------------

def alloc_ranks(n, count, dtype, std, seed0, device):
    import torch
    from fsdp_emulated_ranks_gb300 import inputs as I
    bufs = []
    for r in range(n):
        t = torch.empty(count, dtype=dtype, device=device)
        I.torch_fill_normal_(t, std, seed0 + r)
        bufs.append(t)
    return bufs


def ar_bytes(n, count, esize):
    return 2 * n * count * esize


def run_headline(args, world, rank, device, stream, peak):
    import torch
    from fsdp_emulated_ranks_gb300 import cr
    n, count = 8, 1 << 25
    bufs = alloc_ranks(n, count, torch.bfloat16, 0.02, 0, device)
    # Sample for the CPU baseline before the in-place calls overwrite it.
    sample = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample = [b[:args.cpu_sample].view(torch.int16).cpu().numpy().view("uint16") for b in bufs]

    def step():
        cr.cr_all_reduce(bufs, count, "bf16", "avg", bufs, "bf16", stream)

    sampler = ClockSampler(device)
    total_ms, per = timed(step, args.steps, args.warmup, world, stream, sampler)
    nbytes = ar_bytes(n, count, 2)
    value, ms_step = job_throughput(nbytes, total_ms, args.steps, world, device)
    kern_ms = statistics.mean(per)
    achieved = nbytes / (kern_ms * 1e-3) / 1e9
    out = {
        "ms_per_step": ms_step,
        "value": value,
        "clocks": sampler.summary(),
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak[0],
                     "unit": "GB/s", "frac": round(achieved / peak[0], 4),
                     "traffic": traffic_per_launch("k_fold_vec_allreduce_bf16_8x64MiB"),
                     "kernel": "k_fold_vec<bf16,bf16,AR,8>",
                     "algorithmic_bytes_per_launch": nbytes,
                     "peak_source": peak[1],
                     "kernel_ms_median": statistics.median(per)},
    }
    # End to end through the C ABI from pinned host memory.
    out["e2e"] = None if args.no_e2e else run_e2e(args, bufs, n, count, world, stream, device)
    del bufs
    torch.cuda.empty_cache()
    return out, sample


def run_e2e(args, bufs, n, count, world, stream, device):
    import torch
    from fsdp_emulated_ranks_gb300 import cr
    host_in = [torch.empty(count, dtype=torch.bfloat16, pin_memory=True) for _ in range(n)]
    host_out = [torch.empty(count, dtype=torch.bfloat16, pin_memory=True) for _ in range(n)]
    for h, b in zip(host_in, bufs):
        h.copy_(b)
    torch.cuda.synchronize()

    def step():
        for h, b in zip(host_in, bufs):
            b.copy_(h, non_blocking=True)
        cr.cr_all_reduce(bufs, count, "bf16", "avg", bufs, "bf16", stream)
        for h, b in zip(host_out, bufs):
            h.copy_(b, non_blocking=True)

    steps = max(3, min(args.steps, 50))
    total_ms, _ = timed(step, steps, max(3, min(args.warmup, 5)), world, stream)
    nbytes = ar_bytes(n, count, 2)
    value, ms = job_throughput(nbytes, total_ms, steps, world, device)
    return {"value": round(value, 2), "unit": UNIT,
            "h2d_bytes_per_step": n * count * 2, "d2h_bytes_per_step": n * count * 2,
            "ms_per_step": ms, "steps": steps}


def traffic_per_launch(name):
    """DRAM bytes per launch from the committed ncu summary of this kernel,
    or None if absent or taken on a different build of the library."""
    p = os.path.join(ROOT, "profiles", name + ".md")
    if not os.path.exists(p):
        return None
    vals = {}
    with open(p) as f:
        for line in f:
            if ":" in line and line.strip().startswith(("dram_bytes_per_launch", "libcr_source_hash")):
                k, v = line.split(":", 1)
                vals[k.strip(" -*`")] = v.strip(" `\n")
    try:
        from fsdp_emulated_ranks_gb300 import build as B
        if vals.get("libcr_source_hash") != B.source_hash():
            return None
        return int(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ---- the other rows (N = 1) ------------------------------------------------------------

def row(name, nbytes, per, peak, launches):
    ms = statistics.mean(per) if per else float("nan")
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"name": name, "ms": round(ms, 4), "GB/s": round(gbs, 1),
            "frac": round(gbs / peak[0], 4), "algorithmic_bytes": nbytes,
            "launches_per_call": launches}


def run_rows(args, device, stream, peak):
    import torch
    from fsdp_emulated_ranks_gb300 import cr
    from fsdp_emulated_ranks_gb300 import inputs as I
    rows = []
    K, W = args.row_steps, 3

    # a1-a5 on the headline size: reduce-scatter, all-gather.
    n, count = 8, 1 << 25
    bufs = alloc_ranks(n, count, torch.bfloat16, 0.02, 0, device)
    L = count // n
    shards = [torch.empty(L, dtype=torch.bfloat16, device=device) for _ in range(n)]
    _, per = timed(lambda: cr.cr_reduce_scatter(bufs, count, "bf16", "avg", shards, "bf16", stream),
                   K, W, 1, stream)
    rows.append(row("reduce_scatter_avg_bf16_8x64MiB", n * count * 2 + count * 2, per, peak, 1))
    _, per = timed(lambda: cr.cr_all_gather(shards, count, "bf16", bufs, stream), K, W, 1, stream)
    rows.append(row("all_gather_bf16_8x64MiB", count * 2 + n * count * 2, per, peak, 1))
    del bufs, shards
    torch.cuda.empty_cache()

    # all-reduce SUM fp32, 4 ranks x 2^20 (fits in L2: latency regime).
    n, count = 4, 1 << 20
    bufs = alloc_ranks(n, count, torch.float32, 1.0, 0, device)
    _, per = timed(lambda: cr.cr_all_reduce(bufs, count, "f32", "sum", bufs, "f32", stream),
                   K, W, 1, stream)
    rows.append(row("allreduce_sum_f32_4x4MiB", ar_bytes(n, count, 4), per, peak, 1))
    del bufs
    torch.cuda.empty_cache()

    # a6/a7: DDP buckets, 300 bf16 tensors per rank, 25 MiB buckets.
    n = 8
    numels = [int(k) for k in I.bucket_numels()]
    P = sum(numels)
    plan = cr.cr_bucket_plan(numels, 2, 25 * 1024 * 1024)
    tens = []
    for r in range(n):
        flat = torch.empty(P + 128 * len(numels), dtype=torch.bfloat16, device=device)
        I.torch_fill_normal_(flat, 1e-3, 1000 + r)
        off, row_t = 0, []
        for k in numels:
            row_t.append(flat[off:off + k])
            off += (k + 127) // 128 * 128
        tens.append(row_t)
    bks = []
    for r in range(n):
        sizes = [(int(k) + 127) // 128 * 128 for k in plan.bucket_numel]
        flat = torch.empty(sum(sizes), dtype=torch.bfloat16, device=device)
        off, row_b = 0, []
        for k, s in zip(plan.bucket_numel, sizes):
            row_b.append(flat[off:off + int(k)])
            off += s
        bks.append(row_b)
    flat_t = [x for rr in tens for x in rr]
    flat_b = [x for rr in bks for x in rr]
    copy_launches = -(-n * len(numels) // 1024)
    _, per = timed(lambda: cr.cr_bucket_pack(plan, n, flat_t, flat_b, stream), K, W, 1, stream)
    rows.append(row("bucket_pack_bf16_8x300", 2 * 2 * P * n, per, peak, copy_launches))
    _, per = timed(lambda: cr.cr_bucket_all_reduce(plan, n, flat_b, "bf16", "avg", stream), K, W, 1,
                   stream)
    rows.append(row("bucket_allreduce_avg_bf16_8x300", 2 * 2 * P * n, per, peak, plan.nbuckets))
    _, per = timed(lambda: cr.cr_bucket_unpack(plan, n, flat_b, flat_t, stream), K, W, 1, stream)
    rows.append(row("bucket_unpack_bf16_8x300", 2 * 2 * P * n, per, peak, copy_launches))

    def pipeline():
        cr.cr_bucket_pack(plan, n, flat_t, flat_b, stream)
        cr.cr_bucket_all_reduce(plan, n, flat_b, "bf16", "avg", stream)
        cr.cr_bucket_unpack(plan, n, flat_b, flat_t, stream)
    _, per = timed(pipeline, max(3, K // 2), W, 1, stream)
    rows.append(row("ddp_bucket_pipeline_bf16_8x300", 3 * 2 * 2 * P * n, per, peak,
                    2 * copy_launches + plan.nbuckets))
    rows[-1]["total_params"] = P
    rows[-1]["nbuckets"] = plan.nbuckets
    del tens, bks, flat_t, flat_b
    torch.cuda.empty_cache()

    # a8-a10: fused FSDP step, 8 ranks, flat 1.3e9 parameters.
    if not args.skip_fsdp:
        n, count = 8, 1_300_000_000
        L = count // n
        grads = alloc_ranks(n, count, torch.bfloat16, 1e-3, 1000, device)
        params = [torch.empty(count, dtype=torch.bfloat16, device=device) for _ in range(n)]
        master_full = torch.empty(count, dtype=torch.float32, device=device)
        I.torch_fill_normal_(master_full, 0.02, 2000)
        master = [master_full[j * L:(j + 1) * L] for j in range(n)]
        mv = torch.zeros(2 * count, dtype=torch.float32, device=device)
        m = [mv[j * L:(j + 1) * L] for j in range(n)]
        v = [mv[count + j * L:count + (j + 1) * L] for j in range(n)]
        cfg = cr.adamw_cfg()
        _, per = timed(lambda: cr.cr_fsdp_step(grads, count, master, m, v, cfg, params, stream),
                       max(3, K // 4), W, 1, stream)
        rows.append(row("fsdp_step_bf16_8x1.3e9", (4 * n + 24) * count, per, peak, 1))
        del grads, params, master_full, master, mv, m, v
        torch.cuda.empty_cache()
    return rows


# ---- CPU oracle -------------------------------------------------------------------------

def cpu_oracle_allreduce(sample):
    """Ring all-reduce AVG of the sampled bf16 rank buffers by the CPU oracle
    (single-threaded); returns (GB/s, seconds)."""
    import oracle as O
    n, count = len(sample), sample[0].size
    O.ring_all_reduce(sample[:2], "bf16", "avg")  # load and warm the library
    t0 = time.perf_counter()
    O.ring_all_reduce(sample, "bf16", "avg")
    dt = time.perf_counter() - t0
    return ar_bytes(n, count, 2) / dt / 1e9, dt


def run_reference(args):
    """--impl reference: the CPU oracle on this host, bounded samples of the
    headline workload, same metric and unit."""
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return 0
    import numpy as np
    from fsdp_emulated_ranks_gb300 import inputs as I
    import oracle as O
    n, count = 8, args.ref_sample
    host = [I.np_to_bf16_bits(I.np_normal_f32(count, 0.02, r)) for r in range(n)]
    for _ in range(args.warmup):
        O.ring_all_reduce(host, "bf16", "avg")
    t0 = time.perf_counter()
    for _ in range(args.steps):
        out, _ = O.ring_all_reduce(host, "bf16", "avg")
    dt = time.perf_counter() - t0
    ms = dt * 1e3 / args.steps
    value = ar_bytes(n, count, 2) / (ms * 1e-3) / 1e9
    sample = (f"ring all-reduce AVG of 8 bf16 buffers of {count} elements per step "
              f"(1/{(1 << 25) // count} of the 64 MiB-per-rank workload), oracle/ C code")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32 accumulate, bf16 in/out",
            "data": "synthetic", "config": {"workload": HEADLINE, "ranks": 8,
                                            "elements_per_rank": 1 << 25,
                                            "sampled_elements_per_rank": count},
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---- sweep ----------------------------------------------------------------------------------

def run_sweep(args, device, stream, peak):
    """All-reduce AVG bf16: N = 8 over 1 KiB .. 1 GiB per rank (powers of 4)
    and N in {2,4,8,16,32,64} at 256 MiB per rank; fits T = a + bytes / B to
    the 8-rank points and reports the crossover S* = a * B."""
    import torch
    from fsdp_emulated_ranks_gb300 import cr
    pts = []
    for k in range(11):
        nbytes_rank = 1024 * 4 ** k
        pts.append((8, nbytes_rank // 2))
    for n in (2, 4, 16, 32, 64):
        pts.append((n, (256 << 20) // 2))
    out = []
    for n, count in pts:
        bufs = alloc_ranks(n, count, torch.bfloat16, 1.0, 0, device)
        steps = 50 if count < (1 << 22) else 10
        _, per = timed(lambda: cr.cr_all_reduce(bufs, count, "bf16", "avg", bufs, "bf16", stream),
                       steps, 3, 1, stream)
        ms = statistics.median(per)
        sent, _, _ = cr.cr_comm_elems(cr.COLL_ALL_REDUCE, cr.SCHED_RING, n, count, 0)
        out.append({"n": n, "bytes_per_rank": count * 2, "us": round(ms * 1e3, 2),
                    "GB/s": round(ar_bytes(n, count, 2) / (ms * 1e-3) / 1e9, 1),
                    "ring_bytes_per_rank": sent * 2})
        del bufs
        torch.cuda.empty_cache()
    # least squares on the 8-rank points: t = a + x / B, x = algorithmic bytes
    xs = [ar_bytes(8, p["bytes_per_rank"] // 2, 2) for p in out if p["n"] == 8]
    ts = [p["us"] * 1e-6 for p in out if p["n"] == 8]
    mx, mt = sum(xs) / len(xs), sum(ts) / len(ts)
    slope = sum((x - mx) * (t - mt) for x, t in zip(xs, ts)) / sum((x - mx) ** 2 for x in xs)
    a = mt - slope * mx
    bw = 1 / slope
    return {"points": out, "alpha_us": round(a * 1e6, 3), "bw_GBs": round(bw / 1e9, 1),
            "crossover_bytes": round(a * bw)}


# ---- main ---------------------------------------------------------------------------------

def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--no-rows", action="store_true")
    ap.add_argument("--skip-fsdp", action="store_true")
    ap.add_argument("--row-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-sample", type=int, default=1 << 24,
                    help="elements per rank the CPU oracle reduces for cpu_baseline")
    ap.add_argument("--ref-sample", type=int, default=1 << 21,
                    help="elements per rank per step for --impl reference")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)

    if args.impl == "reference":
        return run_reference(args)

    import torch
    from fsdp_emulated_ranks_gb300 import build as B
    from fsdp_emulated_ranks_gb300 import cr

    world, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (libcr has no CPU path)")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    init_dist(world, "nccl")
    if rank == 0:
        B.build()
    barrier(world)
    B.build()
    cr.lib()
    stream = torch.cuda.current_stream(device)
    peak = measured_peaks()

    if args.sweep:
        res = run_sweep(args, device, stream, peak)
        if rank == 0:
            print(json.dumps({"metric": METRIC, "unit": UNIT, "sweep": res,
                              "config": {"workload": "allreduce_avg_bf16_sweep"}}))
        return 0

    head, sample = run_headline(args, world, rank, device, stream, peak)
    rows = None
    if world == 1 and not args.no_rows:
        rows = run_rows(args, device, stream, peak)
    cpu = None
    if sample is not None:
        gbs, secs = cpu_oracle_allreduce(sample)
        cpu = {"value": round(gbs, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": (f"ring all-reduce AVG of the first {sample[0].size} elements of each "
                          f"of the 8 rank buffers (1/{(1 << 25) // sample[0].size} of the "
                          f"workload), single-threaded C oracle, {secs:.1f} s, host has "
                          f"{os.cpu_count()} cores")}
    if rank == 0:
        line = {"metric": METRIC, "value": round(head["value"], 1), "unit": UNIT,
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": head["ms_per_step"], "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                "data": "synthetic",
                "config": {"workload": HEADLINE, "ranks": 8, "elements_per_rank": 1 << 25,
                           "dtype_in_out": "bf16", "accumulate": "fp32, ring order",
                           "op": "avg, in place", "l2": "inputs 512 MiB > 129 MB L2, no flush",
                           "parallelism": f"{world} GPU(s) x 8 emulated ranks each"},
                "roofline": head["roofline"], "cpu_baseline": cpu, "e2e": head["e2e"],
                "gpu_launches": head["gpu_launches"], "clocks": head["clocks"],
                "frac_of_peak": round(head["value"] / world / peak[0], 4),
                "rows": rows}
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

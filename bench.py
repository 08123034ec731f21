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

Multi-GPU (torchrun, one process per GPU), two modes:
  --split replicas (default): every rank runs its own instance of the
      workload (its own 8 emulated ranks); nothing is exchanged on the data
      path, so scaling is weak and value = sum of all ranks' bytes / max time;
  --split slab: the G ranks share ONE workload (the all-reduce or the
      unclipped FSDP step), rank g holding and processing only slab g of
      every buffer's element range (cr_slab_range, whole chunks while G <= 8)
      through cr_all_reduce_range / cr_fsdp_step_range, which keep the whole
      buffers' chunking and so their fold order; nothing is exchanged either,
      scaling is strong and value = the workload's bytes / max time.

--impl reference times the CPU oracle (the only reference implementation
this method has) on bounded samples of the same workload.
--sweep runs the message-size / rank-count sweep and fits T = a + bytes/B.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import platform
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
FALLBACK_HBM_GBS = 6800.0


# ---- environment ---------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def init_dist(world, backend, timeout_s=600):
    """Process group of the N > 1 run.  Its timeout bounds every barrier and
    collective: a rank that dies or never arrives makes the others fail with
    an error after at most timeout_s instead of waiting forever."""
    import datetime
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend,
                                timeout=datetime.timedelta(seconds=timeout_s))
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


def host_cpu_model():
    """The host CPU's name for the oracle's report: /proc/cpuinfo's model
    name (x86), else lscpu's (Arm, whose /proc/cpuinfo lists part numbers
    only), else the machine type."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.machine()


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
    """W untimed calls, then exactly `steps` calls between two CUDA events on
    the launching stream, bracketed by barrier + synchronize: the total is
    the time of `steps` back-to-back calls, as a caller issues them.
    Returns (total_ms, per_step_ms list).

    The per-step list comes from a second pass of `steps` calls with an
    event recorded after each (outside the bracketed region).  An event
    between two calls keeps the second call's grid from being dispatched
    during the first one's last wave (the kernels are launched as
    programmatic dependents of their predecessor), so per-step times are
    each call on its own, slightly above total / steps.

    The clock sampler starts before the warm-up, so that its thread start
    does not delay the first timed launch, and samples throughout.  Right
    before each first event the stream gets a device-side wait (no memory
    traffic) as long as one host enqueue of a step plus 10 us (the last
    warm-up step's host time; 20-100 us): the first step is queued behind
    it, so the events time device work from the first step on, and a
    host-bound step gets no head start beyond its first enqueue.  (For the
    headline all-reduce the time per call is flat, 153.7-153.8 us, for any
    wait of 20 us or more, and 154.6 us at 5 us.)"""
    import torch
    ctx = sampler if sampler is not None else _Null()
    with ctx:
        host_s = 0.0
        for _ in range(warmup):
            t = time.perf_counter()
            fn()
            host_s = time.perf_counter() - t
        wait_s = min(max(host_s + 10e-6, 20e-6), 100e-6)
        torch.cuda.synchronize()
        barrier(world)
        torch.cuda.synchronize()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        device_wait(stream, wait_s)
        t0.record(stream)
        for _ in range(steps):
            fn()
        t1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    total = t0.elapsed_time(t1)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    device_wait(stream, wait_s)
    ev[0].record(stream)
    for i in range(steps):
        fn()
        ev[i + 1].record(stream)
    torch.cuda.synchronize()
    per = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    return total, per


def device_wait(stream, seconds):
    """About `seconds` of device-side spinning on `stream` (torch's sleep
    kernel, counted in SM cycles at about 2 GHz; nothing if this torch has
    none)."""
    import torch
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is not None:
        with torch.cuda.stream(stream):
            sleep(max(1, int(seconds * 2.0e9)))


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
        I.torch_fill_normal_(t, std, SEED_OFFSET + seed0 + r)
        bufs.append(t)
    return bufs


def ar_bytes(n, count, esize):
    return 2 * n * count * esize


class Workload:
    """One benchmarked call of the hot path: setup() allocates and fills the
    inputs, step(stream) issues the call(s), nbytes is the algorithmic bytes
    per step, launches the kernels one step launches."""
    name = kernel = profile = ""
    nbytes = 0
    launches = 1

    def setup(self, device):
        raise NotImplementedError

    def step(self, stream):
        raise NotImplementedError

    def teardown(self):
        import torch
        for k in list(vars(self)):
            if k.startswith("t_"):
                delattr(self, k)
        torch.cuda.empty_cache()


class AllReduce(Workload):
    """All-reduce of n rank buffers of `count` elements, in place.  slab =
    (lo, hi): this GPU holds and reduces only elements [lo, hi) of every
    rank buffer (cr_all_reduce_range, the whole buffers' chunking); nbytes
    is then this GPU's share and full_nbytes the whole workload's."""

    def __init__(self, n=8, count=1 << 25, dtype="bf16", op="avg", std=0.02, slab=None):
        self.n, self.count, self.dt, self.op, self.std = n, count, dtype, op, std
        es = 2 if dtype == "bf16" else 4
        self.slab = slab
        self.full_nbytes = ar_bytes(n, count, es)
        self.nbytes = ar_bytes(n, slab[1] - slab[0], es) if slab else self.full_nbytes
        mib = count * es >> 20
        self.name = f"allreduce_{op}_{dtype}_{n}ranks_{mib}MiB"
        self.kernel = f"k_fold_vec3<{dtype},{dtype},AR,{n}>"
        self.profile = f"k_fold_vec_allreduce_{dtype}_{n}x{mib}MiB"

    def setup(self, device):
        import torch
        td = torch.bfloat16 if self.dt == "bf16" else torch.float32
        self.t_bufs = alloc_ranks(self.n, self.count, td, self.std, 0, device)
        if self.slab:
            lo, hi = self.slab
            self.t_bufs = [b[lo:hi].clone() for b in self.t_bufs]
            torch.cuda.empty_cache()

    def step(self, stream):
        from fsdp_emulated_ranks_gb300 import cr
        if self.slab:
            lo, hi = self.slab
            cr.cr_all_reduce_range(self.t_bufs, self.count, lo, hi, self.dt, self.op, self.t_bufs,
                                   self.dt, stream)
        else:
            cr.cr_all_reduce(self.t_bufs, self.count, self.dt, self.op, self.t_bufs, self.dt,
                             stream)


def slab_bounds(count, n, world, rank):
    """This GPU's slab of the element range under --split slab: slab `rank`
    of `world` (whole chunks while world <= n)."""
    from fsdp_emulated_ranks_gb300 import cr
    return cr.cr_slab_range(count, n, world, rank)


class AllReduceWire(Workload):
    """The headline all-reduce with its ring messages carried in bf16: each
    forwarded partial rounded before the next rank's fp32 addition."""

    def __init__(self, n=8, count=1 << 25):
        self.n, self.count = n, count
        self.nbytes = ar_bytes(n, count, 2)
        mib = count * 2 >> 20
        self.name = f"allreduce_avg_bf16_bf16wire_{n}ranks_{mib}MiB"
        self.kernel = f"k_fold_vec3<bf16,bf16,AR,{n},wire>"
        self.profile = f"k_fold_vec_allreduce_bf16wire_{n}x{mib}MiB"

    def setup(self, device):
        import torch
        self.t_bufs = alloc_ranks(self.n, self.count, torch.bfloat16, 0.02, 0, device)

    def step(self, stream):
        from fsdp_emulated_ranks_gb300 import cr
        cr.cr_all_reduce_wire(self.t_bufs, self.count, "bf16", "avg", "bf16", self.t_bufs, "bf16",
                              stream)


class Hsdp(Workload):
    """HSDP gradient reduction on an R x S mesh: reduce-scatter inside each
    group of S ranks and all-reduce of every shard across the R groups, one
    pass; reads N*count and writes R*count bf16 elements."""

    def __init__(self, R=2, S=4, count=1 << 25):
        self.R, self.S, self.count = R, S, count
        self.n = n = R * S
        self.nbytes = n * count * 2 + R * count * 2
        mib = count * 2 >> 20
        self.name = f"hsdp_reduce_scatter_avg_bf16_{R}x{S}mesh_{mib}MiB"
        self.kernel = f"k_hsdp_vec4<bf16,bf16,{R},{S},8>"
        self.profile = f"k_hsdp_vec_hsdp_bf16_{R}x{S}x{mib}MiB"

    def setup(self, device):
        import torch
        self.t_bufs = alloc_ranks(self.R * self.S, self.count, torch.bfloat16, 0.02, 0, device)
        L = -(-self.count // self.S)
        self.t_shards = [torch.empty(min(L, self.count - j * L), dtype=torch.bfloat16,
                                     device=device)
                         for _ in range(self.R) for j in range(self.S)]

    def step(self, stream):
        from fsdp_emulated_ranks_gb300 import cr
        cr.cr_hsdp_reduce_scatter(self.t_bufs, self.R, self.S, self.count, "bf16", "avg",
                                  self.t_shards, "bf16", stream)


class ReduceScatter(Workload):
    def __init__(self, n=8, count=1 << 25):
        self.n, self.count = n, count
        self.nbytes = n * count * 2 + count * 2
        self.name = f"reduce_scatter_avg_bf16_{n}ranks_{count * 2 >> 20}MiB"
        self.kernel = f"k_fold_vec3<bf16,bf16,RS,{n}>"
        self.profile = f"k_fold_vec_reduce_scatter_bf16_{n}x{count * 2 >> 20}MiB"

    def setup(self, device):
        import torch
        self.t_bufs = alloc_ranks(self.n, self.count, torch.bfloat16, 0.02, 0, device)
        L = self.count // self.n
        self.t_shards = [torch.empty(L, dtype=torch.bfloat16, device=device) for _ in range(self.n)]

    def step(self, stream):
        from fsdp_emulated_ranks_gb300 import cr
        cr.cr_reduce_scatter(self.t_bufs, self.count, "bf16", "avg", self.t_shards, "bf16", stream)


class AllGather(Workload):
    def __init__(self, n=8, count=1 << 25):
        self.n, self.count = n, count
        self.nbytes = count * 2 + n * count * 2
        self.name = f"all_gather_bf16_{n}ranks_{count * 2 >> 20}MiB"
        self.kernel = "k_gather_vec<2>"
        self.profile = f"k_gather_vec_all_gather_bf16_{n}x{count * 2 >> 20}MiB"

    def setup(self, device):
        import torch
        L = self.count // self.n
        self.t_shards = alloc_ranks(self.n, L, torch.bfloat16, 0.02, 0, device)
        self.t_bufs = [torch.empty(self.count, dtype=torch.bfloat16, device=device)
                       for _ in range(self.n)]

    def step(self, stream):
        from fsdp_emulated_ranks_gb300 import cr
        cr.cr_all_gather(self.t_shards, self.count, "bf16", self.t_bufs, stream)


class Buckets(Workload):
    """DDP bucket fusion: 300 bf16 tensors per rank (log-uniform numel,
    seed 7), 25 MiB buckets; mode pack, allreduce, unpack or pipeline."""

    def __init__(self, mode="pipeline", n=8, ntensors=300, plan=True):
        from fsdp_emulated_ranks_gb300 import inputs as I
        self.mode, self.n = mode, n
        self.numels = [int(k) for k in I.bucket_numels()][:ntensors]
        self.P = sum(self.numels)
        one = 2 * 2 * self.P * n
        self.nbytes = 3 * one if mode == "pipeline" else one
        # The fused all-reduce works on the tensors in place: N reads + N
        # writes per element, the same bytes as one pass over the buckets.
        self.name = f"ddp_bucket_{mode}_bf16_{n}ranks_{ntensors}tensors"
        if not plan:  # name and bytes only (the reference arm)
            return
        from fsdp_emulated_ranks_gb300 import cr
        self.plan = cr.cr_bucket_plan(self.numels, 2, 25 * 1024 * 1024)
        copies = -(-n * len(self.numels) // 1024)
        ar_launches = -(-self.plan.nbuckets // min(128, 2048 // n))
        self.launches = {"pack": copies, "unpack": copies, "allreduce": ar_launches,
                         "pipeline": 2 * copies + ar_launches,
                         "fused": -(-len(self.numels) // min(128, 2048 // n))}[mode]
        self.kernel = {"allreduce": "k_bucket_fused3<bf16,8>",
                       "fused": "k_bucket_fused3<bf16,8>"}.get(mode, "k_copy_segments")
        self.profile = (f"k_bucket_fused_bucket_{mode}_bf16_{n}x{ntensors}"
                        if mode in ("allreduce", "fused")
                        else f"k_copy_segments_bucket_{mode}_bf16_{n}x{ntensors}")

    def setup(self, device):
        import torch
        from fsdp_emulated_ranks_gb300 import inputs as I
        n = self.n
        tens = []
        for r in range(n):
            flat = torch.empty(self.P + 128 * len(self.numels), dtype=torch.bfloat16, device=device)
            I.torch_fill_normal_(flat, 1e-3, SEED_OFFSET + 1000 + r)
            off, row_t = 0, []
            for k in self.numels:
                row_t.append(flat[off:off + k])
                off += (k + 127) // 128 * 128
            tens.append(row_t)
        bks = []
        for r in range(n):
            sizes = [(int(k) + 127) // 128 * 128 for k in self.plan.bucket_numel]
            flat = torch.empty(sum(sizes), dtype=torch.bfloat16, device=device)
            off, row_b = 0, []
            for k, sz in zip(self.plan.bucket_numel, sizes):
                row_b.append(flat[off:off + int(k)])
                off += sz
            bks.append(row_b)
        self.t_flat_t = [x for rr in tens for x in rr]
        self.t_flat_b = [x for rr in bks for x in rr]
        # Device addresses taken once, as a framework with static gradient
        # buffers would: the calls then marshal integers, not 2400 tensors.
        self.p_flat_t = [x.data_ptr() for x in self.t_flat_t]
        self.p_flat_b = [x.data_ptr() for x in self.t_flat_b]

    def step(self, stream):
        from fsdp_emulated_ranks_gb300 import cr
        n = self.n
        if self.mode in ("pack", "pipeline"):
            cr.cr_bucket_pack(self.plan, n, self.p_flat_t, self.p_flat_b, stream)
        if self.mode in ("allreduce", "pipeline"):
            cr.cr_bucket_all_reduce(self.plan, n, self.p_flat_b, "bf16", "avg", stream)
        if self.mode in ("unpack", "pipeline"):
            cr.cr_bucket_unpack(self.plan, n, self.p_flat_b, self.p_flat_t, stream)
        if self.mode == "fused":
            cr.cr_bucket_all_reduce_fused(self.plan, n, self.p_flat_t, "bf16", "avg", stream)


class FsdpStep(Workload):
    """Fused FSDP step: 8 ranks, flat `count` params (1.3e9 by default);
    clip=True adds global grad-norm clipping (max_norm 1.0)."""

    def __init__(self, n=8, count=1_300_000_000, clip=False, slab=None):
        self.n, self.count, self.clip = n, count, clip
        if slab is not None and clip:
            raise SystemExit("the clipped step has no slab form (its norm needs every slab)")
        # slab = (lo, hi): this GPU holds and steps only parameters [lo, hi)
        # of the flat buffer (cr_fsdp_step_range); nbytes is its share
        self.slab = slab
        # clipped, N >= 5: the first pass parks the averaged fp32 gradient in
        # two of the parameter outputs (4 B written, 4 B read back) instead of
        # the update pass folding the N bf16 gradients again (2N B)
        self.stash = clip and n >= 5
        self.nbytes = ((4 * n + 32) if self.stash else ((6 if clip else 4) * n + 24)) * count
        tag = f"{count / 1e9:g}e9" if count >= 10 ** 8 else str(count)
        self.name = f"fsdp_step{'_clipped' if clip else ''}_bf16_{n}ranks_{tag}params"
        if self.stash:
            self.kernel = f"k_fsdp_sumsq<{n},stash> + k_clip_coef + k_fsdp_vec<stash>"
        else:
            self.kernel = f"k_fsdp_vec4<{n}>" + (" + k_fsdp_sumsq + k_clip_coef" if clip else "")
        self.profile = f"k_fsdp_vec_fsdp_step{'_clipped' if clip else ''}_{n}x{tag}"
        self.launches = 3 if clip else 1
        self.full_nbytes = self.nbytes
        if slab is not None:
            self.nbytes = self.nbytes // count * (slab[1] - slab[0])

    def setup(self, device):
        import torch
        from fsdp_emulated_ranks_gb300 import cr
        from fsdp_emulated_ranks_gb300 import inputs as I
        n, count = self.n, self.count
        L = cr.cr_chunk_len(count, n)
        if self.slab is not None:
            return self._setup_slab(device, L)
        self.t_grads = alloc_ranks(n, count, torch.bfloat16, 1e-3, 1000, device)
        self.t_params = [torch.empty(count, dtype=torch.bfloat16, device=device) for _ in range(n)]
        self.t_master_full = torch.empty(count, dtype=torch.float32, device=device)
        I.torch_fill_normal_(self.t_master_full, 0.02, SEED_OFFSET + 2000)
        self.t_mv = torch.zeros(2 * count, dtype=torch.float32, device=device)
        self.t_master = [self.t_master_full[j * L:(j + 1) * L] for j in range(n)]
        self.t_m = [self.t_mv[j * L:(j + 1) * L] for j in range(n)]
        self.t_v = [self.t_mv[count + j * L:count + (j + 1) * L] for j in range(n)]
        self.cfg = cr.adamw_cfg()
        self.ws_bytes = cr.cr_fsdp_clip_workspace_bytes()
        self.t_ws = torch.empty(self.ws_bytes // 8, dtype=torch.float64, device=device)
        self.t_norm = torch.empty(1, dtype=torch.float32, device=device)

    def _setup_slab(self, device, L):
        """The whole workload's values, then only this GPU's slab of the
        grads and params and its parts of the owners' state shards."""
        import torch
        from fsdp_emulated_ranks_gb300 import cr
        from fsdp_emulated_ranks_gb300 import inputs as I
        n, count = self.n, self.count
        lo, hi = self.slab
        self.t_grads = [g[lo:hi].clone() for g in
                        alloc_ranks(n, count, torch.bfloat16, 1e-3, 1000, device)]
        torch.cuda.empty_cache()
        self.t_params = [torch.empty(hi - lo, dtype=torch.bfloat16, device=device)
                         for _ in range(n)]
        full = torch.empty(count, dtype=torch.float32, device=device)
        I.torch_fill_normal_(full, 0.02, SEED_OFFSET + 2000)
        self.t_master, self.t_m, self.t_v = [], [], []
        for j in range(n):
            a, b = max(lo, j * L), min(hi, (j + 1) * L, count)
            k = max(0, b - a)
            self.t_master.append(full[a:a + k].clone() if k else 0)
            self.t_m.append(torch.zeros(k, dtype=torch.float32, device=device) if k else 0)
            self.t_v.append(torch.zeros(k, dtype=torch.float32, device=device) if k else 0)
        del full
        torch.cuda.empty_cache()
        self.cfg = cr.adamw_cfg()

    def step(self, stream):
        from fsdp_emulated_ranks_gb300 import cr
        if self.slab is not None:
            lo, hi = self.slab
            cr.cr_fsdp_step_range(self.t_grads, self.count, lo, hi, self.t_master, self.t_m,
                                  self.t_v, self.cfg, self.t_params, stream)
        elif self.clip:
            cr.cr_fsdp_step_clipped(self.t_grads, self.count, self.t_master, self.t_m, self.t_v,
                                    self.cfg, 1.0, self.t_ws, self.ws_bytes, self.t_params,
                                    self.t_norm, stream)
        else:
            cr.cr_fsdp_step(self.t_grads, self.count, self.t_master, self.t_m, self.t_v,
                            self.cfg, self.t_params, stream)


def transformer_shapes(hidden=2048, layers=24, vocab=32000, ffn=8192):
    """Parameter shapes (dim0, row) of a decoder-only transformer: per layer
    qkv, output, up and down projections and two norms, plus the embedding
    (1.27e9 parameters with the defaults)."""
    shapes = [(vocab, hidden)]
    for _ in range(layers):
        shapes += [(3 * hidden, hidden), (hidden, hidden), (ffn, hidden), (hidden, ffn),
                   (hidden, 1), (hidden, 1)]
    return shapes


class Fsdp2Step(Workload):
    """FSDP2 per-parameter Shard(0) step over a transformer's parameters,
    8 ranks; each rank's grads and params live in one 256-byte-aligned slab
    per rank, the shards' fp32 state in one slab per parameter set."""

    def __init__(self, n=8, layers=24, hidden=2048, planned=True):
        self.n, self.planned = n, planned
        self.shapes = transformer_shapes(hidden=hidden, layers=layers, ffn=4 * hidden)
        self.P = sum(d * r for d, r in self.shapes)
        self.nbytes = (4 * n + 24) * self.P
        tag = "" if planned else "_chained"
        self.name = f"fsdp2{tag}_step_bf16_{n}ranks_{len(self.shapes)}params_{self.P / 1e9:.2f}e9"
        if planned:
            # one launch over the plan's table, uploaded once at setup
            self.kernel = f"k_fsdp2_table<{n}>"
            self.profile = f"k_fsdp2_table_fsdp2_step_{n}x{len(self.shapes)}params"
            self.launches = 1
        else:
            # the pointers in the kernel's parameter block: 64 parameters a launch
            self.kernel = f"k_fsdp2<{n}>"
            self.profile = f"k_fsdp2_fsdp2_step_{n}x{len(self.shapes)}params"
            self.launches = -(-len(self.shapes) // min(64, 2560 // (5 * n)))

    def setup(self, device):
        import torch
        from fsdp_emulated_ranks_gb300 import cr
        from fsdp_emulated_ranks_gb300 import inputs as I
        n, pad = self.n, 128
        sizes = [d * r for d, r in self.shapes]
        offs, o = [], 0
        for k in sizes:
            offs.append(o)
            o += (k + pad - 1) // pad * pad
        self.t_g = [torch.empty(o, dtype=torch.bfloat16, device=device) for _ in range(n)]
        for r, t in enumerate(self.t_g):
            I.torch_fill_normal_(t, 1e-3, SEED_OFFSET + 1000 + r)
        self.t_p = [torch.empty(o, dtype=torch.bfloat16, device=device) for _ in range(n)]
        shard = []
        for (d, rn) in self.shapes:
            Lr = -(-d // n)
            shard.append([max(0, min(d, (j + 1) * Lr) - min(d, j * Lr)) * rn for j in range(n)])
        soffs, so = [], 0
        for row in shard:
            so_row = []
            for k in row:
                so_row.append(so)
                so += (k + pad - 1) // pad * pad
            soffs.append(so_row)
        self.t_state = torch.zeros(3 * so, dtype=torch.float32, device=device)
        I.torch_fill_normal_(self.t_state[:so], 0.02, SEED_OFFSET + 2000)
        self.grads, self.params, self.master, self.m, self.v = [], [], [], [], []
        for p, k in enumerate(sizes):
            for r in range(n):
                self.grads.append(self.t_g[r][offs[p]:offs[p] + k])
                self.params.append(self.t_p[r][offs[p]:offs[p] + k])
                sk, so0 = shard[p][r], soffs[p][r]
                self.master.append(self.t_state[so0:so0 + sk] if sk else 0)
                self.m.append(self.t_state[so + so0:so + so0 + sk] if sk else 0)
                self.v.append(self.t_state[2 * so + so0:2 * so + so0 + sk] if sk else 0)
        # Layout kept for tests that sample elements: parameter p of rank r at
        # t_g/t_p[r][offs[p]:], owner j's shard at t_state[soffs[p][j]:] (m at
        # +so, v at +2 so).
        self.offs, self.soffs, self.so = offs, soffs, so
        # Device addresses taken once (the slabs t_g, t_p, t_state stay alive).
        addr = lambda xs: [x if isinstance(x, int) else x.data_ptr() for x in xs]
        self.grads, self.params = addr(self.grads), addr(self.params)
        self.master, self.m, self.v = addr(self.master), addr(self.m), addr(self.v)
        self.cfg = cr.adamw_cfg()
        self.plan = self.t_table = None
        if self.planned:
            self.plan = cr.cr_fsdp2_plan_create(self.shapes, n, self.grads, self.master, self.m,
                                                self.v, self.params)
            self.t_table = torch.empty(self.plan.table_bytes, dtype=torch.uint8, device=device)
            cr.cr_fsdp2_plan_upload(self.plan, self.t_table)
            torch.cuda.synchronize(device)

    def step(self, stream):
        from fsdp_emulated_ranks_gb300 import cr
        if self.planned:
            cr.cr_fsdp2_step_planned(self.plan, self.t_table, self.cfg, stream)
        else:
            cr.cr_fsdp2_step(self.shapes, self.n, self.grads, self.master, self.m, self.v,
                             self.cfg, self.params, stream)

    def teardown(self):
        self.grads = self.params = self.master = self.m = self.v = None
        self.plan = self.t_table = None
        super().teardown()


class Accumulate(Workload):
    """DDP no_sync micro-steps: 8 ranks' fp32 accumulators of 2^25 elements
    plus a bf16 micro-step gradient each; reduce=True fuses the last
    micro-step's accumulation with the AVG all-reduce."""

    def __init__(self, reduce, n=8, count=1 << 25):
        self.reduce, self.n, self.count = reduce, n, count
        self.nbytes = n * count * (4 + 2 + 4)
        self.name = (f"{'all_reduce_' if reduce else ''}accumulate_bf16_into_f32_{n}ranks_"
                     f"{count * 2 >> 20}MiB")
        self.kernel = f"k_accum_vec<bf16,{n if reduce else 0},8>"
        self.profile = f"k_accum_vec_{'allreduce_' if reduce else ''}accumulate_{n}x{count}"

    def setup(self, device):
        import torch
        self.t_acc = [torch.zeros(self.count, dtype=torch.float32, device=device)
                      for _ in range(self.n)]
        self.t_g = alloc_ranks(self.n, self.count, torch.bfloat16, 1e-3, 0, device)

    def step(self, stream):
        from fsdp_emulated_ranks_gb300 import cr
        if self.reduce:
            cr.cr_all_reduce_accumulate(self.t_acc, self.count, self.t_g, "bf16", "avg", stream)
        else:
            cr.cr_accumulate(self.t_acc, self.count, self.t_g, "bf16", stream)


# Added to every seed of a value draw (--seed); the recipe's seeds at 0.  The
# seeded draw of the bucket workload's tensor sizes is not shifted: the
# workload keeps its shape.
SEED_OFFSET = 0

# --config: the five benchmark configurations (1-4 a workload, 5 the sweep).
CONFIGS = {1: "allreduce_f32", 2: "allreduce", 3: "bucket_pipeline", 4: "fsdp", 5: "sweep"}


def make_workload(name, args, plan=True):
    if name == "allreduce":
        return AllReduce()
    if name == "allreduce_f32":
        return AllReduce(n=4, count=1 << 20, dtype="f32", op="sum", std=1.0)
    if name == "allreduce_wire":
        return AllReduceWire()
    if name == "hsdp":
        return Hsdp()
    if name == "reduce_scatter":
        return ReduceScatter()
    if name == "all_gather":
        return AllGather()
    if name.startswith("bucket_"):
        return Buckets(mode=name[len("bucket_"):], ntensors=args.bucket_ntensors, plan=plan)
    if name == "fsdp":
        return FsdpStep(count=args.fsdp_count)
    if name == "fsdp_clipped":
        return FsdpStep(count=args.fsdp_count, clip=True)
    if name == "fsdp2":
        return Fsdp2Step(layers=args.fsdp2_layers, hidden=args.fsdp2_hidden)
    if name == "fsdp2_chained":
        return Fsdp2Step(layers=args.fsdp2_layers, hidden=args.fsdp2_hidden, planned=False)
    if name == "accumulate":
        return Accumulate(reduce=False)
    if name == "accumulate_allreduce":
        return Accumulate(reduce=True)
    raise SystemExit(f"unknown workload {name}")


ROW_WORKLOADS = ["reduce_scatter", "all_gather", "allreduce_f32", "bucket_pack",
                 "bucket_allreduce", "bucket_unpack", "bucket_pipeline", "bucket_fused", "fsdp", "fsdp_clipped", "fsdp2", "fsdp2_chained", "accumulate",
                 "accumulate_allreduce", "allreduce_wire", "hsdp"]


def workload_config(wl, world):
    """The JSON line's config for workload wl on `world` GPUs (both arms)."""
    config = {"workload": wl.name, "parallelism": f"{world} GPU(s) x {wl.n} emulated ranks each"}
    if isinstance(wl, AllReduce):
        es = 2 if wl.dt == "bf16" else 4
        S = wl.count * es
        config.update({"ranks": wl.n, "elements_per_rank": wl.count, "dtype_in_out": wl.dt,
                       "accumulate": "fp32, ring order" if wl.dt != "i32" else "int32",
                       "op": f"{wl.op}, in place",
                       "l2": ("inputs exceed the 129 MB L2, no flush" if wl.nbytes // 2 > (129 << 20)
                              else "inputs fit in L2 (latency regime), no flush"),
                       # what a real ring and a naive reduce + broadcast would move
                       # (N divides the count): 2(N-1)/N S per rank, 2(N-1) S at the root
                       "ring_bytes_sent_per_rank": 2 * (wl.n - 1) * S // wl.n,
                       "naive_root_bytes_sent_and_received": 2 * (wl.n - 1) * S})
    else:
        config["algorithmic_bytes_per_step"] = wl.nbytes
        config["l2"] = "inputs exceed the 129 MB L2, no flush"
    return config


def run_headline(args, world, rank, device, stream, peak):
    import torch
    wl = make_workload(args.workload, args)
    if args.split == "slab":
        if isinstance(wl, AllReduce):
            wl = AllReduce(wl.n, wl.count, wl.dt, wl.op, wl.std,
                           slab=slab_bounds(wl.count, wl.n, world, rank))
        elif isinstance(wl, FsdpStep) and not wl.clip:
            wl = FsdpStep(wl.n, wl.count, slab=slab_bounds(wl.count, wl.n, world, rank))
        else:
            raise SystemExit("--split slab is built for the all-reduce and FSDP step workloads")
    wl.setup(device)
    # Sample for the CPU baseline before in-place calls overwrite the inputs.
    sample = None
    if (rank == 0 and world == 1 and not args.no_cpu_baseline and isinstance(wl, AllReduce)
            and wl.dt == "bf16"):
        k = min(args.cpu_sample, wl.count)
        sample = [b[:k].view(torch.int16).cpu().numpy().view("uint16") for b in wl.t_bufs]
    sampler = ClockSampler(device)
    total_ms, per = timed(lambda: wl.step(stream), args.steps, args.warmup, world, stream, sampler)
    if getattr(wl, "slab", None) is not None:
        # the ranks' slabs make up one workload: its bytes over the slowest rank's time
        ms_step = max_over_ranks(total_ms, world, device) / args.steps
        value = wl.full_nbytes / (ms_step * 1e-3) / 1e9
    else:
        value, ms_step = job_throughput(wl.nbytes, total_ms, args.steps, world, device)
    kern_ms = total_ms / args.steps   # this GPU's mean launch, back to back
    achieved = wl.nbytes / (kern_ms * 1e-3) / 1e9
    out = {
        "workload": wl,
        "ms_per_step": ms_step,
        "value": value,
        "clocks": sampler.summary(),
        # every GPU launches the same kernels: the job's count, like `value`
        "gpu_launches": world * args.steps * wl.launches,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak[0],
                     "unit": "GB/s", "frac": round(achieved / peak[0], 4),
                     "traffic": traffic_per_launch(wl.profile, wl.launches),
                     "kernel": wl.kernel, "algorithmic_bytes_per_launch": wl.nbytes // wl.launches,
                     "peak_source": peak[1], "step_ms_median": statistics.median(per),
                     **step_quantiles(per)},
    }
    # the same figure from the median of the per-step pass (achieved/frac above:
    # the mean of the back-to-back steps)
    med = statistics.median(per)
    out["roofline"].update({"achieved_median": round(wl.nbytes / (med * 1e-3) / 1e9, 1),
                            "frac_median": round(wl.nbytes / (med * 1e-3) / 1e9 / peak[0], 4)})
    if wl.launches > 1:
        out["roofline"]["launches"] = wl.launches
    out["l2_flushed"] = l2_flushed(wl, stream, device, peak)
    out["e2e"] = None
    if isinstance(wl, AllReduce) and not args.no_e2e:
        out["e2e"] = run_e2e(args, wl.t_bufs, wl.n, wl.count, world, stream, device)
    wl.teardown()
    return out, sample


def l2_flushed(wl, stream, device, peak, steps=20):
    """The workload's step timed one call at a time with L2 flushed before
    each (a write of twice the 129 MB L2 on the same stream, outside the
    timed events): the median step time, as a cross-check that L2 residency
    between back-to-back steps does not inflate the headline figure.

    The write leaves L2 full of dirty lines, which the timed call then
    writes back as its own accesses evict them.  "clean" repeats the
    measurement with an untimed read of the same scratch after the write:
    that read takes the write-backs, and the call starts from an L2 of
    clean lines that hold none of its data."""
    import torch
    scratch = torch.empty(2 * (129 << 20), dtype=torch.uint8, device=device)
    words = scratch.view(torch.int32)

    def median_ms(clean):
        times = []
        with torch.cuda.stream(stream):
            for i in range(steps + 3):
                scratch.fill_(i & 0xff)
                if clean:
                    words.amax()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                wl.step(stream)
                e1.record(stream)
                e1.synchronize()
                if i >= 3:
                    times.append(e0.elapsed_time(e1))
        return statistics.median(times)

    def figures(ms):
        gbs = wl.nbytes / (ms * 1e-3) / 1e9
        return {"ms_median": round(ms, 4), "GB/s": round(gbs, 1), "frac": round(gbs / peak[0], 4)}

    out = {"steps": steps, "flush_bytes": 2 * (129 << 20), **figures(median_ms(False))}
    out["clean"] = figures(median_ms(True))
    del words, scratch
    return out


def run_e2e(args, bufs, n, count, world, stream, device):
    """End to end through the C ABI with the rank buffers in pinned host
    memory: every step moves the 8 inputs host -> GPU, all-reduces them and
    moves the 8 results GPU -> host.  Default API cr_all_reduce_host (the
    kernel reads and writes host memory over the coherent host link, both
    directions at once); --e2e-api staged uses cr_all_reduce_staged (copy
    engines, sliced and pipelined over upload / compute / download streams)."""
    import torch
    from fsdp_emulated_ranks_gb300 import cr
    host_in = [torch.empty(count, dtype=torch.bfloat16, pin_memory=True) for _ in range(n)]
    host_out = [torch.empty(count, dtype=torch.bfloat16, pin_memory=True) for _ in range(n)]
    for h, b in zip(host_in, bufs):
        h.copy_(b)
    torch.cuda.synchronize()
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)

    if args.e2e_api == "host":
        def step():
            cr.cr_all_reduce_host(host_in, host_out, count, "bf16", "avg", stream=stream)
    else:
        def step():
            cr.cr_all_reduce_staged(host_in, host_out, bufs, count, "bf16", "avg",
                                    args.e2e_slice, stream, up, down)

    steps = max(3, min(args.steps, 50))
    total_ms, _ = timed(step, steps, max(3, min(args.warmup, 5)), world, stream)
    nbytes = ar_bytes(n, count, 2)
    value, ms = job_throughput(nbytes, total_ms, steps, world, device)
    out = {"value": round(value, 2), "unit": UNIT,
           "h2d_bytes_per_step": n * count * 2, "d2h_bytes_per_step": n * count * 2,
           "ms_per_step": ms, "steps": steps, "api": f"cr_all_reduce_{args.e2e_api}"}
    if args.e2e_api == "staged":
        out["slice_elems"] = args.e2e_slice or "auto"
    return out


def traffic_per_step(name):
    """DRAM bytes of one step (all its launches) from the committed ncu
    summary, or None if absent or taken on a different build of the kernel."""
    p = os.path.join(ROOT, "profiles", name + ".md")
    if not os.path.exists(p):
        return None
    vals = {}
    with open(p) as f:
        for line in f:
            if ":" in line and line.strip().startswith(
                    ("dram_bytes_per_launch", "dram_bytes_per_step", "kernel_tu",
                     "kernel_source_hash")):
                k, v = line.split(":", 1)
                vals[k.strip(" -*`")] = v.strip(" `\n")
    try:
        from fsdp_emulated_ranks_gb300 import build as B
        if vals.get("kernel_source_hash") != B.kernel_hash(vals["kernel_tu"]):
            return None
        return int(vals.get("dram_bytes_per_step") or vals["dram_bytes_per_launch"])
    except (KeyError, ValueError, OSError):
        return None


def traffic_per_launch(name, launches=1):
    """DRAM bytes per launch from the committed ncu summary of this kernel,
    or None if absent or taken on a different build of its kernel code (the
    summary names the translation unit and its kernel_hash)."""
    p = os.path.join(ROOT, "profiles", name + ".md")
    if not os.path.exists(p) or launches != 1:
        return None
    vals = {}
    with open(p) as f:
        for line in f:
            if ":" in line and line.strip().startswith(
                    ("dram_bytes_per_launch", "kernel_tu", "kernel_source_hash")):
                k, v = line.split(":", 1)
                vals[k.strip(" -*`")] = v.strip(" `\n")
    try:
        from fsdp_emulated_ranks_gb300 import build as B
        if vals.get("kernel_source_hash") != B.kernel_hash(vals["kernel_tu"]):
            return None
        return int(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError, OSError):
        return None


# ---- the other rows (N = 1) ------------------------------------------------------------

def run_rows(args, device, stream, peak, skip=None):
    rows = []
    for name in ROW_WORKLOADS:
        if (name.startswith("fsdp") and args.skip_fsdp) or name == skip:
            continue
        wl = make_workload(name, args)
        wl.setup(device)
        steps = args.row_steps if wl.nbytes < (8 << 30) else max(5, args.row_steps // 2)
        total, per = timed(lambda: wl.step(stream), steps, 3, 1, stream)
        ms = total / steps
        gbs = wl.nbytes / (ms * 1e-3) / 1e9
        rows.append({"name": wl.name, "ms": round(ms, 4), "GB/s": round(gbs, 1),
                     "frac": round(gbs / peak[0], 4), "algorithmic_bytes": wl.nbytes,
                     "steps": steps, **step_quantiles(per),
                     "launches_per_call": wl.launches, "kernel": wl.kernel,
                     "traffic": traffic_per_launch(wl.profile, wl.launches),
                     "traffic_per_step": traffic_per_step(wl.profile)})
        rows[-1]["key"] = name
        if ms < 0.05:
            # host-bound: also the same call prepared once (the C call alone)
            from fsdp_emulated_ranks_gb300 import cr
            prep = cr.prepare(wl.step, stream)
            psteps = max(steps, 200)
            ptot, pper = timed(prep, psteps, 3, 1, stream)
            pms = statistics.median(pper)
            rows[-1].update({"ms_prepared_median": round(pms, 4),
                             "GB/s_prepared": round(wl.nbytes / (pms * 1e-3) / 1e9, 1),
                             # back to back: the host issues the next call
                             # while the device runs this one
                             "ms_prepared": round(ptot / psteps, 4),
                             "frac_prepared": round(wl.nbytes / (ptot / psteps * 1e-3) / 1e9
                                                    / peak[0], 4)})
            del prep
            # and captured in a CUDA graph: device time per call, no host work
            gus = graph_replay_us(wl, device, stream)
            rows[-1].update({"graph_us": round(gus, 2),
                             "GB/s_graph": round(wl.nbytes / (gus * 1e-6) / 1e9, 1),
                             "frac_graph": round(wl.nbytes / (gus * 1e-6) / 1e9 / peak[0], 4)})
            # and one call at a time from cold L2: its inputs come from HBM
            rows[-1]["l2_flushed"] = l2_flushed(wl, stream, device, peak)
        wl.teardown()
    return rows


def graph_replay_us(wl, device, stream, reps=50, replays=10):
    """Per-call time of `reps` back-to-back calls of wl.step captured in one
    CUDA graph (median over `replays` replays): the device time of a call
    whose host work (argument checks, marshalling, launch) would otherwise
    dominate."""
    import torch
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream(device)
    side.wait_stream(torch.cuda.current_stream(device))
    with torch.cuda.graph(g, stream=side):
        for _ in range(reps):
            wl.step(side)
    torch.cuda.current_stream(device).wait_stream(side)
    _, gper = timed(g.replay, replays, 3, 1, stream)
    del g
    return statistics.median(gper) * 1e3 / reps


def rows_summary(head_key, head_roofline, rows, peak):
    """One compact entry per measured row, [ms median, GB/s at the median,
    fraction of the peak at the median, fraction at the mean], keyed by
    workload; host-bound rows add their graph-replay figures
    [us per call, fraction] and their cold-L2 single-call figures
    [ms median, fraction]."""
    out = {head_key: [head_roofline["ms_median"], head_roofline["achieved_median"],
                      head_roofline["frac_median"], head_roofline["frac"]]}
    for r in rows or []:
        gbs = r["algorithmic_bytes"] / (r["ms_median"] * 1e-3) / 1e9
        e = [r["ms_median"], round(gbs, 1), round(gbs / peak[0], 4), r["frac"]]
        if "graph_us" in r:
            e += [r["graph_us"], r["frac_graph"]]
        if "l2_flushed" in r:
            e += [r["l2_flushed"]["ms_median"], r["l2_flushed"]["frac"]]
        out[r["key"]] = e
    return out


def step_quantiles(per):
    """Median, 10th and 90th percentile of the per-step event times (ms)."""
    q = sorted(per)
    at = lambda f: q[min(len(q) - 1, int(round(f * (len(q) - 1))))]
    return {"ms_median": round(statistics.median(q), 4), "ms_p10": round(at(0.1), 4),
            "ms_p90": round(at(0.9), 4)}


# ---- bf16 wire error ----------------------------------------------------------------------

def wire_error(device, n=8, count=1 << 24):
    """What the bf16 wire costs in accuracy, measured on the GPU: the same 8
    bf16 rank buffers (N(0, 0.02^2)) all-reduced (AVG) into fp32, once with
    fp32 partials and once with every forwarded partial rounded to bf16.
    The fp32-partial result is within ~1e-7 relative of the exact sum, so
    the difference is the wire's error; it is reported in bf16 ulps of the
    fp32-partial result, next to the 0.5 ulp that rounding that result to
    bf16 once costs."""
    import torch
    from fsdp_emulated_ranks_gb300 import cr
    bufs = alloc_ranks(n, count, torch.bfloat16, 0.02, 100, device)
    a = [torch.empty(count, dtype=torch.float32, device=device) for _ in range(n)]
    b = [torch.empty(count, dtype=torch.float32, device=device) for _ in range(n)]
    cr.cr_all_reduce(bufs, count, "bf16", "avg", a, "f32")
    cr.cr_all_reduce_wire(bufs, count, "bf16", "avg", "bf16", b, "f32")
    torch.cuda.synchronize()
    ref, got = a[0].double(), b[0].double()
    nz = ref != 0
    ulp = torch.exp2(torch.floor(torch.log2(ref[nz].abs())) - 7)
    err = ((got[nz] - ref[nz]).abs() / ulp).float()
    q = torch.quantile(err[:1 << 20], torch.tensor([0.5, 0.99], device=device)).tolist()
    rel_rms = float(((got - ref) ** 2).mean().sqrt() / (ref ** 2).mean().sqrt())
    out = {"ranks": n, "elements": count, "inputs": "bf16 N(0, 0.02^2), AVG, fp32 output",
           "bf16_ulps_median": round(q[0], 4), "bf16_ulps_p99": round(q[1], 4),
           "bf16_ulps_max": round(float(err.max()), 4), "relative_rms": rel_rms,
           "same_as_fp32_wire_fraction": round(float((err == 0).float().mean()), 4)}
    del bufs, a, b
    torch.cuda.empty_cache()
    return out


# ---- DDP backward / all-reduce overlap ---------------------------------------------------

def run_overlap(args, device, caps=(0, 38, 304)):
    """The reducer's overlap of bucket all-reduces with backward ("AI Infra
    Guide, Chapter 6", 6.2.5): the 300-tensor bucket workload, 8 ranks; the
    emulated backward runs, per bucket, k bf16 4096^3 GEMMs (cuBLAS through
    torch: the stand-in for layer backward, not part of the library) on a
    compute stream and then marks the bucket's tensors ready; the reducer
    all-reduces each bucket on a comm stream with at most `cap` CTAs.  k is
    chosen so that compute alone takes about as long as the all-reduces
    alone, the case where overlap matters most.  hidden = (t_compute +
    t_comm - t_both) / min(t_compute, t_comm)."""
    import torch
    from fsdp_emulated_ranks_gb300 import cr
    wl = Buckets(mode="fused", ntensors=args.bucket_ntensors)
    wl.setup(device)
    plan, n, T = wl.plan, wl.n, wl.plan.ntensors
    members = [[] for _ in range(plan.nbuckets)]
    for t in range(T - 1, -1, -1):
        members[plan.tensor_bucket[t]].append(t)
    compute, comm = torch.cuda.Stream(device), torch.cuda.Stream(device)
    a = torch.randn(4096, 4096, device=device, dtype=torch.bfloat16)
    b = torch.randn(4096, 4096, device=device, dtype=torch.bfloat16)
    c = torch.empty(4096, 4096, device=device, dtype=torch.bfloat16)

    def timed_on(stream, fn, reps):
        fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    def backward(red, k):
        with torch.cuda.stream(compute):
            for bk in range(plan.nbuckets):
                for _ in range(k):
                    torch.mm(a, b, out=c)
                if red is not None:
                    for t in members[bk]:
                        cr.cr_reducer_mark_ready(red, t, compute)
            if red is not None:
                cr.cr_reducer_finalize(red, compute)

    t_gemm = timed_on(compute, lambda: torch.mm(a, b, out=c), 50)
    out = {"workload": wl.name, "buckets": plan.nbuckets, "gemm": "bf16 4096x4096x4096",
           "gemm_ms": round(t_gemm, 4), "caps": []}
    for cap in caps:
        red = cr.cr_reducer_create(plan, n, wl.t_flat_t, "bf16", "avg", cap, comm)
        t_comm = timed_on(compute, lambda: backward(red, 0), 5)
        k = max(1, round(t_comm / (plan.nbuckets * t_gemm)))
        t_comp = timed_on(compute, lambda: backward(None, k), 5)
        t_both = timed_on(compute, lambda: backward(red, k), 5)
        cr.cr_reducer_destroy(red)
        hidden = (t_comp + t_comm - t_both) / min(t_comp, t_comm)
        out["caps"].append({"comm_ctas": cap, "gemms_per_bucket": k,
                            "t_comm_ms": round(t_comm, 3), "t_compute_ms": round(t_comp, 3),
                            "t_both_ms": round(t_both, 3), "hidden": round(hidden, 3),
                            "comm_GBs_alone": round(wl.nbytes / (t_comm * 1e-3) / 1e9, 1)})
    wl.teardown()
    return out


# ---- CPU oracle -------------------------------------------------------------------------

def cpu_oracle_allreduce(sample, min_seconds):
    """Ring all-reduce AVG of the sampled bf16 rank buffers by the CPU oracle
    (single-threaded), repeated until at least `min_seconds` of CPU work;
    returns (GB/s, seconds, passes)."""
    import oracle as O
    n, count = len(sample), sample[0].size
    O.ring_all_reduce([x[:1024] for x in sample], "bf16", "avg")  # load the library
    passes, t0 = 0, time.perf_counter()
    while True:
        O.ring_all_reduce(sample, "bf16", "avg")
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or passes >= 1000:
            break
    return passes * ar_bytes(n, count, 2) / dt / 1e9, dt, passes


class OracleSample:
    """A bounded sample of workload `name` for the CPU oracle, drawn by the
    workload's recipe (numpy's generator on the host): k elements per rank,
    or for the bucket and FSDP2 workloads the same structure scaled down to
    about k elements per rank.  step() runs one step of the workload's
    computation in the oracle; nbytes is that step's algorithmic bytes by
    the workload's own formula; desc says what the sample is."""

    def __init__(self, name, args, k):
        import numpy as np
        import oracle as O
        from fsdp_emulated_ranks_gb300 import inputs as I
        self.full = full = make_workload(name, args, plan=False)
        n = full.n

        def bf16(count, std, seed):
            return I.np_to_bf16_bits(I.np_normal_f32(count, std, SEED_OFFSET + seed))

        def shards(x, parts):
            L = O.chunk_len(x.size, parts)
            return [np.ascontiguousarray(x[min(j * L, x.size):min((j + 1) * L, x.size)])
                    for j in range(parts)]

        if isinstance(full, (AllReduce, AllReduceWire, ReduceScatter, AllGather, Hsdp)):
            k = min(k, full.count)
            dt = getattr(full, "dt", "bf16")
            if dt == "bf16":
                x = [bf16(k, getattr(full, "std", 0.02), r) for r in range(n)]
            else:
                x = [I.np_normal_f32(k, full.std, SEED_OFFSET + r) for r in range(n)]
            if isinstance(full, AllReduce):
                self.step = lambda: O.ring_all_reduce(x, dt, full.op)
                sample = AllReduce(n, k, dt, full.op)
            elif isinstance(full, AllReduceWire):
                self.step = lambda: O.ring_all_reduce_wire(x, "bf16", "avg", "bf16")
                sample = AllReduceWire(n, k)
            elif isinstance(full, ReduceScatter):
                self.step = lambda: O.ring_reduce_scatter(x, "bf16", "avg")
                sample = ReduceScatter(n, k)
            elif isinstance(full, AllGather):
                sh = shards(x[0], n)
                self.step = lambda: O.ring_all_gather(sh, k, "bf16")
                sample = AllGather(n, k)
            else:
                self.step = lambda: O.hsdp_reduce_scatter(x, full.R, full.S, "bf16", "avg")
                sample = Hsdp(full.R, full.S, k)
            self.desc = f"{n} rank buffers of {k} elements"
        elif isinstance(full, Accumulate):
            k = min(k, full.count)
            acc = [np.zeros(k, np.float32) for _ in range(n)]
            g = [bf16(k, 1e-3, r) for r in range(n)]

            def step():
                for r in range(n):
                    O.accumulate(acc[r], g[r], "bf16")
                if full.reduce:
                    out, _ = O.ring_all_reduce(acc, "f32", "avg")
                    for r in range(n):
                        acc[r][:] = out[r]
            self.step = step
            sample = Accumulate(full.reduce, n, k)
            self.desc = f"{n} fp32 accumulators and bf16 gradients of {k} elements"
        elif isinstance(full, FsdpStep):
            k = min(k, full.count)
            grads = [bf16(k, 1e-3, 1000 + r) for r in range(n)]
            master = shards(I.np_normal_f32(k, 0.02, SEED_OFFSET + 2000), n)
            m = [np.zeros_like(a) for a in master]
            v = [np.zeros_like(a) for a in master]
            cfg = O.AdamWConfig()
            if full.clip:
                self.step = lambda: O.fsdp_step_clipped(grads, master, m, v, cfg, 1.0)
            else:
                self.step = lambda: O.fsdp_step(grads, master, m, v, cfg)
            sample = FsdpStep(n, k, full.clip)
            self.desc = f"{k} flat parameters"
        elif isinstance(full, Fsdp2Step):
            # The same architecture at a width whose parameter count is about k.
            hidden = 64
            while hidden < 2048 and Fsdp2Step(n, 1, 2 * hidden).P <= k:
                hidden *= 2
            sample = Fsdp2Step(n, 1, hidden)
            grads = [[bf16(d * rn, 1e-3, 1000 + 8 * p + r) for r in range(n)]
                     for p, (d, rn) in enumerate(sample.shapes)]
            master, m, v = [], [], []
            for p, (d, rn) in enumerate(sample.shapes):
                Lr = O.chunk_len(d, n)
                st = [I.np_normal_f32(max(0, min(d, (j + 1) * Lr) - min(d, j * Lr)) * rn, 0.02,
                                      SEED_OFFSET + 2000 + 8 * p + j) for j in range(n)]
                master.append(st)
                m.append([np.zeros_like(a) for a in st])
                v.append([np.zeros_like(a) for a in st])
            cfg = O.AdamWConfig()
            self.step = lambda: O.fsdp2_step(sample.shapes, grads, master, m, v, cfg)
            self.desc = (f"the same transformer at 1 layer of hidden {hidden} "
                         f"({len(sample.shapes)} parameters, {sample.P} elements)")
        elif isinstance(full, Buckets):
            scale = k / full.P
            numels = [max(1, round(t * scale)) for t in full.numels]
            cap = max(2, round(25 * 1024 * 1024 * scale))
            plan = O.bucket_plan(numels, 2, cap)
            tens = [[bf16(t, 1e-3, 1000 + 1000 * r + i) for i, t in enumerate(numels)]
                    for r in range(n)]
            bks = O.bucket_pack(plan, tens)
            mode = full.mode

            def step():
                if mode == "pack":
                    O.bucket_pack(plan, tens)
                elif mode == "unpack":
                    O.bucket_unpack(plan, bks, np.uint16)
                elif mode == "allreduce":
                    for b in range(plan.nbuckets):
                        O.ring_all_reduce([bks[r][b] for r in range(n)], "bf16", "avg")
                else:  # pipeline, fused: pack, all-reduce per bucket, unpack
                    O.bucketed_all_reduce(plan, tens, "bf16", "avg")
            self.step = step
            P = sum(numels)
            one = 2 * 2 * P * n
            sample = None
            self.nbytes = 3 * one if mode == "pipeline" else one
            self.desc = (f"the {len(numels)} tensor sizes scaled by {scale:.3g} "
                         f"({P} elements per rank, {plan.nbuckets} buckets of a {cap}-byte cap)")
        else:
            raise SystemExit(f"no oracle sample for workload {name}")
        if sample is not None:
            self.nbytes = sample.nbytes
        self.fraction = self.nbytes / full.nbytes


def time_oracle(smp, steps, warmup):
    """Mean seconds per oracle step after `warmup` untimed steps."""
    for _ in range(warmup):
        smp.step()
    t0 = time.perf_counter()
    for _ in range(steps):
        smp.step()
    return (time.perf_counter() - t0) / steps


def run_reference(args):
    """--impl reference: the CPU oracle on this host, timed on a bounded
    sample of the selected workload (the headline by default), with the
    same metric, unit and config as this workload's line."""
    world, rank, _ = dist_env()
    if world > 1 and rank != 0:
        return 0
    smp = OracleSample(args.workload, args, args.ref_sample)
    sec = time_oracle(smp, args.steps, args.warmup)
    config = workload_config(smp.full, world)
    if smp.fraction < 1:
        config["sample"] = smp.desc   # a bounded sample, not the whole workload
    value = smp.nbytes / sec / 1e9
    sample = (f"{smp.desc} per step ({smp.fraction:.3g} of the workload's bytes), "
              f"single-threaded C++ oracle (oracle/); host has {os.cpu_count()} cores")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": config,
            "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1,
                             "kind": "oracle", "sample": sample,
                             "cpu_model": host_cpu_model()},
            "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def cpu_baseline_sampled(args):
    """cpu_baseline of a workload other than the headline all-reduce: the
    oracle on a bounded sample of it (OracleSample), repeated for at least
    --cpu-seconds."""
    smp = OracleSample(args.workload, args, args.ref_sample)
    smp.step()  # loads the library, touches the buffers
    passes, t0 = 0, time.perf_counter()
    while True:
        smp.step()
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= args.cpu_seconds or passes >= 1000:
            break
    return {"value": round(passes * smp.nbytes / dt / 1e9, 4), "unit": UNIT, "cores": 1,
            "kind": "oracle",
            "cpu_model": host_cpu_model(),
            "sample": (f"{passes} step(s) of the workload on {smp.desc} "
                       f"({smp.fraction:.3g} of its bytes), single-threaded C++ oracle, "
                       f"{dt:.1f} s; host has {os.cpu_count()} cores")}


# ---- sweep ----------------------------------------------------------------------------------

def run_sweep(args, device, stream, peak):
    """All-reduce AVG bf16: N = 8 over 1 KiB .. 1 GiB per rank (powers of 4)
    and N in {2,4,8,16,32,64} at 256 MiB per rank; fits T = a + bytes / B to
    the 8-rank points and reports the crossover S* = a * B.  Then the FSDP
    step over the same rank counts (fsdp_rank_sweep)."""
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
        pt = {"n": n, "bytes_per_rank": count * 2, "us": round(ms * 1e3, 2),
              "GB/s": round(ar_bytes(n, count, 2) / (ms * 1e-3) / 1e9, 1),
              "ring_bytes_per_rank": sent * 2}
        if count * 2 <= (16 << 20):
            # the same call prepared once (cr.prepare): the C call alone per step
            prep = cr.prepare(cr.cr_all_reduce, bufs, count, "bf16", "avg", bufs, "bf16", stream)
            _, pper = timed(prep, steps, 3, 1, stream)
            pt["prepared_us"] = round(statistics.median(pper) * 1e3, 2)
            del prep
            # the same calls captured in a CUDA graph: no host work per call
            reps = 50
            g = torch.cuda.CUDAGraph()
            side = torch.cuda.Stream(device)
            side.wait_stream(torch.cuda.current_stream(device))
            with torch.cuda.graph(g, stream=side):
                for _ in range(reps):
                    cr.cr_all_reduce(bufs, count, "bf16", "avg", bufs, "bf16")
            _, gper = timed(g.replay, 10, 3, 1, stream)
            pt["graph_us"] = round(statistics.median(gper) * 1e3 / reps, 2)
            del g
        out.append(pt)
        del bufs
        torch.cuda.empty_cache()
    # least squares on the 8-rank points: t = a + x / B, x = algorithmic bytes
    xs = [ar_bytes(8, p["bytes_per_rank"] // 2, 2) for p in out if p["n"] == 8]
    ts = [p["us"] * 1e-6 for p in out if p["n"] == 8]
    mx, mt = sum(xs) / len(xs), sum(ts) / len(ts)
    slope = sum((x - mx) * (t - mt) for x, t in zip(xs, ts)) / sum((x - mx) ** 2 for x in xs)
    a = mt - slope * mx
    bw = 1 / slope
    g8 = [p["graph_us"] for p in out if p["n"] == 8 and "graph_us" in p]
    return {"points": out, "alpha_us": round(a * 1e6, 3), "bw_GBs": round(bw / 1e9, 1),
            "crossover_bytes": round(a * bw),
            "graph_latency_us_min": min(g8) if g8 else None,
            "fsdp_ranks": fsdp_rank_sweep(device, stream, peak),
            "uneven": uneven_sweep(device, stream, peak)}


def uneven_sweep(device, stream, peak):
    """Shard lengths on and off the vector grid.  The reduce-scatter (bf16
    AVG) and the FSDP step at N = 3, 5 and 8, each once with a count whose
    chunk length L is a multiple of 16 and once with an odd L; and the HSDP
    reduce-scatter (bf16 AVG, 64 MiB per rank) over mesh shapes beyond the
    ones built for a fixed shape."""
    import torch
    from fsdp_emulated_ranks_gb300 import cr
    out = []

    def add(kind, n, count, ms, nbytes, chunks=None, **kw):
        gbs = nbytes / (ms * 1e-3) / 1e9
        out.append({"op": kind, "n": n, "count": count,
                    "L": cr.cr_chunk_len(count, chunks or n), **kw,
                    "ms": round(ms, 4), "GB/s": round(gbs, 1), "frac": round(gbs / peak[0], 4)})

    for n in (3, 5, 8):
        for count in (n << 22, (n << 22) + n):   # L = 2^22, then 2^22 + 1
            bufs = alloc_ranks(n, count, torch.bfloat16, 0.02, 0, device)
            L = cr.cr_chunk_len(count, n)
            shards = [torch.empty(L, dtype=torch.bfloat16, device=device) for _ in range(n)]
            total, _ = timed(lambda: cr.cr_reduce_scatter(bufs, count, "bf16", "avg", shards, "bf16",
                                                          stream), 20, 3, 1, stream)
            add("reduce_scatter", n, count, total / 20, (n + 1) * count * 2)
            del bufs, shards
            torch.cuda.empty_cache()
    for n in (3, 5, 8):
        for count in (n << 24, (n << 24) + n):
            wl = FsdpStep(n=n, count=count)
            wl.setup(device)
            total, _ = timed(lambda: wl.step(stream), 10, 3, 1, stream)
            add("fsdp_step", n, count, total / 10, wl.nbytes)
            wl.teardown()
            torch.cuda.empty_cache()
    count = 1 << 25
    for R, S in ((2, 4), (4, 4), (8, 8), (8, 2), (3, 5)):
        n = R * S
        bufs = alloc_ranks(n, count, torch.bfloat16, 0.02, 0, device)
        L = cr.cr_chunk_len(count, S)
        shards = [torch.empty(L, dtype=torch.bfloat16, device=device) for _ in range(n)]
        total, _ = timed(lambda: cr.cr_hsdp_reduce_scatter(bufs, R, S, count, "bf16", "avg", shards,
                                                           "bf16", stream), 20, 3, 1, stream)
        add("hsdp", n, count, total / 20, (n + R) * count * 2, chunks=S, mesh=f"{R}x{S}")
        del bufs, shards
        torch.cuda.empty_cache()
    return out


def fsdp_rank_sweep(device, stream, peak):
    """The FSDP step, plain and clipped, at N in {2,4,8,16,32,64}: 2, 4 and
    8 ranks run the kernels built for that rank count, the others the
    runtime-N ones.  Parameters per step: 1.3e9 up to 4 ranks, then 2^33 / N
    (every point holds 26-47 GB on the device)."""
    import torch
    out = []
    for clip in (False, True):
        for n in (2, 4, 8, 16, 32, 64):
            count = min((1 << 33) // n, 1_300_000_000)
            wl = FsdpStep(n=n, count=count, clip=clip)
            wl.setup(device)
            total, per = timed(lambda: wl.step(stream), 10, 3, 1, stream)
            ms = total / 10
            gbs = wl.nbytes / (ms * 1e-3) / 1e9
            out.append({"n": n, "clipped": clip, "params": count, "ms": round(ms, 3),
                        "GB/s": round(gbs, 1), "frac": round(gbs / peak[0], 4),
                        "ms_median": round(statistics.median(per), 3)})
            wl.teardown()
            torch.cuda.empty_cache()
    return out


# ---- main ---------------------------------------------------------------------------------

def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", "--iters", dest="steps", type=int, default=200,
                    help="timed steps (--iters is the same flag)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--workload", default="allreduce",
                    help="timed workload: allreduce (headline), allreduce_f32, allreduce_wire, "
                         "reduce_scatter, all_gather, hsdp, "
                         "bucket_{pack,allreduce,unpack,pipeline,fused}, fsdp, fsdp_clipped, "
                         "fsdp2, accumulate, accumulate_allreduce")
    ap.add_argument("--config", type=int, choices=sorted(CONFIGS), default=None,
                    help="1: all-reduce SUM fp32 4 ranks x 2^20; 2: all-reduce AVG bf16 8 x 64 MiB "
                         "(the headline); 3: bucket pack -> all-reduce -> unpack; 4: FSDP step "
                         "1.3e9 x 8; 5: the sweep")
    ap.add_argument("--seed", type=int, default=0,
                    help="offset added to every seed of the input values (0: the recipe)")
    ap.add_argument("--fsdp-count", type=int, default=1_300_000_000)
    ap.add_argument("--bucket-ntensors", type=int, default=300)
    ap.add_argument("--fsdp2-layers", type=int, default=24,
                    help="transformer layers of the fsdp2 workload (1.27e9 parameters at 24)")
    ap.add_argument("--fsdp2-hidden", type=int, default=2048)
    ap.add_argument("--pg-timeout", type=int, default=600,
                    help="seconds after which a barrier or collective of an N > 1 run fails "
                         "when a rank is missing")
    ap.add_argument("--jsonl", default=None,
                    help="also append one JSON record per measured row to this file")
    ap.add_argument("--split", choices=["replicas", "slab"], default="replicas",
                    help="N > 1: every GPU runs the whole workload (replicas, weak scaling) "
                         "or one slab of its element range (slab, strong scaling)")
    ap.add_argument("--no-rows", action="store_true")
    ap.add_argument("--skip-fsdp", action="store_true")
    ap.add_argument("--row-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-api", choices=["host", "staged"], default="host")
    ap.add_argument("--e2e-slice", type=int, default=1 << 22,
                    help="elements per slice of the pipelined host all-reduce (0: auto)")
    ap.add_argument("--cpu-sample", type=int, default=1 << 25,
                    help="elements per rank the CPU oracle reduces for cpu_baseline")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="minimum CPU time of the cpu_baseline measurement")
    ap.add_argument("--ref-sample", type=int, default=1 << 25,
                    help="elements per rank per step for --impl reference (default: the "
                         "headline's whole 2^25, so both arms time the same workload)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)
    global SEED_OFFSET
    SEED_OFFSET = args.seed
    if args.config is not None:
        if CONFIGS[args.config] == "sweep":
            args.sweep = True
        else:
            args.workload = CONFIGS[args.config]

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
    init_dist(world, "nccl", args.pg_timeout)
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
    wl = head["workload"]
    rows = None
    overlap = wire = None
    if world == 1 and not args.no_rows:
        rows = run_rows(args, device, stream, peak, skip=args.workload)
        overlap = run_overlap(args, device)
        wire = wire_error(device)
    cpu = None
    if sample is not None and args.split == "slab":
        sample = None   # the slab run's baseline is the whole workload's; not sampled here
    if sample is not None:
        gbs, secs, passes = cpu_oracle_allreduce(sample, args.cpu_seconds)
        frac = (1 << 25) // sample[0].size
        cpu = {"value": round(gbs, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
               "cpu_model": host_cpu_model(),
               "sample": (f"{passes} pass(es) of the ring all-reduce AVG over the first "
                          f"{sample[0].size} elements of each of the 8 rank buffers "
                          f"({'all' if frac == 1 else '1/%d' % frac} of the workload's bytes), "
                          f"single-threaded C++ oracle, {secs:.1f} s; host has "
                          f"{os.cpu_count()} cores")}
    elif rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline_sampled(args)
    if rank == 0:
        config = workload_config(wl, world)
        if args.split == "slab":
            config["parallelism"] = (f"{world} GPU(s), each the slab of the element range "
                                     f"cr_slab_range gives it, of the same {wl.n} emulated ranks")
        line = {"metric": METRIC, "value": round(head["value"], 1), "unit": UNIT,
                "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
                "ms_per_step": head["ms_per_step"], "higher_is_better": True,
                # the arithmetic: fp32 partial sums (bf16 in and out, see config)
                "scaling": "strong" if args.split == "slab" else "weak",
                "vs_baseline": None, "dtype": "f32",
                "data": "synthetic",
                "config": config,
                "roofline": head["roofline"], "l2_flushed": head["l2_flushed"],
                "cpu_baseline": cpu, "e2e": head["e2e"],
                "gpu_launches": head["gpu_launches"], "clocks": head["clocks"],
                "frac_of_peak": round(head["value"] / world / peak[0], 4),
                "rows": rows, "ddp_overlap": overlap, "wire_error": wire}
        if rows is not None:
            # last on the line, so that the end of stdout carries every row
            line["rows_summary"] = rows_summary(args.workload, head["roofline"], rows, peak)
        print(json.dumps(line))
        if args.jsonl:
            with open(args.jsonl, "a") as f:
                rl = head["roofline"]
                head_rec = {"name": wl.name, "ms": round(head["ms_per_step"], 4),
                            "ms_median": rl["ms_median"], "ms_p10": rl["ms_p10"],
                            "ms_p90": rl["ms_p90"], "GB/s": round(head["value"], 1),
                            "frac": rl["frac"], "algorithmic_bytes": wl.nbytes,
                            "kernel": rl["kernel"], "traffic": rl["traffic"], "n_gpus": world,
                            "cpu_baseline": cpu}
                for rec in [head_rec] + (rows or []):
                    f.write(json.dumps(dict(rec, peak_GBs=peak[0], clocks=head["clocks"],
                                            host_cores=os.cpu_count())) + "\n")
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

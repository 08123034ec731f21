"""Entry points called from several host threads at once.

The library keeps every call's marshalled state (kernel parameter blocks,
the error detail) per thread and guards its caches of device attributes
with a lock, so concurrent calls on different buffers and streams must give
exactly what the same calls give one after another.  Four threads, each on
its own stream, repeat a mix of single-launch and chained calls (the
all-reduce, the same all-reduce again as two range calls over slabs, the
fused bucket all-reduce of 300 tensors in 3 launches, an FSDP2 step in 3
launches, the clipped FSDP step in 3 launches with the thread's own
workspace); every result is compared bit for bit with a single-threaded run
of the same sequence."""
import threading

import pytest
import torch

from fsdp_emulated_ranks_gb300 import build as libbuild
from fsdp_emulated_ranks_gb300 import cr
from fsdp_emulated_ranks_gb300 import inputs as I

pytestmark = pytest.mark.gpu
N = 8


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    libbuild.build()
    cr.lib()


def filled(count, dtype, std, seed):
    t = torch.empty(count, dtype=dtype, device="cuda")
    if count:
        I.torch_fill_normal_(t, std, seed)
    return t


class Job:
    """One thread's buffers and call sequence (seeded by `seed`)."""

    def __init__(self, seed):
        self.count = 8 * 8 * 3000 + 7 * seed
        self.bufs = [filled(self.count, torch.bfloat16, 0.02, seed * 100 + r) for r in range(N)]
        self.numels = [int(k) % 20000 + 1 for k in I.bucket_numels(300, seed=seed)]
        self.plan = cr.cr_bucket_plan(self.numels, 2, 64 * 1024)
        self.tens = [filled(k, torch.bfloat16, 1e-3, seed * 10000 + i)
                     for r in range(N) for i, k in enumerate(self.numels)]
        # FSDP2: 140 small parameters (3 launches of at most 64), uneven rows
        self.shapes = [(3 + (p * 7 + seed) % 13, 1 + p % 5) for p in range(140)]
        self.g2, self.p2, self.m2, self.mm2, self.mv2 = [], [], [], [], []
        for p, (d, rn) in enumerate(self.shapes):
            lr = -(-d // N)
            for r in range(N):
                self.g2.append(filled(d * rn, torch.bfloat16, 1e-3, seed * 7919 + p * N + r))
                self.p2.append(torch.empty(d * rn, dtype=torch.bfloat16, device="cuda"))
                rows = max(0, min(d, (r + 1) * lr) - min(d, r * lr))
                self.m2.append(filled(rows * rn, torch.float32, 0.02, seed * 31 + p * N + r))
                self.mm2.append(torch.zeros(rows * rn, dtype=torch.float32, device="cuda"))
                self.mv2.append(torch.zeros(rows * rn, dtype=torch.float32, device="cuda"))
        # clipped FSDP step: flat, ragged, its own workspace and norm output
        self.fc = 8 * 8 * 2000 + 3 + seed
        L = cr.cr_chunk_len(self.fc, N)
        lens = [max(0, min(self.fc, (j + 1) * L) - min(self.fc, j * L)) for j in range(N)]
        self.fg = [filled(self.fc, torch.bfloat16, 1e-3, seed * 50 + r) for r in range(N)]
        self.fm = [filled(k, torch.float32, 0.02, seed * 60 + j) for j, k in enumerate(lens)]
        self.fmm = [torch.zeros(k, dtype=torch.float32, device="cuda") for k in lens]
        self.fmv = [torch.zeros(k, dtype=torch.float32, device="cuda") for k in lens]
        self.fp = [torch.empty(self.fc, dtype=torch.bfloat16, device="cuda") for _ in range(N)]
        self.ws_bytes = cr.cr_fsdp_clip_workspace_bytes()
        self.ws = torch.empty(self.ws_bytes // 8, dtype=torch.float64, device="cuda")
        self.norm = torch.zeros(1, dtype=torch.float32, device="cuda")
        self.cfg = cr.adamw_cfg()

    def clone(self):
        other = object.__new__(Job)
        for k, v in vars(self).items():
            if isinstance(v, list) and v and isinstance(v[0], torch.Tensor):
                v = [t.clone() for t in v]
            elif isinstance(v, torch.Tensor):
                v = v.clone()
            setattr(other, k, v)
        other.cfg = cr.adamw_cfg()
        return other

    def run(self, stream, iters=4):
        for it in range(iters):
            cr.cr_all_reduce(self.bufs, self.count, "bf16", "avg", self.bufs, "bf16", stream)
            for g in range(2):
                lo, hi = cr.cr_slab_range(self.count, N, 2, g)
                slab = [b[lo:hi] for b in self.bufs]
                cr.cr_all_reduce_range(slab, self.count, lo, hi, "bf16", "avg", slab, "bf16",
                                       stream)
            cr.cr_bucket_all_reduce_fused(self.plan, N, self.tens, "bf16", "avg", stream)
            self.cfg.step = it + 1
            cr.cr_fsdp2_step(self.shapes, N, [None if t.numel() == 0 else t for t in self.g2],
                             [None if t.numel() == 0 else t for t in self.m2],
                             [None if t.numel() == 0 else t for t in self.mm2],
                             [None if t.numel() == 0 else t for t in self.mv2], self.cfg,
                             [None if t.numel() == 0 else t for t in self.p2], stream)
            cr.cr_fsdp_step_clipped(self.fg, self.fc, self.fm, self.fmm, self.fmv, self.cfg, 1e-3,
                                    self.ws, self.ws_bytes, self.fp, self.norm, stream)

    def results(self):
        return (self.bufs + self.tens + self.p2 + self.m2 + self.mm2 + self.mv2 + self.fm
                + self.fmm + self.fmv + self.fp + [self.norm])


def test_concurrent_calls_equal_sequential_calls():
    jobs = [Job(seed) for seed in range(1, 5)]
    refs = [j.clone() for j in jobs]
    torch.cuda.synchronize()
    # one after another, on one stream
    s0 = torch.cuda.Stream()
    for j in refs:
        j.run(s0)
    torch.cuda.synchronize()
    # four threads at once, each on its own stream
    errors = []

    def worker(job):
        try:
            s = torch.cuda.Stream()
            job.run(s)
            s.synchronize()
        except Exception as e:  # reported below
            errors.append(e)
    threads = [threading.Thread(target=worker, args=(j,)) for j in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for j, r in zip(jobs, refs):
        for a, b in zip(j.results(), r.results()):
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8))

"""Seeded synthetic inputs for the emulated-rank collectives.

This module only draws random numbers; it holds none of the collectives'
arithmetic and imports nothing else from the package, so the CUDA path and
the CPU oracle can both be fed from it without sharing any code.

Generators:
  * host draws use numpy's PCG64 (``np.random.default_rng(seed)``);
  * device draws use torch's CUDA Philox generator
    (``torch.Generator("cuda").manual_seed(seed)``), which is what the
    benchmark uses to fill tens of GB quickly.
Parity never depends on which one is used: the exact bytes given to the GPU
path are the ones copied back for the oracle.

Workload recipes (element counts, distributions, seeds):
  * all-reduce SUM, 4 ranks, fp32, 2^20 elements/rank, N(0,1), one stream
    seeded 0 filled rank after rank;
  * all-reduce AVG, 8 ranks, bf16, 2^25 elements/rank, N(0, 0.02^2), rank r
    seeded r;
  * DDP buckets, 8 ranks, 300 bf16 tensors with numel
    floor(exp(U(ln 1024, ln 2^24))) (seed 7), values N(0, 1e-3^2), rank r's
    tensors from one stream seeded 1000 + r;
  * FSDP step, 8 ranks, 1.3e9 flat params, bf16 grads N(0, 1e-3^2) seeded
    1000 + r, fp32 master N(0, 0.02^2) seeded 2000, m = v = 0;
  * sweep, all-reduce AVG bf16, N(0,1), rank r seeded r.
"""
from __future__ import annotations

import math

import numpy as np

BF16_BITS = np.uint16


def np_normal_f32(count: int, std: float, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(count, dtype=np.float32) * np.float32(std))


def np_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even, via torch.

    Used only to shape random inputs; the tested arithmetic never goes
    through here."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def host_rank_buffers(n: int, count: int, dtype: str, std: float = 1.0,
                      seed0: int = 0, one_stream: bool = False):
    """n host buffers of `count` elements each.

    dtype "f32"/"bf16": N(0, std^2); "i32": integers in [-1024, 1024].
    one_stream: draw all ranks from one stream seeded seed0, rank after
    rank; else rank r uses seed seed0 + r."""
    out = []
    if one_stream:
        if dtype == "i32":
            rng = np.random.default_rng(seed0)
            big = rng.integers(-1024, 1025, size=n * count, dtype=np.int32)
        else:
            big = np_normal_f32(n * count, std, seed0)
        for r in range(n):
            out.append(big[r * count:(r + 1) * count].copy())
    else:
        for r in range(n):
            if dtype == "i32":
                rng = np.random.default_rng(seed0 + r)
                out.append(rng.integers(-1024, 1025, size=count, dtype=np.int32))
            else:
                out.append(np_normal_f32(count, std, seed0 + r))
    if dtype == "bf16":
        out = [np_to_bf16_bits(x) for x in out]
    return out


def integer_valued_f32(n: int, count: int, seed: int, bound: int = 1024):
    """fp32 buffers holding integers in [-bound, bound]: every partial sum of
    up to 64 of them is exactly representable, so any summation order gives
    the same result."""
    rng = np.random.default_rng(seed)
    return [rng.integers(-bound, bound + 1, size=count).astype(np.float32)
            for _ in range(n)]


def bucket_numels(ntensors: int = 300, lo: int = 1024, hi: int = 1 << 24,
                  seed: int = 7) -> np.ndarray:
    """Log-uniform element counts in [lo, hi]."""
    rng = np.random.default_rng(seed)
    u = rng.uniform(math.log(lo), math.log(hi), size=ntensors)
    return np.clip(np.floor(np.exp(u)), lo, hi).astype(np.uint64)


# ---- device (torch) draws ---------------------------------------------------

def torch_normal(count: int, std: float, seed: int, dtype, device="cuda"):
    """N(0, std^2) drawn in fp32 by torch's generator on `device`, then cast
    (round to nearest even for bf16)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    x = torch.randn(count, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x if dtype == torch.float32 else x.to(dtype)


def torch_fill_normal_(t, std: float, seed: int):
    """Fill an existing fp32/bf16 tensor with N(0, std^2) in slabs, so that
    multi-GB buffers need no fp32 copy of the whole tensor."""
    import torch
    g = torch.Generator(device=t.device)
    g.manual_seed(seed)
    flat = t.view(-1)
    slab = 1 << 27
    for a in range(0, flat.numel(), slab):
        b = min(flat.numel(), a + slab)
        x = torch.randn(b - a, generator=g, device=t.device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        flat[a:b].copy_(x)
    return t

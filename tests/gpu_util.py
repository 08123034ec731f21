"""Helpers for the GPU parity tests: host<->device copies of the bit
patterns, guarded output buffers (canaries around every output) and bf16
ulp distance."""
from __future__ import annotations

import numpy as np
import torch

GUARD = 64  # elements of canary on each side of an output buffer
_TORCH = {"f32": torch.float32, "bf16": torch.bfloat16, "i32": torch.int32}
_NP = {"f32": np.float32, "bf16": np.uint16, "i32": np.int32}
_PATTERN = {"f32": -7.25, "bf16": -7.25, "i32": -123456789}


def dev():
    return torch.device("cuda")


def to_dev(x: np.ndarray, dt: str, offset: int = 0) -> torch.Tensor:
    """Copy a host array to the device.  offset > 0 places it `offset`
    elements into a larger allocation (so it is not 16-byte aligned)."""
    if dt == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x))
    if offset == 0:
        return t.to(dev())
    base = torch.empty(x.size + offset, dtype=_TORCH[dt], device=dev())
    base[offset:].copy_(t.to(dev()))
    return base[offset:]


def to_host(t: torch.Tensor, dt: str) -> np.ndarray:
    t = t.detach().cpu()
    if dt == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


class Guarded:
    """An output buffer with GUARD canary elements on both sides."""

    def __init__(self, nelem: int, dt: str, offset: int = 0):
        self.dt, self.n = dt, nelem
        self.base = torch.full((nelem + 2 * GUARD + offset,), _PATTERN[dt],
                               dtype=_TORCH[dt], device=dev())
        self.lo = GUARD + offset
        self.view = self.base[self.lo:self.lo + nelem]

    def ptr(self):
        return self.view.data_ptr() if self.n else 0

    def check(self):
        h = self.base.cpu()
        pat = torch.full((1,), _PATTERN[self.dt], dtype=_TORCH[self.dt])
        assert torch.all(h[:self.lo] == pat), "canary before the buffer overwritten"
        assert torch.all(h[self.lo + self.n:] == pat), "canary after the buffer overwritten"

    def host(self):
        return to_host(self.view, self.dt)


def bf16_ulps(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 ulps between two arrays of bf16 bit patterns."""
    def ordered(x):
        x = x.astype(np.int32)
        mag = x & 0x7FFF
        return np.where(x & 0x8000, -mag, mag)
    return np.abs(ordered(a) - ordered(b))


def assert_match(got: np.ndarray, want: np.ndarray, dt: str, what: str = ""):
    """Bit-exact for fp32 and int32; within 1 bf16 ulp for bf16."""
    assert got.shape == want.shape, what
    if dt == "bf16":
        d = bf16_ulps(got, want)
        assert d.size == 0 or int(d.max()) <= 1, f"{what}: max {int(d.max())} bf16 ulps"
    else:
        assert got.tobytes() == want.tobytes(), (
            f"{what}: {int(np.sum(got.view(np.uint32) != want.view(np.uint32)))} elements differ")


def rel_maxabs(got: np.ndarray, want: np.ndarray) -> float:
    """max |got - want| / max |want| (0 when want is all zero and equal)."""
    scale = float(np.max(np.abs(want))) if want.size else 0.0
    err = float(np.max(np.abs(got.astype(np.float64) - want.astype(np.float64)))) if want.size else 0.0
    return err / scale if scale > 0 else err

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
    """Bitwise equality, for every dtype.

    Everything the library computes is deterministic: fp32 partial sums in
    the ring's fixed order, one division by N, one round-to-nearest-even
    cast, AdamW in individually rounded fp32 operations.  So the bits are
    the pass criterion.  The looser bounds of the workload statement (at
    most 1 bf16 ulp after a cast, 1e-6 * max|ref| for fp32 optimizer state)
    are reported in the failure message, not accepted."""
    assert got.shape == want.shape, what
    if got.tobytes() == want.tobytes():
        return
    ndiff = int(np.sum(got.view(np.uint8).reshape(got.size, -1)
                       != want.view(np.uint8).reshape(want.size, -1), axis=1).astype(bool).sum())
    if dt == "bf16":
        detail = f"max {int(bf16_ulps(got, want).max())} bf16 ulps"
    elif dt == "f32":
        detail = f"max-abs error {rel_maxabs(got, want):.3g} of max|ref|"
    else:
        detail = "integers differ"
    raise AssertionError(f"{what}: {ndiff} of {got.size} elements differ ({detail})")


def clip_coefficients(max_norm: float, norm_ref: float, rel: float = 1e-6):
    """The fp32 clip coefficients fl32(min(1, max_norm / (norm + 1e-6)))
    for every norm within `rel` of the oracle's float64 norm, the oracle's
    own coefficient first.

    The library sums the squares of the averaged gradient in fp32 batches
    added in fp64 per CTA, then adds the CTA partials in a fixed order; the
    oracle sums them in float64 in element order.  Both orders are fixed
    and correct, but they round differently, so the fp32 coefficient may sit
    a few ulps apart.  Everything after the coefficient is deterministic, so
    the library's state must equal, bit for bit, the oracle's state at one
    of these coefficients."""
    c0 = np.float32(min(1.0, max_norm / (norm_ref + 1e-6)))
    lo = np.float32(min(1.0, max_norm / (norm_ref * (1 + rel) + 1e-6)))
    hi = np.float32(min(1.0, max_norm / (norm_ref * (1 - rel) + 1e-6)))
    out, c = [c0], lo
    while c <= hi:
        if c != c0:
            out.append(c)
        c = np.nextafter(c, np.float32(np.inf))
    return out


def rel_maxabs(got: np.ndarray, want: np.ndarray) -> float:
    """max |got - want| / max |want| (0 when want is all zero and equal)."""
    scale = float(np.max(np.abs(want))) if want.size else 0.0
    err = float(np.max(np.abs(got.astype(np.float64) - want.astype(np.float64)))) if want.size else 0.0
    return err / scale if scale > 0 else err


def oracle_clipped_at(grads, master, m, v, cfg, coef):
    """The oracle's clipped FSDP step with the clip coefficient given:
    ring reduce-scatter AVG to fp32 shards, g * coef in fp32, AdamW on each
    owner's shard, bf16 cast, ring all-gather.  At the oracle's own
    coefficient this is orc_fsdp_step_clipped (pinned on the CPU).  Updates
    master/m/v in place and returns the per-rank bf16 params."""
    import oracle as O
    count = sum(x.size for x in master)
    gsh, _ = O.ring_reduce_scatter(grads, "bf16", "avg", "f32")
    pshards = []
    for j in range(len(grads)):
        g = (gsh[j] * np.float32(coef)).astype(np.float32)
        O.adamw(master[j], m[j], v[j], g, cfg)
        pshards.append(O.f32_to_bf16(master[j]))
    params, _ = O.ring_all_gather(pshards, count, "bf16")
    return params


def assert_clipped_match(got_state, got_params, grads, master, m, v, cfg, max_norm, norm_ref,
                         what=""):
    """The clipped step's outputs must equal, bitwise, the oracle's at one of
    the fp32 coefficients that clip_coefficients allows.  got_state is
    (master, m, v), each a per-owner list of host arrays; got_params the
    per-rank bf16 params.  master/m/v are the state before the step; they
    are advanced to the matching coefficient's result.  Returns that
    coefficient."""
    for c in clip_coefficients(max_norm, norm_ref):
        ms, mm, vv = [x.copy() for x in master], [x.copy() for x in m], [x.copy() for x in v]
        params = oracle_clipped_at(grads, ms, mm, vv, cfg, c)
        same = all(a.tobytes() == b.tobytes()
                   for got, ref in zip(got_state, (ms, mm, vv)) for a, b in zip(got, ref))
        if same and all(a.tobytes() == b.tobytes() for a, b in zip(got_params, params)):
            for dst, src in zip((master, m, v), (ms, mm, vv)):
                for d, s in zip(dst, src):
                    d[...] = s
            return c
    # Report against the oracle's own coefficient.
    c = clip_coefficients(max_norm, norm_ref)[0]
    ms, mm, vv = [x.copy() for x in master], [x.copy() for x in m], [x.copy() for x in v]
    params = oracle_clipped_at(grads, ms, mm, vv, cfg, c)
    for got, ref, name in zip(got_state, (ms, mm, vv), ("master", "m", "v")):
        for j, (a, b) in enumerate(zip(got, ref)):
            assert_match(a, b, "f32", f"{what} {name}[{j}] (no coefficient in the window fits)")
    for r, (a, b) in enumerate(zip(got_params, params)):
        assert_match(a, b, "bf16", f"{what} params[{r}] (no coefficient in the window fits)")
    raise AssertionError(f"{what}: state and params fit different coefficients")

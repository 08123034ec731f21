"""ctypes bindings to the C++ oracle (``oracle/*.cpp``).

TEST INFRASTRUCTURE ONLY.  This is the plain, slow, single-threaded CPU
statement of what the emulated-rank collectives compute; only ``tests/``, the
smoke check in ``__graft_entry__`` and the CPU-baseline leg of ``bench.py``
import it.  The product library never does, and the two share no code.

Arrays are numpy arrays: fp32 as ``float32``, bf16 as ``uint16`` bit
patterns, int32 as ``int32``.  Dtypes are named ``"f32"``, ``"bf16"``,
``"i32"``; ops ``"sum"``, ``"avg"``.
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass

import numpy as np

from . import build as _build

_DT = {"f32": 0, "bf16": 1, "i32": 2}
_NP = {"f32": np.float32, "bf16": np.uint16, "i32": np.int32}
_OP = {"sum": 0, "avg": 1}
MAX_RANKS = 64

_lib = None


class _Traffic(C.Structure):
    _fields_ = [("sent", C.c_uint64 * MAX_RANKS),
                ("recv", C.c_uint64 * MAX_RANKS),
                ("steps", C.c_int)]


class _AdamCfg(C.Structure):
    _fields_ = [("lr", C.c_double), ("beta1", C.c_double),
                ("beta2", C.c_double), ("eps", C.c_double),
                ("weight_decay", C.c_double), ("step", C.c_long)]


@dataclass
class Traffic:
    """Per-rank element counts of one simulated collective."""
    sent: list
    recv: list
    steps: int


@dataclass
class AdamWConfig:
    lr: float = 1e-4
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01
    step: int = 1


def lib() -> C.CDLL:
    global _lib
    if _lib is None:
        _lib = C.CDLL(_build.build())
        L = _lib
        vp, sz = C.c_void_p, C.c_size_t
        L.orc_chunk_len.restype = sz
        L.orc_chunk_len.argtypes = [sz, C.c_int]
        L.orc_chunk_bounds.argtypes = [sz, C.c_int, C.c_int,
                                       C.POINTER(sz), C.POINTER(sz)]
        L.orc_f32_to_bf16_array.argtypes = [sz, vp, vp]
        L.orc_ring_reduce_scatter.argtypes = [C.c_int, sz, C.c_int, C.c_int,
                                              vp, vp, C.c_int, vp, vp, vp]
        L.orc_fold_reduce_scatter.argtypes = [C.c_int, sz, C.c_int, C.c_int,
                                              vp, vp, C.c_int]
        L.orc_fold_columns.argtypes = [C.c_int, sz, C.c_int, C.c_int, vp, vp,
                                       vp, C.c_int]
        L.orc_ring_all_gather.argtypes = [C.c_int, sz, C.c_int, vp, vp, vp, vp]
        L.orc_ring_all_reduce.argtypes = [C.c_int, sz, C.c_int, C.c_int, vp, vp,
                                          C.c_int, vp]
        L.orc_naive_all_reduce.argtypes = [C.c_int, sz, C.c_int, C.c_int, vp,
                                           vp, C.c_int, vp]
        L.orc_adamw.argtypes = [sz, vp, vp, vp, vp, C.POINTER(_AdamCfg)]
        L.orc_fsdp_step.argtypes = [C.c_int, sz, vp, vp, vp, vp,
                                    C.POINTER(_AdamCfg), vp]
        L.orc_fsdp_step_clipped.argtypes = [C.c_int, sz, vp, vp, vp, vp,
                                            C.POINTER(_AdamCfg), C.c_double, vp,
                                            C.POINTER(C.c_double)]
        L.orc_ring_reduce_scatter_L.argtypes = [C.c_int, sz, sz, C.c_int, C.c_int,
                                                vp, vp, C.c_int, vp, vp, vp]
        L.orc_ring_all_gather_L.argtypes = [C.c_int, sz, sz, C.c_int, vp, vp, vp, vp]
        L.orc_fsdp2_step.argtypes = [C.c_int, vp, C.c_int, vp, vp, vp, vp,
                                     C.POINTER(_AdamCfg), vp]
        L.orc_ring_reduce_scatter_wire.argtypes = [C.c_int, sz, C.c_int, C.c_int, C.c_int,
                                                   vp, vp, C.c_int]
        L.orc_ring_all_reduce_wire.argtypes = [C.c_int, sz, C.c_int, C.c_int, C.c_int, vp, vp,
                                               C.c_int]
        L.orc_hsdp_reduce_scatter.argtypes = [C.c_int, C.c_int, sz, C.c_int, C.c_int, vp, vp,
                                              C.c_int]
        L.orc_accumulate.restype = None
        L.orc_accumulate.argtypes = [sz, vp, vp, C.c_int]
        L.orc_bucket_plan.argtypes = [C.c_int, vp, sz, sz, vp, vp, vp,
                                      C.POINTER(C.c_int)]
        L.orc_bucket_pack.argtypes = [C.c_int, C.c_int, vp, sz, vp, vp, vp, vp]
        L.orc_bucket_unpack.argtypes = [C.c_int, C.c_int, vp, sz, vp, vp, vp,
                                        vp]
        L.orc_alpha_beta_ring_allreduce.restype = C.c_double
        L.orc_alpha_beta_ring_allreduce.argtypes = [C.c_int, C.c_double,
                                                    C.c_double, C.c_double]
    return _lib


class OracleError(RuntimeError):
    pass


def _check(rc: int, what: str) -> None:
    if rc != 0:
        names = {1: "EINVAL", 2: "EUNSUPPORTED", 3: "ENOMEM"}
        raise OracleError(f"{what}: {names.get(rc, rc)}")


def _ptrs(arrays) -> C.Array:
    arr = (C.c_void_p * max(1, len(arrays)))()
    for i, a in enumerate(arrays):
        assert a.flags["C_CONTIGUOUS"]
        arr[i] = a.ctypes.data
    return arr


def _traffic(t: _Traffic, n: int) -> Traffic:
    return Traffic(list(t.sent[:n]), list(t.recv[:n]), t.steps)


def _cfg(c: AdamWConfig) -> _AdamCfg:
    return _AdamCfg(c.lr, c.beta1, c.beta2, c.eps, c.weight_decay, c.step)


# ---- chunking ---------------------------------------------------------------

def chunk_len(count: int, n: int) -> int:
    return lib().orc_chunk_len(count, n)


def chunk_bounds(count: int, n: int, j: int) -> tuple[int, int]:
    lo, hi = C.c_size_t(), C.c_size_t()
    lib().orc_chunk_bounds(count, n, j, C.byref(lo), C.byref(hi))
    return lo.value, hi.value


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().orc_f32_to_bf16_array(x.size, x.ctypes.data, out.ctypes.data)
    return out


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---- ring collectives -------------------------------------------------------

def _shards_out(count, n, dtype):
    out = []
    for j in range(n):
        lo, hi = chunk_bounds(count, n, j)
        out.append(np.zeros(hi - lo, _NP[dtype]))
    return out


def ring_reduce_scatter(bufs, dtype, op="sum", out_dtype=None, trace=False):
    """Literal ring simulation.  Returns (shards, Traffic[, (chunks, values)])."""
    out_dtype = out_dtype or dtype
    n, count = len(bufs), bufs[0].size
    bufs = [np.ascontiguousarray(b, _NP[dtype]) for b in bufs]
    shards = _shards_out(count, n, out_dtype)
    tr = _Traffic()
    tc = np.zeros(max(1, (n - 1) * n), np.int32)
    tv = np.zeros(max(1, (n - 1) * n), np.float64)
    _check(lib().orc_ring_reduce_scatter(
        n, count, _DT[dtype], _OP[op], _ptrs(bufs), _ptrs(shards),
        _DT[out_dtype], C.byref(tr), tc.ctypes.data if trace else None,
        tv.ctypes.data if trace else None), "ring_reduce_scatter")
    res = (shards, _traffic(tr, n))
    if trace:
        res = res + ((tc[:(n - 1) * n].reshape(n - 1, n),
                      tv[:(n - 1) * n].reshape(n - 1, n)),)
    return res


def fold_reduce_scatter(bufs, dtype, op="sum", out_dtype=None):
    out_dtype = out_dtype or dtype
    n, count = len(bufs), bufs[0].size
    bufs = [np.ascontiguousarray(b, _NP[dtype]) for b in bufs]
    shards = _shards_out(count, n, out_dtype)
    _check(lib().orc_fold_reduce_scatter(n, count, _DT[dtype], _OP[op],
                                         _ptrs(bufs), _ptrs(shards),
                                         _DT[out_dtype]), "fold_reduce_scatter")
    return shards


def fold_columns(vals: np.ndarray, chunk: np.ndarray, dtype, op="sum",
                 out_dtype=None) -> np.ndarray:
    """vals: [nsamp, n] values of each sampled element on ranks 0..n-1."""
    out_dtype = out_dtype or dtype
    vals = np.ascontiguousarray(vals, _NP[dtype])
    nsamp, n = vals.shape
    chunk = np.ascontiguousarray(chunk, np.int32)
    out = np.zeros(nsamp, _NP[out_dtype])
    _check(lib().orc_fold_columns(n, nsamp, _DT[dtype], _OP[op],
                                  vals.ctypes.data, chunk.ctypes.data,
                                  out.ctypes.data, _DT[out_dtype]),
           "fold_columns")
    return out


def ring_all_gather(shards, count, dtype, trace=False):
    n = len(shards)
    shards = [np.ascontiguousarray(s, _NP[dtype]) for s in shards]
    bufs = [np.zeros(count, _NP[dtype]) for _ in range(n)]
    tr = _Traffic()
    ta = np.zeros(max(1, (n - 1) * n), np.int32)
    _check(lib().orc_ring_all_gather(n, count, _DT[dtype], _ptrs(shards),
                                     _ptrs(bufs), C.byref(tr),
                                     ta.ctypes.data if trace else None),
           "ring_all_gather")
    res = (bufs, _traffic(tr, n))
    if trace:
        res = res + (ta[:(n - 1) * n].reshape(n - 1, n),)
    return res


def ring_all_reduce(bufs, dtype, op="sum", out_dtype=None):
    out_dtype = out_dtype or dtype
    n, count = len(bufs), bufs[0].size
    bufs = [np.ascontiguousarray(b, _NP[dtype]) for b in bufs]
    out = [np.zeros(count, _NP[out_dtype]) for _ in range(n)]
    tr = _Traffic()
    _check(lib().orc_ring_all_reduce(n, count, _DT[dtype], _OP[op],
                                     _ptrs(bufs), _ptrs(out), _DT[out_dtype],
                                     C.byref(tr)), "ring_all_reduce")
    return out, _traffic(tr, n)


def naive_all_reduce(bufs, dtype, op="sum", out_dtype=None):
    out_dtype = out_dtype or dtype
    n, count = len(bufs), bufs[0].size
    bufs = [np.ascontiguousarray(b, _NP[dtype]) for b in bufs]
    out = [np.zeros(count, _NP[out_dtype]) for _ in range(n)]
    tr = _Traffic()
    _check(lib().orc_naive_all_reduce(n, count, _DT[dtype], _OP[op],
                                      _ptrs(bufs), _ptrs(out), _DT[out_dtype],
                                      C.byref(tr)), "naive_all_reduce")
    return out, _traffic(tr, n)


# ---- AdamW and the FSDP step ------------------------------------------------

def adamw(p, m, v, g, cfg: AdamWConfig) -> None:
    """In-place scalar AdamW on float32 arrays."""
    for a in (p, m, v, g):
        assert a.dtype == np.float32 and a.flags["C_CONTIGUOUS"]
    c = _cfg(cfg)
    lib().orc_adamw(p.size, p.ctypes.data, m.ctypes.data, v.ctypes.data,
                    g.ctypes.data, C.byref(c))


def fsdp_step(grads, master, m, v, cfg: AdamWConfig):
    """grads: n bf16 (uint16) arrays of count; master/m/v: n fp32 shards
    (updated in place).  Returns the n all-gathered bf16 param buffers."""
    n, count = len(grads), grads[0].size
    grads = [np.ascontiguousarray(g, np.uint16) for g in grads]
    params = [np.zeros(count, np.uint16) for _ in range(n)]
    c = _cfg(cfg)
    _check(lib().orc_fsdp_step(n, count, _ptrs(grads), _ptrs(master),
                               _ptrs(m), _ptrs(v), C.byref(c), _ptrs(params)),
           "fsdp_step")
    return params


def fsdp_step_clipped(grads, master, m, v, cfg: AdamWConfig, max_norm: float):
    """FSDP step with global gradient-norm clipping.  Returns (params, norm)."""
    n, count = len(grads), grads[0].size
    grads = [np.ascontiguousarray(g, np.uint16) for g in grads]
    params = [np.zeros(count, np.uint16) for _ in range(n)]
    c = _cfg(cfg)
    norm = C.c_double()
    _check(lib().orc_fsdp_step_clipped(n, count, _ptrs(grads), _ptrs(master),
                                       _ptrs(m), _ptrs(v), C.byref(c),
                                       float(max_norm), _ptrs(params),
                                       C.byref(norm)), "fsdp_step_clipped")
    return params, norm.value


def ring_reduce_scatter_L(bufs, L, dtype, op="sum", out_dtype=None):
    """Ring reduce-scatter with an explicit chunk length L (elements)."""
    out_dtype = out_dtype or dtype
    n, count = len(bufs), bufs[0].size
    bufs = [np.ascontiguousarray(b, _NP[dtype]) for b in bufs]
    shards = [np.zeros(max(0, min(count, (j + 1) * L) - min(count, j * L)), _NP[out_dtype])
              for j in range(n)]
    _check(lib().orc_ring_reduce_scatter_L(n, count, L, _DT[dtype], _OP[op], _ptrs(bufs),
                                           _ptrs(shards), _DT[out_dtype], None, None, None),
           "ring_reduce_scatter_L")
    return shards


def ring_all_reduce_wire(bufs, dtype, op, wire_dtype, out_dtype=None):
    """Ring all-reduce whose messages travel as wire_dtype ("f32" or "bf16")."""
    out_dtype = out_dtype or dtype
    n, count = len(bufs), bufs[0].size
    bufs = [np.ascontiguousarray(b, _NP[dtype]) for b in bufs]
    out = [np.zeros(count, _NP[out_dtype]) for _ in range(n)]
    _check(lib().orc_ring_all_reduce_wire(n, count, _DT[dtype], _OP[op], _DT[wire_dtype],
                                          _ptrs(bufs), _ptrs(out), _DT[out_dtype]),
           "ring_all_reduce_wire")
    return out


def ring_reduce_scatter_wire(bufs, dtype, op, wire_dtype, out_dtype=None):
    out_dtype = out_dtype or dtype
    n, count = len(bufs), bufs[0].size
    bufs = [np.ascontiguousarray(b, _NP[dtype]) for b in bufs]
    shards = _shards_out(count, n, out_dtype)
    _check(lib().orc_ring_reduce_scatter_wire(n, count, _DT[dtype], _OP[op], _DT[wire_dtype],
                                              _ptrs(bufs), _ptrs(shards), _DT[out_dtype]),
           "ring_reduce_scatter_wire")
    return shards


def hsdp_reduce_scatter(bufs, R, S, dtype, op="sum", out_dtype=None):
    """bufs[g*S + s]; returns shards[g*S + j] (shard j of group g)."""
    out_dtype = out_dtype or dtype
    count = bufs[0].size
    bufs = [np.ascontiguousarray(b, _NP[dtype]) for b in bufs]
    shards = [x for _ in range(R) for x in _shards_out(count, S, out_dtype)]
    _check(lib().orc_hsdp_reduce_scatter(R, S, count, _DT[dtype], _OP[op], _ptrs(bufs),
                                         _ptrs(shards), _DT[out_dtype]), "hsdp_reduce_scatter")
    return shards


def fsdp2_shard_rows(dim0: int, n: int, j: int) -> tuple[int, int]:
    """Rows [lo, hi) of dim 0 that rank j owns (torch.chunk-like)."""
    Lr = -(-dim0 // n) if n else 0
    return min(dim0, j * Lr), min(dim0, (j + 1) * Lr)


class _Shape(C.Structure):
    _fields_ = [("dim0", C.c_size_t), ("row_numel", C.c_size_t)]


def fsdp2_step(shapes, grads, master, m, v, cfg: AdamWConfig):
    """shapes: [(dim0, row_numel)] per parameter; grads[p][r]: full bf16
    gradient of parameter p on rank r; master/m/v[p][j]: fp32 shard j
    (updated in place).  Returns params[p][r], the all-gathered bf16."""
    n = len(grads[0]) if grads else 1
    P = len(shapes)
    sh = (_Shape * max(1, P))(*[_Shape(d, rn) for d, rn in shapes])
    flat_g = [np.ascontiguousarray(g, np.uint16) for row in grads for g in row]
    params = [[np.zeros(d * rn, np.uint16) for _ in range(n)] for d, rn in shapes]
    flat_p = [x for row in params for x in row]
    flat = lambda xs: [x for row in xs for x in row]
    c = _cfg(cfg)
    _check(lib().orc_fsdp2_step(P, sh, n, _ptrs(flat_g), _ptrs(flat(master)), _ptrs(flat(m)),
                                _ptrs(flat(v)), C.byref(c), _ptrs(flat_p)), "fsdp2_step")
    return params


def accumulate(acc: np.ndarray, g: np.ndarray, dtype: str) -> None:
    """acc += g in fp32 (g: f32 or bf16 bits), in place."""
    assert acc.dtype == np.float32 and acc.flags["C_CONTIGUOUS"]
    g = np.ascontiguousarray(g, _NP[dtype])
    lib().orc_accumulate(acc.size, acc.ctypes.data, g.ctypes.data, _DT[dtype])


# ---- DDP buckets ------------------------------------------------------------

@dataclass
class BucketPlan:
    tensor_bucket: np.ndarray   # int32 [T]
    tensor_offset: np.ndarray   # uint64 [T], elements
    bucket_numel: np.ndarray    # uint64 [B]
    numels: np.ndarray          # uint64 [T]
    esize: int

    @property
    def nbuckets(self) -> int:
        return int(self.bucket_numel.size)


def bucket_plan(numels, esize: int, cap_bytes: int) -> BucketPlan:
    numels = np.ascontiguousarray(numels, np.uint64)
    t = numels.size
    tb = np.zeros(max(1, t), np.int32)
    to = np.zeros(max(1, t), np.uint64)
    bn = np.zeros(max(1, t), np.uint64)
    nb = C.c_int()
    _check(lib().orc_bucket_plan(t, numels.ctypes.data, esize, cap_bytes,
                                 tb.ctypes.data, to.ctypes.data,
                                 bn.ctypes.data, C.byref(nb)), "bucket_plan")
    return BucketPlan(tb[:t].copy(), to[:t].copy(), bn[:nb.value].copy(),
                      numels, esize)


def bucket_pack(plan: BucketPlan, tensors_per_rank):
    """tensors_per_rank[r][t] -> buckets_per_rank[r][b]."""
    n, t = len(tensors_per_rank), plan.numels.size
    dt = tensors_per_rank[0][0].dtype if t else np.uint16
    buckets = [[np.zeros(int(bn), dt) for bn in plan.bucket_numel]
               for _ in range(n)]
    flat_t = [np.ascontiguousarray(x) for row in tensors_per_rank for x in row]
    flat_b = [b for row in buckets for b in row]
    lib().orc_bucket_pack(n, t, plan.numels.ctypes.data, plan.esize,
                          plan.tensor_bucket.ctypes.data,
                          plan.tensor_offset.ctypes.data, _ptrs(flat_t),
                          _ptrs(flat_b))
    return buckets


def bucket_unpack(plan: BucketPlan, buckets_per_rank, dtype):
    n, t = len(buckets_per_rank), plan.numels.size
    tensors = [[np.zeros(int(k), dtype) for k in plan.numels] for _ in range(n)]
    flat_b = [np.ascontiguousarray(x) for row in buckets_per_rank for x in row]
    flat_t = [x for row in tensors for x in row]
    lib().orc_bucket_unpack(n, t, plan.numels.ctypes.data, plan.esize,
                            plan.tensor_bucket.ctypes.data,
                            plan.tensor_offset.ctypes.data, _ptrs(flat_b),
                            _ptrs(flat_t))
    return tensors


def bucketed_all_reduce(plan: BucketPlan, tensors_per_rank, dtype, op="avg"):
    """DDP bucket pipeline: pack, ring all-reduce of each bucket, unpack."""
    buckets = bucket_pack(plan, tensors_per_rank)
    n = len(tensors_per_rank)
    for b in range(plan.nbuckets):
        out, _ = ring_all_reduce([buckets[r][b] for r in range(n)], dtype, op)
        for r in range(n):
            buckets[r][b] = out[r]
    return bucket_unpack(plan, buckets, _NP[dtype])


# ---- communication accounting -----------------------------------------------

def alpha_beta_ring_allreduce(n: int, nbytes: float, alpha_s: float,
                              bw_bytes_per_s: float) -> float:
    return lib().orc_alpha_beta_ring_allreduce(n, nbytes, alpha_s,
                                               bw_bytes_per_s)

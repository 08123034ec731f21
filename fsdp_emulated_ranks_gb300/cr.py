"""ctypes binding of libcr (include/cr.h): argument marshalling only.

Every function here has the name of the C entry point it calls and does
nothing but turn Python arguments (torch tensors or integer device
pointers, dtype names, a stream) into the C call and raise on a non-OK
status.  All computation happens in libcr's CUDA kernels; there is no
fallback: if libcr.so is missing, the first call raises.
"""
from __future__ import annotations

import ctypes as C
import os
import struct
import threading
from typing import Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "_build", "libcr.so")
# CR_LIBRARY=<path> loads another build of the library (the tests' checked
# variant, with device-side index checks).
LIB_PATH = os.environ.get("CR_LIBRARY", LIB_PATH)
MAX_RANKS = 64

F32, BF16, I32 = 0, 1, 2
SUM, AVG = 0, 1
COLL_REDUCE_SCATTER, COLL_ALL_GATHER, COLL_ALL_REDUCE = 0, 1, 2
SCHED_RING, SCHED_NAIVE = 0, 1

_DTYPES = {"f32": F32, "float32": F32, "bf16": BF16, "bfloat16": BF16,
           "i32": I32, "int32": I32}
_OPS = {"sum": SUM, "avg": AVG}
STATUS = {0: "CR_OK", 1: "CR_ERR_INVALID_ARG", 2: "CR_ERR_UNSUPPORTED",
          3: "CR_ERR_ALIGNMENT", 4: "CR_ERR_CUDA", 5: "CR_ERR_TIMEOUT"}

# Every symbol include/cr.h declares.
EXPORTS = ["cr_status_string", "cr_last_error", "cr_version", "cr_chunk_len",
           "cr_shard_range", "cr_reduce_scatter", "cr_all_gather",
           "cr_all_reduce", "cr_all_reduce_host", "cr_all_reduce_staged", "cr_bucket_plan", "cr_bucket_plan_free",
           "cr_bucket_pack", "cr_bucket_unpack", "cr_bucket_all_reduce",
           "cr_bucket_all_reduce_fused", "cr_fsdp_step",
           "cr_fsdp_clip_workspace_bytes", "cr_fsdp_step_clipped",
           "cr_fsdp_step_clipped_noalloc", "cr_fsdp2_step", "cr_fsdp2_plan_create",
           "cr_fsdp2_plan_table_bytes", "cr_fsdp2_plan_upload", "cr_fsdp2_step_planned",
           "cr_fsdp2_plan_free", "cr_slab_range", "cr_all_reduce_range",
           "cr_reduce_scatter_range", "cr_fsdp_step_range", "cr_accumulate",
           "cr_all_reduce_accumulate", "cr_adamw_step", "cr_comm_elems",
           "cr_reduce_scatter_wire", "cr_all_reduce_wire",
           "cr_hsdp_reduce_scatter", "cr_reducer_create", "cr_reducer_mark_ready",
           "cr_reducer_launched", "cr_reducer_finalize", "cr_reducer_destroy",
           "cr_comm_create", "cr_comm_all_reduce", "cr_comm_reduce_scatter",
           "cr_comm_all_gather", "cr_comm_broken", "cr_comm_destroy",
           "cr_check_word", "cr_check_selftest"]

_lib = None


class CRError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        super().__init__(f"{where}: {STATUS.get(status, status)}: {detail}")
        self.status = status


class AdamWCfg(C.Structure):
    _fields_ = [("lr", C.c_double), ("beta1", C.c_double),
                ("beta2", C.c_double), ("eps", C.c_double),
                ("weight_decay", C.c_double), ("step", C.c_int64)]


class ParamShape(C.Structure):
    _fields_ = [("dim0", C.c_size_t), ("row_numel", C.c_size_t)]


class BucketPlanT(C.Structure):
    _fields_ = [("ntensors", C.c_int), ("nbuckets", C.c_int),
                ("elem_size", C.c_size_t), ("cap_bytes", C.c_size_t),
                ("numels", C.POINTER(C.c_size_t)),
                ("tensor_bucket", C.POINTER(C.c_int)),
                ("tensor_offset", C.POINTER(C.c_size_t)),
                ("bucket_numel", C.POINTER(C.c_size_t))]


_tls = threading.local()  # .recorder: set while prepare() runs a wrapper
_recording = 0            # threads inside prepare(); lib() skips _tls while 0
_recording_lock = threading.Lock()


def lib() -> C.CDLL:
    """Open libcr.so (built by fsdp_emulated_ranks_gb300.build)."""
    global _lib
    if _recording:
        rec = getattr(_tls, "recorder", None)
        if rec is not None:
            return rec
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"libcr.so not found at {LIB_PATH}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = C.CDLL(LIB_PATH)
    vp, sz, i = C.c_void_p, C.c_size_t, C.c_int
    L.cr_reducer_destroy.restype = None
    L.cr_comm_destroy.restype = None
    L.cr_status_string.restype = C.c_char_p
    L.cr_status_string.argtypes = [i]
    L.cr_last_error.restype = C.c_char_p
    L.cr_last_error.argtypes = []
    L.cr_version.restype = i
    L.cr_chunk_len.restype = sz
    L.cr_chunk_len.argtypes = [sz, i]
    L.cr_shard_range.argtypes = [sz, i, i, C.POINTER(sz), C.POINTER(sz)]
    L.cr_reduce_scatter.argtypes = [vp, i, sz, i, i, vp, i, vp]
    L.cr_all_gather.argtypes = [vp, i, sz, i, vp, vp]
    L.cr_all_reduce.argtypes = [vp, i, sz, i, i, vp, i, vp]
    L.cr_reduce_scatter_wire.argtypes = [vp, i, sz, i, i, i, vp, i, vp]
    L.cr_all_reduce_wire.argtypes = [vp, i, sz, i, i, i, vp, i, vp]
    L.cr_hsdp_reduce_scatter.argtypes = [vp, i, i, sz, i, i, vp, i, vp]
    L.cr_reducer_create.argtypes = [C.POINTER(BucketPlanT), i, vp, i, i, i, vp,
                                    C.POINTER(vp)]
    L.cr_reducer_mark_ready.argtypes = [vp, i, vp]
    L.cr_reducer_launched.argtypes = [vp]
    L.cr_reducer_launched.restype = i
    L.cr_reducer_finalize.argtypes = [vp, vp]
    L.cr_reducer_destroy.argtypes = [vp]
    L.cr_comm_create.argtypes = [i, i, vp, C.POINTER(vp)]
    L.cr_comm_all_reduce.argtypes = [vp, i, vp, sz, i, i]
    L.cr_comm_reduce_scatter.argtypes = [vp, i, vp, vp, sz, i, i, i]
    L.cr_comm_all_gather.argtypes = [vp, i, vp, vp, sz, i]
    L.cr_comm_broken.argtypes = [vp]
    L.cr_comm_destroy.argtypes = [vp]
    L.cr_check_word.argtypes = [i]
    L.cr_check_word.restype = C.c_longlong
    L.cr_check_selftest.argtypes = [vp]
    L.cr_all_reduce_host.argtypes = [vp, vp, vp, i, sz, i, i, vp]
    L.cr_all_reduce_staged.argtypes = [vp, vp, vp, i, sz, i, i, sz, vp, vp, vp]
    L.cr_bucket_plan.argtypes = [vp, i, sz, sz, C.POINTER(C.POINTER(BucketPlanT))]
    L.cr_bucket_plan_free.restype = None
    L.cr_bucket_plan_free.argtypes = [C.POINTER(BucketPlanT)]
    L.cr_bucket_pack.argtypes = [C.POINTER(BucketPlanT), i, vp, vp, vp]
    L.cr_bucket_unpack.argtypes = [C.POINTER(BucketPlanT), i, vp, vp, vp]
    L.cr_bucket_all_reduce.argtypes = [C.POINTER(BucketPlanT), i, vp, i, i, vp]
    L.cr_bucket_all_reduce_fused.argtypes = [C.POINTER(BucketPlanT), i, vp, i, i, vp]
    L.cr_fsdp_step.argtypes = [vp, i, sz, vp, vp, vp, C.POINTER(AdamWCfg), vp, vp]
    L.cr_fsdp_clip_workspace_bytes.restype = sz
    L.cr_fsdp_clip_workspace_bytes.argtypes = []
    L.cr_fsdp_step_clipped.argtypes = [vp, i, sz, vp, vp, vp, C.POINTER(AdamWCfg), C.c_double,
                                       vp, sz, vp, vp, vp]
    L.cr_fsdp_step_clipped_noalloc.argtypes = [vp, i, sz, vp, vp, vp, C.POINTER(AdamWCfg),
                                               C.c_double, vp, vp, vp]
    L.cr_fsdp2_step.argtypes = [vp, i, i, vp, vp, vp, vp, C.POINTER(AdamWCfg), vp, vp]
    L.cr_fsdp2_plan_create.argtypes = [vp, i, i, vp, vp, vp, vp, vp, C.POINTER(vp)]
    L.cr_fsdp2_plan_table_bytes.restype = sz
    L.cr_fsdp2_plan_table_bytes.argtypes = [vp]
    L.cr_fsdp2_plan_upload.argtypes = [vp, vp, sz, vp]
    L.cr_fsdp2_step_planned.argtypes = [vp, vp, C.POINTER(AdamWCfg), vp]
    L.cr_fsdp2_plan_free.restype = None
    L.cr_fsdp2_plan_free.argtypes = [vp]
    L.cr_slab_range.argtypes = [sz, i, i, i, C.POINTER(sz), C.POINTER(sz)]
    L.cr_all_reduce_range.argtypes = [vp, i, sz, sz, sz, i, i, vp, i, vp]
    L.cr_reduce_scatter_range.argtypes = [vp, i, sz, sz, sz, i, i, vp, i, vp]
    L.cr_fsdp_step_range.argtypes = [vp, i, sz, sz, sz, vp, vp, vp, C.POINTER(AdamWCfg), vp, vp]
    L.cr_accumulate.argtypes = [vp, i, sz, vp, i, vp]
    L.cr_all_reduce_accumulate.argtypes = [vp, i, sz, vp, i, i, vp]
    L.cr_adamw_step.argtypes = [sz, vp, vp, vp, vp, C.POINTER(AdamWCfg), vp, vp]
    L.cr_comm_elems.argtypes = [i, i, i, sz, i, C.POINTER(C.c_uint64),
                                C.POINTER(C.c_uint64), C.POINTER(i)]
    for name in EXPORTS:
        getattr(L, name).restype = getattr(L, name).restype or i
    L.cr_status_string.restype = C.c_char_p
    L.cr_last_error.restype = C.c_char_p
    L.cr_chunk_len.restype = sz
    L.cr_bucket_plan_free.restype = None
    L.cr_fsdp_clip_workspace_bytes.restype = sz
    L.cr_fsdp2_plan_table_bytes.restype = sz
    L.cr_fsdp2_plan_free.restype = None
    _lib = L
    return L


# ---- marshalling helpers --------------------------------------------------------

def _ptr(x) -> int:
    if x is None:
        return 0
    if isinstance(x, int):
        return x
    return x.data_ptr()


_PACK = {}  # length -> struct packer of that many native 64-bit pointers


def _ptr_array(xs: Sequence):
    """Host array of device pointers for a call, as a bytes object of native
    64-bit words: ctypes passes a bytes argument to a void* parameter as the
    address of its buffer, which lives until the call returns (the library
    copies the table before returning).  Packing with struct is about three
    times faster than filling a ctypes array element by element, which
    matters for short calls whose host cost is the call itself.  An empty
    list still yields a valid (one zero entry) table."""
    ptrs = [x if type(x) is int else (0 if x is None else x.data_ptr()) for x in xs]
    n = len(ptrs)
    if n == 0:
        ptrs, n = [0], 1
    pack = _PACK.get(n)
    if pack is None:
        pack = struct.Struct(f"={n}Q").pack
        if len(_PACK) < 256:  # a bounded cache: callers use few table lengths
            _PACK[n] = pack
    return pack(*ptrs)


def _dtype(d) -> int:
    if isinstance(d, int):
        return d
    k = _DTYPES.get(d)
    return k if k is not None else _DTYPES[str(d).replace("torch.", "")]


def _op(o) -> int:
    return o if isinstance(o, int) else _OPS[o]


_torch = None
_raw_stream = None  # torch's C-level current-stream query, when it has one


def _current_stream() -> int:
    """Handle of torch's current CUDA stream on the current device."""
    global _torch, _raw_stream
    if _torch is None:
        import torch
        _torch = torch
        get_raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
        get_dev = getattr(torch._C, "_cuda_getDevice", None)
        if get_raw is not None and get_dev is not None:
            _raw_stream = lambda: get_raw(get_dev())
    if _raw_stream is not None:
        return _raw_stream()
    return _torch.cuda.current_stream().cuda_stream


def _stream(stream) -> int:
    if stream is None:
        return _current_stream()
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(status: int, where: str) -> None:
    if status != 0:
        raise CRError(status, where, lib().cr_last_error().decode())


# ---- entry points -----------------------------------------------------------------

def cr_version() -> int:
    return lib().cr_version()


def cr_chunk_len(count: int, nranks: int) -> int:
    return lib().cr_chunk_len(count, nranks)


def cr_shard_range(count: int, nranks: int, j: int) -> tuple[int, int]:
    lo, hi = C.c_size_t(), C.c_size_t()
    _check(lib().cr_shard_range(count, nranks, j, C.byref(lo), C.byref(hi)),
           "cr_shard_range")
    return lo.value, hi.value


def cr_reduce_scatter(bufs, count, in_dtype, op, out_shards, out_dtype,
                      stream=None) -> None:
    _check(lib().cr_reduce_scatter(_ptr_array(bufs), len(bufs), count,
                                   _dtype(in_dtype), _op(op),
                                   _ptr_array(out_shards), _dtype(out_dtype),
                                   _stream(stream)), "cr_reduce_scatter")


def cr_all_gather(shards, count, dtype, bufs, stream=None) -> None:
    _check(lib().cr_all_gather(_ptr_array(shards), len(shards), count,
                               _dtype(dtype), _ptr_array(bufs),
                               _stream(stream)), "cr_all_gather")


def cr_all_reduce(inbufs, count, in_dtype, op, outbufs, out_dtype,
                  stream=None) -> None:
    _check(lib().cr_all_reduce(_ptr_array(inbufs), len(inbufs), count,
                               _dtype(in_dtype), _op(op), _ptr_array(outbufs),
                               _dtype(out_dtype), _stream(stream)),
           "cr_all_reduce")


def cr_reduce_scatter_wire(bufs, count, in_dtype, op, wire_dtype, out_shards, out_dtype,
                           stream=None) -> None:
    _check(lib().cr_reduce_scatter_wire(_ptr_array(bufs), len(bufs), count,
                                        _dtype(in_dtype), _op(op), _dtype(wire_dtype),
                                        _ptr_array(out_shards), _dtype(out_dtype),
                                        _stream(stream)), "cr_reduce_scatter_wire")


def cr_all_reduce_wire(inbufs, count, in_dtype, op, wire_dtype, outbufs, out_dtype,
                       stream=None) -> None:
    _check(lib().cr_all_reduce_wire(_ptr_array(inbufs), len(inbufs), count,
                                    _dtype(in_dtype), _op(op), _dtype(wire_dtype),
                                    _ptr_array(outbufs), _dtype(out_dtype),
                                    _stream(stream)), "cr_all_reduce_wire")


def cr_hsdp_reduce_scatter(bufs, R, S, count, in_dtype, op, out_shards, out_dtype,
                           stream=None) -> None:
    """bufs[g*S + s]: rank (g, s)'s buffer; out_shards[g*S + j]: shard j of group g."""
    _check(lib().cr_hsdp_reduce_scatter(_ptr_array(bufs), R, S, count, _dtype(in_dtype),
                                        _op(op), _ptr_array(out_shards), _dtype(out_dtype),
                                        _stream(stream)), "cr_hsdp_reduce_scatter")


def cr_all_reduce_host(host_in, host_out, count, dtype, op, dev_out=None, stream=None) -> None:
    _check(lib().cr_all_reduce_host(_ptr_array(host_in), _ptr_array(host_out),
                                    _ptr_array(dev_out) if dev_out is not None else None,
                                    len(host_in), count, _dtype(dtype), _op(op), _stream(stream)),
           "cr_all_reduce_host")


def cr_all_reduce_staged(host_in, host_out, dev_bufs, count, dtype, op,
                         slice_elems=0, compute_stream=None, h2d_stream=None,
                         d2h_stream=None) -> None:
    sc = _stream(compute_stream)
    sh = sc if h2d_stream is None else _stream(h2d_stream)
    sd = sc if d2h_stream is None else _stream(d2h_stream)
    _check(lib().cr_all_reduce_staged(_ptr_array(host_in), _ptr_array(host_out),
                                      _ptr_array(dev_bufs), len(dev_bufs), count,
                                      _dtype(dtype), _op(op), slice_elems, sc, sh, sd),
           "cr_all_reduce_staged")


class BucketPlan:
    """Owns a cr_bucket_plan_t; freed with cr_bucket_plan_free."""

    def __init__(self, ptr):
        self._ptr = ptr
        p = ptr.contents
        self.ntensors = p.ntensors
        self.nbuckets = p.nbuckets
        self.elem_size = p.elem_size
        self.tensor_bucket = [p.tensor_bucket[t] for t in range(p.ntensors)]
        self.tensor_offset = [p.tensor_offset[t] for t in range(p.ntensors)]
        self.bucket_numel = [p.bucket_numel[b] for b in range(p.nbuckets)]
        self.numels = [p.numels[t] for t in range(p.ntensors)]

    @property
    def ptr(self):
        return self._ptr

    def __del__(self):
        if getattr(self, "_ptr", None) is not None and _lib is not None:
            _lib.cr_bucket_plan_free(self._ptr)
            self._ptr = None


def cr_bucket_plan(numels: Sequence[int], elem_size: int, cap_bytes: int) -> BucketPlan:
    arr = (C.c_size_t * max(1, len(numels)))(*[int(k) for k in numels])
    out = C.POINTER(BucketPlanT)()
    _check(lib().cr_bucket_plan(arr, len(numels), elem_size, cap_bytes,
                                C.byref(out)), "cr_bucket_plan")
    return BucketPlan(out)


def cr_bucket_pack(plan: BucketPlan, nranks: int, tensors, buckets,
                   stream=None) -> None:
    _check(lib().cr_bucket_pack(plan.ptr, nranks, _ptr_array(tensors),
                                _ptr_array(buckets), _stream(stream)),
           "cr_bucket_pack")


def cr_bucket_unpack(plan: BucketPlan, nranks: int, buckets, tensors,
                     stream=None) -> None:
    _check(lib().cr_bucket_unpack(plan.ptr, nranks, _ptr_array(buckets),
                                  _ptr_array(tensors), _stream(stream)),
           "cr_bucket_unpack")


def cr_bucket_all_reduce(plan: BucketPlan, nranks: int, buckets, dtype, op,
                         stream=None) -> None:
    _check(lib().cr_bucket_all_reduce(plan.ptr, nranks, _ptr_array(buckets),
                                      _dtype(dtype), _op(op), _stream(stream)),
           "cr_bucket_all_reduce")


def cr_bucket_all_reduce_fused(plan: BucketPlan, nranks: int, tensors, dtype, op,
                               stream=None) -> None:
    _check(lib().cr_bucket_all_reduce_fused(plan.ptr, nranks, _ptr_array(tensors),
                                            _dtype(dtype), _op(op), _stream(stream)),
           "cr_bucket_all_reduce_fused")


class Reducer:
    """Owns a cr_reducer_t, the DDP reducer (bucket all-reduces started as
    gradients become ready); released by cr_reducer_destroy or when
    collected."""

    def __init__(self, ptr: int):
        self._ptr = ptr

    @property
    def ptr(self):
        return self._ptr

    def __del__(self):
        if getattr(self, "_ptr", None) and _lib is not None:
            _lib.cr_reducer_destroy(self._ptr)
            self._ptr = None


def cr_reducer_create(plan: BucketPlan, nranks: int, tensors, dtype, op, comm_ctas=0,
                      comm_stream=None) -> Reducer:
    """tensors[r*T + t]: rank r's tensor t."""
    out = C.c_void_p()
    _check(lib().cr_reducer_create(plan.ptr, nranks, _ptr_array(tensors), _dtype(dtype),
                                   _op(op), comm_ctas, _stream(comm_stream), C.byref(out)),
           "cr_reducer_create")
    return Reducer(out.value)


def cr_reducer_mark_ready(red: Reducer, tensor: int, compute_stream=None) -> None:
    _check(lib().cr_reducer_mark_ready(red.ptr, tensor, _stream(compute_stream)),
           "cr_reducer_mark_ready")


def cr_reducer_launched(red: Reducer) -> int:
    return lib().cr_reducer_launched(red.ptr)


def cr_reducer_finalize(red: Reducer, compute_stream=None) -> None:
    _check(lib().cr_reducer_finalize(red.ptr, _stream(compute_stream)), "cr_reducer_finalize")


def cr_reducer_destroy(red: Reducer) -> None:
    if red.ptr:
        lib().cr_reducer_destroy(red.ptr)
        red._ptr = None


class Comm:
    """Owns a cr_comm_t: N emulated ranks, one host thread each (ctypes
    releases the GIL during the blocking calls)."""

    def __init__(self, ptr: int):
        self._ptr = ptr

    @property
    def ptr(self):
        return self._ptr

    def __del__(self):
        if getattr(self, "_ptr", None) and _lib is not None:
            _lib.cr_comm_destroy(self._ptr)
            self._ptr = None


def cr_comm_create(nranks: int, timeout_ms: int, stream=None) -> Comm:
    out = C.c_void_p()
    _check(lib().cr_comm_create(nranks, timeout_ms, _stream(stream), C.byref(out)),
           "cr_comm_create")
    return Comm(out.value)


def cr_comm_all_reduce(comm: Comm, rank: int, buf, count, dtype, op) -> None:
    _check(lib().cr_comm_all_reduce(comm.ptr, rank, _ptr(buf), count, _dtype(dtype), _op(op)),
           "cr_comm_all_reduce")


def cr_comm_reduce_scatter(comm: Comm, rank: int, buf, shard, count, in_dtype, op,
                           out_dtype) -> None:
    _check(lib().cr_comm_reduce_scatter(comm.ptr, rank, _ptr(buf), _ptr(shard), count,
                                        _dtype(in_dtype), _op(op), _dtype(out_dtype)),
           "cr_comm_reduce_scatter")


def cr_comm_all_gather(comm: Comm, rank: int, shard, buf, count, dtype) -> None:
    _check(lib().cr_comm_all_gather(comm.ptr, rank, _ptr(shard), _ptr(buf), count,
                                    _dtype(dtype)), "cr_comm_all_gather")


def cr_comm_broken(comm: Comm) -> int:
    return lib().cr_comm_broken(comm.ptr)


def cr_comm_destroy(comm: Comm) -> None:
    if comm.ptr:
        lib().cr_comm_destroy(comm.ptr)
        comm._ptr = None


def cr_check_word(clear: bool = False) -> int:
    """Device error word of the checked build (-1: the loaded library was
    built without device checks; -2: reading it failed)."""
    return lib().cr_check_word(1 if clear else 0)


def cr_check_selftest(stream=None) -> None:
    _check(lib().cr_check_selftest(_stream(stream)), "cr_check_selftest")


def adamw_cfg(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01,
              step=1) -> AdamWCfg:
    return AdamWCfg(lr, beta1, beta2, eps, weight_decay, step)


def cr_fsdp_step(grads, count, master, m, v, cfg: AdamWCfg, params,
                 stream=None) -> None:
    _check(lib().cr_fsdp_step(_ptr_array(grads), len(grads), count,
                              _ptr_array(master), _ptr_array(m), _ptr_array(v),
                              C.byref(cfg), _ptr_array(params), _stream(stream)),
           "cr_fsdp_step")


def cr_fsdp_clip_workspace_bytes() -> int:
    return lib().cr_fsdp_clip_workspace_bytes()


def cr_fsdp_step_clipped(grads, count, master, m, v, cfg: AdamWCfg, max_norm, workspace,
                         workspace_bytes, params, norm_out=None, stream=None) -> None:
    _check(lib().cr_fsdp_step_clipped(_ptr_array(grads), len(grads), count,
                                      _ptr_array(master), _ptr_array(m), _ptr_array(v),
                                      C.byref(cfg), float(max_norm), _ptr(workspace),
                                      workspace_bytes, _ptr_array(params), _ptr(norm_out),
                                      _stream(stream)), "cr_fsdp_step_clipped")


def cr_fsdp_step_clipped_noalloc(grads, count, master, m, v, cfg: AdamWCfg, max_norm, params,
                                 norm_out=None, stream=None) -> None:
    """cr_fsdp_step_clipped with the library's static scratch instead of a
    caller workspace, for callers that cannot allocate device memory."""
    _check(lib().cr_fsdp_step_clipped_noalloc(_ptr_array(grads), len(grads), count,
                                              _ptr_array(master), _ptr_array(m), _ptr_array(v),
                                              C.byref(cfg), float(max_norm), _ptr_array(params),
                                              _ptr(norm_out), _stream(stream)),
           "cr_fsdp_step_clipped_noalloc")


def cr_fsdp2_step(shapes, nranks, grads, master, m, v, cfg: AdamWCfg, params,
                  stream=None) -> None:
    """shapes: [(dim0, row_numel)]; the pointer lists are flat, index p*N + r."""
    arr = (ParamShape * max(1, len(shapes)))(*[ParamShape(d, rn) for d, rn in shapes])
    _check(lib().cr_fsdp2_step(arr, len(shapes), nranks, _ptr_array(grads), _ptr_array(master),
                               _ptr_array(m), _ptr_array(v), C.byref(cfg), _ptr_array(params),
                               _stream(stream)), "cr_fsdp2_step")


def cr_slab_range(count: int, nranks: int, nslabs: int, g: int) -> tuple[int, int]:
    lo, hi = C.c_size_t(), C.c_size_t()
    _check(lib().cr_slab_range(count, nranks, nslabs, g, C.byref(lo), C.byref(hi)),
           "cr_slab_range")
    return lo.value, hi.value


def cr_all_reduce_range(inp, count, begin, end, in_dtype, op, out, out_dtype,
                        stream=None) -> None:
    """inp/out: per-rank slab buffers (element `begin` first)."""
    _check(lib().cr_all_reduce_range(_ptr_array(inp), len(inp), count, begin, end,
                                     _dtype(in_dtype), _op(op), _ptr_array(out),
                                     _dtype(out_dtype), _stream(stream)), "cr_all_reduce_range")


def cr_reduce_scatter_range(bufs, count, begin, end, in_dtype, op, out_shards, out_dtype,
                            stream=None) -> None:
    """out_shards[j]: shard j's part inside [begin, end) (or 0 if none)."""
    _check(lib().cr_reduce_scatter_range(_ptr_array(bufs), len(bufs), count, begin, end,
                                         _dtype(in_dtype), _op(op), _ptr_array(out_shards),
                                         _dtype(out_dtype), _stream(stream)),
           "cr_reduce_scatter_range")


def cr_fsdp_step_range(grads, count, begin, end, master, m, v, cfg: AdamWCfg, params,
                       stream=None) -> None:
    _check(lib().cr_fsdp_step_range(_ptr_array(grads), len(grads), count, begin, end,
                                    _ptr_array(master), _ptr_array(m), _ptr_array(v),
                                    C.byref(cfg), _ptr_array(params), _stream(stream)),
           "cr_fsdp_step_range")


class Fsdp2Plan:
    """Owns a cr_fsdp2_plan_t; freed with cr_fsdp2_plan_free."""

    def __init__(self, ptr: int):
        self._ptr = ptr
        self.table_bytes = int(lib().cr_fsdp2_plan_table_bytes(ptr))

    @property
    def ptr(self):
        return self._ptr

    def __del__(self):
        if getattr(self, "_ptr", None) and _lib is not None:
            _lib.cr_fsdp2_plan_free(self._ptr)
            self._ptr = None


def cr_fsdp2_plan_create(shapes, nranks, grads, master, m, v, params) -> Fsdp2Plan:
    """shapes: [(dim0, row_numel)]; the pointer lists are flat, index p*N + r."""
    arr = (ParamShape * max(1, len(shapes)))(*[ParamShape(d, rn) for d, rn in shapes])
    out = C.c_void_p()
    _check(lib().cr_fsdp2_plan_create(arr, len(shapes), nranks, _ptr_array(grads),
                                      _ptr_array(master), _ptr_array(m), _ptr_array(v),
                                      _ptr_array(params), C.byref(out)), "cr_fsdp2_plan_create")
    return Fsdp2Plan(out.value)


def cr_fsdp2_plan_table_bytes(plan: Fsdp2Plan) -> int:
    return int(lib().cr_fsdp2_plan_table_bytes(plan.ptr if plan is not None else None))


def cr_fsdp2_plan_upload(plan: Fsdp2Plan, table, table_bytes=None, stream=None) -> None:
    """table: a device tensor or pointer of at least plan.table_bytes bytes."""
    nbytes = table_bytes if table_bytes is not None else table.numel() * table.element_size()
    _check(lib().cr_fsdp2_plan_upload(plan.ptr, _ptr(table), nbytes, _stream(stream)),
           "cr_fsdp2_plan_upload")


def cr_fsdp2_step_planned(plan: Fsdp2Plan, table, cfg: AdamWCfg, stream=None) -> None:
    _check(lib().cr_fsdp2_step_planned(plan.ptr if plan is not None else None, _ptr(table),
                                       C.byref(cfg), _stream(stream)), "cr_fsdp2_step_planned")


def cr_accumulate(acc, count, grads, grad_dtype, stream=None) -> None:
    _check(lib().cr_accumulate(_ptr_array(acc), len(acc), count, _ptr_array(grads),
                               _dtype(grad_dtype), _stream(stream)), "cr_accumulate")


def cr_all_reduce_accumulate(acc, count, grads, grad_dtype, op, stream=None) -> None:
    _check(lib().cr_all_reduce_accumulate(_ptr_array(acc), len(acc), count, _ptr_array(grads),
                                          _dtype(grad_dtype), _op(op), _stream(stream)),
           "cr_all_reduce_accumulate")


def cr_adamw_step(n, master, m, v, grad, cfg: AdamWCfg, param_bf16=None,
                  stream=None) -> None:
    _check(lib().cr_adamw_step(n, _ptr(master), _ptr(m), _ptr(v), _ptr(grad),
                               C.byref(cfg), _ptr(param_bf16), _stream(stream)),
           "cr_adamw_step")


def cr_comm_elems(coll: int, sched: int, nranks: int, count: int,
                  rank: int) -> tuple[int, int, int]:
    sent, recv, steps = C.c_uint64(), C.c_uint64(), C.c_int()
    _check(lib().cr_comm_elems(coll, sched, nranks, count, rank, C.byref(sent),
                               C.byref(recv), C.byref(steps)), "cr_comm_elems")
    return sent.value, recv.value, steps.value


# ---- prepared calls -----------------------------------------------------------------

# Entry points that launch work on a stream: the ones prepare() can record.
_PREPARABLE = frozenset([
    "cr_reduce_scatter", "cr_all_gather", "cr_all_reduce", "cr_reduce_scatter_wire",
    "cr_all_reduce_wire", "cr_hsdp_reduce_scatter", "cr_all_reduce_host",
    "cr_all_reduce_staged", "cr_bucket_pack", "cr_bucket_unpack", "cr_bucket_all_reduce",
    "cr_bucket_all_reduce_fused", "cr_fsdp_step", "cr_fsdp_step_clipped",
    "cr_fsdp_step_clipped_noalloc", "cr_fsdp2_step", "cr_fsdp2_plan_upload",
    "cr_fsdp2_step_planned", "cr_all_reduce_range", "cr_reduce_scatter_range",
    "cr_fsdp_step_range", "cr_accumulate", "cr_all_reduce_accumulate", "cr_adamw_step"])
# Functions without side effects that a wrapper may call while it marshals.
_PURE = frozenset(["cr_last_error", "cr_status_string", "cr_chunk_len", "cr_version",
                   "cr_fsdp_clip_workspace_bytes", "cr_shard_range", "cr_slab_range",
                   "cr_comm_elems", "cr_fsdp2_plan_table_bytes"])


class _Recorder:
    """Stands in for the library while prepare() runs a wrapper: a launching
    entry point is recorded with its marshalled arguments instead of being
    called, the pure helpers are the library's, and anything else (a call
    with side effects that prepare() must not make) raises."""

    def __init__(self, real):
        self._real = real
        self.calls = []

    def __getattr__(self, name):
        fn = getattr(self._real, name)
        if name in _PURE:
            return fn
        if name not in _PREPARABLE:
            raise TypeError(f"prepare() records launching entry points only, not {name}")

        def record(*args):
            self.calls.append((name, fn, args))
            return 0
        return record


class Prepared:
    """One marshalled call of a launching entry point; see prepare()."""

    __slots__ = ("name", "_calls", "_keep")

    def __init__(self, name, calls, keep):
        # keep: the wrapper's arguments, so that the tensors and the bucket
        # plan whose addresses were recorded outlive the prepared call
        self.name, self._calls, self._keep = name, calls, keep

    def __call__(self) -> None:
        for name, fn, args in self._calls:
            status = fn(*args)
            if status != 0:
                _check(status, name)


def prepare(wrapper, *args, **kwargs) -> Prepared:
    """Marshal one call of a launching wrapper (cr_all_reduce, cr_fsdp_step,
    ...) once and return a callable that issues the same C call again: the
    same device pointers, sizes, dtypes and stream, with none of the Python
    argument conversion per invocation.  Meant for loops that repeat a call
    on fixed buffers (a training step on static gradient buffers, a latency
    measurement).

    The stream is fixed at preparation: the one given, else the current
    stream then.  The library validates every invocation as it does a
    direct call.  A cr_adamw_cfg is passed by reference and read at each
    invocation, so advancing cfg.step between invocations takes effect.
    The prepared call holds references to the arguments, so the tensors and
    the bucket plan it addresses stay allocated while it exists."""
    global _recording
    if getattr(_tls, "recorder", None) is not None:
        raise RuntimeError("prepare() cannot be nested")
    rec = _Recorder(lib())
    with _recording_lock:
        _recording += 1
    _tls.recorder = rec
    try:
        wrapper(*args, **kwargs)
    finally:
        _tls.recorder = None
        with _recording_lock:
            _recording -= 1
    name = getattr(wrapper, "__name__", "call")
    if not rec.calls:
        raise ValueError(f"{name} launches nothing that prepare() could record")
    return Prepared(name, rec.calls, (args, kwargs))

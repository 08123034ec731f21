// api.cu -- the extern "C" entry points of libcr (include/cr.h): argument
// validation on the host, then one launch per call (bucket copies: one per
// 1024 ranges; bucket all-reduce: one per bucket).
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "cr_internal.cuh"

using namespace cr;

namespace {

thread_local char g_err[512] = "";

cr_status fail(cr_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

cr_status ok() {
  g_err[0] = '\0';
  return CR_OK;
}

cr_status cuda_fail(cudaError_t e, const char* what) {
  return fail(CR_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e),
              cudaGetErrorString(e));
}

size_t esize_of(cr_dtype d) {
  switch (d) {
    case CR_F32: return 4;
    case CR_BF16: return 2;
    case CR_I32: return 4;
  }
  return 0;
}

bool is_float(cr_dtype d) { return d == CR_F32 || d == CR_BF16; }

// Byte interval of one buffer argument.
struct Span {
  uintptr_t a, b;  // [a, b)
  int kind;        // 0 input, 1 output
  int rank;
};

bool overlaps(const Span& x, const Span& y) {
  return x.a < y.b && y.a < x.b && x.a < x.b && y.a < y.b;
}

uint64_t chunk_lo(uint64_t count, uint64_t L, int j) {
  uint64_t a = L * (uint64_t)j;
  return a < count ? a : count;
}

uint64_t chunk_size(uint64_t count, uint64_t L, int j) {
  uint64_t a = chunk_lo(count, L, j);
  uint64_t b = L * (uint64_t)(j + 1);
  if (b > count) b = count;
  return b - a;
}

bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Rejects ranks out of range and counts whose byte size overflows.
cr_status check_common(int nranks, size_t count, const void* arr1,
                       const void* arr2) {
  if (nranks < 1 || nranks > CR_MAX_RANKS)
    return fail(CR_ERR_INVALID_ARG, "nranks=%d outside [1, %d]", nranks, CR_MAX_RANKS);
  if (!arr1 || !arr2) return fail(CR_ERR_INVALID_ARG, "pointer array is NULL");
  if (count > (SIZE_MAX / 8)) return fail(CR_ERR_INVALID_ARG, "count=%zu too large", count);
  return CR_OK;
}

cr_status check_pair(cr_dtype in, cr_op op, cr_dtype out) {
  if (esize_of(in) == 0 || esize_of(out) == 0)
    return fail(CR_ERR_INVALID_ARG, "unknown dtype (%d, %d)", (int)in, (int)out);
  if (op != CR_SUM && op != CR_AVG) return fail(CR_ERR_INVALID_ARG, "unknown op %d", (int)op);
  if (op == CR_AVG && !is_float(in))
    return fail(CR_ERR_UNSUPPORTED, "AVG needs a floating-point dtype");
  const bool supported = (in == CR_F32 && out == CR_F32) || (in == CR_BF16 && out == CR_BF16) ||
                         (in == CR_BF16 && out == CR_F32) || (in == CR_I32 && out == CR_I32);
  if (!supported)
    return fail(CR_ERR_UNSUPPORTED, "dtype pair (%d -> %d) not supported", (int)in, (int)out);
  return CR_OK;
}

// Every buffer: non-NULL if non-empty and aligned to its element size.
cr_status check_buf(const void* p, uint64_t nelem, size_t es, const char* what, int r) {
  if (nelem == 0) return CR_OK;
  if (!p) return fail(CR_ERR_INVALID_ARG, "%s[%d] is NULL", what, r);
  if (!aligned(p, es))
    return fail(CR_ERR_ALIGNMENT, "%s[%d]=%p not aligned to %zu bytes", what, r, p, es);
  return CR_OK;
}

// No output may overlap another buffer, except the pairs allow(i, o) marks.
template <typename Allow>
cr_status check_overlaps(const std::vector<Span>& spans, Allow allow) {
  for (size_t x = 0; x < spans.size(); ++x) {
    if (spans[x].kind != 1) continue;
    for (size_t y = 0; y < spans.size(); ++y) {
      if (x == y || !overlaps(spans[x], spans[y])) continue;
      if (spans[y].kind == 0 && allow(spans[y], spans[x])) continue;
      return fail(CR_ERR_INVALID_ARG, "%s %d overlaps %s %d",
                  "output", spans[x].rank, spans[y].kind ? "output" : "input",
                  spans[y].rank);
    }
  }
  return CR_OK;
}

// Many buffers, none of which may overlap another: sort by start address.
cr_status check_disjoint(std::vector<Span> spans) {
  std::sort(spans.begin(), spans.end(), [](const Span& x, const Span& y) { return x.a < y.a; });
  for (size_t k = 1; k < spans.size(); ++k)
    if (spans[k].a < spans[k - 1].b)
      return fail(CR_ERR_INVALID_ARG, "buffer %d overlaps buffer %d", spans[k].rank,
                  spans[k - 1].rank);
  return CR_OK;
}

Span span_of(const void* p, uint64_t bytes, int kind, int rank) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Span{a, a + bytes, kind, rank};
}

// Widest vector access every buffer of a call allows: 32 or 16 bytes, or
// 0 for the element-wise kernels.
struct Width {
  bool w16 = true, w32 = true;
  void ptr(const void* p) {
    w16 = w16 && aligned(p, 16);
    w32 = w32 && aligned(p, 32);
  }
  void bytes(uint64_t b) {
    w16 = w16 && b % 16 == 0;
    w32 = w32 && b % 32 == 0;
  }
  int get() const { return w32 ? 32 : (w16 ? 16 : 0); }
};

float exact_inv_n(int n) {
  return (n & (n - 1)) == 0 ? 1.0f / (float)n : 0.0f;
}

AdamScalars adam_scalars(const cr_adamw_cfg& c) {
  AdamScalars s;
  s.lr = (float)c.lr;
  s.eps = (float)c.eps;
  s.b1 = (float)c.beta1;
  s.b2 = (float)c.beta2;
  s.omb1 = (float)(1.0 - c.beta1);
  s.omb2 = (float)(1.0 - c.beta2);
  s.decay = (float)(1.0 - c.lr * c.weight_decay);
  s.bc1 = (float)(1.0 - pow(c.beta1, (double)c.step));
  s.bc2 = (float)(1.0 - pow(c.beta2, (double)c.step));
  return s;
}

cr_status check_adam_cfg(const cr_adamw_cfg* cfg) {
  if (!cfg) return fail(CR_ERR_INVALID_ARG, "cfg is NULL");
  if (cfg->step < 1) return fail(CR_ERR_INVALID_ARG, "cfg->step=%lld < 1", (long long)cfg->step);
  if (!(cfg->beta1 >= 0.0 && cfg->beta1 < 1.0) || !(cfg->beta2 >= 0.0 && cfg->beta2 < 1.0))
    return fail(CR_ERR_INVALID_ARG, "betas must lie in [0, 1)");
  if (!(cfg->eps >= 0.0) || !(cfg->lr >= 0.0) || !(cfg->weight_decay >= 0.0))
    return fail(CR_ERR_INVALID_ARG, "lr, eps and weight_decay must be >= 0");
  return CR_OK;
}

// The wire type of a ring whose messages may travel in low precision.
cr_status check_wire(cr_dtype in, cr_dtype wire, bool* bf16) {
  if (wire == CR_F32) {
    *bf16 = false;
    return CR_OK;
  }
  if (wire == CR_BF16) {
    if (!is_float(in)) return fail(CR_ERR_UNSUPPORTED, "a bf16 wire needs a floating-point dtype");
    *bf16 = true;
    return CR_OK;
  }
  return fail(CR_ERR_INVALID_ARG, "wire dtype %d is neither CR_F32 nor CR_BF16", (int)wire);
}

cr_status all_reduce_impl(const void* const* in, int nranks, size_t count,
                          cr_dtype in_dtype, cr_op op, void* const* out,
                          cr_dtype out_dtype, cudaStream_t stream, bool wire_bf16 = false) {
  cr_status st = check_common(nranks, count, in, out);
  if (st) return st;
  if ((st = check_pair(in_dtype, op, out_dtype))) return st;
  const size_t is = esize_of(in_dtype), os = esize_of(out_dtype);
  std::vector<Span> spans;
  Width vw;
  for (int r = 0; r < nranks; ++r) {
    if ((st = check_buf(in[r], count, is, "in", r))) return st;
    if ((st = check_buf(out[r], count, os, "out", r))) return st;
    if (count) {
      spans.push_back(span_of(in[r], count * is, 0, r));
      spans.push_back(span_of(out[r], count * os, 1, r));
      vw.ptr(in[r]);
      vw.ptr(out[r]);
    }
  }
  const bool same = in_dtype == out_dtype;
  st = check_overlaps(spans, [&](const Span& i, const Span& o) {
    return same && i.rank == o.rank && i.a == o.a && i.b == o.b;
  });
  if (st) return st;
  if (count == 0) return ok();
  FoldArgs a;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < nranks; ++r) {
    a.in[r] = in[r];
    a.out[r] = out[r];
  }
  a.count = count;
  a.L = (count + nranks - 1) / nranks;
  a.Ld = fastdiv_make(a.L, count ? count - 1 : 0);
  a.begin = 0;
  a.end = count;
  a.n = nranks;
  a.n_out = nranks;
  a.avg = op == CR_AVG;
  a.inv_n = exact_inv_n(nranks);
  a.wire_bf16 = wire_bf16 ? 1 : 0;
  cudaError_t e = launch_fold(in_dtype, out_dtype, kAR, a, vw.get(), stream);
  if (e != cudaSuccess) return cuda_fail(e, "all_reduce launch");
  return ok();
}

}  // namespace

void cr::report_error(cr_status status, const char* msg) { fail(status, "%s", msg); }

extern "C" {

const char* cr_status_string(cr_status s) {
  switch (s) {
    case CR_OK: return "CR_OK";
    case CR_ERR_INVALID_ARG: return "CR_ERR_INVALID_ARG";
    case CR_ERR_UNSUPPORTED: return "CR_ERR_UNSUPPORTED";
    case CR_ERR_ALIGNMENT: return "CR_ERR_ALIGNMENT";
    case CR_ERR_CUDA: return "CR_ERR_CUDA";
    case CR_ERR_TIMEOUT: return "CR_ERR_TIMEOUT";
  }
  return "CR_ERR_UNKNOWN";
}

const char* cr_last_error(void) { return g_err; }

int cr_version(void) { return 100; }

size_t cr_chunk_len(size_t count, int nranks) {
  if (nranks < 1) return 0;
  return count / (size_t)nranks + (count % (size_t)nranks ? 1 : 0);
}

cr_status cr_shard_range(size_t count, int nranks, int j, size_t* lo, size_t* hi) {
  if (nranks < 1 || nranks > CR_MAX_RANKS)
    return fail(CR_ERR_INVALID_ARG, "nranks=%d outside [1, %d]", nranks, CR_MAX_RANKS);
  if (j < 0 || j >= nranks) return fail(CR_ERR_INVALID_ARG, "j=%d outside [0, %d)", j, nranks);
  if (!lo || !hi) return fail(CR_ERR_INVALID_ARG, "lo/hi is NULL");
  const uint64_t L = cr_chunk_len(count, nranks);
  *lo = chunk_lo(count, L, j);
  *hi = *lo + chunk_size(count, L, j);
  return ok();
}

}  // extern "C"

namespace {

cr_status reduce_scatter_impl(const void* const* bufs, int nranks, size_t count,
                              cr_dtype in_dtype, cr_op op, void* const* out_shards,
                              cr_dtype out_dtype, cudaStream_t stream, bool wire_bf16) {
  cr_status st = check_common(nranks, count, bufs, out_shards);
  if (st) return st;
  if ((st = check_pair(in_dtype, op, out_dtype))) return st;
  const size_t is = esize_of(in_dtype), os = esize_of(out_dtype);
  const uint64_t L = cr_chunk_len(count, nranks);
  std::vector<Span> spans;
  Width vw;
  vw.bytes(L * is);
  vw.bytes(L * os);
  for (int r = 0; r < nranks; ++r) {
    const uint64_t len = chunk_size(count, L, r);
    if ((st = check_buf(bufs[r], count, is, "bufs", r))) return st;
    if ((st = check_buf(out_shards[r], len, os, "out_shards", r))) return st;
    if (count) {
      spans.push_back(span_of(bufs[r], count * is, 0, r));
      vw.ptr(bufs[r]);
    }
    if (len) {
      spans.push_back(span_of(out_shards[r], len * os, 1, r));
      vw.ptr(out_shards[r]);
    }
  }
  const bool same = in_dtype == out_dtype;
  st = check_overlaps(spans, [&](const Span& i, const Span& o) {
    // In place: shard j is exactly chunk j of rank j's own buffer.
    return same && i.rank == o.rank && o.a == i.a + L * (uint64_t)o.rank * is;
  });
  if (st) return st;
  if (count == 0) return ok();
  FoldArgs a;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < nranks; ++r) {
    a.in[r] = bufs[r];
    a.out[r] = out_shards[r];
  }
  a.count = count;
  a.L = L;
  a.Ld = fastdiv_make(a.L, count ? count - 1 : 0);
  a.begin = 0;
  a.end = count;
  a.n = nranks;
  a.n_out = nranks;
  a.avg = op == CR_AVG;
  a.inv_n = exact_inv_n(nranks);
  a.wire_bf16 = wire_bf16 ? 1 : 0;
  cudaError_t e = launch_fold(in_dtype, out_dtype, kRS, a, vw.get(), stream);
  if (e != cudaSuccess) return cuda_fail(e, "reduce_scatter launch");
  return ok();
}

}  // namespace

extern "C" {

cr_status cr_reduce_scatter(const void* const* bufs, int nranks, size_t count,
                            cr_dtype in_dtype, cr_op op, void* const* out_shards,
                            cr_dtype out_dtype, cr_stream_t stream) {
  return reduce_scatter_impl(bufs, nranks, count, in_dtype, op, out_shards, out_dtype,
                             (cudaStream_t)stream, false);
}

cr_status cr_reduce_scatter_wire(const void* const* bufs, int nranks, size_t count,
                                 cr_dtype in_dtype, cr_op op, cr_dtype wire_dtype,
                                 void* const* out_shards, cr_dtype out_dtype,
                                 cr_stream_t stream) {
  bool bf16 = false;
  cr_status st = check_wire(in_dtype, wire_dtype, &bf16);
  if (st) return st;
  return reduce_scatter_impl(bufs, nranks, count, in_dtype, op, out_shards, out_dtype,
                             (cudaStream_t)stream, bf16);
}

cr_status cr_hsdp_reduce_scatter(const void* const* bufs, int R, int S, size_t count,
                                 cr_dtype in_dtype, cr_op op, void* const* out_shards,
                                 cr_dtype out_dtype, cr_stream_t stream) {
  if (R < 1 || S < 1 || R > CR_MAX_RANKS || S > CR_MAX_RANKS || R * S > CR_MAX_RANKS)
    return fail(CR_ERR_INVALID_ARG, "mesh %d x %d outside [1, %d] ranks", R, S, CR_MAX_RANKS);
  const int n = R * S;
  cr_status st = check_common(n, count, bufs, out_shards);
  if (st) return st;
  if ((st = check_pair(in_dtype, op, out_dtype))) return st;
  const size_t is = esize_of(in_dtype), os = esize_of(out_dtype);
  const uint64_t L = cr_chunk_len(count, S);
  std::vector<Span> spans;
  Width vw;
  vw.bytes(L * is);
  vw.bytes(L * os);
  for (int r = 0; r < n; ++r) {
    const uint64_t len = chunk_size(count, L, r % S);
    if ((st = check_buf(bufs[r], count, is, "bufs", r))) return st;
    if ((st = check_buf(out_shards[r], len, os, "out_shards", r))) return st;
    if (count) {
      spans.push_back(span_of(bufs[r], count * is, 0, r));
      vw.ptr(bufs[r]);
    }
    if (len) {
      spans.push_back(span_of(out_shards[r], len * os, 1, r));
      vw.ptr(out_shards[r]);
    }
  }
  const bool same = in_dtype == out_dtype;
  st = check_overlaps(spans, [&](const Span& i, const Span& o) {
    // In place: shard j of group g is chunk j of rank (g, j)'s own buffer.
    return same && i.rank == o.rank && o.a == i.a + L * (uint64_t)(o.rank % S) * is;
  });
  if (st) return st;
  if (count == 0) return ok();
  HsdpArgs a;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < n; ++r) {
    a.in[r] = bufs[r];
    a.out[r] = out_shards[r];
  }
  a.count = count;
  a.L = L;
  a.jlast = (count - 1) / L;
  const uint64_t len_last = count - a.jlast * L;
  a.L2 = (L + R - 1) / R;
  a.L2last = (len_last + R - 1) / R;
  a.Ld = fastdiv_make(L, count - 1);
  a.L2d = fastdiv_make(a.L2, L - 1);
  a.L2lastd = fastdiv_make(a.L2last, len_last - 1);
  a.R = R;
  a.S = S;
  a.avg = op == CR_AVG;
  a.inv_n = exact_inv_n(n);
  cudaError_t e = launch_hsdp(in_dtype, out_dtype, a, vw.get(), (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "hsdp_reduce_scatter launch");
  return ok();
}

cr_status cr_all_gather(const void* const* shards, int nranks, size_t count,
                        cr_dtype dtype, void* const* bufs, cr_stream_t stream) {
  cr_status st = check_common(nranks, count, shards, bufs);
  if (st) return st;
  const size_t es = esize_of(dtype);
  if (!es) return fail(CR_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
  const uint64_t L = cr_chunk_len(count, nranks);
  std::vector<Span> spans;
  Width vw;
  vw.bytes(L * es);
  uint64_t inplace = 0;
  for (int r = 0; r < nranks; ++r) {
    const uint64_t len = chunk_size(count, L, r);
    if ((st = check_buf(shards[r], len, es, "shards", r))) return st;
    if ((st = check_buf(bufs[r], count, es, "bufs", r))) return st;
    if (len) {
      spans.push_back(span_of(shards[r], len * es, 0, r));
      vw.ptr(shards[r]);
      if (count && reinterpret_cast<uintptr_t>(shards[r]) ==
                       reinterpret_cast<uintptr_t>(bufs[r]) + L * (uint64_t)r * es)
        inplace |= 1ull << r;
    }
    if (count) {
      spans.push_back(span_of(bufs[r], count * es, 1, r));
      vw.ptr(bufs[r]);
    }
  }
  st = check_overlaps(spans, [&](const Span& i, const Span& o) {
    return i.rank == o.rank && ((inplace >> i.rank) & 1ull);
  });
  if (st) return st;
  if (count == 0) return ok();
  GatherArgs a;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < nranks; ++r) {
    a.shards[r] = shards[r];
    a.bufs[r] = bufs[r];
  }
  a.count = count;
  a.L = L;
  a.Ld = fastdiv_make(L, count - 1);
  a.n = nranks;
  a.inplace_mask = inplace;
  cudaError_t e = launch_gather(es, a, vw.get(), (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "all_gather launch");
  return ok();
}

cr_status cr_all_reduce(const void* const* in, int nranks, size_t count,
                        cr_dtype in_dtype, cr_op op, void* const* out,
                        cr_dtype out_dtype, cr_stream_t stream) {
  return all_reduce_impl(in, nranks, count, in_dtype, op, out, out_dtype,
                         (cudaStream_t)stream);
}

cr_status cr_all_reduce_wire(const void* const* in, int nranks, size_t count,
                             cr_dtype in_dtype, cr_op op, cr_dtype wire_dtype,
                             void* const* out, cr_dtype out_dtype, cr_stream_t stream) {
  bool bf16 = false;
  cr_status st = check_wire(in_dtype, wire_dtype, &bf16);
  if (st) return st;
  return all_reduce_impl(in, nranks, count, in_dtype, op, out, out_dtype,
                         (cudaStream_t)stream, bf16);
}

// Device address of a host buffer the GPU can read and write directly
// (pinned with cudaHostAlloc / cudaHostRegister, or managed memory).
static cr_status host_view(const void* p, const char* what, int r, void** dptr) {
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) return cuda_fail(e, "cudaPointerGetAttributes");
  if ((at.type != cudaMemoryTypeHost && at.type != cudaMemoryTypeManaged) || !at.devicePointer)
    return fail(CR_ERR_INVALID_ARG, "%s[%d]=%p is not pinned (page-locked, mapped) host memory",
                what, r, p);
  *dptr = at.devicePointer;
  return CR_OK;
}

cr_status cr_all_reduce_host(const void* const* host_in, void* const* host_out,
                             void* const* dev_out, int nranks, size_t count, cr_dtype dtype,
                             cr_op op, cr_stream_t stream) {
  cr_status st = check_common(nranks, count, host_in, host_out);
  if (st) return st;
  if ((st = check_pair(dtype, op, dtype))) return st;
  if (dev_out && nranks > CR_MAX_RANKS / 2)
    return fail(CR_ERR_UNSUPPORTED, "dev_out needs nranks <= %d", CR_MAX_RANKS / 2);
  const size_t es = esize_of(dtype);
  std::vector<Span> spans;
  for (int r = 0; r < nranks; ++r) {
    if ((st = check_buf(host_in[r], count, es, "host_in", r))) return st;
    if ((st = check_buf(host_out[r], count, es, "host_out", r))) return st;
    if (dev_out && (st = check_buf(dev_out[r], count, es, "dev_out", r))) return st;
    if (count) {
      spans.push_back(span_of(host_in[r], count * es, 0, r));
      spans.push_back(span_of(host_out[r], count * es, 1, r));
      if (dev_out) spans.push_back(span_of(dev_out[r], count * es, 1, 100 + r));
    }
  }
  st = check_overlaps(spans, [](const Span& i, const Span& o) {
    return i.rank == o.rank && i.a == o.a && i.b == o.b;  // in place per rank
  });
  if (st) return st;
  if (count == 0) return ok();
  FoldArgs a;
  memset(&a, 0, sizeof(a));
  Width vw;
  for (int r = 0; r < nranks; ++r) {
    void* din = nullptr;
    void* dout = nullptr;
    if ((st = host_view(host_in[r], "host_in", r, &din))) return st;
    if ((st = host_view(host_out[r], "host_out", r, &dout))) return st;
    a.in[r] = din;
    a.out[r] = dout;
    if (dev_out) a.out[nranks + r] = dev_out[r];
    vw.ptr(din);
    vw.ptr(dout);
    if (dev_out) vw.ptr(dev_out[r]);
  }
  a.count = count;
  a.L = (count + nranks - 1) / nranks;
  a.Ld = fastdiv_make(a.L, count ? count - 1 : 0);
  a.begin = 0;
  a.end = count;
  a.n = nranks;
  a.n_out = dev_out ? 2 * nranks : nranks;
  a.avg = op == CR_AVG;
  a.inv_n = exact_inv_n(nranks);
  // Over the host link 16-byte accesses from a grid of 4 CTAs per SM keep
  // the link busiest (32-byte accesses and larger grids measured 5-17 %
  // slower on a GB300).
  int sms = 0;
  cudaError_t e = sm_count(&sms);
  if (e != cudaSuccess) return cuda_fail(e, "all_reduce_host SM count");
  a.max_ctas = 4u * (uint32_t)sms;
  e = launch_fold(dtype, dtype, kAR, a, vw.get() ? 16 : 0, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "all_reduce_host launch");
  return ok();
}

cr_status cr_all_reduce_staged(const void* const* host_in, void* const* host_out,
                               void* const* dev_bufs, int nranks, size_t count,
                               cr_dtype dtype, cr_op op, size_t slice_elems,
                               cr_stream_t compute_stream, cr_stream_t h2d_stream,
                               cr_stream_t d2h_stream) {
  cr_status st = check_common(nranks, count, host_in, dev_bufs);
  if (st) return st;
  if (!host_out) return fail(CR_ERR_INVALID_ARG, "host_out is NULL");
  if ((st = check_pair(dtype, op, dtype))) return st;
  const size_t es = esize_of(dtype);
  std::vector<Span> dev_spans, out_spans;
  Width vw;
  for (int r = 0; r < nranks; ++r) {
    if ((st = check_buf(host_in[r], count, es, "host_in", r))) return st;
    if ((st = check_buf(host_out[r], count, es, "host_out", r))) return st;
    if ((st = check_buf(dev_bufs[r], count, es, "dev_bufs", r))) return st;
    if (count) {
      dev_spans.push_back(span_of(dev_bufs[r], count * es, 1, r));
      out_spans.push_back(span_of(host_out[r], count * es, 1, r));
      vw.ptr(dev_bufs[r]);
    }
  }
  auto never = [](const Span&, const Span&) { return false; };
  if ((st = check_overlaps(dev_spans, never))) return st;
  if ((st = check_overlaps(out_spans, never))) return st;
  if (count == 0) return ok();

  const cudaStream_t sc = (cudaStream_t)compute_stream, sh = (cudaStream_t)h2d_stream,
                     sd = (cudaStream_t)d2h_stream;
  uint64_t slice = slice_elems;
  if (slice == 0) {
    slice = (count + 15) / 16;
    if (slice < (1u << 18)) slice = 1u << 18;
  }
  slice = (slice + 63) / 64 * 64;
  const uint64_t nslices = (count + slice - 1) / slice;

  FoldArgs a;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < nranks; ++r) {
    a.in[r] = dev_bufs[r];
    a.out[r] = dev_bufs[r];
  }
  a.count = count;
  a.L = (count + nranks - 1) / nranks;
  a.Ld = fastdiv_make(a.L, count - 1);
  a.n = nranks;
  a.n_out = nranks;
  a.avg = op == CR_AVG;
  a.inv_n = exact_inv_n(nranks);

  // Events are released with cudaEventDestroy right after being waited on;
  // the runtime frees each once it has completed.
  std::vector<cudaEvent_t> events;
  auto new_event = [&](cudaEvent_t* ev) -> cudaError_t {
    cudaError_t e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    if (e == cudaSuccess) events.push_back(*ev);
    return e;
  };
  auto release = [&]() {
    for (cudaEvent_t ev : events) cudaEventDestroy(ev);
    events.clear();
  };
  cudaError_t e = cudaSuccess;
  cudaEvent_t ev_start;
  if ((e = new_event(&ev_start)) != cudaSuccess) return cuda_fail(e, "staged: event");
  e = cudaEventRecord(ev_start, sc);
  if (e == cudaSuccess && sh != sc) e = cudaStreamWaitEvent(sh, ev_start, 0);
  if (e == cudaSuccess && sd != sc) e = cudaStreamWaitEvent(sd, ev_start, 0);
  for (uint64_t k = 0; k < nslices && e == cudaSuccess; ++k) {
    const uint64_t lo = k * slice, hi = lo + slice < count ? lo + slice : count;
    const size_t off = lo * es, bytes = (hi - lo) * es;
    for (int r = 0; r < nranks && e == cudaSuccess; ++r)
      e = cudaMemcpyAsync(static_cast<unsigned char*>(dev_bufs[r]) + off,
                          static_cast<const unsigned char*>(host_in[r]) + off, bytes,
                          cudaMemcpyHostToDevice, sh);
    cudaEvent_t ev_in, ev_out;
    if (e == cudaSuccess) e = new_event(&ev_in);
    if (e == cudaSuccess) e = cudaEventRecord(ev_in, sh);
    if (e == cudaSuccess && sc != sh) e = cudaStreamWaitEvent(sc, ev_in, 0);
    if (e == cudaSuccess) {
      a.begin = lo;
      a.end = hi;
      e = launch_fold(dtype, dtype, kAR, a, vw.get(), sc);
    }
    if (e == cudaSuccess) e = new_event(&ev_out);
    if (e == cudaSuccess) e = cudaEventRecord(ev_out, sc);
    if (e == cudaSuccess && sd != sc) e = cudaStreamWaitEvent(sd, ev_out, 0);
    for (int r = 0; r < nranks && e == cudaSuccess; ++r)
      e = cudaMemcpyAsync(static_cast<unsigned char*>(host_out[r]) + off,
                          static_cast<const unsigned char*>(dev_bufs[r]) + off, bytes,
                          cudaMemcpyDeviceToHost, sd);
  }
  cudaEvent_t ev_done;
  if (e == cudaSuccess) e = new_event(&ev_done);
  if (e == cudaSuccess) e = cudaEventRecord(ev_done, sd);
  if (e == cudaSuccess && sc != sd) e = cudaStreamWaitEvent(sc, ev_done, 0);
  release();
  if (e != cudaSuccess) return cuda_fail(e, "all_reduce_staged");
  return ok();
}

}  // extern "C"

namespace {

// Shared argument checks of the FSDP step entry points; fills `a` and the
// vector width `vw`.
cr_status fsdp_prepare(const void* const* grads_bf16, int nranks, size_t count,
                       float* const* master, float* const* m, float* const* v,
                       const cr_adamw_cfg* cfg, void* const* params_bf16,
                       std::vector<Span>& spans, FsdpArgs& a, int& vw) {
  cr_status st = check_common(nranks, count, grads_bf16, params_bf16);
  if (st) return st;
  if (!master || !m || !v) return fail(CR_ERR_INVALID_ARG, "master/m/v array is NULL");
  if ((st = check_adam_cfg(cfg))) return st;
  const uint64_t L = cr_chunk_len(count, nranks);
  // Vector path: 16-byte bf16 grads/params and 16- (or 32-) byte fp32
  // state vectors of 8 elements, which needs L % 8 == 0.
  Width gw, sw;
  gw.bytes(L * 2);
  sw.bytes(L * 4);
  for (int r = 0; r < nranks; ++r) {
    const uint64_t len = chunk_size(count, L, r);
    if ((st = check_buf(grads_bf16[r], count, 2, "grads", r))) return st;
    if ((st = check_buf(params_bf16[r], count, 2, "params", r))) return st;
    if ((st = check_buf(master[r], len, 4, "master", r))) return st;
    if ((st = check_buf(m[r], len, 4, "m", r))) return st;
    if ((st = check_buf(v[r], len, 4, "v", r))) return st;
    if (count) {
      // Every buffer is written or must not be written, so each is an
      // "output" span: no two may overlap.
      spans.push_back(span_of(grads_bf16[r], count * 2, 1, r));
      spans.push_back(span_of(params_bf16[r], count * 2, 1, r));
      gw.ptr(grads_bf16[r]);
      gw.ptr(params_bf16[r]);
    }
    if (len) {
      spans.push_back(span_of(master[r], len * 4, 1, r));
      spans.push_back(span_of(m[r], len * 4, 1, r));
      spans.push_back(span_of(v[r], len * 4, 1, r));
      sw.ptr(master[r]);
      sw.ptr(m[r]);
      sw.ptr(v[r]);
    }
  }
  vw = (gw.w16 && sw.w16) ? (sw.w32 ? 32 : 16) : 0;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < nranks; ++r) {
    a.grads[r] = grads_bf16[r];
    a.params[r] = params_bf16[r];
    a.master[r] = master[r];
    a.m[r] = m[r];
    a.v[r] = v[r];
  }
  a.count = count;
  a.L = L;
  a.Ld = fastdiv_make(L, count ? count - 1 : 0);
  a.n = nranks;
  a.inv_n = exact_inv_n(nranks);
  a.a = adam_scalars(*cfg);
  return CR_OK;
}

}  // namespace

extern "C" {

cr_status cr_fsdp_step(const void* const* grads_bf16, int nranks, size_t count,
                       float* const* master, float* const* m, float* const* v,
                       const cr_adamw_cfg* cfg, void* const* params_bf16,
                       cr_stream_t stream) {
  std::vector<Span> spans;
  FsdpArgs a;
  int vw = 0;
  cr_status st = fsdp_prepare(grads_bf16, nranks, count, master, m, v, cfg, params_bf16,
                              spans, a, vw);
  if (st) return st;
  if ((st = check_overlaps(spans, [](const Span&, const Span&) { return false; }))) return st;
  if (count == 0) return ok();
  cudaError_t e = launch_fsdp(a, vw, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "fsdp_step launch");
  return ok();
}

size_t cr_fsdp_clip_workspace_bytes(void) {
  return (size_t)(kMaxNormParts + 1) * sizeof(double);
}

cr_status cr_fsdp_step_clipped(const void* const* grads_bf16, int nranks, size_t count,
                               float* const* master, float* const* m, float* const* v,
                               const cr_adamw_cfg* cfg, double max_norm, void* workspace,
                               size_t workspace_bytes, void* const* params_bf16,
                               float* norm_out, cr_stream_t stream) {
  std::vector<Span> spans;
  FsdpArgs a;
  int vw = 0;
  cr_status st = fsdp_prepare(grads_bf16, nranks, count, master, m, v, cfg, params_bf16,
                              spans, a, vw);
  if (st) return st;
  if (!(max_norm > 0.0) || !isfinite(max_norm))
    return fail(CR_ERR_INVALID_ARG, "max_norm must be finite and > 0");
  if (!workspace) return fail(CR_ERR_INVALID_ARG, "workspace is NULL");
  if (!aligned(workspace, 8)) return fail(CR_ERR_ALIGNMENT, "workspace not 8-byte aligned");
  if (workspace_bytes < 2 * sizeof(double))
    return fail(CR_ERR_INVALID_ARG, "workspace_bytes=%zu too small", workspace_bytes);
  if (norm_out && !aligned(norm_out, 4)) return fail(CR_ERR_ALIGNMENT, "norm_out not aligned");
  // Slot 0: the clip coefficient; slots 1..max_parts: the partial sums.
  const size_t max_parts = workspace_bytes / sizeof(double) - 1 < (size_t)kMaxNormParts
                               ? workspace_bytes / sizeof(double) - 1
                               : (size_t)kMaxNormParts;
  spans.push_back(span_of(workspace, (max_parts + 1) * sizeof(double), 1, 1000));
  if (norm_out) spans.push_back(span_of(norm_out, sizeof(float), 1, 1001));
  if ((st = check_overlaps(spans, [](const Span&, const Span&) { return false; }))) return st;
  if (count == 0) {
    if (norm_out) {
      cudaError_t e = cudaMemsetAsync(norm_out, 0, sizeof(float), (cudaStream_t)stream);
      if (e != cudaSuccess) return cuda_fail(e, "fsdp_step_clipped norm_out");
    }
    return ok();
  }
  float* coef = static_cast<float*>(workspace);
  double* partials = static_cast<double*>(workspace) + 1;
  int nparts = 0;
  cudaError_t e = launch_fsdp_sumsq(a, vw != 0, partials, (int)max_parts, &nparts,
                                    (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "fsdp_step_clipped sum-of-squares launch");
  e = launch_clip_coef(partials, nparts, max_norm, coef, norm_out, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "fsdp_step_clipped coefficient launch");
  a.coef = coef;
  e = launch_fsdp(a, vw, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "fsdp_step_clipped launch");
  return ok();
}

cr_status cr_adamw_step(size_t n, float* master, float* m, float* v,
                        const float* grad, const cr_adamw_cfg* cfg,
                        void* param_bf16, cr_stream_t stream) {
  cr_status st = check_adam_cfg(cfg);
  if (st) return st;
  if (n > SIZE_MAX / 8) return fail(CR_ERR_INVALID_ARG, "n=%zu too large", n);
  if ((st = check_buf(master, n, 4, "master", 0))) return st;
  if ((st = check_buf(m, n, 4, "m", 0))) return st;
  if ((st = check_buf(v, n, 4, "v", 0))) return st;
  if ((st = check_buf(grad, n, 4, "grad", 0))) return st;
  if (param_bf16 && (st = check_buf(param_bf16, n, 2, "param_bf16", 0))) return st;
  if (n == 0) return ok();
  std::vector<Span> spans = {span_of(master, n * 4, 1, 0), span_of(m, n * 4, 1, 1),
                             span_of(v, n * 4, 1, 2), span_of(grad, n * 4, 1, 3)};
  if (param_bf16) spans.push_back(span_of(param_bf16, n * 2, 1, 4));
  st = check_overlaps(spans, [](const Span&, const Span&) { return false; });
  if (st) return st;
  AdamArgs a;
  a.master = master;
  a.m = m;
  a.v = v;
  a.g = grad;
  a.param_bf16 = param_bf16;
  a.n = n;
  a.a = adam_scalars(*cfg);
  const bool vec = aligned(master, 16) && aligned(m, 16) && aligned(v, 16) &&
                   aligned(grad, 16) && (!param_bf16 || aligned(param_bf16, 8));
  cudaError_t e = launch_adamw(a, vec, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "adamw launch");
  return ok();
}

// ---- buckets ---------------------------------------------------------------

static cr_status check_plan(const cr_bucket_plan_t* plan, int nranks) {
  if (!plan) return fail(CR_ERR_INVALID_ARG, "plan is NULL");
  if (nranks < 1 || nranks > CR_MAX_RANKS)
    return fail(CR_ERR_INVALID_ARG, "nranks=%d outside [1, %d]", nranks, CR_MAX_RANKS);
  if (plan->ntensors < 0 || plan->nbuckets < 0 || plan->elem_size == 0)
    return fail(CR_ERR_INVALID_ARG, "malformed plan");
  return CR_OK;
}

// Copies for pack (to_bucket) or unpack, batched kMaxSegsPerLaunch per launch.
static cr_status bucket_copy(const cr_bucket_plan_t* plan, int nranks,
                             const void* const* tensors, void* const* buckets,
                             bool to_bucket, cudaStream_t stream) {
  cr_status st = check_plan(plan, nranks);
  if (st) return st;
  const int T = plan->ntensors, B = plan->nbuckets;
  const size_t es = plan->elem_size;
  if (T > 0 && (!tensors || !buckets)) return fail(CR_ERR_INVALID_ARG, "pointer array is NULL");
  for (int r = 0; r < nranks; ++r) {
    for (int b = 0; b < B; ++b)
      if ((st = check_buf(buckets[(size_t)r * B + b], plan->bucket_numel[b], es, "buckets",
                          r * B + b)))
        return st;
    for (int t = 0; t < T; ++t)
      if ((st = check_buf(tensors[(size_t)r * T + t], plan->numels[t], es, "tensors",
                          r * T + t)))
        return st;
  }
  static thread_local CopyArgs args;  // ~28 KB: kept off the stack
  uint32_t ntiles = 0;
  int launches = 0;  // launches after the first are chained to their predecessor
  args.nseg = 0;
  auto flush = [&]() -> cr_status {
    if (args.nseg == 0) return CR_OK;
    args.tile_start[args.nseg] = ntiles;
    cudaError_t e = launch_copy(args, ntiles, launches++ > 0, stream);
    args.nseg = 0;
    ntiles = 0;
    if (e != cudaSuccess) return cuda_fail(e, "bucket copy launch");
    return CR_OK;
  };
  for (int r = 0; r < nranks; ++r) {
    for (int t = 0; t < T; ++t) {
      const uint64_t bytes = (uint64_t)plan->numels[t] * es;
      if (bytes == 0) continue;
      const int b = plan->tensor_bucket[t];
      unsigned char* bk = static_cast<unsigned char*>(buckets[(size_t)r * B + b]) +
                          plan->tensor_offset[t] * es;
      unsigned char* tp =
          static_cast<unsigned char*>(const_cast<void*>(tensors[(size_t)r * T + t]));
      CopySeg sg;
      sg.src = to_bucket ? tp : bk;
      sg.dst = to_bucket ? bk : tp;
      sg.bytes = bytes;
      const uintptr_t d0 = reinterpret_cast<uintptr_t>(sg.dst);
      const uintptr_t da = (d0 + 15) & ~uintptr_t(15), de = (d0 + bytes) & ~uintptr_t(15);
      const uint64_t nint = de > da ? (de - da) / 16 : 0;
      const uint64_t tiles64 = nint == 0 ? 1 : (nint + kCopyTileBytes / 16 - 1) / (kCopyTileBytes / 16);
      if (args.nseg == kMaxSegsPerLaunch || (uint64_t)ntiles + tiles64 > 0x7fffffffull) {
        if ((st = flush())) return st;
      }
      args.seg[args.nseg] = sg;
      args.tile_start[args.nseg] = ntiles;
      args.nseg += 1;
      ntiles += (uint32_t)tiles64;
    }
  }
  if ((st = flush())) return st;
  return ok();
}

cr_status cr_bucket_pack(const cr_bucket_plan_t* plan, int nranks,
                         const void* const* tensors, void* const* buckets,
                         cr_stream_t stream) {
  return bucket_copy(plan, nranks, tensors, buckets, true, (cudaStream_t)stream);
}

cr_status cr_bucket_unpack(const cr_bucket_plan_t* plan, int nranks,
                           const void* const* buckets, void* const* tensors,
                           cr_stream_t stream) {
  return bucket_copy(plan, nranks, const_cast<const void* const*>(tensors),
                     const_cast<void* const*>(buckets), false, (cudaStream_t)stream);
}

}  // extern "C"

namespace {

// Runs the fused bucket kernel over `nitems` items (tensors, or whole
// buckets): item(k, &numel, &offset in bucket, &bucket numel, rank ptrs).
// One launch per kFusedMaxTensors items (fewer when N > 16).
template <typename Item>
cr_status fused_run(int nitems, int nranks, cr_dtype dtype, cr_op op, cudaStream_t stream,
                    Item item, uint32_t max_ctas = 0) {
  static thread_local FusedArgs args;  // ~24 KB: kept off the stack
  const int per_launch = std::min(kFusedMaxTensors, kFusedMaxPtrs / nranks);
  const uint64_t tile = fused_tile_elems(dtype);
  uint32_t ntiles = 0;
  int launches = 0;  // launches after the first are chained to their predecessor
  args.ntens = 0;
  args.max_ctas = max_ctas;
  args.n = nranks;
  args.avg = op == CR_AVG;
  args.inv_n = exact_inv_n(nranks);
  auto flush = [&]() -> cr_status {
    if (args.ntens == 0) return CR_OK;
    args.tile_start[args.ntens] = ntiles;
    cudaError_t e = launch_bucket_fused(dtype, args, ntiles, launches++ > 0, stream);
    args.ntens = 0;
    ntiles = 0;
    if (e != cudaSuccess) return cuda_fail(e, "fused bucket all-reduce launch");
    return CR_OK;
  };
  cr_status st = CR_OK;
  void* ptrs[CR_MAX_RANKS];
  for (int t = 0; t < nitems; ++t) {
    uint64_t numel = 0, off = 0, bnumel = 0;
    item(t, &numel, &off, &bnumel, ptrs);
    if (numel == 0) continue;
    const uint64_t tiles = (numel + tile - 1) / tile;
    if (args.ntens == per_launch || (uint64_t)ntiles + tiles > 0x7fffffffull)
      if ((st = flush())) return st;
    const int k = args.ntens;
    FusedTensor& d = args.t[k];
    d.numel = numel;
    d.off = off;
    d.Lb = cr_chunk_len(bnumel, nranks);
    d.Lbd = fastdiv_make(d.Lb, bnumel ? bnumel - 1 : 0);
    d.ptr0 = (uint32_t)(k * nranks);
    Width w;
    for (int r = 0; r < nranks; ++r) {
      args.ptrs[k * nranks + r] = ptrs[r];
      w.ptr(ptrs[r]);
    }
    d.vw = (uint32_t)w.get();
    args.tile_start[k] = ntiles;
    args.ntens += 1;
    ntiles += (uint32_t)tiles;
  }
  if ((st = flush())) return st;
  return ok();
}

}  // namespace

// Arguments of cr_bucket_all_reduce_fused: plan, dtype, and N*T aligned,
// pairwise disjoint tensors.
cr_status cr::bucket_fused_check(const cr_bucket_plan_t* plan, int nranks, void* const* tensors,
                                 cr_dtype dtype, cr_op op) {
  cr_status st = check_plan(plan, nranks);
  if (st) return st;
  if ((st = check_pair(dtype, op, dtype))) return st;
  const size_t es = esize_of(dtype);
  if (es != plan->elem_size)
    return fail(CR_ERR_INVALID_ARG, "dtype size %zu != plan elem_size %zu", es, plan->elem_size);
  const int T = plan->ntensors;
  if (T > 0 && !tensors) return fail(CR_ERR_INVALID_ARG, "tensors is NULL");
  std::vector<Span> spans;
  for (int r = 0; r < nranks; ++r)
    for (int t = 0; t < T; ++t) {
      const void* p = tensors[(size_t)r * T + t];
      if ((st = check_buf(p, plan->numels[t], es, "tensors", r * T + t))) return st;
      if (plan->numels[t]) spans.push_back(span_of(p, plan->numels[t] * es, 1, r * T + t));
    }
  return check_disjoint(spans);
}

// The fused in-place all-reduce of tensors list[0..nlist) of the plan (all
// T tensors when list is NULL), on at most max_ctas CTAs (0: no cap).
cr_status cr::bucket_fused_tensors(const cr_bucket_plan_t* plan, int nranks,
                                   void* const* tensors, cr_dtype dtype, cr_op op,
                                   const int* list, int nlist, uint32_t max_ctas,
                                   cudaStream_t stream) {
  const int T = plan->ntensors;
  return fused_run(nlist, nranks, dtype, op, stream,
                   [&](int i, uint64_t* numel, uint64_t* off, uint64_t* bnumel, void** ptrs) {
                     const int t = list ? list[i] : i;
                     *numel = plan->numels[t];
                     *off = plan->tensor_offset[t];
                     *bnumel = plan->bucket_numel[plan->tensor_bucket[t]];
                     for (int r = 0; r < nranks; ++r) ptrs[r] = tensors[(size_t)r * T + t];
                   },
                   max_ctas);
}

extern "C" {

cr_status cr_bucket_all_reduce_fused(const cr_bucket_plan_t* plan, int nranks,
                                     void* const* tensors, cr_dtype dtype, cr_op op,
                                     cr_stream_t stream) {
  cr_status st = cr::bucket_fused_check(plan, nranks, tensors, dtype, op);
  if (st) return st;
  return cr::bucket_fused_tensors(plan, nranks, tensors, dtype, op, nullptr, plan->ntensors, 0,
                                  (cudaStream_t)stream);
}

// Every bucket of every rank all-reduced in place, all buckets in one
// launch (per 128): each bucket is one item of the fused kernel, offset 0,
// chunked over its own element count -- the same result as one
// cr_all_reduce per bucket.
cr_status cr_bucket_all_reduce(const cr_bucket_plan_t* plan, int nranks,
                               void* const* buckets, cr_dtype dtype, cr_op op,
                               cr_stream_t stream) {
  cr_status st = check_plan(plan, nranks);
  if (st) return st;
  if ((st = check_pair(dtype, op, dtype))) return st;
  const size_t es = esize_of(dtype);
  if (es != plan->elem_size)
    return fail(CR_ERR_INVALID_ARG, "dtype size %zu != plan elem_size %zu", es, plan->elem_size);
  const int B = plan->nbuckets;
  if (B > 0 && !buckets) return fail(CR_ERR_INVALID_ARG, "buckets is NULL");
  std::vector<Span> spans;
  for (int r = 0; r < nranks; ++r)
    for (int b = 0; b < B; ++b) {
      const void* p = buckets[(size_t)r * B + b];
      if ((st = check_buf(p, plan->bucket_numel[b], es, "buckets", r * B + b))) return st;
      if (plan->bucket_numel[b]) spans.push_back(span_of(p, plan->bucket_numel[b] * es, 1, r * B + b));
    }
  if ((st = check_disjoint(spans))) return st;
  return fused_run(B, nranks, dtype, op, (cudaStream_t)stream,
                   [&](int b, uint64_t* numel, uint64_t* off, uint64_t* bnumel, void** ptrs) {
                     *numel = plan->bucket_numel[b];
                     *off = 0;
                     *bnumel = plan->bucket_numel[b];
                     for (int r = 0; r < nranks; ++r) ptrs[r] = buckets[(size_t)r * B + b];
                   });
}

// ---- FSDP2 per-parameter step -------------------------------------------

cr_status cr_fsdp2_step(const cr_param_shape* shapes, int nparams, int nranks,
                        const void* const* grads_bf16, float* const* master, float* const* m,
                        float* const* v, const cr_adamw_cfg* cfg, void* const* params_bf16,
                        cr_stream_t stream) {
  if (nranks < 1 || nranks > CR_MAX_RANKS)
    return fail(CR_ERR_INVALID_ARG, "nranks=%d outside [1, %d]", nranks, CR_MAX_RANKS);
  if (nparams < 0 || (nparams > 0 && (!shapes || !grads_bf16 || !master || !m || !v ||
                                      !params_bf16)))
    return fail(CR_ERR_INVALID_ARG, "NULL array or nparams < 0");
  cr_status st = check_adam_cfg(cfg);
  if (st) return st;
  const int n = nranks;
  std::vector<Span> spans;
  for (int p = 0; p < nparams; ++p) {
    const uint64_t d0 = shapes[p].dim0, rn = shapes[p].row_numel;
    if (rn && d0 > (SIZE_MAX / 8) / rn) return fail(CR_ERR_INVALID_ARG, "param %d too large", p);
    const uint64_t numel = d0 * rn;
    const uint64_t L = cr_chunk_len(d0, n) * rn;
    for (int r = 0; r < n; ++r) {
      const size_t k = (size_t)p * n + r;
      const uint64_t len = chunk_size(numel, L, r);
      if ((st = check_buf(grads_bf16[k], numel, 2, "grads", (int)k))) return st;
      if ((st = check_buf(params_bf16[k], numel, 2, "params", (int)k))) return st;
      if ((st = check_buf(master[k], len, 4, "master", (int)k))) return st;
      if ((st = check_buf(m[k], len, 4, "m", (int)k))) return st;
      if ((st = check_buf(v[k], len, 4, "v", (int)k))) return st;
      if (numel) {
        spans.push_back(span_of(grads_bf16[k], numel * 2, 1, (int)k));
        spans.push_back(span_of(params_bf16[k], numel * 2, 1, (int)k));
      }
      if (len) {
        spans.push_back(span_of(master[k], len * 4, 1, (int)k));
        spans.push_back(span_of(m[k], len * 4, 1, (int)k));
        spans.push_back(span_of(v[k], len * 4, 1, (int)k));
      }
    }
  }
  if ((st = check_disjoint(spans))) return st;
  static thread_local Fsdp2Args args;  // ~24 KB: kept off the stack
  const int per_launch = std::min(kFsdp2MaxParams, kFsdp2MaxPtrs / (5 * n));
  uint32_t ntiles = 0;
  int launches = 0;  // launches after the first are chained to their predecessor
  args.nparams = 0;
  args.n = n;
  args.inv_n = exact_inv_n(n);
  args.a = adam_scalars(*cfg);
  auto flush = [&]() -> cr_status {
    if (args.nparams == 0) return CR_OK;
    args.tile_start[args.nparams] = ntiles;
    cudaError_t e = launch_fsdp2(args, ntiles, launches++ > 0, (cudaStream_t)stream);
    args.nparams = 0;
    ntiles = 0;
    if (e != cudaSuccess) return cuda_fail(e, "fsdp2_step launch");
    return CR_OK;
  };
  for (int p = 0; p < nparams; ++p) {
    const uint64_t numel = shapes[p].dim0 * shapes[p].row_numel;
    if (numel == 0) continue;
    const uint64_t tiles = (numel + kFsdp2TileElems - 1) / kFsdp2TileElems;
    if (args.nparams == per_launch || (uint64_t)ntiles + tiles > 0x7fffffffull)
      if ((st = flush())) return st;
    const int q = args.nparams;
    Fsdp2Param& d = args.p[q];
    d.numel = numel;
    d.L = cr_chunk_len(shapes[p].dim0, n) * shapes[p].row_numel;
    d.Ld = fastdiv_make(d.L, numel - 1);
    d.ptr0 = (uint32_t)(q * 5 * n);
    Width gw, sw;
    gw.bytes(d.L * 2);
    sw.bytes(d.L * 4);
    for (int r = 0; r < n; ++r) {
      const size_t k = (size_t)p * n + r;
      args.ptrs[d.ptr0 + r] = const_cast<void*>(grads_bf16[k]);
      args.ptrs[d.ptr0 + n + r] = params_bf16[k];
      args.ptrs[d.ptr0 + 2 * n + r] = master[k];
      args.ptrs[d.ptr0 + 3 * n + r] = m[k];
      args.ptrs[d.ptr0 + 4 * n + r] = v[k];
      gw.ptr(grads_bf16[k]);
      gw.ptr(params_bf16[k]);
      if (chunk_size(numel, d.L, r)) {  // empty shards' pointers do not matter
        sw.ptr(master[k]);
        sw.ptr(m[k]);
        sw.ptr(v[k]);
      }
    }
    d.vw = (gw.w16 && sw.w16) ? (sw.w32 ? 32u : 16u) : 0u;
    args.tile_start[q] = ntiles;
    args.nparams += 1;
    ntiles += (uint32_t)tiles;
  }
  if ((st = flush())) return st;
  return ok();
}

// ---- gradient accumulation (no_sync) ------------------------------------

static cr_status accumulate_impl(float* const* acc, int nranks, size_t count,
                                 const void* const* grads, cr_dtype grad_dtype, int reduce,
                                 cr_op op, cudaStream_t stream) {
  cr_status st = check_common(nranks, count, acc, grads);
  if (st) return st;
  if (grad_dtype != CR_F32 && grad_dtype != CR_BF16)
    return fail(CR_ERR_UNSUPPORTED, "grad_dtype must be CR_F32 or CR_BF16");
  if (op != CR_SUM && op != CR_AVG) return fail(CR_ERR_INVALID_ARG, "unknown op %d", (int)op);
  const size_t gs = esize_of(grad_dtype);
  std::vector<Span> spans;
  Width aw, gw;
  for (int r = 0; r < nranks; ++r) {
    if ((st = check_buf(acc[r], count, 4, "acc", r))) return st;
    if ((st = check_buf(grads[r], count, gs, "grads", r))) return st;
    if (count) {
      spans.push_back(span_of(acc[r], count * 4, 1, r));
      spans.push_back(span_of(grads[r], count * gs, 1, 100 + r));
      aw.ptr(acc[r]);
      gw.ptr(grads[r]);
    }
  }
  if ((st = check_disjoint(spans))) return st;
  if (count == 0) return ok();
  AccumArgs a;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < nranks; ++r) {
    a.acc[r] = acc[r];
    a.grads[r] = grads[r];
  }
  a.count = count;
  a.L = cr_chunk_len(count, nranks);
  a.Ld = fastdiv_make(a.L, count - 1);
  a.n = nranks;
  a.reduce = reduce;
  a.avg = op == CR_AVG;
  a.inv_n = exact_inv_n(nranks);
  const int vw = (aw.w16 && gw.w16) ? (aw.w32 ? 32 : 16) : 0;
  cudaError_t e = launch_accum(grad_dtype, a, vw, stream);
  if (e != cudaSuccess) return cuda_fail(e, "accumulate launch");
  return ok();
}

cr_status cr_accumulate(float* const* acc, int nranks, size_t count, const void* const* grads,
                        cr_dtype grad_dtype, cr_stream_t stream) {
  return accumulate_impl(acc, nranks, count, grads, grad_dtype, 0, CR_SUM,
                         (cudaStream_t)stream);
}

cr_status cr_all_reduce_accumulate(float* const* acc, int nranks, size_t count,
                                   const void* const* grads, cr_dtype grad_dtype, cr_op op,
                                   cr_stream_t stream) {
  return accumulate_impl(acc, nranks, count, grads, grad_dtype, 1, op, (cudaStream_t)stream);
}

}  // extern "C"

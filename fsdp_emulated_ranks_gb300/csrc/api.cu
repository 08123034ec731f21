// api.cu -- the extern "C" collectives of libcr (include/cr.h): reduce-
// scatter, all-gather and all-reduce (fp32 and bf16 wires), HSDP, the
// host-memory all-reduces, and the status / chunking helpers.  Host-side
// argument checks (api_host.h), then one launch per call.
#include "api_host.h"

using namespace cr;
using namespace cr::host;

namespace {

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
cr_status cr::report_cuda_error(cudaError_t e, const char* what) { return cuda_fail(e, what); }

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
  Width vw, vin;  // every buffer and L; the inputs alone
  vw.bytes(L * is);
  vw.bytes(L * os);
  for (int r = 0; r < nranks; ++r) {
    const uint64_t len = chunk_size(count, L, r);
    if ((st = check_buf(bufs[r], count, is, "bufs", r))) return st;
    if ((st = check_buf(out_shards[r], len, os, "out_shards", r))) return st;
    if (count) {
      spans.push_back(span_of(bufs[r], count * is, 0, r));
      vw.ptr(bufs[r]);
      vin.ptr(bufs[r]);
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
  // Shards off the vector grid (L or a shard pointer): vector loads, element
  // stores, rather than element loads too.
  int w = vw.get();
  if (w == 0 && vin.get() != 0) {
    w = vin.get();
    a.out_scalar = 1;
  }
  cudaError_t e = launch_fold(in_dtype, out_dtype, kRS, a, w, stream);
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
  Width vw, vin;  // every buffer and L; the inputs alone
  vw.bytes(L * is);
  vw.bytes(L * os);
  for (int r = 0; r < n; ++r) {
    const uint64_t len = chunk_size(count, L, r % S);
    if ((st = check_buf(bufs[r], count, is, "bufs", r))) return st;
    if ((st = check_buf(out_shards[r], len, os, "out_shards", r))) return st;
    if (count) {
      spans.push_back(span_of(bufs[r], count * is, 0, r));
      vw.ptr(bufs[r]);
      vin.ptr(bufs[r]);
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
  int w = vw.get();
  if (w == 0 && vin.get() != 0) {  // shards off the vector grid: element stores
    w = vin.get();
    a.out_scalar = 1;
  }
  cudaError_t e = launch_hsdp(in_dtype, out_dtype, a, w, (cudaStream_t)stream);
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

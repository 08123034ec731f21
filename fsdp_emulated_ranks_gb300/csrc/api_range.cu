// api_range.cu -- range forms of the collectives (include/cr.h): the
// all-reduce and reduce-scatter of elements [begin, end) of the rank
// buffers, with the whole buffers' chunks and so the whole buffers' fold
// order, and the slab split that hands each of G GPUs one such range.
//
// Each output element of a reduce-scatter or all-reduce depends only on the
// same element of every rank ("Distributed Training for Large Models",
// section 2, All-Reduce: the sum is taken element-wise across ranks), so
// the element range [0, count) can be cut into slabs that are reduced
// independently, on different GPUs, with no exchange between them.  What
// must not change is the chunking: element e belongs to chunk e / L with
// L = ceil(count / N) of the whole buffer, which fixes where its ring fold
// starts.  Calling the whole-buffer entry points on a slab would re-chunk
// the slab; these calls keep count (and so L) and take the range apart.
#include "api_host.h"

using namespace cr;
using namespace cr::host;

extern "C" {

cr_status cr_slab_range(size_t count, int nranks, int nslabs, int g, size_t* begin,
                        size_t* end) {
  if (nranks < 1 || nranks > CR_MAX_RANKS)
    return fail(CR_ERR_INVALID_ARG, "nranks=%d outside [1, %d]", nranks, CR_MAX_RANKS);
  if (nslabs < 1) return fail(CR_ERR_INVALID_ARG, "nslabs=%d < 1", nslabs);
  if (g < 0 || g >= nslabs) return fail(CR_ERR_INVALID_ARG, "g=%d outside [0, %d)", g, nslabs);
  if (!begin || !end) return fail(CR_ERR_INVALID_ARG, "begin/end is NULL");
  if (count > SIZE_MAX / 8) return fail(CR_ERR_INVALID_ARG, "count=%zu too large", count);
  auto bound = [&](uint64_t k) -> uint64_t {  // start of slab k (k = nslabs: count)
    uint64_t b;
    if (nslabs <= nranks) {
      // whole chunks: slab k starts at chunk floor(k * N / G)
      const uint64_t L = cr_chunk_len(count, nranks);
      b = L * ((k * (uint64_t)nranks) / (uint64_t)nslabs);
    } else {
      // more slabs than chunks: 16-element boundaries
      const uint64_t units = (count + 15) / 16;
      b = 16 * ((k * units) / (uint64_t)nslabs);
    }
    return b < count ? b : count;
  };
  *begin = bound((uint64_t)g);
  *end = bound((uint64_t)g + 1);
  return ok();
}

cr_status cr_all_reduce_range(const void* const* in, int nranks, size_t count, size_t begin,
                              size_t end, cr_dtype in_dtype, cr_op op, void* const* out,
                              cr_dtype out_dtype, cr_stream_t stream) {
  cr_status st = check_common(nranks, count, in, out);
  if (st) return st;
  if ((st = check_pair(in_dtype, op, out_dtype))) return st;
  if (begin > end || end > count)
    return fail(CR_ERR_INVALID_ARG, "range [%zu, %zu) outside [0, %zu)", begin, end, count);
  const size_t is = esize_of(in_dtype), os = esize_of(out_dtype);
  const uint64_t nslab = end - begin;
  std::vector<Span> spans;
  Width vw;
  FoldArgs a;
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < nranks; ++r) {
    if ((st = check_buf(in[r], nslab, is, "in", r))) return st;
    if ((st = check_buf(out[r], nslab, os, "out", r))) return st;
    a.in[r] = shift_back(in[r], begin, is);
    a.out[r] = shift_back(out[r], begin, os);
    if (nslab) {
      spans.push_back(span_of(in[r], nslab * is, 0, r));
      spans.push_back(span_of(out[r], nslab * os, 1, r));
      vw.ptr(a.in[r]);
      vw.ptr(a.out[r]);
    }
  }
  const bool same = in_dtype == out_dtype;
  st = check_overlaps(spans, [&](const Span& i, const Span& o) {
    return same && i.rank == o.rank && i.a == o.a && i.b == o.b;
  });
  if (st) return st;
  if (nslab == 0) return ok();
  a.count = count;
  a.L = cr_chunk_len(count, nranks);
  a.Ld = fastdiv_make(a.L, count - 1);
  a.begin = begin;
  a.end = end;
  a.n = nranks;
  a.n_out = nranks;
  a.avg = op == CR_AVG;
  a.inv_n = exact_inv_n(nranks);
  cudaError_t e = launch_fold(in_dtype, out_dtype, kAR, a, vw.get(), (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "all_reduce_range launch");
  return ok();
}

cr_status cr_reduce_scatter_range(const void* const* bufs, int nranks, size_t count,
                                  size_t begin, size_t end, cr_dtype in_dtype, cr_op op,
                                  void* const* out_shards, cr_dtype out_dtype,
                                  cr_stream_t stream) {
  cr_status st = check_common(nranks, count, bufs, out_shards);
  if (st) return st;
  if ((st = check_pair(in_dtype, op, out_dtype))) return st;
  if (begin > end || end > count)
    return fail(CR_ERR_INVALID_ARG, "range [%zu, %zu) outside [0, %zu)", begin, end, count);
  const size_t is = esize_of(in_dtype), os = esize_of(out_dtype);
  const uint64_t L = cr_chunk_len(count, nranks);
  const uint64_t nslab = end - begin;
  std::vector<Span> spans;
  std::vector<uint64_t> part_lo(nranks, 0);  // first element of shard j's part
  Width vw, vin;  // every buffer and L; the inputs alone
  vw.bytes(L * is);
  vw.bytes(L * os);
  FoldArgs a;
  memset(&a, 0, sizeof(a));
  for (int j = 0; j < nranks; ++j) {
    const uint64_t c0 = chunk_lo(count, L, j);
    const uint64_t lo = std::max<uint64_t>(begin, c0);
    const uint64_t hi = std::min<uint64_t>(end, c0 + chunk_size(count, L, j));
    const uint64_t len = hi > lo ? hi - lo : 0;
    part_lo[j] = lo;
    if ((st = check_buf(bufs[j], nslab, is, "bufs", j))) return st;
    if ((st = check_buf(out_shards[j], len, os, "out_shards", j))) return st;
    a.in[j] = shift_back(bufs[j], begin, is);
    // out[j] + (e - jL) * os must be element e's place in shard j
    a.out[j] = len ? shift_back(out_shards[j], lo - L * (uint64_t)j, os) : nullptr;
    if (nslab) {
      spans.push_back(span_of(bufs[j], nslab * is, 0, j));
      vw.ptr(a.in[j]);
      vin.ptr(a.in[j]);
    }
    if (len) {
      spans.push_back(span_of(out_shards[j], len * os, 1, j));
      vw.ptr(a.out[j]);
    }
  }
  const bool same = in_dtype == out_dtype;
  st = check_overlaps(spans, [&](const Span& i, const Span& o) {
    // In place: shard j's part is exactly where its elements sit in rank
    // j's own slab.
    return same && i.rank == o.rank && o.a == i.a + (part_lo[o.rank] - begin) * is;
  });
  if (st) return st;
  if (nslab == 0) return ok();
  a.count = count;
  a.L = L;
  a.Ld = fastdiv_make(L, count - 1);
  a.begin = begin;
  a.end = end;
  a.n = nranks;
  a.n_out = nranks;
  a.avg = op == CR_AVG;
  a.inv_n = exact_inv_n(nranks);
  int w = vw.get();
  if (w == 0 && vin.get() != 0) {  // as cr_reduce_scatter: element stores
    w = vin.get();
    a.out_scalar = 1;
  }
  cudaError_t e = launch_fold(in_dtype, out_dtype, kRS, a, w, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "reduce_scatter_range launch");
  return ok();
}

}  // extern "C"

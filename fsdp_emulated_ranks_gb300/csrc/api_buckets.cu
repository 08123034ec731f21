// api_buckets.cu -- the extern "C" DDP bucket entry points (include/cr.h):
// pack / unpack (one launch per 1024 ranges), the per-bucket all-reduce and
// the fused all-reduce on the tensors (one launch per 128 items, chained),
// and the fused run the reducer uses.
#include "api_host.h"

using namespace cr;
using namespace cr::host;

extern "C" {

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
  st = check_disjoint(spans);
  if (st) return st;
  return fused_run(B, nranks, dtype, op, (cudaStream_t)stream,
                   [&](int b, uint64_t* numel, uint64_t* off, uint64_t* bnumel, void** ptrs) {
                     *numel = plan->bucket_numel[b];
                     *off = 0;
                     *bnumel = plan->bucket_numel[b];
                     for (int r = 0; r < nranks; ++r) ptrs[r] = buckets[(size_t)r * B + b];
                   });
}

}  // extern "C"

// api_optim.cu -- the extern "C" optimizer-side entry points (include/cr.h):
// the fused FSDP step (plain, clipped), stand-alone AdamW, the FSDP2
// per-parameter step and the no_sync accumulation.
#include <memory>
#include <new>

#include "api_host.h"

using namespace cr;
using namespace cr::host;

namespace {

// Shared argument checks of the FSDP step entry points; fills `a` and the
// vector width `vw`.  The step covers elements [begin, end) of the flat
// buffer of `count` elements (the whole buffer: 0, count).  grads/params
// point at element `begin` of each rank's buffer (slabs of end - begin
// elements); master/m/v[j] at the first element of owner j's shard that
// lies in the range (any value, NULL included, for a shard the range does
// not reach).  The kernel addresses elements by their index in the whole
// buffer, so the pointers it gets are shifted back by the offsets of the
// slab and of each shard's part.
cr_status fsdp_prepare(const void* const* grads_bf16, int nranks, size_t count,
                       float* const* master, float* const* m, float* const* v,
                       const cr_adamw_cfg* cfg, void* const* params_bf16,
                       std::vector<Span>& spans, FsdpArgs& a, int& vw,
                       size_t begin, size_t end) {
  cr_status st = check_common(nranks, count, grads_bf16, params_bf16);
  if (st) return st;
  if (!master || !m || !v) return fail(CR_ERR_INVALID_ARG, "master/m/v array is NULL");
  if ((st = check_adam_cfg(cfg))) return st;
  if (begin > end || end > count)
    return fail(CR_ERR_INVALID_ARG, "range [%zu, %zu) outside [0, %zu)", begin, end, count);
  const uint64_t L = cr_chunk_len(count, nranks);
  const uint64_t nslab = end - begin;
  // Vector path: 16-byte bf16 grads/params and 16- (or 32-) byte fp32
  // state vectors of 8 elements, which needs L % 8 == 0.  With L (or a
  // state pointer) off that grid, the grads/params still move as vectors
  // and the state element by element (vw = 1).
  Width gw, sw, gp;
  gw.bytes(L * 2);
  sw.bytes(L * 4);
  memset(&a, 0, sizeof(a));
  for (int r = 0; r < nranks; ++r) {
    // owner r's part of the range: shard elements [lo - rL, hi - rL)
    const uint64_t lo = std::max<uint64_t>(begin, chunk_lo(count, L, r));
    const uint64_t hi = std::min<uint64_t>(end, chunk_lo(count, L, r) + chunk_size(count, L, r));
    const uint64_t len = hi > lo ? hi - lo : 0;
    if ((st = check_buf(grads_bf16[r], nslab, 2, "grads", r))) return st;
    if ((st = check_buf(params_bf16[r], nslab, 2, "params", r))) return st;
    if ((st = check_buf(master[r], len, 4, "master", r))) return st;
    if ((st = check_buf(m[r], len, 4, "m", r))) return st;
    if ((st = check_buf(v[r], len, 4, "v", r))) return st;
    const uint64_t soff = len ? lo - L * (uint64_t)r : 0;  // offset of the part in shard r
    a.grads[r] = shift_back(grads_bf16[r], begin, 2);
    a.params[r] = shift_back(params_bf16[r], begin, 2);
    a.master[r] = len ? shift_back(master[r], soff, 4) : nullptr;
    a.m[r] = len ? shift_back(m[r], soff, 4) : nullptr;
    a.v[r] = len ? shift_back(v[r], soff, 4) : nullptr;
    if (nslab) {
      // Every buffer is written or must not be written, so each is an
      // "output" span: no two may overlap.
      spans.push_back(span_of(grads_bf16[r], nslab * 2, 1, r));
      spans.push_back(span_of(params_bf16[r], nslab * 2, 1, r));
      gw.ptr(a.grads[r]);
      gw.ptr(a.params[r]);
      gp.ptr(a.grads[r]);
      gp.ptr(a.params[r]);
    }
    if (len) {
      spans.push_back(span_of(master[r], len * 4, 1, r));
      spans.push_back(span_of(m[r], len * 4, 1, r));
      spans.push_back(span_of(v[r], len * 4, 1, r));
      sw.ptr(a.master[r]);
      sw.ptr(a.m[r]);
      sw.ptr(a.v[r]);
    }
  }
  vw = (gw.w16 && sw.w16) ? (sw.w32 ? 32 : 16) : (gp.w16 ? 1 : 0);
  a.count = count;
  a.L = L;
  a.Ld = fastdiv_make(L, count ? count - 1 : 0);
  a.begin = begin;
  a.end = end;
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
                              spans, a, vw, 0, count);
  if (st) return st;
  if ((st = check_overlaps(spans, [](const Span&, const Span&) { return false; }))) return st;
  if (count == 0) return ok();
  cudaError_t e = launch_fsdp(a, vw, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "fsdp_step launch");
  return ok();
}

cr_status cr_fsdp_step_range(const void* const* grads_bf16, int nranks, size_t count,
                             size_t begin, size_t end, float* const* master, float* const* m,
                             float* const* v, const cr_adamw_cfg* cfg,
                             void* const* params_bf16, cr_stream_t stream) {
  std::vector<Span> spans;
  FsdpArgs a;
  int vw = 0;
  cr_status st = fsdp_prepare(grads_bf16, nranks, count, master, m, v, cfg, params_bf16,
                              spans, a, vw, begin, end);
  if (st) return st;
  if ((st = check_overlaps(spans, [](const Span&, const Span&) { return false; }))) return st;
  if (end == begin) return ok();
  cudaError_t e = launch_fsdp(a, vw, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "fsdp_step_range launch");
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
                              spans, a, vw, 0, count);
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
  // Park the averaged gradient in params[0]/params[1] between the passes
  // when that moves fewer bytes: 4N + 32 per element against 6N + 24.
  a.stash = (vw != 0 && nranks >= 5) ? 1 : 0;
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

// ---- FSDP2 per-parameter step -------------------------------------------

}  // extern "C"

namespace {

// Argument checks shared by cr_fsdp2_step and cr_fsdp2_plan_create: sizes,
// alignment and NULLs of every buffer, and no two buffers overlapping.
cr_status fsdp2_check(const cr_param_shape* shapes, int nparams, int nranks,
                      const void* const* grads_bf16, float* const* master, float* const* m,
                      float* const* v, void* const* params_bf16) {
  if (nranks < 1 || nranks > CR_MAX_RANKS)
    return fail(CR_ERR_INVALID_ARG, "nranks=%d outside [1, %d]", nranks, CR_MAX_RANKS);
  if (nparams < 0 || (nparams > 0 && (!shapes || !grads_bf16 || !master || !m || !v ||
                                      !params_bf16)))
    return fail(CR_ERR_INVALID_ARG, "NULL array or nparams < 0");
  cr_status st;
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
  return check_disjoint(spans);
}

// Descriptor of parameter p (numel > 0) whose 5N pointers start at ptr0;
// writes the pointers to ptrs[ptr0 ...].
Fsdp2Param fsdp2_param(const cr_param_shape& shape, int n, size_t p, uint32_t ptr0,
                       const void* const* grads_bf16, float* const* master, float* const* m,
                       float* const* v, void* const* params_bf16, void** ptrs) {
  Fsdp2Param d;
  memset(&d, 0, sizeof(d));
  d.numel = shape.dim0 * shape.row_numel;
  d.L = cr_chunk_len(shape.dim0, n) * shape.row_numel;
  d.Ld = fastdiv_make(d.L, d.numel - 1);
  d.ptr0 = ptr0;
  Width gw, sw;
  gw.bytes(d.L * 2);
  sw.bytes(d.L * 4);
  for (int r = 0; r < n; ++r) {
    const size_t k = p * n + r;
    ptrs[ptr0 + r] = const_cast<void*>(grads_bf16[k]);
    ptrs[ptr0 + n + r] = params_bf16[k];
    ptrs[ptr0 + 2 * n + r] = master[k];
    ptrs[ptr0 + 3 * n + r] = m[k];
    ptrs[ptr0 + 4 * n + r] = v[k];
    gw.ptr(grads_bf16[k]);
    gw.ptr(params_bf16[k]);
    if (chunk_size(d.numel, d.L, r)) {  // empty shards' pointers do not matter
      sw.ptr(master[k]);
      sw.ptr(m[k]);
      sw.ptr(v[k]);
    }
  }
  d.vw = (gw.w16 && sw.w16) ? (sw.w32 ? 32u : 16u) : 0u;
  return d;
}

}  // namespace

// A parameter set's FSDP2 table, built on the host (see cr_internal.cuh for
// the layout the kernel reads).
struct cr_fsdp2_plan {
  int n;
  uint32_t nparams;  // parameters with at least one element
  uint32_t ntiles;
  uint64_t p_off, ptr_off;
  std::vector<unsigned char> table;
};

extern "C" {

cr_status cr_fsdp2_step(const cr_param_shape* shapes, int nparams, int nranks,
                        const void* const* grads_bf16, float* const* master, float* const* m,
                        float* const* v, const cr_adamw_cfg* cfg, void* const* params_bf16,
                        cr_stream_t stream) {
  cr_status st = check_adam_cfg(cfg);
  if (st) return st;
  if ((st = fsdp2_check(shapes, nparams, nranks, grads_bf16, master, m, v, params_bf16)))
    return st;
  const int n = nranks;
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
    args.p[q] = fsdp2_param(shapes[p], n, (size_t)p, (uint32_t)(q * 5 * n), grads_bf16, master,
                            m, v, params_bf16, args.ptrs);
    args.tile_start[q] = ntiles;
    args.nparams += 1;
    ntiles += (uint32_t)tiles;
  }
  if ((st = flush())) return st;
  return ok();
}

cr_status cr_fsdp2_plan_create(const cr_param_shape* shapes, int nparams, int nranks,
                               const void* const* grads_bf16, float* const* master,
                               float* const* m, float* const* v, void* const* params_bf16,
                               cr_fsdp2_plan_t** plan) {
  if (!plan) return fail(CR_ERR_INVALID_ARG, "plan is NULL");
  *plan = nullptr;
  cr_status st = fsdp2_check(shapes, nparams, nranks, grads_bf16, master, m, v, params_bf16);
  if (st) return st;
  const int n = nranks;
  std::vector<uint32_t> tile_start;
  std::vector<int> keep;
  uint64_t ntiles = 0;
  for (int p = 0; p < nparams; ++p) {
    const uint64_t numel = shapes[p].dim0 * shapes[p].row_numel;
    if (numel == 0) continue;
    tile_start.push_back((uint32_t)ntiles);
    keep.push_back(p);
    ntiles += (numel + kFsdp2TileElems - 1) / kFsdp2TileElems;
    if (ntiles > 0x7fffffffull)
      return fail(CR_ERR_INVALID_ARG, "more than 2^31 tiles of %llu elements",
                  (unsigned long long)kFsdp2TileElems);
  }
  tile_start.push_back((uint32_t)ntiles);
  const uint64_t np = keep.size();
  if (np * 5 * (uint64_t)n > 0xffffffffull)
    return fail(CR_ERR_INVALID_ARG, "too many parameters for one table");
  auto up16 = [](uint64_t x) { return (x + 15) & ~uint64_t(15); };
  std::unique_ptr<cr_fsdp2_plan> pl(new (std::nothrow) cr_fsdp2_plan);
  if (!pl) return fail(CR_ERR_INVALID_ARG, "out of host memory");
  pl->n = n;
  pl->nparams = (uint32_t)np;
  pl->ntiles = (uint32_t)ntiles;
  pl->p_off = up16(tile_start.size() * sizeof(uint32_t));
  pl->ptr_off = pl->p_off + np * sizeof(Fsdp2Param);
  try {
    pl->table.assign(pl->ptr_off + np * 5 * n * sizeof(void*), 0);
  } catch (const std::bad_alloc&) {
    return fail(CR_ERR_INVALID_ARG, "out of host memory");
  }
  unsigned char* t = pl->table.data();
  memcpy(t, tile_start.data(), tile_start.size() * sizeof(uint32_t));
  Fsdp2Param* desc = reinterpret_cast<Fsdp2Param*>(t + pl->p_off);
  void** ptrs = reinterpret_cast<void**>(t + pl->ptr_off);
  for (uint64_t q = 0; q < np; ++q)
    desc[q] = fsdp2_param(shapes[keep[q]], n, (size_t)keep[q], (uint32_t)(q * 5 * n), grads_bf16,
                          master, m, v, params_bf16, ptrs);
  *plan = pl.release();
  return ok();
}

size_t cr_fsdp2_plan_table_bytes(const cr_fsdp2_plan_t* plan) {
  return plan ? plan->table.size() : 0;
}

cr_status cr_fsdp2_plan_upload(const cr_fsdp2_plan_t* plan, void* table, size_t table_bytes,
                               cr_stream_t stream) {
  if (!plan || !table) return fail(CR_ERR_INVALID_ARG, "plan or table is NULL");
  if (!aligned(table, 16)) return fail(CR_ERR_ALIGNMENT, "table not 16-byte aligned");
  if (table_bytes < plan->table.size())
    return fail(CR_ERR_INVALID_ARG, "table_bytes=%zu below the plan's %zu", table_bytes,
                plan->table.size());
  cudaError_t e = cudaMemcpyAsync(table, plan->table.data(), plan->table.size(),
                                  cudaMemcpyHostToDevice, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "fsdp2_plan_upload copy");
  return ok();
}

cr_status cr_fsdp2_step_planned(const cr_fsdp2_plan_t* plan, const void* table,
                                const cr_adamw_cfg* cfg, cr_stream_t stream) {
  if (!plan || !table) return fail(CR_ERR_INVALID_ARG, "plan or table is NULL");
  if (!aligned(table, 16)) return fail(CR_ERR_ALIGNMENT, "table not 16-byte aligned");
  cr_status st = check_adam_cfg(cfg);
  if (st) return st;
  Fsdp2TableArgs a;
  memset(&a, 0, sizeof(a));
  a.table = static_cast<const unsigned char*>(table);
  a.p_off = plan->p_off;
  a.ptr_off = plan->ptr_off;
  a.nparams = plan->nparams;
  a.ntiles = plan->ntiles;
  a.n = plan->n;
  a.inv_n = exact_inv_n(plan->n);
  a.a = adam_scalars(*cfg);
  cudaError_t e = launch_fsdp2_table(a, (cudaStream_t)stream);
  if (e != cudaSuccess) return cuda_fail(e, "fsdp2_step_planned launch");
  return ok();
}

void cr_fsdp2_plan_free(cr_fsdp2_plan_t* plan) { delete plan; }

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
  st = check_disjoint(spans);
  if (st) return st;
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


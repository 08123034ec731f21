// api_host.h -- host-side argument checks shared by the entry points
// (api.cu: collectives; api_buckets.cu: DDP buckets; api_optim.cu: the
// FSDP / AdamW / accumulation steps).  Inline; every TU that defines
// entry points includes it.
#pragma once

#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "cr_internal.cuh"

namespace cr {
namespace host {

// Detail of the last failure on this thread (cr_last_error).
inline thread_local char g_err[512] = "";



inline cr_status fail(cr_status st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return st;
}

inline cr_status ok() {
  g_err[0] = '\0';
  return CR_OK;
}

inline cr_status cuda_fail(cudaError_t e, const char* what) {
  return fail(CR_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e),
              cudaGetErrorString(e));
}

inline size_t esize_of(cr_dtype d) {
  switch (d) {
    case CR_F32: return 4;
    case CR_BF16: return 2;
    case CR_I32: return 4;
  }
  return 0;
}

inline bool is_float(cr_dtype d) { return d == CR_F32 || d == CR_BF16; }

// Byte interval of one buffer argument.
struct Span {
  uintptr_t a, b;  // [a, b)
  int kind;        // 0 input, 1 output
  int rank;
};

inline bool overlaps(const Span& x, const Span& y) {
  return x.a < y.b && y.a < x.b && x.a < x.b && y.a < y.b;
}

inline uint64_t chunk_lo(uint64_t count, uint64_t L, int j) {
  uint64_t a = L * (uint64_t)j;
  return a < count ? a : count;
}

inline uint64_t chunk_size(uint64_t count, uint64_t L, int j) {
  uint64_t a = chunk_lo(count, L, j);
  uint64_t b = L * (uint64_t)(j + 1);
  if (b > count) b = count;
  return b - a;
}

// p moved back by `elems` elements of `es` bytes: the address element 0 of
// a buffer would have if p is where its element `elems` sits.  Range calls
// hand kernels such addresses; the kernels only touch elements >= elems.
template <typename T>
inline T* shift_back(T* p, uint64_t elems, size_t es) {
  return reinterpret_cast<T*>(reinterpret_cast<uintptr_t>(p) - elems * es);
}

inline bool aligned(const void* p, size_t a) {
  return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

// Rejects ranks out of range and counts whose byte size overflows.
inline cr_status check_common(int nranks, size_t count, const void* arr1,
                       const void* arr2) {
  if (nranks < 1 || nranks > CR_MAX_RANKS)
    return fail(CR_ERR_INVALID_ARG, "nranks=%d outside [1, %d]", nranks, CR_MAX_RANKS);
  if (!arr1 || !arr2) return fail(CR_ERR_INVALID_ARG, "pointer array is NULL");
  if (count > (SIZE_MAX / 8)) return fail(CR_ERR_INVALID_ARG, "count=%zu too large", count);
  return CR_OK;
}

inline cr_status check_pair(cr_dtype in, cr_op op, cr_dtype out) {
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
inline cr_status check_buf(const void* p, uint64_t nelem, size_t es, const char* what, int r) {
  if (nelem == 0) return CR_OK;
  if (!p) return fail(CR_ERR_INVALID_ARG, "%s[%d] is NULL", what, r);
  if (!aligned(p, es))
    return fail(CR_ERR_ALIGNMENT, "%s[%d]=%p not aligned to %zu bytes", what, r, p, es);
  return CR_OK;
}

// No output may overlap another buffer, except the pairs allow(i, o) marks.
template <typename Allow>
inline cr_status check_overlaps(const std::vector<Span>& spans, Allow allow) {
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
inline cr_status check_disjoint(std::vector<Span> spans) {
  std::sort(spans.begin(), spans.end(), [](const Span& x, const Span& y) { return x.a < y.a; });
  for (size_t k = 1; k < spans.size(); ++k)
    if (spans[k].a < spans[k - 1].b)
      return fail(CR_ERR_INVALID_ARG, "buffer %d overlaps buffer %d", spans[k].rank,
                  spans[k - 1].rank);
  return CR_OK;
}

inline Span span_of(const void* p, uint64_t bytes, int kind, int rank) {
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

inline float exact_inv_n(int n) {
  return (n & (n - 1)) == 0 ? 1.0f / (float)n : 0.0f;
}

inline AdamScalars adam_scalars(const cr_adamw_cfg& c) {
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

inline cr_status check_adam_cfg(const cr_adamw_cfg* cfg) {
  if (!cfg) return fail(CR_ERR_INVALID_ARG, "cfg is NULL");
  if (cfg->step < 1) return fail(CR_ERR_INVALID_ARG, "cfg->step=%lld < 1", (long long)cfg->step);
  if (!(cfg->beta1 >= 0.0 && cfg->beta1 < 1.0) || !(cfg->beta2 >= 0.0 && cfg->beta2 < 1.0))
    return fail(CR_ERR_INVALID_ARG, "betas must lie in [0, 1)");
  if (!(cfg->eps >= 0.0) || !(cfg->lr >= 0.0) || !(cfg->weight_decay >= 0.0))
    return fail(CR_ERR_INVALID_ARG, "lr, eps and weight_decay must be >= 0");
  return CR_OK;
}

// The wire type of a ring whose messages may travel in low precision.
inline cr_status check_wire(cr_dtype in, cr_dtype wire, bool* bf16) {
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

}  // namespace host
}  // namespace cr

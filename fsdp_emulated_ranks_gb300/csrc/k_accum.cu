// k_accum.cu -- gradient accumulation for DDP's no_sync().
//
// "AI Infra Guide, Chapter 6", 6.2.6: inside model.no_sync() a micro-step
// only adds its gradient to the accumulated one, with no all-reduce; the
// last micro-step's backward accumulates too and then all-reduces the sum.
// k_accum does the first (acc[r] += g[r], every rank, in fp32); with
// `reduce` set it does the second in the same pass: each element's N sums
// acc[r] + g[r] are folded over the ranks in ring order (chunk j from rank
// j+1 to its owner j, as every collective here), averaged if asked, and
// written back to every rank's accumulator -- the result of accumulating
// and then all-reducing, bit for bit, without writing and re-reading the
// accumulators in between.
#include "check.cuh"
#include "cr_internal.cuh"
#include "fold.cuh"
#include "pdl.cuh"

namespace cr {

template <int GD>
__device__ __forceinline__ float grad_elem(const void* g, uint64_t e) {
  return ld_elem<GD>(g, e);
}

// 8 gradient elements at element e0 as fp32 (bf16: one 16-byte vector).
template <int GD>
__device__ __forceinline__ void grad8(const void* g, uint64_t e0, float* out) {
  if constexpr (GD == CR_BF16) {
    const uint4 v = ld16(static_cast<const uint16_t*>(g) + e0);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      out[2 * i] = bf16_lo(w[i]);
      out[2 * i + 1] = bf16_hi(w[i]);
    }
  } else {
    const float* p = static_cast<const float*>(g) + e0;
    const uint4 a = ld16(p), b = ld16(p + 4);
    out[0] = __uint_as_float(a.x), out[1] = __uint_as_float(a.y);
    out[2] = __uint_as_float(a.z), out[3] = __uint_as_float(a.w);
    out[4] = __uint_as_float(b.x), out[5] = __uint_as_float(b.y);
    out[6] = __uint_as_float(b.z), out[7] = __uint_as_float(b.w);
  }
}

template <int SW>
__device__ __forceinline__ void acc8_load(const float* p, float* out) {
  uint32_t w[8];
  if constexpr (SW == 8) {
    const Words<8> v = ldv<8>(p);
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = v.w[i];
  } else {
    const uint4 a = ld16(p), b = ld16(p + 4);
    w[0] = a.x, w[1] = a.y, w[2] = a.z, w[3] = a.w, w[4] = b.x, w[5] = b.y, w[6] = b.z, w[7] = b.w;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) out[i] = __uint_as_float(w[i]);
}

template <int SW>
__device__ __forceinline__ void acc8_store(float* p, const float* x) {
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = __float_as_uint(x[i]);
  st_words<32, SW * 4>(p, w);
}

// Element e: accumulate on every rank, then (reduce) fold in ring order.
template <int GD>
__device__ __forceinline__ void accum_elem(const AccumArgs& a, int n, uint64_t e) {
  if (!a.reduce) {
    for (int r = 0; r < n; ++r) a.acc[r][e] = __fadd_rn(a.acc[r][e], grad_elem<GD>(a.grads[r], e));
    return;
  }
  const int j = (int)fastdiv_div(a.Ld, e);
  CR_DCHECK(e < a.count && (uint64_t)j == e / a.L && j < n, kChkAccum);
  int r = (j + 1 == n) ? 0 : j + 1;
  float sum = __fadd_rn(a.acc[r][e], grad_elem<GD>(a.grads[r], e));
  for (int k = 1; k < n; ++k) {
    r = (r + 1 == n) ? 0 : r + 1;
    sum = __fadd_rn(sum, __fadd_rn(a.acc[r][e], grad_elem<GD>(a.grads[r], e)));
  }
  if (a.avg) sum = finish_avg(sum, n, a.inv_n);
  for (int q = 0; q < n; ++q) a.acc[q][e] = sum;
}

template <int GD, int NT, int SW>
__global__ void __launch_bounds__(kBlock)
    k_accum_vec(const __grid_constant__ AccumArgs a) {
  pdl_enter();
  const int n = NT > 0 ? NT : a.n;
  const uint64_t nvec = a.count / 8;
  const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  if (!a.reduce) {
    // blockIdx.y is the rank: ranks are independent without the reduce.
    const int r = blockIdx.y;
    for (uint64_t iv = tid; iv < nvec; iv += stride) {
      const uint64_t e0 = iv * 8;
      float x[8], g[8];
      acc8_load<SW>(a.acc[r] + e0, x);
      grad8<GD>(a.grads[r], e0, g);
#pragma unroll
      for (int i = 0; i < 8; ++i) x[i] = __fadd_rn(x[i], g[i]);
      acc8_store<SW>(a.acc[r] + e0, x);
    }
    const uint64_t e = nvec * 8 + tid;
    if (e < a.count) a.acc[r][e] = __fadd_rn(a.acc[r][e], grad_elem<GD>(a.grads[r], e));
    return;
  }
  for (uint64_t iv = tid; iv < nvec; iv += stride) {
    const uint64_t e0 = iv * 8;
    const uint64_t j64 = fastdiv_div(a.Ld, e0);
    if (e0 + 8 > (j64 + 1) * a.L) {  // straddles a chunk boundary
      for (int i = 0; i < 8; ++i) accum_elem<GD>(a, n, e0 + i);
      continue;
    }
    const int j = (int)j64;
    CR_DCHECK(e0 + 8 <= a.count && j64 == e0 / a.L && j < n, kChkAccum);
    int r = (j + 1 == n) ? 0 : j + 1;
    float sum[8];
#pragma unroll
    for (int k = 0; k < (NT > 0 ? NT : kMaxRanks); ++k) {
      if (NT == 0 && k >= n) break;
      float x[8], g[8];
      acc8_load<SW>(a.acc[r] + e0, x);
      grad8<GD>(a.grads[r], e0, g);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float xi = __fadd_rn(x[i], g[i]);
        sum[i] = k == 0 ? xi : __fadd_rn(sum[i], xi);
      }
      r = (r + 1 == n) ? 0 : r + 1;
    }
    if (a.avg) {
#pragma unroll
      for (int i = 0; i < 8; ++i) sum[i] = finish_avg(sum[i], n, a.inv_n);
    }
#pragma unroll 8
    for (int q = 0; q < n; ++q) acc8_store<SW>(a.acc[q] + e0, sum);
  }
  const uint64_t e = nvec * 8 + tid;
  if (e < a.count) accum_elem<GD>(a, n, e);
}

template <int GD>
__global__ void __launch_bounds__(kBlock)
    k_accum_elem(const __grid_constant__ AccumArgs a) {
  pdl_enter();
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t e = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; e < a.count; e += stride)
    accum_elem<GD>(a, a.n, e);
}

template <int GD, int SW>
static cudaError_t accum_dispatch(const AccumArgs& a, cudaStream_t s) {
  const dim3 grid(flat_grid(a.count / 8 + 1), a.reduce ? 1 : a.n);
  clear_stale_error();
  switch (a.reduce ? a.n : 0) {
    case 2: return launch_pdl(k_accum_vec<GD, 2, SW>, grid, kBlock, s, a);
    case 4: return launch_pdl(k_accum_vec<GD, 4, SW>, grid, kBlock, s, a);
    case 8: return launch_pdl(k_accum_vec<GD, 8, SW>, grid, kBlock, s, a);
    default: return launch_pdl(k_accum_vec<GD, 0, SW>, grid, kBlock, s, a);
  }
}

template <int GD>
static cudaError_t accum_by_width(const AccumArgs& a, int vw, cudaStream_t s) {
  if (vw == 32) return accum_dispatch<GD, 8>(a, s);
  if (vw == 16) return accum_dispatch<GD, 4>(a, s);
  clear_stale_error();
  return launch_pdl(k_accum_elem<GD>, dim3(flat_grid(a.count)), kBlock, s, a);
}

cudaError_t launch_accum(cr_dtype grad_dtype, const AccumArgs& a, int vw, cudaStream_t s) {
  if (a.count == 0) return cudaSuccess;
  if (grad_dtype == CR_BF16) return accum_by_width<CR_BF16>(a, vw, s);
  if (grad_dtype == CR_F32) return accum_by_width<CR_F32>(a, vw, s);
  return cudaErrorInvalidValue;
}

}  // namespace cr

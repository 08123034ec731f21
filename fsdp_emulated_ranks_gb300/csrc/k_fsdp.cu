// k_fsdp.cu -- the fused FSDP / ZeRO-3 step and the stand-alone AdamW.
//
// One pass over the flat parameter buffer does what the FSDP1 unit lifecycle
// of "Distributed Training for Large Models: Collectives, FSDP/ZeRO,
// DeviceMesh, and Multi-Dimensional Parallelism" (section 4; ZeRO-3 flow
// steps 5-6) spreads over three phases:
//   backward post-hook  reduce-scatter of the bf16 grads, fp32 partials in
//                       ring order, / N (reduce_dtype fp32, "AI Infra Guide,
//                       Chapter 6", 6.3.4);
//   optimizer step      AdamW on owner j's fp32 master/m/v shard;
//   next forward        bf16 cast and all-gather to every rank's params.
// Element e belongs to shard j = e / L, so the thread that folds e's
// gradient is the one that owns e's optimizer state: nothing is staged in
// HBM between the phases.  Per element: N bf16 grad loads, 12 B of fp32
// state read and written, N bf16 param stores -- (4N + 24) bytes.
//
// The clipped step needs the global gradient norm before any update, so it
// makes two passes: a sum-of-squares pass, then this one with the clip
// coefficient.  For N >= 5 the first pass parks each averaged fp32 gradient
// in two of the parameter outputs (16 bits in each) and this pass reads it
// back, (4N + 32) bytes per element in all instead of the (6N + 24) of
// folding the N gradients twice.
//
// AdamW uses only correctly rounded fp32 operations (__fmul_rn & co. are
// never contracted into FMAs), in the order of the textbook decoupled-
// weight-decay rule stated in include/cr.h.
#include "check.cuh"
#include "cr_internal.cuh"
#include "fold.cuh"
#include "pdl.cuh"
#include "fsdp_body.cuh"

namespace cr {

// Clip coefficient of clip_grad_norm_, computed once per step by one warp:
// the partial sums are added in a fixed order (lane-strided, then a fixed
// shuffle tree), so the norm is reproducible run to run.
__global__ void k_clip_coef(const double* partials, int nparts, double max_norm, float* coef,
                            float* norm_out) {
  pdl_enter();
  double t = 0.0;
  for (int i = threadIdx.x; i < nparts; i += 32) t += partials[i];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) t += __shfl_down_sync(0xffffffffu, t, off);
  if (threadIdx.x == 0) {
    const double norm = sqrt(t);
    double c = max_norm / (norm + 1e-6);
    if (c > 1.0) c = 1.0;
    *coef = (float)c;
    if (norm_out) *norm_out = (float)norm;
  }
}

cudaError_t launch_clip_coef(const double* partials, int nparts, double max_norm, float* coef,
                             float* norm_out, cudaStream_t s) {
  clear_stale_error();
  return launch_pdl(k_clip_coef, dim3(1), 32, s, partials, nparts, max_norm, coef, norm_out);
}

__device__ __forceinline__ float clip_coef(const FsdpArgs& a) {
  return a.coef ? __ldg(a.coef) : 1.0f;
}

// Sum of squares of the averaged fp32 gradient, one fp64 partial per CTA
// (fp64 per thread and across threads, fp32 within batches of 8 squares).
// STASH: also park every averaged gradient in params[0] / params[1] (low /
// high 16 bits) for the update pass -- 4 bytes written per element so that
// the update pass reads 4 bytes instead of the 2N of a second fold.
// STRADDLE: L is not a multiple of 8, so a vector may straddle two shards.
template <int NT, bool VEC, bool STASH = false, bool STRADDLE = false>
__global__ void __launch_bounds__(kBlock)
    k_fsdp_sumsq(const __grid_constant__ FsdpArgs a, double* partials) {
  __shared__ double s_warp[kBlock / 32];
  pdl_enter();
  const int n = NT > 0 ? NT : a.n;
  const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  double t = 0.0;
  uint64_t e_elem = 0;  // first element the element-wise loop covers
  if constexpr (VEC) {
    const uint64_t nvec = a.count / 8;
    for (uint64_t iv = tid; iv < nvec; iv += stride) {
      const uint64_t e0 = iv * 8;
      const uint64_t j64 = fastdiv_div(a.Ld, e0);
      if (STRADDLE && e0 + 8 > (j64 + 1) * a.L) {
        // the vector straddles two shards (L not a multiple of 8): each
        // element in its own shard's fold order
        for (int i = 0; i < 8; ++i) {
          const uint64_t e = e0 + i;
          const float gf =
              finish_avg(fold_elem<CR_BF16>(a.grads, n, (int)fastdiv_div(a.Ld, e), e), n, a.inv_n);
          if constexpr (STASH) stash_put(a.params, e, gf);
          t += (double)gf * (double)gf;
        }
        continue;
      }
      float g[8];
      fold_vec16<CR_BF16, NT>(a.grads, n, (int)j64, e0 * 2, g);
      // Eight squares summed in fp32, the batch added in fp64: GB300's fp64
      // rate is far below its fp32 rate, and the norm only needs ~1e-7.
      float s8 = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        g[i] = finish_avg(g[i], n, a.inv_n);
        s8 = fmaf(g[i], g[i], s8);
      }
      t += (double)s8;
      if constexpr (STASH) {
        uint32_t lo[4], hi[4];
        stash_split(g, lo, hi);
        st16(static_cast<unsigned char*>(a.params[0]) + e0 * 2, make_uint4(lo[0], lo[1], lo[2], lo[3]));
        st16(static_cast<unsigned char*>(a.params[1]) + e0 * 2, make_uint4(hi[0], hi[1], hi[2], hi[3]));
      }
    }
    e_elem = nvec * 8;
  }
  for (uint64_t e = e_elem + tid; e < a.count; e += stride) {
    const float gf = finish_avg(fold_elem<CR_BF16>(a.grads, n, (int)fastdiv_div(a.Ld, e), e), n, a.inv_n);
    if constexpr (STASH) stash_put(a.params, e, gf);
    const double gi = gf;
    t += gi * gi;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) t += __shfl_down_sync(0xffffffffu, t, off);
  if ((threadIdx.x & 31) == 0) s_warp[threadIdx.x >> 5] = t;
  __syncthreads();
  if (threadIdx.x == 0) {
    double b = 0.0;
    for (int w = 0; w < kBlock / 32; ++w) b += s_warp[w];
    partials[blockIdx.x] = b;
  }
}

// Vector path: 8 elements (one 16-byte bf16 vector per rank) per thread and
// iteration; SW = 8 moves the fp32 state in 32-byte accesses, SW = 4 in
// 16-byte ones, SW = 1 element by element (a shard length that is not a
// multiple of 8).  The body of k_fsdp_vec and k_fsdp_vec4, which differ
// only in their launch bounds.
template <int NT, bool STASH>
__device__ __forceinline__ void fsdp_one(const FsdpArgs& a, int n, float coef, uint64_t e) {
  CR_DCHECK(e >= a.begin && e < a.end && fastdiv_div(a.Ld, e) == e / a.L && e / a.L < (uint64_t)n,
            kChkFsdp);
  fsdp_element<STASH>(a.grads, a.params, a.master, a.m, a.v, n, a.L, a.Ld, a.inv_n, a.a, coef, e);
}

template <int NT, int SW, bool STASH>
__device__ __forceinline__ void fsdp_range(const FsdpArgs& a) {
  pdl_enter();
  const int n = NT > 0 ? NT : a.n;
  const float coef = clip_coef(a);
  const uint64_t vbeg = (a.begin + 7) / 8, vend = a.end / 8;
  const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t iv = vbeg + tid; iv < vend; iv += stride) {
    if constexpr (SW == 1) {
      // L off the vector grid: a vector may straddle two shards, and then
      // each element takes its own shard's fold order and state
      const uint64_t e0 = iv * 8;
      if (e0 + 8 > (fastdiv_div(a.Ld, e0) + 1) * a.L) {
        for (int i = 0; i < 8; ++i) fsdp_one<NT, STASH>(a, n, coef, e0 + i);
        continue;
      }
    }
    // the 8 elements lie in one shard, inside that shard's length
    CR_DCHECK(fastdiv_div(a.Ld, iv * 8) == iv * 8 / a.L && iv * 8 / a.L < (uint64_t)n &&
                  iv * 8 % a.L + 8 <= a.L && iv * 8 + 8 <= a.end,
              kChkFsdp);
    fsdp_vector<NT, SW, STASH>(a.grads, a.params, a.master, a.m, a.v, n, a.L, a.Ld, a.inv_n, a.a,
                               coef, iv * 8);
  }
  // Ragged ends: fewer than 8 elements before the first and after the last
  // whole vector of the range (threads 0-7 and 8-15).
  if (vbeg <= vend) {
    const uint64_t head = vbeg * 8 - a.begin, tail = a.end - vend * 8;
    if (tid < head) fsdp_one<NT, STASH>(a, n, coef, a.begin + tid);
    if (tid >= 8 && tid - 8 < tail) fsdp_one<NT, STASH>(a, n, coef, vend * 8 + (tid - 8));
  } else if (tid < a.end - a.begin) {
    fsdp_one<NT, STASH>(a, n, coef, a.begin + tid);
  }
}

// A runtime rank count: built for 3 CTAs per SM (80 registers, 32-72 bytes
// of spills).  At N = 16 and 2^27 parameters GB300 runs it at 6,600 GB/s,
// against 6,190 under the 4-CTA bound (216-260 bytes of spills) and 5,710
// with default bounds (87-89 registers, 2 CTAs per SM).
template <int NT, int SW, bool STASH = false>
__global__ void __launch_bounds__(kBlock, 3) k_fsdp_vec(const __grid_constant__ FsdpArgs a) {
  fsdp_range<NT, SW, STASH>(a);
}

// A compile-time rank count, registers capped for 4 resident CTAs per SM
// (63 per thread, no spills), which GB300 runs about 1 % faster than the
// 3 CTAs that 70 registers allow.
template <int NT, int SW, bool STASH = false>
__global__ void __launch_bounds__(kBlock, 4) k_fsdp_vec4(const __grid_constant__ FsdpArgs a) {
  fsdp_range<NT, SW, STASH>(a);
}

__global__ void __launch_bounds__(kBlock)
    k_fsdp_elem(const __grid_constant__ FsdpArgs a) {
  pdl_enter();
  const float coef = clip_coef(a);
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t e = a.begin + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; e < a.end;
       e += stride) {
    CR_DCHECK(fastdiv_div(a.Ld, e) == e / a.L && e / a.L < (uint64_t)a.n, kChkFsdp);
    fsdp_element(a.grads, a.params, a.master, a.m, a.v, a.n, a.L, a.Ld, a.inv_n, a.a, coef, e);
  }
}

// ---- stand-alone AdamW on an fp32 shard ------------------------------------

__global__ void __launch_bounds__(kBlock)
    k_adamw_vec(const __grid_constant__ AdamArgs a) {
  pdl_enter();
  const uint64_t nvec = a.n / 4;
  const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t iv = tid; iv < nvec; iv += stride) {
    const uint64_t e0 = iv * 4;
    const uint4 p = ld16(a.master + e0), m = ld16(a.m + e0), v = ld16(a.v + e0);
    const uint4 g = ld16(a.g + e0);
    const uint32_t pw[4] = {p.x, p.y, p.z, p.w}, mw[4] = {m.x, m.y, m.z, m.w};
    const uint32_t vw[4] = {v.x, v.y, v.z, v.w}, gw[4] = {g.x, g.y, g.z, g.w};
    uint32_t po[4], mo[4], vo[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const AdamOut o = adamw_elem(__uint_as_float(pw[i]), __uint_as_float(mw[i]),
                                   __uint_as_float(vw[i]), __uint_as_float(gw[i]), a.a);
      po[i] = __float_as_uint(o.p);
      mo[i] = __float_as_uint(o.m);
      vo[i] = __float_as_uint(o.v);
    }
    st16(a.master + e0, make_uint4(po[0], po[1], po[2], po[3]));
    st16(a.m + e0, make_uint4(mo[0], mo[1], mo[2], mo[3]));
    st16(a.v + e0, make_uint4(vo[0], vo[1], vo[2], vo[3]));
    if (a.param_bf16) {
      const uint32_t w[2] = {pack_bf16x2(__uint_as_float(po[0]), __uint_as_float(po[1])),
                             pack_bf16x2(__uint_as_float(po[2]), __uint_as_float(po[3]))};
      st_words<8, 16>(static_cast<unsigned char*>(a.param_bf16) + e0 * 2, w);
    }
  }
  const uint64_t e = nvec * 4 + tid;
  if (e < a.n) {
    const AdamOut o = adamw_elem(a.master[e], a.m[e], a.v[e], a.g[e], a.a);
    a.master[e] = o.p;
    a.m[e] = o.m;
    a.v[e] = o.v;
    if (a.param_bf16) st_elem<CR_BF16>(a.param_bf16, e, o.p);
  }
}

__global__ void __launch_bounds__(kBlock)
    k_adamw_elem(const __grid_constant__ AdamArgs a) {
  pdl_enter();
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t e = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; e < a.n;
       e += stride) {
    const AdamOut o = adamw_elem(a.master[e], a.m[e], a.v[e], a.g[e], a.a);
    a.master[e] = o.p;
    a.m[e] = o.m;
    a.v[e] = o.v;
    if (a.param_bf16) st_elem<CR_BF16>(a.param_bf16, e, o.p);
  }
}

template <typename K, typename A>
static cudaError_t launch_flat(K kernel, const A& args, uint64_t threads, cudaStream_t s) {
  clear_stale_error();
  return launch_pdl(kernel, dim3(flat_grid(threads)), kBlock, s, args);
}

template <int SW>
static cudaError_t fsdp_dispatch(const FsdpArgs& a, cudaStream_t s) {
  const uint64_t threads = (a.end - a.begin) / 8 + 16;
  // The update pass of the parked gradient folds nothing, so one runtime-N
  // build serves every N (the 4-CTA bound would spill here).
  if (a.stash) return launch_flat(k_fsdp_vec<0, SW, true>, a, threads, s);
  switch (a.n) {
    case 2: return launch_flat(k_fsdp_vec4<2, SW>, a, threads, s);
    case 3: return launch_flat(k_fsdp_vec4<3, SW>, a, threads, s);
    case 4: return launch_flat(k_fsdp_vec4<4, SW>, a, threads, s);
    case 5: return launch_flat(k_fsdp_vec4<5, SW>, a, threads, s);
    case 6: return launch_flat(k_fsdp_vec4<6, SW>, a, threads, s);
    case 7: return launch_flat(k_fsdp_vec4<7, SW>, a, threads, s);
    case 8: return launch_flat(k_fsdp_vec4<8, SW>, a, threads, s);
    default: return launch_flat(k_fsdp_vec<0, SW>, a, threads, s);
  }
}

cudaError_t launch_fsdp(const FsdpArgs& a, int vw, cudaStream_t s) {
  if (vw == 32) return fsdp_dispatch<8>(a, s);
  if (vw == 16) return fsdp_dispatch<4>(a, s);
  if (vw == 1) return fsdp_dispatch<1>(a, s);
  return launch_flat(k_fsdp_elem, a, a.end - a.begin, s);
}

cudaError_t launch_adamw(const AdamArgs& a, bool vec, cudaStream_t s) {
  return vec ? launch_flat(k_adamw_vec, a, a.n / 4 + 1, s)
             : launch_flat(k_adamw_elem, a, a.n, s);
}

template <int NT, bool VEC, bool STASH = false, bool STRADDLE = false>
static cudaError_t sumsq_launch(const FsdpArgs& a, double* partials, int max_parts,
                                int* nparts, cudaStream_t s) {
  const uint64_t threads = VEC ? a.count / 8 + 1 : a.count;
  int grid = 0;
  cudaError_t err = persistent_grid(
      reinterpret_cast<const void*>(k_fsdp_sumsq<NT, VEC, STASH, STRADDLE>), threads, &grid);
  if (err != cudaSuccess) return err;
  if (grid > max_parts) grid = max_parts;
  *nparts = grid;
  clear_stale_error();
  return launch_pdl(k_fsdp_sumsq<NT, VEC, STASH, STRADDLE>, dim3(grid), kBlock, s, a, partials);
}

cudaError_t launch_fsdp_sumsq(const FsdpArgs& a, bool vec, double* partials,
                              int max_parts, int* nparts, cudaStream_t s) {
  if (!vec) return sumsq_launch<0, false>(a, partials, max_parts, nparts, s);
  if (a.L % 8 != 0) {  // vectors may straddle shards: the runtime-N builds
    return a.stash ? sumsq_launch<0, true, true, true>(a, partials, max_parts, nparts, s)
                   : sumsq_launch<0, true, false, true>(a, partials, max_parts, nparts, s);
  }
  if (a.stash) {
    switch (a.n) {
      case 5: return sumsq_launch<5, true, true>(a, partials, max_parts, nparts, s);
      case 6: return sumsq_launch<6, true, true>(a, partials, max_parts, nparts, s);
      case 7: return sumsq_launch<7, true, true>(a, partials, max_parts, nparts, s);
      case 8: return sumsq_launch<8, true, true>(a, partials, max_parts, nparts, s);
      default: return sumsq_launch<0, true, true>(a, partials, max_parts, nparts, s);
    }
  }
  switch (a.n) {
    case 2: return sumsq_launch<2, true>(a, partials, max_parts, nparts, s);
    case 3: return sumsq_launch<3, true>(a, partials, max_parts, nparts, s);
    case 4: return sumsq_launch<4, true>(a, partials, max_parts, nparts, s);
    case 8: return sumsq_launch<8, true>(a, partials, max_parts, nparts, s);
    default: return sumsq_launch<0, true>(a, partials, max_parts, nparts, s);
  }
}


}  // namespace cr

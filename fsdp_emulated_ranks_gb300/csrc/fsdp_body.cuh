// fsdp_body.cuh -- per-vector and per-element work of the fused FSDP step,
// shared by the flat-buffer kernel (k_fsdp.cu) and the per-parameter FSDP2
// kernel (k_fsdp2.cu).
#pragma once

#include "cr_internal.cuh"
#include "fold.cuh"

namespace cr {

struct AdamOut {
  float p, m, v;
};

__device__ __forceinline__ AdamOut adamw_elem(float p, float m, float v,
                                              float g, const AdamScalars& a) {
  AdamOut o;
  const float pd = __fmul_rn(p, a.decay);
  o.m = __fadd_rn(__fmul_rn(a.b1, m), __fmul_rn(a.omb1, g));
  o.v = __fadd_rn(__fmul_rn(a.b2, v), __fmul_rn(a.omb2, __fmul_rn(g, g)));
  const float mh = __fdiv_rn(o.m, a.bc1);
  const float vh = __fdiv_rn(o.v, a.bc2);
  const float denom = __fadd_rn(__fsqrt_rn(vh), a.eps);
  o.p = __fsub_rn(pd, __fmul_rn(a.lr, __fdiv_rn(mh, denom)));
  return o;
}

// 8 fp32 state words at p: one 32-byte access (SW == 8), two 16-byte ones
// (SW == 4), or eight 4-byte ones (SW == 1: a shard length off the vector
// grid puts the state of a vector at any 4-byte offset).
template <int SW>
__device__ __forceinline__ void ld_state8(const float* p, uint32_t* w) {
  if constexpr (SW == 8) {
    const Words<8> v = ldv<8>(p);
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = v.w[i];
  } else if constexpr (SW == 4) {
    const uint4 a = ld16(p), b = ld16(p + 4);
    w[0] = a.x, w[1] = a.y, w[2] = a.z, w[3] = a.w;
    w[4] = b.x, w[5] = b.y, w[6] = b.z, w[7] = b.w;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = __float_as_uint(p[i]);
  }
}
template <int SW>
__device__ __forceinline__ void st_state8(float* p, const uint32_t* w) {
  if constexpr (SW == 8) {
    st32(p, w);
  } else if constexpr (SW == 4) {
    st16(p, make_uint4(w[0], w[1], w[2], w[3]));
    st16(p + 4, make_uint4(w[4], w[5], w[6], w[7]));
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i) p[i] = __uint_as_float(w[i]);
  }
}

// The master/m/v stores of one 8-element vector whose shard offset is off
// the vector grid (SW == 1).  Each thread's 8 floats sit in one 32-byte
// sector at most two sectors apart from its neighbour's, so plain stores
// would split every warp store across 32 sectors.  When the whole warp
// holds consecutive vectors of one shard, each array goes through shared
// memory and the warp writes 32 consecutive floats per store instruction;
// otherwise each thread stores its own elements.
__device__ __forceinline__ void st_state3_offgrid(float* mp, float* mm, float* mv,
                                                  const uint32_t* po, const uint32_t* mo,
                                                  const uint32_t* vo, int j, uint64_t e0) {
  __shared__ __align__(16) uint32_t s_st[kBlock / 32][32 * 8];
  const unsigned act = __activemask();
  const int lane = threadIdx.x & 31;
  bool whole = act == 0xffffffffu;
  if (whole) {
    const uint64_t e_first = __shfl_sync(0xffffffffu, e0, 0);
    const int j_first = __shfl_sync(0xffffffffu, j, 0);
    whole = __all_sync(0xffffffffu, j == j_first && e0 == e_first + 8ull * lane);
  }
  float* const dst[3] = {mp, mm, mv};
  const uint32_t* const src[3] = {po, mo, vo};
  if (!whole) {
#pragma unroll
    for (int t = 0; t < 3; ++t) {
#pragma unroll
      for (int i = 0; i < 8; ++i) dst[t][i] = __uint_as_float(src[t][i]);
    }
    return;
  }
  uint32_t* buf = s_st[threadIdx.x >> 5];
#pragma unroll
  for (int t = 0; t < 3; ++t) {
    uint4* bv = reinterpret_cast<uint4*>(buf) + lane * 2;
    bv[0] = make_uint4(src[t][0], src[t][1], src[t][2], src[t][3]);
    bv[1] = make_uint4(src[t][4], src[t][5], src[t][6], src[t][7]);
    __syncwarp();
    float* d0 = reinterpret_cast<float*>(
        __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(dst[t]), 0));
#pragma unroll
    for (int i = 0; i < 8; ++i) d0[i * 32 + lane] = __uint_as_float(buf[i * 32 + lane]);
    __syncwarp();  // the buffer is reused for the next array
  }
}

// The averaged fp32 gradient parked in two bf16 parameter buffers: its low
// half in `lo`, its high half in `hi`, at the element's own index.
__device__ __forceinline__ void stash_split(const float* g, uint32_t* lo, uint32_t* hi) {
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    lo[i] = __byte_perm(__float_as_uint(g[2 * i]), __float_as_uint(g[2 * i + 1]), 0x5410);
    hi[i] = __byte_perm(__float_as_uint(g[2 * i]), __float_as_uint(g[2 * i + 1]), 0x7632);
  }
}
__device__ __forceinline__ void stash_join(uint4 lo, uint4 hi, float* g) {
  const uint32_t l[4] = {lo.x, lo.y, lo.z, lo.w}, h[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    g[2 * i] = __uint_as_float(__byte_perm(l[i], h[i], 0x5410));
    g[2 * i + 1] = __uint_as_float(__byte_perm(l[i], h[i], 0x7632));
  }
}
__device__ __forceinline__ void stash_put(void* const* params, uint64_t e, float g) {
  static_cast<uint16_t*>(params[0])[e] = (uint16_t)(__float_as_uint(g) & 0xffffu);
  static_cast<uint16_t*>(params[1])[e] = (uint16_t)(__float_as_uint(g) >> 16);
}
__device__ __forceinline__ float stash_get(void* const* params, uint64_t e) {
  const uint32_t lo = static_cast<const uint16_t*>(params[0])[e];
  const uint32_t hi = static_cast<const uint16_t*>(params[1])[e];
  return __uint_as_float(lo | (hi << 16));
}

// Element e0..e0+7 of a flat buffer (e0 % 8 == 0; the vector lies inside
// chunk j = e0 / L, i.e. L % 8 == 0): fold the n bf16 gradients in ring
// order, average, clip, AdamW on owner j's fp32 state, bf16 cast, write
// the parameter to every rank.  SW = 8: 32-byte state accesses.  STASH:
// the averaged gradient is read back from params[0] / params[1], where the
// sum-of-squares pass of the clipped step parked it, instead of folded.
template <int NT, int SW, bool STASH = false>
__device__ __forceinline__ void fsdp_vector(const void* const* grads, void* const* params,
                                            float* const* master, float* const* m,
                                            float* const* v, int n, uint64_t L,
                                            const FastDiv& Ld, float inv_n,
                                            const AdamScalars& as, float coef, uint64_t e0) {
  const uint64_t j64 = fastdiv_div(Ld, e0);
  const int j = (int)j64;
  const uint64_t k = e0 - j64 * L;  // offset inside shard j
  float g[8];
  if constexpr (STASH) {
    stash_join(ld16(static_cast<const unsigned char*>(params[0]) + e0 * 2),
               ld16(static_cast<const unsigned char*>(params[1]) + e0 * 2), g);
  } else {
    fold_vec16<CR_BF16, NT>(grads, n, j, e0 * 2, g);
#pragma unroll
    for (int i = 0; i < 8; ++i) g[i] = finish_avg(g[i], n, inv_n);
  }
  float* mp = master[j] + k;
  float* mm = m[j] + k;
  float* mv = v[j] + k;
  uint32_t pw[8], mw[8], vw[8];
  ld_state8<SW>(mp, pw);
  ld_state8<SW>(mm, mw);
  ld_state8<SW>(mv, vw);
  uint32_t po[8], mo[8], vo[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float gi = __fmul_rn(g[i], coef);
    const AdamOut o = adamw_elem(__uint_as_float(pw[i]), __uint_as_float(mw[i]),
                                 __uint_as_float(vw[i]), gi, as);
    po[i] = __float_as_uint(o.p);
    mo[i] = __float_as_uint(o.m);
    vo[i] = __float_as_uint(o.v);
  }
  if constexpr (SW == 1) {
    st_state3_offgrid(mp, mm, mv, po, mo, vo, j, e0);
  } else {
    st_state8<SW>(mp, po);
    st_state8<SW>(mm, mo);
    st_state8<SW>(mv, vo);
  }
  const uint4 pb = make_uint4(pack_bf16x2(__uint_as_float(po[0]), __uint_as_float(po[1])),
                              pack_bf16x2(__uint_as_float(po[2]), __uint_as_float(po[3])),
                              pack_bf16x2(__uint_as_float(po[4]), __uint_as_float(po[5])),
                              pack_bf16x2(__uint_as_float(po[6]), __uint_as_float(po[7])));
#pragma unroll 8
  for (int r = 0; r < n; ++r) st16(static_cast<unsigned char*>(params[r]) + e0 * 2, pb);
}

// The same for one element e (any alignment, any chunk).
template <bool STASH = false>
__device__ __forceinline__ void fsdp_element(const void* const* grads, void* const* params,
                                             float* const* master, float* const* m,
                                             float* const* v, int n, uint64_t L,
                                             const FastDiv& Ld, float inv_n,
                                             const AdamScalars& as, float coef, uint64_t e) {
  const uint64_t j64 = fastdiv_div(Ld, e);
  const int j = (int)j64;
  const uint64_t k = e - j64 * L;
  const float gavg = STASH ? stash_get(params, e)
                           : finish_avg(fold_elem<CR_BF16>(grads, n, j, e), n, inv_n);
  const float gi = __fmul_rn(gavg, coef);
  const AdamOut o = adamw_elem(master[j][k], m[j][k], v[j][k], gi, as);
  master[j][k] = o.p;
  m[j][k] = o.m;
  v[j][k] = o.v;
  for (int r = 0; r < n; ++r) st_elem<CR_BF16>(params[r], e, o.p);
}

}  // namespace cr

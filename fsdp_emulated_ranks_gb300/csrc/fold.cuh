// fold.cuh -- device building blocks of the ring-ordered reduction.
//
// The ring reduce-scatter of the distributed-training tutorial (section 2,
// Reduce-Scatter, N=4 schedule) sends chunk j's partial from rank j+1 around
// the ring to its owner j, each hop adding the receiver's contribution.  With
// every rank's buffer in one GPU's HBM the hops collapse into one thread
// that loads element e of every rank and adds them in that same order:
//     acc = x[(j+1)%N][e]; acc += x[(j+2)%N][e]; ...; acc += x[j][e]
// so the result equals the ring's bit for bit.  Partials are fp32 for fp32
// and bf16 inputs, uint32 (two's-complement wrap) for int32.
#pragma once

#include <type_traits>

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "cr.h"
#include "cr_internal.cuh"

namespace cr {

template <int D> struct Elem;
template <> struct Elem<CR_F32> {
  using Acc = float;
  static constexpr int kSize = 4;
};
template <> struct Elem<CR_BF16> {
  using Acc = float;
  static constexpr int kSize = 2;
};
template <> struct Elem<CR_I32> {
  using Acc = uint32_t;
  static constexpr int kSize = 4;
};

// ---- global memory access ------------------------------------------------
// Every byte is touched once per call, so loads and stores bypass L1
// (16-byte: cache-streaming .cs; 32-byte: .L1::no_allocate).  They are
// ordinary coherent accesses (not the read-only path) because in-place
// calls write buffers the same kernel reads.  Two widths: 16-byte
// (.v4.u32) and, where the buffers are 32-byte aligned, 32-byte accesses
// (.v8.u32, sm_100 and newer), which halve the memory instructions and
// measurably raise DRAM efficiency.

__device__ __forceinline__ uint4 ld16(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st16(void* p, uint4 v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}

template <int NW>
struct Words {
  uint32_t w[NW];
};

template <int NW>
__device__ __forceinline__ Words<NW> ldv(const void* p) {
  Words<NW> r;
  if constexpr (NW == 4) {
    const uint4 v = ld16(p);
    r.w[0] = v.x, r.w[1] = v.y, r.w[2] = v.z, r.w[3] = v.w;
  } else {
    static_assert(NW == 8, "vector width");
    asm volatile("ld.global.L1::no_allocate.v8.u32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]),
                   "=r"(r.w[5]), "=r"(r.w[6]), "=r"(r.w[7])
                 : "l"(p));
  }
  return r;
}

__device__ __forceinline__ void st32(void* p, const uint32_t* w) {
  asm volatile("st.global.L1::no_allocate.v8.u32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
               :: "l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]),
                  "r"(w[6]), "r"(w[7])
               : "memory");
}

// Store BYTES = 8, 16, 32 or 64 bytes of words at p, which is known to be
// ALIGN-byte aligned (16 or 32): 32-byte stores are used only when ALIGN
// is 32, otherwise the bytes go out as 16-byte stores.
template <int BYTES, int ALIGN>
__device__ __forceinline__ void st_words(void* p, const uint32_t* w) {
  static_assert(ALIGN == 16 || ALIGN == 32, "store alignment");
  unsigned char* b = static_cast<unsigned char*>(p);
  if constexpr (BYTES == 8) {
    __stcs(reinterpret_cast<uint2*>(p), make_uint2(w[0], w[1]));
  } else if constexpr (BYTES == 16) {
    st16(p, make_uint4(w[0], w[1], w[2], w[3]));
  } else if constexpr (ALIGN == 32) {
    static_assert(BYTES == 32 || BYTES == 64, "vector store width");
    st32(b, w);
    if constexpr (BYTES == 64) st32(b + 32, w + 8);
  } else {
    static_assert(BYTES == 32 || BYTES == 64, "vector store width");
#pragma unroll
    for (int q = 0; q < BYTES / 16; ++q)
      st16(b + 16 * q, make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]));
  }
}

// ---- conversions -----------------------------------------------------------

__device__ __forceinline__ float bf16_lo(uint32_t w) {
  return __uint_as_float(w << 16);
}
__device__ __forceinline__ float bf16_hi(uint32_t w) {
  return __uint_as_float(w & 0xffff0000u);
}
// Two fp32 -> packed bf16x2, each rounded to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Elements of type D in NW 32-bit words.
template <int D, int NW>
constexpr int elems_per() {
  return NW * 4 / Elem<D>::kSize;
}

// Input words -> accumulators (first contribution of the fold).
template <int D, int NW>
__device__ __forceinline__ void acc_init(typename Elem<D>::Acc* acc, const Words<NW>& v) {
  if constexpr (D == CR_BF16) {
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      acc[2 * i] = bf16_lo(v.w[i]);
      acc[2 * i + 1] = bf16_hi(v.w[i]);
    }
  } else if constexpr (D == CR_F32) {
#pragma unroll
    for (int i = 0; i < NW; ++i) acc[i] = __uint_as_float(v.w[i]);
  } else {
#pragma unroll
    for (int i = 0; i < NW; ++i) acc[i] = v.w[i];
  }
}

// acc += input words (the next rank's contribution).
template <int D, int NW>
__device__ __forceinline__ void acc_add(typename Elem<D>::Acc* acc, const Words<NW>& v) {
  if constexpr (D == CR_BF16) {
#pragma unroll
    for (int i = 0; i < NW; ++i) {
      acc[2 * i] = __fadd_rn(acc[2 * i], bf16_lo(v.w[i]));
      acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], bf16_hi(v.w[i]));
    }
  } else if constexpr (D == CR_F32) {
#pragma unroll
    for (int i = 0; i < NW; ++i) acc[i] = __fadd_rn(acc[i], __uint_as_float(v.w[i]));
  } else {
#pragma unroll
    for (int i = 0; i < NW; ++i) acc[i] += v.w[i];
  }
}

// AVG: one fp32 division of the finished sum by n.  For a power-of-two n the
// product with the exact reciprocal is the same correctly rounded value.
__device__ __forceinline__ float finish_avg(float x, int n, float inv_n) {
  return inv_n != 0.0f ? __fmul_rn(x, inv_n) : __fdiv_rn(x, (float)n);
}

// Accumulators of VEC elements -> output words (VEC * size(DO) / 4 words).
template <int DI, int DO, int VEC>
__device__ __forceinline__ void acc_pack(const typename Elem<DI>::Acc* acc, uint32_t* w) {
  if constexpr (DO == CR_BF16) {
#pragma unroll
    for (int i = 0; i < VEC / 2; ++i) w[i] = pack_bf16x2(acc[2 * i], acc[2 * i + 1]);
  } else if constexpr (DO == CR_F32) {
#pragma unroll
    for (int i = 0; i < VEC; ++i) w[i] = __float_as_uint(acc[i]);
  } else {
#pragma unroll
    for (int i = 0; i < VEC; ++i) w[i] = acc[i];
  }
}

// Low-precision wire: the partial sum a rank forwards is rounded to bf16
// (nearest even) before the next rank adds its contribution in fp32.
__device__ __forceinline__ float wire_round(float x) {
  return __bfloat162float(__float2bfloat16_rn(x));
}

template <int D, int NW, bool WIRE>
__device__ __forceinline__ void wire_round_acc(typename Elem<D>::Acc* acc) {
  if constexpr (WIRE && D != CR_I32) {
    constexpr int VEC = elems_per<D, NW>();
#pragma unroll
    for (int i = 0; i < VEC; ++i) acc[i] = wire_round(acc[i]);
  }
}

// Ring-ordered fold of one NW-word vector at byte offset byte_off of chunk
// j.  NT > 0: the rank count is a compile-time constant and all NT loads are
// issued before the first add; NT == 0: runtime n, loads in groups of 8.
// WIRE: the partial is rounded to bf16 before every add (a bf16 wire).
template <int D, int NT, int NW, bool WIRE = false>
__device__ __forceinline__ void fold_vec(const void* const* in, int n, int j,
                                         uint64_t byte_off, typename Elem<D>::Acc* acc) {
  if constexpr (NT > 0) {
    Words<NW> v[NT];
    int r = (j + 1 == NT) ? 0 : j + 1;
#pragma unroll
    for (int k = 0; k < NT; ++k) {
      v[k] = ldv<NW>(static_cast<const unsigned char*>(in[r]) + byte_off);
      r = (r + 1 == NT) ? 0 : r + 1;
    }
    acc_init<D, NW>(acc, v[0]);
#pragma unroll
    for (int k = 1; k < NT; ++k) {
      wire_round_acc<D, NW, WIRE>(acc);
      acc_add<D, NW>(acc, v[k]);
    }
  } else {
    int r = (j + 1 == n) ? 0 : j + 1;
    for (int k0 = 0; k0 < n; k0 += 8) {
      const int cnt = min(8, n - k0);
      Words<NW> v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (k < cnt) {
          v[k] = ldv<NW>(static_cast<const unsigned char*>(in[r]) + byte_off);
          r = (r + 1 == n) ? 0 : r + 1;
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (k < cnt) {
          if (k0 == 0 && k == 0) {
            acc_init<D, NW>(acc, v[0]);
          } else {
            wire_round_acc<D, NW, WIRE>(acc);
            acc_add<D, NW>(acc, v[k]);
          }
        }
      }
    }
  }
}

// The 16-byte fold (kept for the kernels that stage 16-byte vectors).
template <int D, int NT>
__device__ __forceinline__ void fold_vec16(const void* const* in, int n, int j,
                                           uint64_t byte_off, typename Elem<D>::Acc* acc) {
  fold_vec<D, NT, 4>(in, n, j, byte_off, acc);
}

// ---- one element at a time (unaligned buffers, ragged tails) -------------

template <int D>
__device__ __forceinline__ typename Elem<D>::Acc ld_elem(const void* p,
                                                         uint64_t e) {
  if constexpr (D == CR_BF16) {
    const uint16_t b = static_cast<const uint16_t*>(p)[e];
    return __uint_as_float((uint32_t)b << 16);
  } else if constexpr (D == CR_F32) {
    return static_cast<const float*>(p)[e];
  } else {
    return (uint32_t)static_cast<const int32_t*>(p)[e];
  }
}

template <int D>
__device__ __forceinline__ void st_elem(void* p, uint64_t e,
                                        typename Elem<D>::Acc x) {
  if constexpr (D == CR_BF16) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    static_cast<uint16_t*>(p)[e] = *reinterpret_cast<uint16_t*>(&h);
  } else if constexpr (D == CR_F32) {
    static_cast<float*>(p)[e] = x;
  } else {
    static_cast<int32_t*>(p)[e] = (int32_t)x;
  }
}

// Store of one vector's VEC results into a shard whose offsets are off the
// vector grid (the reduce-scatters' out_scalar: L or a shard pointer not a
// multiple of the vector).  Element stores straight from each thread would
// put every lane of a warp store in a different 32-byte sector.  When the
// whole warp holds VEC-element vectors that follow one another in one
// shard, the warp instead passes its 32 * VEC results through shared
// memory and writes them lane by lane, each store instruction covering 32
// consecutive elements.  Otherwise (a partial warp, a warp across a chunk
// boundary) each thread stores its own elements.  e0: the vector's first
// element in the rank buffers; k0: its offset in shard j.
template <int DI, int DO, int NW>
__device__ __forceinline__ void store_offgrid(void* out, uint64_t e0, uint64_t k0, int j,
                                                 const typename Elem<DI>::Acc* acc) {
  constexpr int VEC = elems_per<DI, NW>();
  constexpr int OB = VEC * Elem<DO>::kSize;
  static_assert(OB % 16 == 0, "whole 16-byte words per thread in the staging buffer");
  using T = typename std::conditional<DO == CR_BF16, uint16_t, uint32_t>::type;
  __shared__ __align__(16) T s_out[kBlock / 32][32 * VEC];
  const unsigned act = __activemask();
  const int lane = threadIdx.x & 31;
  bool whole = act == 0xffffffffu;
  if (whole) {
    const uint64_t e_first = __shfl_sync(0xffffffffu, e0, 0);
    const int j_first = __shfl_sync(0xffffffffu, j, 0);
    whole = __all_sync(0xffffffffu, j == j_first && e0 == e_first + (uint64_t)lane * VEC);
  }
  if (!whole) {
#pragma unroll
    for (int i = 0; i < VEC; ++i) st_elem<DO>(out, k0 + i, acc[i]);
    return;
  }
  uint32_t w[OB / 4];
  acc_pack<DI, DO, VEC>(acc, w);
  T* buf = s_out[threadIdx.x >> 5];
  uint4* bv = reinterpret_cast<uint4*>(buf) + lane * (OB / 16);
#pragma unroll
  for (int q = 0; q < OB / 16; ++q) bv[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  __syncwarp();
  T* dst = static_cast<T*>(out) + __shfl_sync(0xffffffffu, k0, 0);
#pragma unroll
  for (int i = 0; i < VEC; ++i) dst[i * 32 + lane] = buf[i * 32 + lane];
  __syncwarp();  // the buffer is reused by this warp's next vector
}

template <int D>
__device__ __forceinline__ typename Elem<D>::Acc acc_plus(
    typename Elem<D>::Acc a, typename Elem<D>::Acc b) {
  if constexpr (D == CR_I32) return a + b;
  else return __fadd_rn(a, b);
}

// Ring-ordered fold of element e (chunk j) over n ranks (WIRE: a bf16 wire).
template <int D, bool WIRE = false>
__device__ __forceinline__ typename Elem<D>::Acc fold_elem(
    const void* const* in, int n, int j, uint64_t e) {
  int r = (j + 1 == n) ? 0 : j + 1;
  typename Elem<D>::Acc acc = ld_elem<D>(in[r], e);
  for (int k = 1; k < n; ++k) {
    r = (r + 1 == n) ? 0 : r + 1;
    if constexpr (WIRE && D != CR_I32) acc = wire_round(acc);
    acc = acc_plus<D>(acc, ld_elem<D>(in[r], e));
  }
  return acc;
}

}  // namespace cr

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

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "cr.h"

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
// Streaming (evict-first) 128-bit loads and stores: every byte is touched
// once per call.  These are ordinary coherent accesses (not the read-only
// path) because in-place calls write buffers the same kernel reads.

__device__ __forceinline__ uint4 ld16(const void* p) {
  return __ldcs(reinterpret_cast<const uint4*>(p));
}
__device__ __forceinline__ void st16(void* p, uint4 v) {
  __stcs(reinterpret_cast<uint4*>(p), v);
}

template <int BYTES>
__device__ __forceinline__ void st_words(void* p, const uint32_t* w) {
  if constexpr (BYTES == 8) {
    __stcs(reinterpret_cast<uint2*>(p), make_uint2(w[0], w[1]));
  } else if constexpr (BYTES == 16) {
    st16(p, make_uint4(w[0], w[1], w[2], w[3]));
  } else {
    static_assert(BYTES == 32, "vector store width");
    st16(p, make_uint4(w[0], w[1], w[2], w[3]));
    st16(static_cast<unsigned char*>(p) + 16, make_uint4(w[4], w[5], w[6], w[7]));
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

// 16 input bytes -> accumulators (first contribution of the fold).
template <int D>
__device__ __forceinline__ void acc_init(typename Elem<D>::Acc* acc, uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if constexpr (D == CR_BF16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] = bf16_lo(w[i]);
      acc[2 * i + 1] = bf16_hi(w[i]);
    }
  } else if constexpr (D == CR_F32) {
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = __uint_as_float(w[i]);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = w[i];
  }
}

// acc += 16 input bytes (the next rank's contribution).
template <int D>
__device__ __forceinline__ void acc_add(typename Elem<D>::Acc* acc, uint4 v) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  if constexpr (D == CR_BF16) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      acc[2 * i] = __fadd_rn(acc[2 * i], bf16_lo(w[i]));
      acc[2 * i + 1] = __fadd_rn(acc[2 * i + 1], bf16_hi(w[i]));
    }
  } else if constexpr (D == CR_F32) {
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = __fadd_rn(acc[i], __uint_as_float(w[i]));
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] += w[i];
  }
}

// AVG: one fp32 division of the finished sum by n.  For a power-of-two n the
// product with the exact reciprocal is the same correctly rounded value.
__device__ __forceinline__ float finish_avg(float x, int n, float inv_n) {
  return inv_n != 0.0f ? __fmul_rn(x, inv_n) : __fdiv_rn(x, (float)n);
}

// Accumulators -> output words.
template <int DI, int DO>
__device__ __forceinline__ void acc_pack(const typename Elem<DI>::Acc* acc,
                                         uint32_t* w) {
  constexpr int VEC = 16 / Elem<DI>::kSize;
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

// Ring-ordered fold of one 16-byte vector at element e0 of chunk j.  NT > 0:
// the rank count is a compile-time constant and all NT loads are issued
// before the first add; NT == 0: runtime n, loads issued in groups of 8.
template <int D, int NT>
__device__ __forceinline__ void fold_vec16(const void* const* in, int n, int j,
                                           uint64_t byte_off,
                                           typename Elem<D>::Acc* acc) {
  if constexpr (NT > 0) {
    uint4 v[NT];
    int r = (j + 1 == NT) ? 0 : j + 1;
#pragma unroll
    for (int k = 0; k < NT; ++k) {
      v[k] = ld16(static_cast<const unsigned char*>(in[r]) + byte_off);
      r = (r + 1 == NT) ? 0 : r + 1;
    }
    acc_init<D>(acc, v[0]);
#pragma unroll
    for (int k = 1; k < NT; ++k) acc_add<D>(acc, v[k]);
  } else {
    int r = (j + 1 == n) ? 0 : j + 1;
    for (int k0 = 0; k0 < n; k0 += 8) {
      const int cnt = min(8, n - k0);
      uint4 v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (k < cnt) {
          v[k] = ld16(static_cast<const unsigned char*>(in[r]) + byte_off);
          r = (r + 1 == n) ? 0 : r + 1;
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        if (k < cnt) {
          if (k0 == 0 && k == 0) acc_init<D>(acc, v[0]);
          else acc_add<D>(acc, v[k]);
        }
      }
    }
  }
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

template <int D>
__device__ __forceinline__ typename Elem<D>::Acc acc_plus(
    typename Elem<D>::Acc a, typename Elem<D>::Acc b) {
  if constexpr (D == CR_I32) return a + b;
  else return __fadd_rn(a, b);
}

// Ring-ordered fold of element e (chunk j) over n ranks.
template <int D>
__device__ __forceinline__ typename Elem<D>::Acc fold_elem(
    const void* const* in, int n, int j, uint64_t e) {
  int r = (j + 1 == n) ? 0 : j + 1;
  typename Elem<D>::Acc acc = ld_elem<D>(in[r], e);
  for (int k = 1; k < n; ++k) {
    r = (r + 1 == n) ? 0 : r + 1;
    acc = acc_plus<D>(acc, ld_elem<D>(in[r], e));
  }
  return acc;
}

}  // namespace cr

// k_collectives.cu -- reduce-scatter, all-reduce and all-gather kernels.
//
// Reduce-scatter / all-reduce: k_fold_vec (k_fold_vec3 for a compile-time
// rank count with 32-byte vectors, the same body built for 3 CTAs per SM)
// reads element e of every rank buffer with 16- or 32-byte streaming
// loads, folds them in ring order
// (fold.cuh), applies the AVG / cast epilogue in registers and writes either
// shard j (reduce-scatter, [DT] section 2 Reduce-Scatter) or every rank
// buffer (all-reduce = reduce-scatter + all-gather fused, [DT] section 2
// All-Reduce).  No intermediate touches HBM: per element the kernel moves
// N input and 1 (RS) or N (AR) output elements, the algorithmic minimum.
//
// All-gather: k_gather_vec writes each shard element to every rank buffer
// at its chunk offset ([DT] section 2 All-Gather), one CTA per span and
// destination buffer; the CTAs of a span share its shard reads through L2,
// so each shard byte comes from DRAM once.
//
// [DT] = "Distributed Training for Large Models: Collectives, FSDP/ZeRO,
// DeviceMesh, and Multi-Dimensional Parallelism".
//
// Launch shape (fold): one vector per thread, as many CTAs as vectors need
// (a grid-stride loop covers any remainder).  On a GB300 this beats a
// persistent grid of resident CTAs by 5-8 %: there is no per-thread
// sequence of dependent iterations and the last wave is short.  Ragged
// ends and buffers that are not 16-byte aligned go through the
// element-wise kernels.
#include "check.cuh"
#include "cr_internal.cuh"
#include "fold.cuh"
#include "pdl.cuh"

namespace cr {

// Fold, finish and store element e (any chunk, any alignment).
template <int DI, int DO, int MODE, bool WIRE>
__device__ __forceinline__ void fold_store_elem(const FoldArgs& a, int n, uint64_t e) {
  using Acc = typename Elem<DI>::Acc;
  const int j = (int)(fastdiv_div(a.Ld, e));
  CR_DCHECK(e < a.count && (uint64_t)j == e / a.L && j < n, kChkFoldChunk);
  Acc x = fold_elem<DI, WIRE>(a.in, n, j, e);
  if constexpr (DI != CR_I32) {
    if (a.avg) x = finish_avg(x, n, a.inv_n);
  }
  if constexpr (MODE == kRS) {
    st_elem<DO>(a.out[j], e - (uint64_t)j * a.L, x);
  } else {
    for (int r = 0; r < a.n_out; ++r) st_elem<DO>(a.out[r], e, x);
  }
}

// Elements [a.begin, a.end) of every rank buffer; chunks (and so the fold
// order) are those of the whole buffer of a.count elements.  NW: 4 or 8
// words per vector (16 or 32 bytes of input).  The body of k_fold_vec and
// k_fold_vec3, which differ only in their launch bounds.
template <int DI, int DO, int MODE, int NT, int NW, bool WIRE>
__device__ __forceinline__ void fold_range(const FoldArgs& a) {
  using Acc = typename Elem<DI>::Acc;
  constexpr int IS = Elem<DI>::kSize;
  constexpr int OS = Elem<DO>::kSize;
  constexpr int VEC = elems_per<DI, NW>();
  constexpr int OB = VEC * OS;
  pdl_enter();
  const int n = NT > 0 ? NT : a.n;
  const uint64_t vbeg = (a.begin + VEC - 1) / VEC;
  const uint64_t vend = a.end / VEC;
  const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;

  for (uint64_t iv = vbeg + tid; iv < vend; iv += stride) {
    const uint64_t e0 = iv * VEC;
    const uint64_t j64 = fastdiv_div(a.Ld, e0);
    const int j = (int)j64;
    CR_DCHECK(e0 + VEC <= a.end && j64 == e0 / a.L && j < n, kChkFoldChunk);
    // A reduce-scatter with vector stores has L a multiple of VEC.
    CR_DCHECK(MODE == kAR || a.out_scalar || e0 + VEC <= (j64 + 1) * a.L, kChkFoldShard);
    if ((MODE == kAR || a.out_scalar) && e0 + VEC > (j64 + 1) * a.L) {
      // The vector straddles a chunk boundary (L % VEC != 0): each element
      // takes its own chunk's ring order.
      for (int i = 0; i < VEC; ++i) fold_store_elem<DI, DO, MODE, WIRE>(a, n, e0 + i);
      continue;
    }
    Acc acc[VEC];
    fold_vec<DI, NT, NW, WIRE>(a.in, n, j, e0 * IS, acc);
    if constexpr (DI != CR_I32) {
      if (a.avg) {
#pragma unroll
        for (int i = 0; i < VEC; ++i) acc[i] = finish_avg(acc[i], n, a.inv_n);
      }
    }
    if constexpr (MODE == kRS) {
      if (a.out_scalar) {  // the shard offset of e0 is off the vector grid
        store_offgrid<DI, DO, NW>(a.out[j], e0, e0 - j64 * a.L, j, acc);
        continue;
      }
    }
    uint32_t w[OB / 4];
    acc_pack<DI, DO, VEC>(acc, w);
    if constexpr (MODE == kRS) {
      st_words<OB, NW * 4>(static_cast<unsigned char*>(a.out[j]) + (e0 - j64 * a.L) * OS, w);
    } else {
      const int n_out = NT > 0 && NT <= 32 && a.n_out == NT ? NT : a.n_out;
#pragma unroll 8
      for (int r = 0; r < n_out; ++r)
        st_words<OB, NW * 4>(static_cast<unsigned char*>(a.out[r]) + e0 * OS, w);
    }
  }

  // Ragged ends: fewer than VEC elements before the first and after the
  // last whole vector of the range.
  if (vbeg <= vend) {
    const uint64_t head = vbeg * VEC - a.begin, tail = a.end - vend * VEC;
    if (tid < head) fold_store_elem<DI, DO, MODE, WIRE>(a, n, a.begin + tid);
    if (tid >= VEC && tid - VEC < tail) fold_store_elem<DI, DO, MODE, WIRE>(a, n, vend * VEC + (tid - VEC));
  } else if (tid < a.end - a.begin) {
    fold_store_elem<DI, DO, MODE, WIRE>(a, n, a.begin + tid);
  }
}

template <int DI, int DO, int MODE, int NT, int NW, bool WIRE>
__global__ void __launch_bounds__(kBlock) k_fold_vec(const __grid_constant__ FoldArgs a) {
  fold_range<DI, DO, MODE, NT, NW, WIRE>(a);
}

// The same kernel built for 3 resident CTAs per SM (up to 85 registers),
// for a compile-time rank count and 32-byte vectors.  Left to itself
// ptxas gives the kernel 42-48 registers and interleaves the adds with the
// N loads; at the larger budget it keeps more of them in flight, and the
// 8 x 64 MiB bf16 reduce-scatter runs 2.4 % faster on a GB300 (86.3
// against 88.5 us; the all-reduce is unchanged).  The runtime-N kernels,
// which would spill, and the 16-byte ones, which the host-memory path runs
// at 4 CTAs per SM, keep the default bounds (an explicit minimum of one
// CTA is not the same to ptxas: it raises their registers).
template <int DI, int DO, int MODE, int NT, int NW, bool WIRE>
__global__ void __launch_bounds__(kBlock, 3) k_fold_vec3(const __grid_constant__ FoldArgs a) {
  fold_range<DI, DO, MODE, NT, NW, WIRE>(a);
}

template <int DI, int DO, int MODE, bool WIRE>
__global__ void __launch_bounds__(kBlock)
    k_fold_elem(const __grid_constant__ FoldArgs a) {
  pdl_enter();
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t e = a.begin + (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; e < a.end;
       e += stride)
    fold_store_elem<DI, DO, MODE, WIRE>(a, a.n, e);
}

// ---- all-gather ----------------------------------------------------------

// Vectors per span: each CTA writes one span of one destination buffer,
// two vectors per thread.
constexpr int kGatherSpanVecs = 2 * kBlock;

// Grid (n, spans): CTA x of span (y + z * gridDim.y) writes that span of
// destination buffer x.  Blocks start x-fastest, so the n CTAs of a span
// run together and the shard data they all read comes from DRAM once and
// from L2 for the rest; each CTA writes one contiguous run into one
// buffer.  On a GB300 this is 1.7 % faster than one thread writing its
// vector to all n buffers (8 x 64 MiB bf16: 90.3 against 91.8 us),
// provided 8 CTAs stay resident per SM (32 registers).  Vectors never
// straddle a shard (L is a whole number of vectors on this path); the last
// count % VEC elements are written by the CTAs of span 0, each for its own
// destination.
template <int ES, int NW>
__global__ void __launch_bounds__(kBlock, 8)
    k_gather_vec(const __grid_constant__ GatherArgs a) {
  pdl_enter();
  constexpr int VEC = NW * 4 / ES;
  const uint64_t nvec = a.count / VEC;
  const int dest = blockIdx.x;
  const uint64_t span = (uint64_t)blockIdx.z * gridDim.y + blockIdx.y;
  const bool own_inplace = (a.inplace_mask >> dest) & 1ull;
  unsigned char* const out = static_cast<unsigned char*>(a.bufs[dest]);
  Words<NW> v[2];
  uint64_t e0[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const uint64_t iv = span * kGatherSpanVecs + (uint64_t)k * kBlock + threadIdx.x;
    e0[k] = iv < nvec ? iv * VEC : a.count;  // a.count: nothing to do
    if (e0[k] < a.count) {
      const uint64_t j64 = fastdiv_div(a.Ld, e0[k]);
      CR_DCHECK(j64 == e0[k] / a.L && j64 < (uint64_t)a.n && e0[k] + VEC <= (j64 + 1) * a.L &&
                    e0[k] + VEC <= a.count,
                kChkGather);
      if ((int)j64 == dest && own_inplace) {
        e0[k] = a.count;  // rank dest's own chunk is already in place
      } else {
        v[k] = ldv<NW>(static_cast<const unsigned char*>(a.shards[j64]) +
                       (e0[k] - j64 * a.L) * ES);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < 2; ++k)
    if (e0[k] < a.count) st_words<NW * 4, NW * 4>(out + e0[k] * ES, v[k].w);
  const uint64_t e = nvec * VEC + threadIdx.x;
  if (span == 0 && e < a.count) {
    const uint64_t j64 = fastdiv_div(a.Ld, e);
    CR_DCHECK(j64 == e / a.L && j64 < (uint64_t)a.n, kChkGather);
    if (!((int)j64 == dest && own_inplace)) {
      const unsigned char* src =
          static_cast<const unsigned char*>(a.shards[j64]) + (e - j64 * a.L) * ES;
      if constexpr (ES == 2)
        *reinterpret_cast<uint16_t*>(out + e * ES) = *reinterpret_cast<const uint16_t*>(src);
      else
        *reinterpret_cast<uint32_t*>(out + e * ES) = *reinterpret_cast<const uint32_t*>(src);
    }
  }
}

template <int ES>
__global__ void __launch_bounds__(kBlock)
    k_gather_elem(const __grid_constant__ GatherArgs a) {
  pdl_enter();
  using W = typename std::conditional<ES == 2, uint16_t, uint32_t>::type;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t e = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
       e < a.count; e += stride) {
    const uint64_t j64 = fastdiv_div(a.Ld, e);
    const int j = (int)j64;
    CR_DCHECK(j64 == e / a.L && j < a.n, kChkGather);
    const W x = static_cast<const W*>(a.shards[j])[e - j64 * a.L];
    const bool skip_own = (a.inplace_mask >> j) & 1ull;
    for (int r = 0; r < a.n; ++r) {
      if (skip_own && r == j) continue;
      static_cast<W*>(a.bufs[r])[e] = x;
    }
  }
}

// ---- launchers -------------------------------------------------------------

template <typename K, typename A>
static cudaError_t launch_flat(K kernel, const A& args, uint64_t threads, cudaStream_t s) {
  clear_stale_error();
  return launch_pdl(kernel, dim3(flat_grid(threads)), kBlock, s, args);
}

template <typename K>
static cudaError_t launch_fold_kernel(K kernel, const FoldArgs& a, uint64_t threads,
                                      cudaStream_t s) {
  unsigned grid = flat_grid(threads);
  if (a.max_ctas && grid > a.max_ctas) grid = a.max_ctas;
  clear_stale_error();
  return launch_pdl(kernel, dim3(grid), kBlock, s, a);
}

// A compile-time rank count: 32-byte vectors take the kernel built for 3
// CTAs per SM, 16-byte ones the default.
template <int DI, int DO, int MODE, int NT, int NW, bool WIRE>
static cudaError_t launch_fixed_n(const FoldArgs& a, uint64_t threads, cudaStream_t s) {
  if constexpr (NW == 8)
    return launch_fold_kernel(k_fold_vec3<DI, DO, MODE, NT, NW, WIRE>, a, threads, s);
  else
    return launch_fold_kernel(k_fold_vec<DI, DO, MODE, NT, NW, WIRE>, a, threads, s);
}

template <int DI, int DO, int MODE, int NW, bool WIRE>
static cudaError_t fold_dispatch_nw(const FoldArgs& a, cudaStream_t s) {
  constexpr int VEC = elems_per<DI, NW>();
  const uint64_t threads = (a.end - a.begin) / VEC + 2 * VEC;
  if constexpr (NW == 8) {
    // Rank counts below 8 that are not a power of two: with the rank count
    // a runtime value a thread has only its 3-7 loads in flight at 2 CTAs
    // per SM; built for the count, at 3 CTAs per SM.
    switch (a.n) {
      case 3: return launch_fixed_n<DI, DO, MODE, 3, NW, WIRE>(a, threads, s);
      case 5: return launch_fixed_n<DI, DO, MODE, 5, NW, WIRE>(a, threads, s);
      case 6: return launch_fixed_n<DI, DO, MODE, 6, NW, WIRE>(a, threads, s);
      case 7: return launch_fixed_n<DI, DO, MODE, 7, NW, WIRE>(a, threads, s);
      default: break;
    }
  }
  switch (a.n) {
    case 2: return launch_fixed_n<DI, DO, MODE, 2, NW, WIRE>(a, threads, s);
    case 4: return launch_fixed_n<DI, DO, MODE, 4, NW, WIRE>(a, threads, s);
    case 8: return launch_fixed_n<DI, DO, MODE, 8, NW, WIRE>(a, threads, s);
    default: return launch_fold_kernel(k_fold_vec<DI, DO, MODE, 0, NW, WIRE>, a, threads, s);
  }
}

template <int DI, int DO, int MODE, bool WIRE>
static cudaError_t fold_dispatch(const FoldArgs& a, int vw, cudaStream_t s) {
  if (vw == 32) return fold_dispatch_nw<DI, DO, MODE, 8, WIRE>(a, s);
  if (vw == 16) return fold_dispatch_nw<DI, DO, MODE, 4, WIRE>(a, s);
  return launch_fold_kernel(k_fold_elem<DI, DO, MODE, WIRE>, a, a.end - a.begin, s);
}

template <int MODE>
static cudaError_t fold_by_type(cr_dtype in, cr_dtype out, const FoldArgs& a,
                                int vw, cudaStream_t s) {
  if (a.wire_bf16) {
    if (in == CR_F32 && out == CR_F32) return fold_dispatch<CR_F32, CR_F32, MODE, true>(a, vw, s);
    if (in == CR_BF16 && out == CR_BF16) return fold_dispatch<CR_BF16, CR_BF16, MODE, true>(a, vw, s);
    if (in == CR_BF16 && out == CR_F32) return fold_dispatch<CR_BF16, CR_F32, MODE, true>(a, vw, s);
    return cudaErrorInvalidValue;
  }
  if (in == CR_F32 && out == CR_F32) return fold_dispatch<CR_F32, CR_F32, MODE, false>(a, vw, s);
  if (in == CR_BF16 && out == CR_BF16) return fold_dispatch<CR_BF16, CR_BF16, MODE, false>(a, vw, s);
  if (in == CR_BF16 && out == CR_F32) return fold_dispatch<CR_BF16, CR_F32, MODE, false>(a, vw, s);
  if (in == CR_I32 && out == CR_I32) return fold_dispatch<CR_I32, CR_I32, MODE, false>(a, vw, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_fold(cr_dtype in, cr_dtype out, FoldMode mode,
                        const FoldArgs& a, int vw, cudaStream_t s) {
  return mode == kRS ? fold_by_type<kRS>(in, out, a, vw, s)
                     : fold_by_type<kAR>(in, out, a, vw, s);
}

// One CTA per destination and span: grid (n, ny, nz) with ny * nz >= the
// number of spans (at least one, whose CTAs write the tail); CTAs of a
// span past the last do nothing.
template <int ES, int NW>
static cudaError_t launch_gather_vec(const GatherArgs& a, cudaStream_t s) {
  constexpr int VEC = NW * 4 / ES;
  const uint64_t nvec = a.count / VEC;
  const uint64_t nspans = nvec ? (nvec + kGatherSpanVecs - 1) / kGatherSpanVecs : 1;
  const uint64_t ny = nspans < 65535 ? nspans : 65535, nz = (nspans + ny - 1) / ny;
  if (nz > 65535) return cudaErrorInvalidValue;  // beyond 2^52 elements
  const dim3 grid((unsigned)a.n, (unsigned)ny, (unsigned)nz);
  clear_stale_error();
  return launch_pdl(k_gather_vec<ES, NW>, grid, kBlock, s, a);
}

cudaError_t launch_gather(size_t esize, const GatherArgs& a, int vw,
                          cudaStream_t s) {
  if (esize == 2) {
    if (vw == 32) return launch_gather_vec<2, 8>(a, s);
    if (vw == 16) return launch_gather_vec<2, 4>(a, s);
    return launch_flat(k_gather_elem<2>, a, a.count, s);
  }
  if (vw == 32) return launch_gather_vec<4, 8>(a, s);
  if (vw == 16) return launch_gather_vec<4, 4>(a, s);
  return launch_flat(k_gather_elem<4>, a, a.count, s);
}

}  // namespace cr

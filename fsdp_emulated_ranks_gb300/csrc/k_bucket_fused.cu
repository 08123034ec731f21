// k_bucket_fused.cu -- DDP bucket all-reduce straight on the gradient
// tensors, without packing them into bucket buffers.
//
// "AI Infra Guide, Chapter 6", 6.2.4 lets gradients alias bucket storage
// (gradient_as_bucket_view) so that no copy is made; on one GPU the same
// idea removes the pack and unpack passes entirely: element i of tensor t
// sits at bucket position p = off_t + i of bucket b = bucket(t), and is
// reduced over the ranks in the ring order of p's chunk, j = p / L_b with
// L_b = ceil(numel_b / N), exactly as the all-reduce of the packed bucket
// would reduce it.  The result, written back in place into every rank's
// tensor, is bit-identical to pack -> all-reduce -> unpack, at a third of
// the HBM traffic (N reads + N writes per element instead of three times
// that).
//
// One launch covers up to kFusedMaxTensors tensors whose N rank pointers
// (kFusedMaxPtrs in all) travel in the __grid_constant__ parameter block;
// each CTA takes one tile of kFusedTileElems elements of one tensor, in
// 32-byte vectors when all of that tensor's rank pointers allow it.
#include "check.cuh"
#include "cr_internal.cuh"
#include "fold.cuh"
#include "pdl.cuh"

namespace cr {

template <int D>
__device__ __forceinline__ void fused_elem(const FusedArgs& a, const FusedTensor& t,
                                           uint64_t i) {
  using Acc = typename Elem<D>::Acc;
  const int n = a.n;
  const int j = (int)fastdiv_div(t.Lbd, t.off + i);
  CR_DCHECK(i < t.numel && (uint64_t)j == (t.off + i) / t.Lb && j < n, kChkFused);
  int r = (j + 1 == n) ? 0 : j + 1;
  Acc acc = ld_elem<D>(a.ptrs[t.ptr0 + r], i);
  for (int k = 1; k < n; ++k) {
    r = (r + 1 == n) ? 0 : r + 1;
    acc = acc_plus<D>(acc, ld_elem<D>(a.ptrs[t.ptr0 + r], i));
  }
  if constexpr (D != CR_I32) {
    if (a.avg) acc = finish_avg(acc, n, a.inv_n);
  }
  for (int q = 0; q < n; ++q) st_elem<D>(a.ptrs[t.ptr0 + q], i, acc);
}

// Vectors of NW words over tensor elements [e_lo, e_hi) of one tile; the
// ragged end of the tensor (fewer than a vector) goes element by element.
template <int D, int NT, int NW>
__device__ __forceinline__ void fused_tile(const FusedArgs& a, const FusedTensor& t, int n,
                                           uint64_t e_lo, uint64_t e_hi) {
  using Acc = typename Elem<D>::Acc;
  constexpr int IS = Elem<D>::kSize;
  constexpr int VEC = elems_per<D, NW>();
  constexpr int OB = VEC * IS;
  const uint64_t v_hi = e_hi / VEC;  // e_lo is a multiple of VEC
  for (uint64_t iv = e_lo / VEC + threadIdx.x; iv < v_hi; iv += kBlock) {
    const uint64_t e0 = iv * VEC;
    const uint64_t p0 = t.off + e0;
    const uint64_t j64 = fastdiv_div(t.Lbd, p0);
    if (p0 + VEC > (j64 + 1) * t.Lb) {  // straddles a chunk of the bucket
      for (int q = 0; q < VEC; ++q) fused_elem<D>(a, t, e0 + q);
      continue;
    }
    CR_DCHECK(e0 + VEC <= t.numel && j64 == p0 / t.Lb && j64 < (uint64_t)n, kChkFused);
    Acc acc[VEC];
    fold_vec<D, NT, NW>(a.ptrs + t.ptr0, n, (int)j64, e0 * IS, acc);
    if constexpr (D != CR_I32) {
      if (a.avg) {
#pragma unroll
        for (int q = 0; q < VEC; ++q) acc[q] = finish_avg(acc[q], n, a.inv_n);
      }
    }
    uint32_t w[OB / 4];
    acc_pack<D, D, VEC>(acc, w);
#pragma unroll 8
    for (int q = 0; q < n; ++q)
      st_words<OB, NW * 4>(static_cast<unsigned char*>(a.ptrs[t.ptr0 + q]) + e0 * IS, w);
  }
  if (e_hi == t.numel) {
    const uint64_t i = v_hi * VEC + threadIdx.x;
    if (i < e_hi && i >= e_lo) fused_elem<D>(a, t, i);
  }
}

// The tiles of one launch (grid-strided); the body of k_bucket_fused and
// k_bucket_fused3, which differ only in their launch bounds.
template <int D, int NT>
__device__ __forceinline__ void fused_tiles(const FusedArgs& a, uint32_t ntiles) {
  pdl_launch_dependents();
  const int n = NT > 0 ? NT : a.n;
  for (uint32_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    int lo = 0, hi = a.ntens;  // tile_start[lo] <= tile < tile_start[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (a.tile_start[mid] <= tile) lo = mid;
      else hi = mid;
    }
    CR_DCHECK(lo < a.ntens && a.tile_start[lo] <= tile && tile < a.tile_start[lo + 1], kChkFused);
    const FusedTensor& t = a.t[lo];
    const uint64_t e_lo = (uint64_t)(tile - a.tile_start[lo]) * kFusedTileElems;
    const uint64_t e_hi = e_lo + kFusedTileElems < t.numel ? e_lo + kFusedTileElems : t.numel;
    if (t.vw == 32) {
      fused_tile<D, NT, 8>(a, t, n, e_lo, e_hi);
    } else if (t.vw == 16) {
      fused_tile<D, NT, 4>(a, t, n, e_lo, e_hi);
    } else {
      for (uint64_t i = e_lo + threadIdx.x; i < e_hi; i += kBlock) fused_elem<D>(a, t, i);
    }
  }
  pdl_wait_prerequisites();
}

// A runtime rank count: built for 2 CTAs per SM (126-128 registers, 128-160
// bytes of spills).  At
// N = 16 (100 tensors of the DDP workload) GB300 runs it at 6,690 GB/s,
// against 6,240 with default bounds (162-164 registers, 1 CTA per SM) and
// 5,210 when built for 3.
template <int D, int NT>
__global__ void __launch_bounds__(kBlock, 2)
    k_bucket_fused(const __grid_constant__ FusedArgs a, uint32_t ntiles) {
  fused_tiles<D, NT>(a, ntiles);
}

// The same kernel built for 3 resident CTAs per SM (64-80 registers), for a
// compile-time rank count.  As with the fold kernels, the larger register
// budget keeps more of the N loads in flight: on a GB300 the 52-bucket
// all-reduce of the DDP workload runs at 7,046 against 6,803 GB/s, the
// fused all-reduce of its 300 tensors at 6,982 against 6,752 (A/B on one
// box).  The runtime-N kernel, above, spills too much under this bound
// and is built for 2.
template <int D, int NT>
__global__ void __launch_bounds__(kBlock, 3)
    k_bucket_fused3(const __grid_constant__ FusedArgs a, uint32_t ntiles) {
  fused_tiles<D, NT>(a, ntiles);
}

template <int D>
static cudaError_t fused_dispatch(const FusedArgs& a, uint32_t ntiles, bool chained,
                                  cudaStream_t s) {
  unsigned grid = flat_grid((uint64_t)ntiles * kBlock);
  if (a.max_ctas && grid > a.max_ctas) grid = a.max_ctas;  // tiles are grid-strided
  switch (a.n) {
    case 2: return launch_chained(k_bucket_fused3<D, 2>, grid, kBlock, s, chained, a, ntiles);
    case 4: return launch_chained(k_bucket_fused3<D, 4>, grid, kBlock, s, chained, a, ntiles);
    case 8: return launch_chained(k_bucket_fused3<D, 8>, grid, kBlock, s, chained, a, ntiles);
    default: return launch_chained(k_bucket_fused<D, 0>, grid, kBlock, s, chained, a, ntiles);
  }
}

cudaError_t launch_bucket_fused(cr_dtype d, const FusedArgs& a, uint32_t ntiles, bool chained,
                                cudaStream_t s) {
  if (ntiles == 0) return cudaSuccess;
  switch (d) {
    case CR_F32: return fused_dispatch<CR_F32>(a, ntiles, chained, s);
    case CR_BF16: return fused_dispatch<CR_BF16>(a, ntiles, chained, s);
    case CR_I32: return fused_dispatch<CR_I32>(a, ntiles, chained, s);
  }
  return cudaErrorInvalidValue;
}

uint64_t fused_tile_elems(cr_dtype) { return kFusedTileElems; }

}  // namespace cr

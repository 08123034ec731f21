// k_fsdp2.cu -- the fused FSDP step for FSDP2-style per-parameter shards.
//
// FSDP2 ("Distributed Training for Large Models: Collectives, FSDP/ZeRO,
// DeviceMesh, and Multi-Dimensional Parallelism", section 4, FSDP2) keeps
// every parameter as its own DTensor with placement Shard(0): rank j owns
// rows [j*Lr, min((j+1)*Lr, dim0)), Lr = ceil(dim0 / N), so shards may be
// uneven or empty, and a parameter's gradient is reduce-scattered along the
// same row boundaries.  Per parameter this is the flat FSDP step of
// k_fsdp.cu with chunk length L = Lr * row_numel; one launch runs it for up
// to kFsdp2MaxParams parameters, whose 5N pointers travel in the
// __grid_constant__ parameter block.  Each CTA takes one tile of
// kFsdp2TileElems elements of one parameter.
#include "check.cuh"
#include "cr_internal.cuh"
#include "fold.cuh"
#include "fsdp_body.cuh"
#include "pdl.cuh"

namespace cr {

template <int NT>
__global__ void __launch_bounds__(kBlock)
    k_fsdp2(const __grid_constant__ Fsdp2Args a, uint32_t ntiles) {
  pdl_launch_dependents();
  const int n = NT > 0 ? NT : a.n;
  for (uint32_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
    int lo = 0, hi = a.nparams;  // tile_start[lo] <= tile < tile_start[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (a.tile_start[mid] <= tile) lo = mid;
      else hi = mid;
    }
    CR_DCHECK(lo < a.nparams && a.tile_start[lo] <= tile && tile < a.tile_start[lo + 1],
              kChkFsdp2);
    const Fsdp2Param& p = a.p[lo];
    const void* const* grads = a.ptrs + p.ptr0;
    void* const* params = a.ptrs + p.ptr0 + n;
    float* const* master = reinterpret_cast<float* const*>(a.ptrs + p.ptr0 + 2 * n);
    float* const* m = reinterpret_cast<float* const*>(a.ptrs + p.ptr0 + 3 * n);
    float* const* v = reinterpret_cast<float* const*>(a.ptrs + p.ptr0 + 4 * n);
    const uint64_t e_lo = (uint64_t)(tile - a.tile_start[lo]) * kFsdp2TileElems;
    const uint64_t e_hi = e_lo + kFsdp2TileElems < p.numel ? e_lo + kFsdp2TileElems : p.numel;
    if (p.vw) {
      const uint64_t v_hi = e_hi / 8;  // e_lo is a multiple of 8
      for (uint64_t iv = e_lo / 8 + threadIdx.x; iv < v_hi; iv += kBlock) {
        CR_DCHECK(fastdiv_div(p.Ld, iv * 8) == iv * 8 / p.L && iv * 8 / p.L < (uint64_t)n &&
                      iv * 8 % p.L + 8 <= p.L && iv * 8 + 8 <= p.numel,
                  kChkFsdp2);
        if (p.vw == 32)
          fsdp_vector<NT, 8>(grads, params, master, m, v, n, p.L, p.Ld, a.inv_n, a.a, 1.0f, iv * 8);
        else
          fsdp_vector<NT, 4>(grads, params, master, m, v, n, p.L, p.Ld, a.inv_n, a.a, 1.0f, iv * 8);
      }
      const uint64_t e = v_hi * 8 + threadIdx.x;  // ragged end of the parameter
      if (e_hi == p.numel && e < e_hi && e >= e_lo)
        fsdp_element(grads, params, master, m, v, n, p.L, p.Ld, a.inv_n, a.a, 1.0f, e);
    } else {
      for (uint64_t e = e_lo + threadIdx.x; e < e_hi; e += kBlock)
        fsdp_element(grads, params, master, m, v, n, p.L, p.Ld, a.inv_n, a.a, 1.0f, e);
    }
  }
  pdl_wait_prerequisites();
}

cudaError_t launch_fsdp2(const Fsdp2Args& a, uint32_t ntiles, bool chained, cudaStream_t s) {
  if (ntiles == 0) return cudaSuccess;
  const unsigned grid = flat_grid((uint64_t)ntiles * kBlock);
  switch (a.n) {
    case 2: return launch_chained(k_fsdp2<2>, grid, kBlock, s, chained, a, ntiles);
    case 4: return launch_chained(k_fsdp2<4>, grid, kBlock, s, chained, a, ntiles);
    case 8: return launch_chained(k_fsdp2<8>, grid, kBlock, s, chained, a, ntiles);
    default: return launch_chained(k_fsdp2<0>, grid, kBlock, s, chained, a, ntiles);
  }
}

}  // namespace cr

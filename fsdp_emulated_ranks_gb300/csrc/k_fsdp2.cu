// k_fsdp2.cu -- the fused FSDP step for FSDP2-style per-parameter shards.
//
// FSDP2 ("Distributed Training for Large Models: Collectives, FSDP/ZeRO,
// DeviceMesh, and Multi-Dimensional Parallelism", section 4, FSDP2) keeps
// every parameter as its own DTensor with placement Shard(0): rank j owns
// rows [j*Lr, min((j+1)*Lr, dim0)), Lr = ceil(dim0 / N), so shards may be
// uneven or empty, and a parameter's gradient is reduce-scattered along the
// same row boundaries.  Per parameter this is the flat FSDP step of
// k_fsdp.cu with chunk length L = Lr * row_numel.  Each CTA takes one tile
// of kFsdp2TileElems elements of one parameter.  Two forms:
//   k_fsdp2        up to kFsdp2MaxParams parameters per launch, their 5N
//                  pointers in the __grid_constant__ parameter block
//                  (cr_fsdp2_step: several chained launches for a model);
//   k_fsdp2_table  the parameters, tile prefix sums and pointers in a table
//                  in device memory, built once per parameter set by a plan
//                  (cr_fsdp2_step_planned: one launch for any model).
#include "check.cuh"
#include "cr_internal.cuh"
#include "fold.cuh"
#include "fsdp_body.cuh"
#include "pdl.cuh"

namespace cr {

// One tile of parameter p: elements [e_lo, min(e_lo + kFsdp2TileElems,
// numel)).  ptr holds the parameter's 5N pointers: grads[0..N),
// params[N..2N), master[2N..3N), m[3N..4N), v[4N..5N).
template <int NT>
__device__ __forceinline__ void fsdp2_tile(const Fsdp2Param& p, void* const* ptr, int n,
                                           float inv_n, const AdamScalars& as, uint64_t e_lo) {
  const void* const* grads = ptr;
  void* const* params = ptr + n;
  float* const* master = reinterpret_cast<float* const*>(ptr + 2 * n);
  float* const* m = reinterpret_cast<float* const*>(ptr + 3 * n);
  float* const* v = reinterpret_cast<float* const*>(ptr + 4 * n);
  const uint64_t e_hi = e_lo + kFsdp2TileElems < p.numel ? e_lo + kFsdp2TileElems : p.numel;
  if (p.vw) {
    const uint64_t v_hi = e_hi / 8;  // e_lo is a multiple of 8
    for (uint64_t iv = e_lo / 8 + threadIdx.x; iv < v_hi; iv += kBlock) {
      CR_DCHECK(fastdiv_div(p.Ld, iv * 8) == iv * 8 / p.L && iv * 8 / p.L < (uint64_t)n &&
                    iv * 8 % p.L + 8 <= p.L && iv * 8 + 8 <= p.numel,
                kChkFsdp2);
      if (p.vw == 32)
        fsdp_vector<NT, 8>(grads, params, master, m, v, n, p.L, p.Ld, inv_n, as, 1.0f, iv * 8);
      else
        fsdp_vector<NT, 4>(grads, params, master, m, v, n, p.L, p.Ld, inv_n, as, 1.0f, iv * 8);
    }
    const uint64_t e = v_hi * 8 + threadIdx.x;  // ragged end of the parameter
    if (e_hi == p.numel && e < e_hi && e >= e_lo)
      fsdp_element(grads, params, master, m, v, n, p.L, p.Ld, inv_n, as, 1.0f, e);
  } else {
    for (uint64_t e = e_lo + threadIdx.x; e < e_hi; e += kBlock)
      fsdp_element(grads, params, master, m, v, n, p.L, p.Ld, inv_n, as, 1.0f, e);
  }
}

// The parameter whose tiles include `tile`: tile_start[lo] <= tile <
// tile_start[lo + 1], by binary search over the nparams + 1 prefix sums.
__device__ __forceinline__ int fsdp2_param_of(const uint32_t* tile_start, int nparams,
                                              uint32_t tile) {
  int lo = 0, hi = nparams;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(tile_start + mid) <= tile) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Parameters, tiles and pointers in the __grid_constant__ parameter block
// (up to kFsdp2MaxParams parameters per launch).
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
    fsdp2_tile<NT>(p, a.ptrs + p.ptr0, n, a.inv_n, a.a,
                   (uint64_t)(tile - a.tile_start[lo]) * kFsdp2TileElems);
  }
  pdl_wait_prerequisites();
}

// The same step with the parameter table in device memory (a plan's table,
// uploaded once per parameter set): any number of parameters in one launch.
// Each CTA finds its tile's parameter in the table, stages that parameter's
// 5N pointers in shared memory and runs the tile.
// Registers capped for 4 resident CTAs per SM with a compile-time N (as
// k_fsdp2 gets without a cap) and 2 with a runtime N.
template <int NT>
__global__ void __launch_bounds__(kBlock, NT > 0 ? 4 : 2)
    k_fsdp2_table(const __grid_constant__ Fsdp2TableArgs a) {
  pdl_enter();
  __shared__ void* s_ptr[5 * kMaxRanks];
  __shared__ uint4 s_desc[3];  // the tile's Fsdp2Param (48 bytes)
  static_assert(sizeof(Fsdp2Param) == sizeof(s_desc), "descriptor size");
  const int n = NT > 0 ? NT : a.n;
  const uint32_t* tile_start = reinterpret_cast<const uint32_t*>(a.table);
  const uint4* prm = reinterpret_cast<const uint4*>(a.table + a.p_off);
  const unsigned long long* ptrs = reinterpret_cast<const unsigned long long*>(a.table + a.ptr_off);
  for (uint32_t tile = blockIdx.x; tile < a.ntiles; tile += gridDim.x) {
    const int q = fsdp2_param_of(tile_start, a.nparams, tile);
    const uint32_t t0 = __ldg(tile_start + q);
    CR_DCHECK(q < a.nparams && t0 <= tile && tile < __ldg(tile_start + q + 1), kChkFsdp2);
    __syncthreads();  // every thread is done with the previous tile's descriptor
    // the descriptor as three read-only 16-byte loads (the table places it
    // 16-byte aligned), then its 5N pointers
    if (threadIdx.x < 3) s_desc[threadIdx.x] = __ldg(prm + 3 * q + threadIdx.x);
    __syncthreads();
    const Fsdp2Param& p = *reinterpret_cast<const Fsdp2Param*>(s_desc);
    for (int t = threadIdx.x; t < 5 * n; t += kBlock)
      s_ptr[t] = reinterpret_cast<void*>(__ldg(ptrs + p.ptr0 + t));
    __syncthreads();
    fsdp2_tile<NT>(p, s_ptr, n, a.inv_n, a.a, (uint64_t)(tile - t0) * kFsdp2TileElems);
  }
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

cudaError_t launch_fsdp2_table(const Fsdp2TableArgs& a, cudaStream_t s) {
  if (a.ntiles == 0) return cudaSuccess;
  const unsigned grid = flat_grid((uint64_t)a.ntiles * kBlock);
  clear_stale_error();
  switch (a.n) {
    case 2: return launch_pdl(k_fsdp2_table<2>, dim3(grid), kBlock, s, a);
    case 4: return launch_pdl(k_fsdp2_table<4>, dim3(grid), kBlock, s, a);
    case 8: return launch_pdl(k_fsdp2_table<8>, dim3(grid), kBlock, s, a);
    default: return launch_pdl(k_fsdp2_table<0>, dim3(grid), kBlock, s, a);
  }
}

}  // namespace cr

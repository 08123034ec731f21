// k_hsdp.cu -- HSDP gradient reduction: shard inside a group, replicate
// across groups.
//
// Hybrid sharding ("AI Infra Guide, Chapter 6", 6.3.6; "Distributed
// Training" section 4, a 2-D device mesh with one sharded and one
// replicated dimension) reduces a gradient over N = R*S ranks in two
// rings: a reduce-scatter over the S ranks of each group (shard j =
// elements [jL, (j+1)L), L = ceil(count/S)), then, for every shard j, an
// all-reduce over the R groups of their shard-j partial sums.  The outer
// all-reduce has its own chunks: shard j has len_j elements, cut into R
// chunks of L2_j = ceil(len_j / R), and its chunk i is folded starting at
// group i+1.
//
// On one GPU both rings collapse into one pass.  Element e of shard j
// (offset k = e - jL, outer chunk i = k / L2_j) is
//     sum over groups g = i+1, i+2, ..., i (mod R) of
//         P_g = sum over ranks s = j+1, j+2, ..., j (mod S) of x_{g,s}[e]
// with fp32 partials (int32 wraps), each parenthesised left to right, then
// AVG (one division by N) and the output cast, stored at k in every
// group's shard j.  Each element is read once from every rank and written
// once per group: N*in + R*out bytes, the roofline bound of this pass.
#include "check.cuh"
#include "cr_internal.cuh"
#include "fold.cuh"
#include "pdl.cuh"

namespace cr {

// Outer chunk of offset k within shard j.
__device__ __forceinline__ uint64_t hsdp_outer_chunk(const HsdpArgs& a, uint64_t j, uint64_t k) {
  return j == a.jlast ? fastdiv_div(a.L2lastd, k) : fastdiv_div(a.L2d, k);
}

template <int DI, int DO>
__device__ __forceinline__ void hsdp_elem(const HsdpArgs& a, int R, int S, uint64_t e) {
  using Acc = typename Elem<DI>::Acc;
  const uint64_t j = fastdiv_div(a.Ld, e);
  const uint64_t k = e - j * a.L;
  const int i = (int)hsdp_outer_chunk(a, j, k);
  CR_DCHECK(e < a.count && j == e / a.L && j < (uint64_t)S && i < R &&
                (uint64_t)i == k / (j == a.jlast ? a.L2last : a.L2),
            kChkHsdp);
  int g = (i + 1 == R) ? 0 : i + 1;
  Acc acc = fold_elem<DI>(a.in + g * S, S, (int)j, e);
  for (int q = 1; q < R; ++q) {
    g = (g + 1 == R) ? 0 : g + 1;
    acc = acc_plus<DI>(acc, fold_elem<DI>(a.in + g * S, S, (int)j, e));
  }
  if constexpr (DI != CR_I32) {
    if (a.avg) acc = finish_avg(acc, R * S, a.inv_n);
  }
  for (int q = 0; q < R; ++q) st_elem<DO>(a.out[q * S + (int)j], k, acc);
}

// One vector of VEC elements per thread over [0, count); RT/ST > 0 fix the
// mesh shape at compile time (ST > 0 alone: the group size, so that the S
// loads of each group are issued together).  The body of k_hsdp_vec,
// k_hsdp_vec3 and k_hsdp_vec4, which differ only in their launch bounds.
template <int DI, int DO, int RT, int ST, int NW>
__device__ __forceinline__ void hsdp_range(const HsdpArgs& a) {
  using Acc = typename Elem<DI>::Acc;
  constexpr int IS = Elem<DI>::kSize;
  constexpr int OS = Elem<DO>::kSize;
  constexpr int VEC = elems_per<DI, NW>();
  constexpr int OB = VEC * OS;
  const int R = RT > 0 ? RT : a.R;
  const int S = ST > 0 ? ST : a.S;
  const uint64_t nvec = a.count / VEC;
  const uint64_t tid = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;

  for (uint64_t iv = tid; iv < nvec; iv += stride) {
    const uint64_t e0 = iv * VEC;
    const uint64_t j = fastdiv_div(a.Ld, e0);
    const uint64_t k0 = e0 - j * a.L;
    const uint64_t L2 = j == a.jlast ? a.L2last : a.L2;
    const uint64_t i = hsdp_outer_chunk(a, j, k0);
    if (k0 + VEC > a.L || k0 + VEC > (i + 1) * L2) {
      // The vector straddles a shard or an outer chunk: element by element.
      for (int q = 0; q < VEC; ++q) hsdp_elem<DI, DO>(a, R, S, e0 + q);
      continue;
    }
    CR_DCHECK(e0 + VEC <= a.count && j == e0 / a.L && j < (uint64_t)S && i < (uint64_t)R &&
                  i == k0 / L2,
              kChkHsdp);
    Acc acc[VEC], part[VEC];
    int g = ((int)i + 1 == R) ? 0 : (int)i + 1;
    fold_vec<DI, ST, NW>(a.in + g * S, S, (int)j, e0 * IS, acc);
    auto add_group = [&]() {
      g = (g + 1 == R) ? 0 : g + 1;
      fold_vec<DI, ST, NW>(a.in + g * S, S, (int)j, e0 * IS, part);
#pragma unroll
      for (int t = 0; t < VEC; ++t) acc[t] = acc_plus<DI>(acc[t], part[t]);
    };
    if constexpr (RT > 0) {
#pragma unroll
      for (int q = 1; q < RT; ++q) add_group();
    } else {
      for (int q = 1; q < R; ++q) add_group();
    }
    if constexpr (DI != CR_I32) {
      if (a.avg) {
#pragma unroll
        for (int t = 0; t < VEC; ++t) acc[t] = finish_avg(acc[t], R * S, a.inv_n);
      }
    }
    if (a.out_scalar) {
      // shard offsets off the vector grid (L or a shard pointer)
      for (int q = 0; q < R; ++q) store_offgrid<DI, DO, NW>(a.out[q * S + (int)j], e0, k0, (int)j, acc);
      continue;
    }
    uint32_t w[OB / 4];
    acc_pack<DI, DO, VEC>(acc, w);
#pragma unroll 4
    for (int q = 0; q < R; ++q)
      st_words<OB, NW * 4>(static_cast<unsigned char*>(a.out[q * S + (int)j]) + k0 * OS, w);
  }
  // The last count % VEC elements.
  const uint64_t tail = a.count - nvec * VEC;
  if (tid < tail) hsdp_elem<DI, DO>(a, R, S, nvec * VEC + tid);
}

// A runtime mesh shape: built for 2 CTAs per SM (125-128 registers; the
// 32-byte versions spill up to 576 bytes and are still the fastest).  On
// a 4 x 4 mesh of 64 MiB bf16 ranks GB300 ran it at 5,160 GB/s, against
// 4,550 with default bounds (200-240 registers, 1 CTA per SM) and 2,450
// under the 4-CTA bound (which spills over a kilobyte).  Only group sizes
// other than 2, 4 and 8 take it now (k_hsdp_vec3).
template <int DI, int DO, int RT, int ST, int NW>
__global__ void __launch_bounds__(kBlock, 2) k_hsdp_vec(const __grid_constant__ HsdpArgs a) {
  pdl_enter();
  hsdp_range<DI, DO, RT, ST, NW>(a);
}

// A compile-time group size S with a runtime group count R, for 3 CTAs per
// SM: the S loads of the inner fold are issued together, and the R groups
// are added one after another into one partial, so the registers do not
// grow with R (60-80, no spills).  On 64 MiB bf16 ranks GB300 runs meshes
// of 4 x 4, 8 x 8, 2 x 8, 4 x 8 and 16 x 4 at 7,070-7,330 GB/s (8 x 2:
// 6,870), against 4,900-6,130 for the runtime-shape kernel.
template <int DI, int DO, int RT, int ST, int NW>
__global__ void __launch_bounds__(kBlock, 3) k_hsdp_vec3(const __grid_constant__ HsdpArgs a) {
  pdl_enter();
  hsdp_range<DI, DO, RT, ST, NW>(a);
}

// A compile-time mesh shape, registers capped for 4 resident CTAs per SM
// (64 per thread, no spills): on GB300 that is 6 % faster than the 3 CTAs
// that 68 allow.
template <int DI, int DO, int RT, int ST, int NW>
__global__ void __launch_bounds__(kBlock, 4) k_hsdp_vec4(const __grid_constant__ HsdpArgs a) {
  pdl_enter();
  hsdp_range<DI, DO, RT, ST, NW>(a);
}

template <int DI, int DO>
__global__ void __launch_bounds__(kBlock)
    k_hsdp_elem(const __grid_constant__ HsdpArgs a) {
  pdl_enter();
  const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
  for (uint64_t e = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; e < a.count; e += stride)
    hsdp_elem<DI, DO>(a, a.R, a.S, e);
}

template <typename K>
static cudaError_t launch_flat_hsdp(K kernel, const HsdpArgs& a, uint64_t threads,
                                    cudaStream_t s) {
  clear_stale_error();
  return launch_pdl(kernel, dim3(flat_grid(threads)), kBlock, s, a);
}

template <int DI, int DO, int NW>
static cudaError_t hsdp_dispatch_nw(const HsdpArgs& a, cudaStream_t s) {
  constexpr int VEC = elems_per<DI, NW>();
  const uint64_t threads = a.count / VEC + VEC;
  if (a.R == 2 && a.S == 4) return launch_flat_hsdp(k_hsdp_vec4<DI, DO, 2, 4, NW>, a, threads, s);
  if (a.R == 4 && a.S == 2) return launch_flat_hsdp(k_hsdp_vec4<DI, DO, 4, 2, NW>, a, threads, s);
  if (a.R == 2 && a.S == 2) return launch_flat_hsdp(k_hsdp_vec4<DI, DO, 2, 2, NW>, a, threads, s);
  if (a.S == 2) return launch_flat_hsdp(k_hsdp_vec3<DI, DO, 0, 2, NW>, a, threads, s);
  if (a.S == 4) return launch_flat_hsdp(k_hsdp_vec3<DI, DO, 0, 4, NW>, a, threads, s);
  if (a.S == 8) return launch_flat_hsdp(k_hsdp_vec3<DI, DO, 0, 8, NW>, a, threads, s);
  return launch_flat_hsdp(k_hsdp_vec<DI, DO, 0, 0, NW>, a, threads, s);
}

template <int DI, int DO>
static cudaError_t hsdp_dispatch(const HsdpArgs& a, int vw, cudaStream_t s) {
  if (vw == 32) return hsdp_dispatch_nw<DI, DO, 8>(a, s);
  if (vw == 16) return hsdp_dispatch_nw<DI, DO, 4>(a, s);
  return launch_flat_hsdp(k_hsdp_elem<DI, DO>, a, a.count, s);
}

cudaError_t launch_hsdp(cr_dtype in, cr_dtype out, const HsdpArgs& a, int vw, cudaStream_t s) {
  if (in == CR_F32 && out == CR_F32) return hsdp_dispatch<CR_F32, CR_F32>(a, vw, s);
  if (in == CR_BF16 && out == CR_BF16) return hsdp_dispatch<CR_BF16, CR_BF16>(a, vw, s);
  if (in == CR_BF16 && out == CR_F32) return hsdp_dispatch<CR_BF16, CR_F32>(a, vw, s);
  if (in == CR_I32 && out == CR_I32) return hsdp_dispatch<CR_I32, CR_I32>(a, vw, s);
  return cudaErrorInvalidValue;
}

}  // namespace cr

// k_bucket.cu -- batched byte copies for the DDP bucket packer.
//
// Packing gradient tensors into fixed-size buckets ("AI Infra Guide,
// Chapter 6", 6.2.4 bucketing and 6.2.6 Horovod Tensor Fusion) is a gather
// of many contiguous byte ranges into others.  One launch copies up to
// kMaxSegsPerLaunch ranges, described in its __grid_constant__ parameter
// block (no device-side table, no allocation).  Work is cut into tiles of
// kCopyTileBytes of destination, one per CTA; a CTA finds its tile's range
// by binary search over the per-range tile prefix sum.
//
// Inside a range the destination is written in aligned 16-byte vectors.
// When the source is misaligned relative to the destination (bucket offsets
// are arbitrary multiples of the element size), each vector is assembled
// from the two aligned 16-byte source granules it straddles with a funnel
// shift; both granules hold bytes of the range, so no load leaves it.  The
// unaligned head and tail bytes of the destination (< 16 each) are copied
// one byte at a time by the range's first tile.
#include "check.cuh"
#include "cr_internal.cuh"
#include "fold.cuh"
#include "pdl.cuh"

namespace cr {

constexpr int kVecPerTile = kCopyTileBytes / 16;
constexpr int kVecPerThread = kVecPerTile / kBlock;
static_assert(kVecPerTile % kBlock == 0, "tile must split evenly over a CTA");

// Bytes [sh, sh + 16) of the 32-byte concatenation lo:hi (0 < sh < 16).
__device__ __forceinline__ uint4 shift_window(uint4 lo, uint4 hi, int sh) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  const int q = sh >> 2;
  const uint32_t bits = (uint32_t)(sh & 3) * 8u;
  uint32_t s[5];
#pragma unroll
  for (int i = 0; i < 5; ++i) {
    // w[q + i] with q in 0..3 and i in 0..4 (index <= 7), by selects.
    const uint32_t a0 = w[i], a1 = w[i + 1 < 8 ? i + 1 : 7];
    const uint32_t a2 = w[i + 2 < 8 ? i + 2 : 7], a3 = w[i + 3 < 8 ? i + 3 : 7];
    s[i] = q == 0 ? a0 : q == 1 ? a1 : q == 2 ? a2 : a3;
  }
  uint4 o;
  o.x = __funnelshift_r(s[0], s[1], bits);
  o.y = __funnelshift_r(s[1], s[2], bits);
  o.z = __funnelshift_r(s[2], s[3], bits);
  o.w = __funnelshift_r(s[3], s[4], bits);
  return o;
}

__device__ __forceinline__ uint4 ld16_ro(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

__global__ void __launch_bounds__(kBlock)
    k_copy_segments(const __grid_constant__ CopyArgs a, uint32_t ntiles) {
  pdl_launch_dependents();
  for (uint32_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    // Range s holds tile t iff tile_start[s] <= t < tile_start[s + 1].
    int lo = 0, hi = a.nseg;  // invariant: tile_start[lo] <= t < tile_start[hi]
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (a.tile_start[mid] <= t) lo = mid;
      else hi = mid;
    }
    CR_DCHECK(lo < a.nseg && a.tile_start[lo] <= t && t < a.tile_start[lo + 1], kChkCopy);
    const CopySeg sg = a.seg[lo];
    const uint32_t tile = t - a.tile_start[lo];
    const uintptr_t d0 = reinterpret_cast<uintptr_t>(sg.dst);
    const uintptr_t d_end = d0 + sg.bytes;
    const uintptr_t da = (d0 + 15) & ~uintptr_t(15);
    const uintptr_t de = d_end & ~uintptr_t(15);
    if (da >= de) {
      // No whole aligned vector: the range is copied byte by byte.
      if (tile == 0) {
        for (uint64_t b = threadIdx.x; b < sg.bytes; b += blockDim.x) sg.dst[b] = sg.src[b];
      }
      continue;
    }
    if (tile == 0) {
      const uint64_t head = da - d0, tail = d_end - de;
      if (threadIdx.x < head) sg.dst[threadIdx.x] = sg.src[threadIdx.x];
      if (threadIdx.x >= 32 && threadIdx.x - 32 < tail) {
        const uint64_t b = (de - d0) + (threadIdx.x - 32);
        sg.dst[b] = sg.src[b];
      }
    }
    const uint64_t nint = (de - da) / 16;
    const unsigned char* s0 = sg.src + (da - d0);  // source byte of vector 0
    const int sh = (int)(reinterpret_cast<uintptr_t>(s0) & 15);
    const unsigned char* sa = s0 - sh;             // aligned granule of vector 0
    unsigned char* dst = reinterpret_cast<unsigned char*>(da);
    const uint64_t v0 = (uint64_t)tile * kVecPerTile;
    if (sh == 0) {
      uint4 v[kVecPerThread];
#pragma unroll
      for (int k = 0; k < kVecPerThread; ++k) {
        const uint64_t i = v0 + (uint64_t)k * kBlock + threadIdx.x;
        if (i < nint) v[k] = ld16_ro(sa + i * 16);
      }
#pragma unroll
      for (int k = 0; k < kVecPerThread; ++k) {
        const uint64_t i = v0 + (uint64_t)k * kBlock + threadIdx.x;
        if (i < nint) st16(dst + i * 16, v[k]);
      }
    } else {
      uint4 lo_v[kVecPerThread], hi_v[kVecPerThread];
#pragma unroll
      for (int k = 0; k < kVecPerThread; ++k) {
        const uint64_t i = v0 + (uint64_t)k * kBlock + threadIdx.x;
        if (i < nint) {
          // both granules hold bytes of the source range
          CR_DCHECK(sa + i * 16 + 16 < sg.src + sg.bytes && sa + i * 16 + 16 > sg.src, kChkCopy);
          lo_v[k] = ld16_ro(sa + i * 16);
          hi_v[k] = ld16_ro(sa + i * 16 + 16);
        }
      }
#pragma unroll
      for (int k = 0; k < kVecPerThread; ++k) {
        const uint64_t i = v0 + (uint64_t)k * kBlock + threadIdx.x;
        if (i < nint) st16(dst + i * 16, shift_window(lo_v[k], hi_v[k], sh));
      }
    }
  }
  pdl_wait_prerequisites();
}

cudaError_t launch_copy(const CopyArgs& a, uint32_t ntiles, bool chained, cudaStream_t s) {
  if (ntiles == 0) return cudaSuccess;
  return launch_chained(k_copy_segments, flat_grid((uint64_t)ntiles * kBlock), kBlock, s, chained,
                        a, ntiles);
}

}  // namespace cr

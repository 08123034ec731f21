// cr_internal.cuh -- types shared by the host API layer and the kernels of
// libcr (never installed; the public interface is include/cr.h).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "cr.h"

namespace cr {

constexpr int kMaxRanks = CR_MAX_RANKS;
constexpr int kBlock = 256;  // threads per CTA for every streaming kernel

// Arguments of the reduce kernels (reduce-scatter and all-reduce).  Passed
// by value as a __grid_constant__ kernel parameter: the per-rank pointer
// table lives in the constant bank and is indexed with the ring offset.
struct FoldArgs {
  const void* in[kMaxRanks];
  void* out[kMaxRanks];
  uint64_t count;  // elements per rank buffer
  uint64_t L;      // chunk length ceil(count / n)
  int n;           // ranks
  int avg;         // 1: divide the finished sum by n
  float inv_n;     // 1/n when n is a power of two (exact), else 0
};

struct GatherArgs {
  const void* shards[kMaxRanks];
  void* bufs[kMaxRanks];
  uint64_t count;
  uint64_t L;
  int n;
  uint64_t inplace_mask;  // bit j: shards[j] is chunk j of bufs[j]
};

// AdamW scalars, each formed in double on the host and rounded once.
struct AdamScalars {
  float lr, eps, b1, b2, omb1, omb2, decay, bc1, bc2;
};

struct FsdpArgs {
  const void* grads[kMaxRanks];
  void* params[kMaxRanks];
  float* master[kMaxRanks];
  float* m[kMaxRanks];
  float* v[kMaxRanks];
  uint64_t count;
  uint64_t L;
  int n;
  float inv_n;
  AdamScalars a;
};

struct AdamArgs {
  float* master;
  float* m;
  float* v;
  const float* g;
  void* param_bf16;  // may be null
  uint64_t n;
  AdamScalars a;
};

// One contiguous byte copy of the bucket packer.
struct CopySeg {
  const unsigned char* src;
  unsigned char* dst;
  uint64_t bytes;
};

constexpr int kMaxSegsPerLaunch = 1024;
constexpr int kCopyTileBytes = 32768;  // bytes of destination per CTA tile

struct CopyArgs {
  int nseg;
  uint32_t tile_start[kMaxSegsPerLaunch + 1];  // prefix sum of tiles per seg
  CopySeg seg[kMaxSegsPerLaunch];
};

enum FoldMode { kRS = 0, kAR = 1 };

// Launchers (defined next to their kernels).  `vec` selects the 16-byte
// vector kernel; the host layer has checked its preconditions.
cudaError_t launch_fold(cr_dtype in, cr_dtype out, FoldMode mode,
                        const FoldArgs& a, bool vec, cudaStream_t s);
cudaError_t launch_gather(size_t esize, const GatherArgs& a, bool vec,
                          cudaStream_t s);
cudaError_t launch_fsdp(const FsdpArgs& a, bool vec, cudaStream_t s);
cudaError_t launch_adamw(const AdamArgs& a, bool vec, cudaStream_t s);
cudaError_t launch_copy(const CopyArgs& a, uint32_t ntiles, cudaStream_t s);

// Persistent-grid size for a kBlock-thread kernel that needs `threads`
// threads of work: min(SMs on the current device * CTAs of `kernel` resident
// per SM, ceil(threads / kBlock)), at least 1.  Occupancy is queried once
// per (kernel, device) and cached.
cudaError_t persistent_grid(const void* kernel, uint64_t threads, int* grid);

}  // namespace cr

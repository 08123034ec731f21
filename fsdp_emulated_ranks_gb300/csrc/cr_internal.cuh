// cr_internal.cuh -- types shared by the host API layer and the kernels of
// libcr (never installed; the public interface is include/cr.h).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "cr.h"
#include "fastdiv.h"

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
  FastDiv Ld;      // division by L
  uint64_t begin;  // the call covers elements [begin, end) of each buffer
  uint64_t end;
  int n;           // ranks
  int n_out;       // all-reduce: output buffers written (n, or 2n when the
                   // result also goes to a second set of buffers)
  int avg;         // 1: divide the finished sum by n
  float inv_n;     // 1/n when n is a power of two (exact), else 0
  uint32_t max_ctas;  // cap on the grid (0: one vector per thread)
  int wire_bf16;      // 1: round every forwarded partial to bf16 (a bf16 wire)
  int out_scalar;     // reduce-scatter: 1 when the chunk length or the shard
                      // pointers are off the vector grid; the inputs still
                      // take vector loads, each shard element its own store
};

struct GatherArgs {
  const void* shards[kMaxRanks];
  void* bufs[kMaxRanks];
  uint64_t count;
  uint64_t L;
  FastDiv Ld;
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
  FastDiv Ld;
  uint64_t begin;  // the update covers elements [begin, end) of the flat
  uint64_t end;    // buffer (the whole buffer's chunks and fold order)
  int n;
  float inv_n;
  AdamScalars a;
  // Gradient-norm clipping (clip_grad_norm_): when non-null, the device
  // address of the coefficient min(1, max_norm / (norm + 1e-6)) by which
  // every averaged gradient is scaled (written by k_clip_coef).
  const float* coef;
  // Clipped step only (n >= 2, vector path): 1 when the sum-of-squares pass
  // parks each averaged fp32 gradient in the parameter outputs -- its low
  // 16 bits at element e of params[0], its high 16 bits at element e of
  // params[1] -- and the update pass reads it back from there instead of
  // folding the n bf16 gradients a second time.
  int stash;
};

// Upper bound on the per-CTA partial sums of the sum-of-squares pass; the
// clip workspace holds the coefficient in its first 8 bytes, then these.
constexpr int kMaxNormParts = 4095;

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
constexpr int kCopyTileBytes = 8192;  // bytes of destination per CTA tile

struct CopyArgs {
  int nseg;
  uint32_t tile_start[kMaxSegsPerLaunch + 1];  // prefix sum of tiles per seg
  CopySeg seg[kMaxSegsPerLaunch];
};

// Fused bucket all-reduce: one tensor of a launch.
struct FusedTensor {
  uint64_t numel;  // elements of the tensor
  uint64_t off;    // element offset of the tensor inside its bucket
  uint64_t Lb;     // chunk length of its bucket, ceil(bucket numel / N)
  FastDiv Lbd;     // division by Lb
  uint32_t ptr0;   // index of rank 0's pointer in FusedArgs::ptrs
  uint32_t vw;     // vector bytes all N rank pointers allow: 32, 16 or 0
};

constexpr int kFusedMaxTensors = 128;
constexpr int kFusedMaxPtrs = 2048;
constexpr uint64_t kFusedTileElems = 4096;  // elements of a tensor per CTA

struct FusedArgs {
  int ntens;
  int n;
  int avg;
  float inv_n;
  uint32_t max_ctas;  // cap on the grid (0: one CTA per tile)
  uint32_t tile_start[kFusedMaxTensors + 1];
  FusedTensor t[kFusedMaxTensors];
  void* ptrs[kFusedMaxPtrs];  // rank q of tensor k at ptrs[t[k].ptr0 + q]
};

// FSDP2 step: one parameter of a launch.  Its 5N pointers sit in
// Fsdp2Args::ptrs from ptr0: grads[0..N), params[N..2N), master[2N..3N),
// m[3N..4N), v[4N..5N).
struct Fsdp2Param {
  uint64_t numel;  // dim0 * row_numel
  uint64_t L;      // shard length: ceil(dim0 / N) rows * row_numel
  FastDiv Ld;      // division by L
  uint32_t ptr0;
  uint32_t vw;     // 32: vector path with 32-byte state, 16: 16-byte, 0: elements
};

constexpr int kFsdp2MaxParams = 64;
constexpr int kFsdp2MaxPtrs = 2560;
constexpr uint64_t kFsdp2TileElems = 4096;  // elements of a parameter per CTA

struct Fsdp2Args {
  int nparams;
  int n;
  float inv_n;
  AdamScalars a;
  uint32_t tile_start[kFsdp2MaxParams + 1];
  Fsdp2Param p[kFsdp2MaxParams];
  void* ptrs[kFsdp2MaxPtrs];
};

// FSDP2 step over a plan's table in device memory.  Table layout (built on
// the host by cr_fsdp2_plan_create, uploaded by cr_fsdp2_plan_upload):
//   [0, p_off)          uint32 tile_start[nparams + 1] (prefix sums of the
//                       parameters' tiles), zero-padded to 16 bytes
//   [p_off, ptr_off)    Fsdp2Param p[nparams], 48 bytes each
//   [ptr_off, ...)      void* ptrs[5 * n * nparams], parameter q's from
//                       p[q].ptr0 in the order of Fsdp2Param
struct Fsdp2TableArgs {
  const unsigned char* table;
  uint64_t p_off;
  uint64_t ptr_off;
  uint32_t nparams;  // parameters in the table (empty ones left out)
  uint32_t ntiles;   // tile_start[nparams]
  int n;
  float inv_n;
  AdamScalars a;
};

// Gradient accumulation (no_sync) and the fused accumulate + all-reduce.
struct AccumArgs {
  float* acc[kMaxRanks];
  const void* grads[kMaxRanks];
  uint64_t count;
  uint64_t L;
  FastDiv Ld;
  int n;
  int reduce;  // 0: acc[r] += g[r] only; 1: then all-reduce the sums in place
  int avg;
  float inv_n;
};

enum FoldMode { kRS = 0, kAR = 1 };

// Launchers (defined next to their kernels).  `vw` is the vector width in
// bytes the host layer has checked the buffers allow: 32, 16, or 0 for the
// element-wise kernels; launch_fsdp also takes 1 (vector grads and params,
// fp32 state element by element).
// HSDP gradient reduction over an R x S mesh (rank (g, s) at g*S + s): the
// ring reduce-scatter inside each group of S ranks, then the ring
// all-reduce of every shard across the R groups.
struct HsdpArgs {
  const void* in[CR_MAX_RANKS];  // rank g*S + s's full buffer
  void* out[CR_MAX_RANKS];       // shard j of group g at g*S + j
  uint64_t count;
  uint64_t L;       // shard length ceil(count / S)
  uint64_t L2;      // outer chunk length of a full shard: ceil(L / R)
  uint64_t L2last;  // outer chunk length of the last non-empty shard
  uint64_t jlast;   // index of the last non-empty shard
  FastDiv Ld, L2d, L2lastd;
  int R, S;
  int avg;
  float inv_n;     // 1/(R*S) when exact, else 0 (divide)
  int out_scalar;  // 1: shard offsets off the vector grid, element stores
};

// The fused bucket all-reduce (api.cu), for the DDP reducer: argument
// checks, and the launch over a list of the plan's tensors.
cr_status bucket_fused_check(const cr_bucket_plan_t* plan, int nranks, void* const* tensors,
                             cr_dtype dtype, cr_op op);
cr_status bucket_fused_tensors(const cr_bucket_plan_t* plan, int nranks, void* const* tensors,
                               cr_dtype dtype, cr_op op, const int* list, int nlist,
                               uint32_t max_ctas, cudaStream_t stream);

cudaError_t launch_hsdp(cr_dtype in, cr_dtype out, const HsdpArgs& a, int vw,
                        cudaStream_t s);
cudaError_t launch_fold(cr_dtype in, cr_dtype out, FoldMode mode,
                        const FoldArgs& a, int vw, cudaStream_t s);
cudaError_t launch_gather(size_t esize, const GatherArgs& a, int vw,
                          cudaStream_t s);
cudaError_t launch_fsdp(const FsdpArgs& a, int vw, cudaStream_t s);
// Sum-of-squares pass of the clipped step: writes *nparts (<= max_parts)
// fp64 partials to `partials`.
cudaError_t launch_fsdp_sumsq(const FsdpArgs& a, bool vec, double* partials,
                              int max_parts, int* nparts, cudaStream_t s);
// One warp: sums the nparts partials in a fixed order, writes the clip
// coefficient to *coef and the norm to *norm_out (if non-null).
cudaError_t launch_clip_coef(const double* partials, int nparts, double max_norm, float* coef,
                             float* norm_out, cudaStream_t s);
cudaError_t launch_adamw(const AdamArgs& a, bool vec, cudaStream_t s);
// chained: launched as the programmatic dependent of the call's previous
// launch (pdl.cuh).
cudaError_t launch_copy(const CopyArgs& a, uint32_t ntiles, bool chained, cudaStream_t s);
cudaError_t launch_bucket_fused(cr_dtype d, const FusedArgs& a, uint32_t ntiles, bool chained,
                                cudaStream_t s);
uint64_t fused_tile_elems(cr_dtype d);  // elements of a tensor per CTA tile
cudaError_t launch_fsdp2(const Fsdp2Args& a, uint32_t ntiles, bool chained, cudaStream_t s);
cudaError_t launch_fsdp2_table(const Fsdp2TableArgs& a, cudaStream_t s);
// grad_dtype CR_F32 or CR_BF16; vw as for the other launchers (16-byte
// grads and 32- or 16-byte accumulators).
cudaError_t launch_accum(cr_dtype grad_dtype, const AccumArgs& a, int vw, cudaStream_t s);

// Records `msg` as the detail cr_last_error() returns on this thread.
void report_error(cr_status status, const char* msg);
// CR_ERR_CUDA with `what` and the CUDA error's name and text as the detail.
cr_status report_cuda_error(cudaError_t e, const char* what);

// Persistent-grid size for a kBlock-thread kernel that needs `threads`
// threads of work: min(SMs on the current device * CTAs of `kernel` resident
// per SM, ceil(threads / kBlock)), at least 1.  Occupancy is queried once
// per (kernel, device) and cached.
cudaError_t persistent_grid(const void* kernel, uint64_t threads, int* grid);

// Streaming multiprocessors of the current device (cached per device).
cudaError_t sm_count(int* sms);

// Grid of ceil(threads / kBlock) CTAs (at least 1, at most 2^30; kernels
// keep a grid-stride loop for anything beyond).
inline unsigned flat_grid(uint64_t threads) {
  uint64_t g = (threads + kBlock - 1) / kBlock;
  if (g < 1) g = 1;
  if (g > (1ull << 30)) g = 1ull << 30;
  return (unsigned)g;
}

// cudart is linked statically, so its last-error word belongs to this
// library alone, but it also keeps errors that earlier calls returned
// directly (a failed cudaLaunchKernelEx, cudaEventRecord, ...).  Every
// <<<>>> launch clears it first, so that cudaGetLastError() after the
// launch reports that launch alone.  A sticky error of the context is
// reported again whatever is cleared.
inline void clear_stale_error() { (void)cudaGetLastError(); }

}  // namespace cr

// fsdp_noalloc.cu -- the clipped FSDP step for callers that cannot allocate.
//
// cr_fsdp_step_clipped needs a small device workspace for the per-CTA
// partial sums of its first (sum-of-squares) pass, and leaves it to the
// caller to provide one.  Some callers have no way to get device memory:
// a plugin handed only its tensors by a host framework that owns the whole
// device budget through its own allocator, or latency-critical code where a
// cudaMalloc would synchronise the device.  cr_fsdp_step_clipped_noalloc
// serves them with a workspace that lives in this file, as a static device
// array loaded with the library.
#include <cuda.h>

#include <map>
#include <mutex>
#include <utility>

#include "cr_internal.cuh"

namespace {

// The clip coefficient (first 8 bytes) and one fp64 partial sum per CTA of
// the first pass: 4096 x 8 B = 32 KiB, resident on every GPU that loads the
// library until the process exits.  cr_fsdp_step_clipped caps the first
// pass at as many CTAs as the workspace has partial slots (4095 here), so
// any GPU fits.
constexpr int kScratchParts = 4096;
static __device__ __align__(256) double g_clip_scratch[kScratchParts];

// Identity of the current context: the driver's context ID, unique for the
// life of the process (a context created after a cudaDeviceReset gets a new
// one).  The two driver calls are looked up through the runtime, so the
// library does not link libcuda itself.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

std::mutex g_mu;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
// (device, context ID) -> device address of g_clip_scratch in that context
std::map<std::pair<int, unsigned long long>, void*> g_scratch_addr;

cudaError_t current_context_id(unsigned long long* id) {
  if (!g_ctx_get_current || !g_ctx_get_id) {
    cudaDriverEntryPointQueryResult q1, q2;
    void* f1 = nullptr;
    void* f2 = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000,
                                                     cudaEnableDefault, &q1);
    if (e == cudaSuccess)
      e = cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2);
    if (e != cudaSuccess) return e;
    if (q1 != cudaDriverEntryPointSuccess || q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
      return cudaErrorSymbolNotFound;
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f2);
  }
  CUcontext ctx = nullptr;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorDeviceUninitialized;
  if (g_ctx_get_id(ctx, id) != CUDA_SUCCESS) return cudaErrorContextIsDestroyed;
  return cudaSuccess;
}

// Device address of the scratch array in the current device's current
// context, looked up once per (device, context) with that device current
// and cached; a new context (after a device reset) gets a fresh lookup.
cudaError_t scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  unsigned long long ctx_id = 0;
  cudaError_t e = current_context_id(&ctx_id);
  if (e != cudaSuccess) return e;
  const auto key = std::make_pair(dev, ctx_id);
  auto it = g_scratch_addr.find(key);
  if (it != g_scratch_addr.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  void* ptr = nullptr;
  e = cudaGetSymbolAddress(&ptr, g_clip_scratch);
  if (e != cudaSuccess) return e;
  g_scratch_addr[key] = ptr;
  *out = ptr;
  return cudaSuccess;
}

}  // namespace

extern "C" cr_status cr_fsdp_step_clipped_noalloc(
    const void* const* grads_bf16, int nranks, size_t count, float* const* master,
    float* const* m, float* const* v, const cr_adamw_cfg* cfg, double max_norm,
    void* const* params_bf16, float* norm_out, cr_stream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    return cr::report_cuda_error(e, "fsdp_step_clipped_noalloc: cudaGetDevice");
  }
  // cudaGetDevice does not create the primary context; cudaSetDevice on the
  // current device does (CUDA 12 and later), so that the context lookup
  // below sees the context the launches will use.
  e = cudaSetDevice(dev);
  if (e != cudaSuccess) {
    return cr::report_cuda_error(e, "fsdp_step_clipped_noalloc: context initialisation");
  }
  void* scratch = nullptr;
  e = scratch_address(dev, &scratch);
  if (e != cudaSuccess) {
    return cr::report_cuda_error(e, "fsdp_step_clipped_noalloc: scratch address lookup");
  }
  return cr_fsdp_step_clipped(grads_bf16, nranks, count, master, m, v, cfg, max_norm, scratch,
                              sizeof(g_clip_scratch), params_bf16, norm_out, stream);
}

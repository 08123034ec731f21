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
#include <map>
#include <mutex>

#include "cr_internal.cuh"

namespace {

// The clip coefficient (first 8 bytes) and one fp64 partial sum per CTA of
// the first pass: 4096 x 8 B = 32 KiB, resident on every GPU that loads the
// library until the process exits.
constexpr int kScratchParts = 4096;
static __device__ __align__(256) double g_clip_scratch[kScratchParts];

// A CTA of 256 threads, at most 2048 threads per SM: 8 CTAs per SM.
constexpr int kMaxCtasPerSm = 8;

std::mutex g_mu;
std::map<int, void*> g_scratch_addr;  // device -> address of g_clip_scratch

// Device address of the scratch array on the current device, looked up
// once per device (with that device current) and cached.
cudaError_t scratch_address(int dev, void** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_scratch_addr.find(dev);
  if (it != g_scratch_addr.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  void* ptr = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&ptr, g_clip_scratch);
  if (e != cudaSuccess) return e;
  g_scratch_addr[dev] = ptr;
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
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) {
    return cr::report_cuda_error(e, "fsdp_step_clipped_noalloc: SM count query");
  }
  if ((long long)sms * kMaxCtasPerSm > kScratchParts - 1) {
    cr::report_error(CR_ERR_UNSUPPORTED,
                     "fsdp_step_clipped_noalloc: this GPU's first pass may need more "
                     "partial sums than the 4095 the static scratch holds");
    return CR_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  e = scratch_address(dev, &scratch);
  if (e != cudaSuccess) {
    return cr::report_cuda_error(e, "fsdp_step_clipped_noalloc: cudaGetSymbolAddress");
  }
  return cr_fsdp_step_clipped(grads_bf16, nranks, count, master, m, v, cfg, max_norm, scratch,
                              sizeof(g_clip_scratch), params_bf16, norm_out, stream);
}

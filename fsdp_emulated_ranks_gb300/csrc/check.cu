// check.cu -- the device error word of the checked build and its host side.
#include "cr_internal.cuh"
#include "check.cuh"

namespace cr {

#if defined(CR_DEVICE_CHECKS)
__device__ unsigned int g_check_word = 0;
#endif

// Sets kChkSelfTest through the same path a failed check takes.
__global__ void k_check_selftest() { CR_DCHECK(false, kChkSelfTest); }

}  // namespace cr

extern "C" {

long long cr_check_word(int clear) {
#if defined(CR_DEVICE_CHECKS)
  unsigned int w = 0;
  if (cudaMemcpyFromSymbol(&w, cr::g_check_word, sizeof(w)) != cudaSuccess) return -2;
  if (clear) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(cr::g_check_word, &zero, sizeof(zero)) != cudaSuccess) return -2;
  }
  return (long long)w;
#else
  (void)clear;
  return -1;
#endif
}

cr_status cr_check_selftest(cr_stream_t stream) {
#if defined(CR_DEVICE_CHECKS)
  cr::clear_stale_error();
  cr::k_check_selftest<<<1, 1, 0, (cudaStream_t)stream>>>();
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cr::report_cuda_error(e, "check self-test launch");
  return CR_OK;
#else
  (void)stream;
  cr::report_error(CR_ERR_UNSUPPORTED, "the library was built without device checks");
  return CR_ERR_UNSUPPORTED;
#endif
}

}  // extern "C"

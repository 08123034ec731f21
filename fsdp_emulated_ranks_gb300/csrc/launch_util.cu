// launch_util.cu -- grid sizing shared by the launchers (SM counts and
// occupancy, cached per device).
#include <map>
#include <mutex>
#include <utility>

#include "cr_internal.cuh"

namespace cr {

namespace {
std::mutex g_mu;
std::map<std::pair<const void*, int>, int> g_ctas_per_sm;  // (kernel, device)
std::map<int, int> g_sms;                                  // device -> SMs
}  // namespace

cudaError_t sm_count(int* sms) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_sms.find(dev);
  if (it != g_sms.end()) {
    *sms = it->second;
    return cudaSuccess;
  }
  err = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (err == cudaSuccess) g_sms[dev] = *sms;
  return err;
}

cudaError_t persistent_grid(const void* kernel, uint64_t threads, int* grid) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  int sms = 0, per_sm = 0;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    auto it = g_sms.find(dev);
    if (it == g_sms.end()) {
      err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
      if (err != cudaSuccess) return err;
      g_sms[dev] = sms;
    } else {
      sms = it->second;
    }
    auto key = std::make_pair(kernel, dev);
    auto jt = g_ctas_per_sm.find(key);
    if (jt == g_ctas_per_sm.end()) {
      err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kBlock, 0);
      if (err != cudaSuccess) return err;
      if (per_sm < 1) per_sm = 1;
      g_ctas_per_sm[key] = per_sm;
    } else {
      per_sm = jt->second;
    }
  }
  const uint64_t full = (uint64_t)sms * (uint64_t)per_sm;
  const uint64_t need = (threads + kBlock - 1) / kBlock;
  uint64_t g = need < full ? need : full;
  if (g < 1) g = 1;
  *grid = (int)g;
  return cudaSuccess;
}

}  // namespace cr

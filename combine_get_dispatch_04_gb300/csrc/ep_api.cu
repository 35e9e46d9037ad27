// ep_api.cu -- status strings and the per-device property cache used by the
// launchers (SM count for persistent grids, opt-in shared memory for the
// combine pipeline).
#include <mutex>

#include "ep_common.cuh"

namespace ep {

bool device_props(DeviceProps* out) {
  static std::mutex mu;
  static DeviceProps cache[64];
  static bool have[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return false;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 64 && have[dev]) {
    *out = cache[dev];
    return true;
  }
  DeviceProps p;
  if (cudaDeviceGetAttribute(&p.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return false;
  if (cudaDeviceGetAttribute(&p.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
      cudaSuccess)
    return false;
  if (cudaDeviceGetAttribute(&p.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
      cudaSuccess)
    return false;
  if (dev < 64) {
    cache[dev] = p;
    have[dev] = true;
  }
  *out = p;
  return true;
}

}  // namespace ep

extern "C" const char* ep_status_string(ep_status_t status) {
  switch (status) {
    case EP_OK:
      return "EP_OK";
    case EP_ERR_INVALID_ARG:
      return "EP_ERR_INVALID_ARG: an argument check failed; nothing was enqueued";
    case EP_ERR_CAPACITY:
      return "EP_ERR_CAPACITY: a caller-provided buffer is too small";
    case EP_ERR_CUDA:
      return "EP_ERR_CUDA: a CUDA runtime call failed";
    case EP_ERR_TIMEOUT:
      return "EP_ERR_TIMEOUT: a bounded device wait ran out";
  }
  return "unknown ep_status_t";
}

// Host-side helpers: device property cache, CUDA error text, status strings.
#include <string.h>

#include <mutex>

#include "pa_host.h"

namespace pa {

namespace {
constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
bool g_have[kMaxDevices];
std::mutex g_mu;
thread_local char g_last_err[256];
}  // namespace

bool current_device_info(DeviceInfo *out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_have[dev]) {
    DeviceInfo d;
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return false;
    if (cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
        cudaSuccess)
      return false;
    if (cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
        cudaSuccess)
      return false;
    g_info[dev] = d;
    g_have[dev] = true;
  }
  *out = g_info[dev];
  return true;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

pa_status cuda_fail(cudaError_t err) {
  const char *s = cudaGetErrorString(err);
  strncpy(g_last_err, s ? s : "unknown CUDA error", sizeof(g_last_err) - 1);
  g_last_err[sizeof(g_last_err) - 1] = '\0';
  return PA_ERR_CUDA;
}

}  // namespace pa

extern "C" const char *pa_status_string(pa_status status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_DEVICE_CHECK: return "device-side check failed";
    case PA_ERR_OUT_OF_BLOCKS: return "out of blocks";
  }
  return "unknown status";
}

extern "C" const char *pa_last_cuda_error(void) { return pa::g_last_err; }

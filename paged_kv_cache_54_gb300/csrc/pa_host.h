// Host-side helpers shared by the libpa entry points.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

struct DeviceInfo {
  int sm_count = 0;
  int max_smem_optin = 0;  // bytes of dynamic shared memory a block may opt into
  int smem_per_sm = 0;     // bytes of shared memory per SM
};

// Properties of the current device, queried once per device.
bool current_device_info(DeviceInfo *out);

// Record the text of a failed CUDA call for pa_last_cuda_error() and return
// PA_ERR_CUDA.
pa_status cuda_fail(cudaError_t err);

// cuTensorMapEncodeTiled from the driver (looked up once through the
// runtime, so the library needs no link to libcuda); null if unavailable.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool valid_cache_desc(const pa_cache_desc *c) {
  if (c == nullptr) return false;
  if (c->num_blocks <= 0 || c->kv_heads <= 0 || c->block_size <= 0 || c->head_dim <= 0) return false;
  if (c->dtype < PA_F16 || c->dtype > PA_INT8) return false;
  if (c->dtype >= PA_FP8_E4M3) {
    if (!(c->k_scale > 0.f) || !(c->v_scale > 0.f)) return false;
    if (c->k_scale > 3.0e38f || c->v_scale > 3.0e38f) return false;
    if ((reinterpret_cast<uintptr_t>(c->k_head_scales) & 3u) ||
        (reinterpret_cast<uintptr_t>(c->v_head_scales) & 3u))
      return false;
    // one pointer without the other would leave a tensor without scales
    if ((c->k_head_scales == nullptr) != (c->v_head_scales == nullptr)) return false;
  } else if (c->k_head_scales != nullptr || c->v_head_scales != nullptr) {
    return false;  // 16-bit caches have no scales
  }
  return true;
}

inline bool supported_cache_shape(const pa_cache_desc *c) {
  return (c->block_size == 8 || c->block_size == 16 || c->block_size == 32) &&
         (c->head_dim == 64 || c->head_dim == 128);
}

}  // namespace pa

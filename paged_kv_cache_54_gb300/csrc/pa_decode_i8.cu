// Decode instantiations for INT8 KV caches.
#include "pa_decode.cuh"

namespace pa {

pa_status dispatch_decode_i8(int q_dtype, int head_dim, int group, DecodeParams p,
                            const DeviceInfo &dev, cudaStream_t stream) {
  if (q_dtype == kF16) return launch_by_dim<kI8, kF16>(head_dim, group, p, dev, stream);
  if (q_dtype == kBF16) return launch_by_dim<kI8, kBF16>(head_dim, group, p, dev, stream);
  return PA_ERR_UNSUPPORTED;
}

}  // namespace pa

// Decode instantiations for f16 KV caches.
#include "pa_decode.cuh"

namespace pa {

pa_status dispatch_decode_f16(int q_dtype, int head_dim, int group, DecodeParams p,
                              const DeviceInfo &dev, cudaStream_t stream) {
  if (q_dtype != kF16) return PA_ERR_UNSUPPORTED;
  return launch_by_dim<kF16, kF16>(head_dim, group, p, dev, stream);
}

}  // namespace pa

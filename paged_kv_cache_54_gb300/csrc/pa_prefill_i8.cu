// Prefill instantiations for i8 KV caches.
#include "pa_prefill.cuh"

namespace pa {

pa_status dispatch_prefill_i8(int q_dtype, int head_dim, int G, const PrefillParams &p, int num_seqs,
                             int max_q_len, cudaStream_t s) {
  return dispatch_prefill<kI8>(q_dtype, head_dim, G, p, num_seqs, max_q_len, s);
}

}  // namespace pa

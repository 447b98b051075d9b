// pa_decode_static_scratch: pa_decode without a caller-supplied workspace.
//
// Some callers cannot allocate device memory when they need to decode: a
// plugin running inside a host framework that owns every byte of the GPU
// through its own pool (a stray cudaMalloc bypasses the pool's accounting
// and can fail once the KV pool has been sized to fill the device), or a
// latency-critical serving loop that forbids allocation after start-up
// because cudaMalloc may synchronise the device and stall other streams.
// This entry point needs no allocation from them: its scratch is a
// file-scope device array of fixed size that every GPU loading the library
// holds until the process exits.
#include <mutex>

#include "pa_decode_params.h"

namespace pa {
namespace {

// The decode scratch (claim counter, work list, split-sequence partials).
// Host code must not use this name as an address: it is a host-side stand-in
// for the symbol.  The device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) uint8_t g_decode_scratch[PA_DECODE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
pa_status scratch_for_current_device(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return cuda_fail(e);
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" pa_status pa_decode_static_scratch(
    void *out, const void *q, int32_t q_dtype, int32_t num_seqs, int32_t num_q_heads,
    const void *k_cache, const void *v_cache, const pa_cache_desc *cache,
    const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *seq_lens,
    int32_t max_seq_len, float scale, int32_t partition_size, int *device_error,
    pa_stream_t stream) {
  if (!pa::valid_cache_desc(cache)) return PA_ERR_INVALID;
  if (num_seqs == 0) return PA_OK;
  const size_t need = pa_decode_workspace_size(num_seqs, num_q_heads, cache->kv_heads,
                                               cache->head_dim, max_seq_len, partition_size);
  if (need == 0) return PA_ERR_INVALID;
  if (need > static_cast<size_t>(PA_DECODE_STATIC_SCRATCH_BYTES)) return PA_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  const pa_status st = pa::scratch_for_current_device(&scratch);
  if (st != PA_OK) return st;
  return pa_decode(out, q, q_dtype, num_seqs, num_q_heads, k_cache, v_cache, cache,
                   block_tables, max_blocks_per_seq, seq_lens, max_seq_len, scale,
                   partition_size, scratch, static_cast<size_t>(PA_DECODE_STATIC_SCRATCH_BYTES),
                   device_error, stream);
}

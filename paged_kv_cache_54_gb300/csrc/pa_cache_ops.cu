// Cache write through a slot mapping, and whole-block copies for
// copy-on-write.  Both are bandwidth-bound element moves: one thread moves
// one 16-byte vector of the destination per iteration of a grid-stride loop,
// so reads and writes of a warp are contiguous 512-byte runs.
#include "pa_common.cuh"
#include "pa_host.h"

namespace pa {
namespace {

// INT8 code of an already-divided value: nearest integer, ties to even,
// saturated to [-128, 127]; NaN stores 0.
__device__ __forceinline__ uint32_t int8_code(float y) {
  if (y != y) return 0u;
  y = fminf(fmaxf(y, -128.f), 127.f);
  return static_cast<uint32_t>(__float2int_rn(y)) & 0xFFu;
}

// Token t, head h, destination chunk c (16 bytes of the cache row).
template <int SRC, int DST>
__global__ void __launch_bounds__(256) reshape_and_cache_kernel(
    const uint8_t *__restrict__ key, const uint8_t *__restrict__ value,
    const int64_t *__restrict__ slots, int num_tokens, int kv_heads, int head_dim,
    int block_size, long long num_slots, uint8_t *__restrict__ k_cache,
    uint8_t *__restrict__ v_cache, float k_scale, float v_scale,
    const float *__restrict__ k_head_scales, const float *__restrict__ v_head_scales, int *err) {
  // A pa_decode enqueued next may start its plan now: the plan reads only the
  // block tables and lengths, which this kernel never writes, and the decode
  // itself runs after this grid has completed.
  launch_dependents();
  constexpr int DE = elt_bytes(DST);
  constexpr int CE = 16 / DE;  // elements per destination chunk
  const int cpr = head_dim / CE;
  const long long total = static_cast<long long>(num_tokens) * kv_heads * cpr;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c = static_cast<int>(i % cpr);
    const long long th = i / cpr;
    const int h = static_cast<int>(th % kv_heads);
    const long long t = th / kv_heads;
    const long long slot = __ldg(slots + t);
    if (slot < 0) continue;  // padding row
    if (slot >= num_slots) {
      if (h == 0 && c == 0) record_error(err, kErrSlot);
      continue;
    }
    const long long blk = slot / block_size;
    const int off = static_cast<int>(slot - blk * block_size);
    const size_t dst = ((static_cast<size_t>(blk) * kv_heads + h) * block_size + off) * head_dim +
                       static_cast<size_t>(c) * CE;
    const size_t src = (static_cast<size_t>(t) * kv_heads + h) * head_dim + static_cast<size_t>(c) * CE;
    if constexpr (DE == 2) {
      *reinterpret_cast<uint4 *>(k_cache + dst * 2) = __ldg(reinterpret_cast<const uint4 *>(key + src * 2));
      *reinterpret_cast<uint4 *>(v_cache + dst * 2) =
          __ldg(reinterpret_cast<const uint4 *>(value + src * 2));
    } else {
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint8_t *in = (which == 0 ? key : value) + src * 2;
        const float *head_scales = which == 0 ? k_head_scales : v_head_scales;
        const float scale = head_scales != nullptr ? __ldg(head_scales + h) : (which == 0 ? k_scale : v_scale);
        const uint4 a = __ldg(reinterpret_cast<const uint4 *>(in));
        const uint4 b = __ldg(reinterpret_cast<const uint4 *>(in + 16));
        const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        uint32_t o[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          uint32_t packed = 0;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float2 f = half2_bits_to_float2<SRC>(w[2 * k + half]);
            // stored = value / scale, in IEEE float32 (division rounded to nearest)
            f.x = __fdiv_rn(f.x, scale);
            f.y = __fdiv_rn(f.y, scale);
            if constexpr (DST == kI8) {
              packed |= (int8_code(f.x) | (int8_code(f.y) << 8)) << (16 * half);
            } else {
              const __nv_fp8_interpretation_t interp = (DST == kE4M3) ? __NV_E4M3 : __NV_E5M2;
              const __nv_fp8x2_storage_t q = __nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE, interp);
              packed |= static_cast<uint32_t>(q) << (16 * half);
            }
          }
          o[k] = packed;
        }
        uint8_t *outp = (which == 0 ? k_cache : v_cache) + dst;
        *reinterpret_cast<uint4 *>(outp) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
}

__global__ void __launch_bounds__(256) copy_blocks_kernel(uint8_t *__restrict__ k_cache,
                                                          uint8_t *__restrict__ v_cache,
                                                          const int64_t *__restrict__ mapping,
                                                          int num_pairs, long long block_bytes,
                                                          long long num_blocks, int *err) {
  launch_dependents();  // as in reshape_and_cache_kernel: no block table or length is written here
  const long long vecs = block_bytes / 16;
  const long long total = static_cast<long long>(num_pairs) * 2 * vecs;
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long pair = i / (2 * vecs);
    const long long r = i - pair * 2 * vecs;
    const int which = r >= vecs;
    const long long v = r - which * vecs;
    const long long src = __ldg(mapping + 2 * pair);
    const long long dst = __ldg(mapping + 2 * pair + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
      if (v == 0 && which == 0) record_error(err, kErrCopyIndex);
      continue;
    }
    uint8_t *base = which ? v_cache : k_cache;
    const uint4 x = *reinterpret_cast<const uint4 *>(base + src * block_bytes + v * 16);
    *reinterpret_cast<uint4 *>(base + dst * block_bytes + v * 16) = x;
  }
}

// Whole-block moves between two pools of one block shape (the device caches
// and a pool in host memory, either way).  Thread t of CTA b handles four
// 16-byte vectors kUnroll * blockDim apart per round, issuing the four loads
// before the four stores so that enough reads are in flight to cover the
// latency of a host-memory link.  (pair, K|V, vector) is the flat index.
constexpr int kSwapUnroll = 4;

__global__ void __launch_bounds__(256) swap_blocks_kernel(
    const uint8_t *__restrict__ src_k, const uint8_t *__restrict__ src_v, uint8_t *__restrict__ dst_k,
    uint8_t *__restrict__ dst_v, const int64_t *__restrict__ mapping, int num_pairs, long long block_bytes,
    long long src_blocks, long long dst_blocks, int *err) {
  const long long vecs = block_bytes / 16;
  const long long total = static_cast<long long>(num_pairs) * 2 * vecs;
  const long long step = static_cast<long long>(gridDim.x) * blockDim.x * kSwapUnroll;
  for (long long base = static_cast<long long>(blockIdx.x) * blockDim.x * kSwapUnroll + threadIdx.x; base < total;
       base += step) {
    uint4 x[kSwapUnroll];
    uint8_t *to[kSwapUnroll];
#pragma unroll
    for (int u = 0; u < kSwapUnroll; ++u) {
      to[u] = nullptr;
      const long long i = base + static_cast<long long>(u) * blockDim.x;
      if (i >= total) continue;
      const long long pair = i / (2 * vecs);
      const long long r = i - pair * 2 * vecs;
      const int which = r >= vecs;
      const long long v = r - which * vecs;
      const long long s = __ldg(mapping + 2 * pair);
      const long long d = __ldg(mapping + 2 * pair + 1);
      if (s < 0 || s >= src_blocks || d < 0 || d >= dst_blocks) {
        if (v == 0 && which == 0) record_error(err, kErrCopyIndex);
        continue;
      }
      x[u] = *reinterpret_cast<const uint4 *>((which ? src_v : src_k) + s * block_bytes + v * 16);
      to[u] = (which ? dst_v : dst_k) + d * block_bytes + v * 16;
    }
#pragma unroll
    for (int u = 0; u < kSwapUnroll; ++u)
      if (to[u] != nullptr) *reinterpret_cast<uint4 *>(to[u]) = x[u];
  }
}

// Device address of memory the current device can address: its own memory
// (returned as is) or page-locked host memory (its mapped device address).
bool device_view(void *p, int device, uint8_t **out) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();  // clear the error the query recorded
    return false;
  }
  if ((a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) && a.device == device) {
    *out = static_cast<uint8_t *>(p);
    return true;
  }
  if (a.type == cudaMemoryTypeHost && a.devicePointer != nullptr) {
    *out = static_cast<uint8_t *>(a.devicePointer);
    return true;
  }
  return false;
}

// An mbarrier that expects one arrival which never comes: the bounded wait
// gives up after its time limit and the kernel reports a timeout.
__global__ void selftest_wait_kernel(int *err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, nullptr)) record_error(err, kErrTimeout);
}

int grid_for(long long work_items, int threads) {
  DeviceInfo info;
  int sms = current_device_info(&info) ? info.sm_count : 148;
  long long blocks = (work_items + threads - 1) / threads;
  long long cap = static_cast<long long>(sms) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<int>(blocks);
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" pa_status pa_reshape_and_cache(const void *key, const void *value, int32_t src_dtype,
                                          const int64_t *slot_mapping, int32_t num_tokens,
                                          void *k_cache, void *v_cache, const pa_cache_desc *cache,
                                          int *device_error, pa_stream_t stream) {
  if (!valid_cache_desc(cache) || num_tokens < 0) return PA_ERR_INVALID;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PA_ERR_INVALID;
  if (src_dtype != PA_F16 && src_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  if (!supported_cache_shape(cache)) return PA_ERR_UNSUPPORTED;
  const int dst = cache->dtype;
  if ((dst == PA_F16 || dst == PA_BF16) && dst != src_dtype) return PA_ERR_UNSUPPORTED;

  const int H = cache->kv_heads, D = cache->head_dim, bs = cache->block_size;
  const long long nslots = static_cast<long long>(cache->num_blocks) * bs;
  const int CE = 16 / elt_bytes(dst);
  const long long work = static_cast<long long>(num_tokens) * H * (D / CE);
  const int threads = 256;
  const int blocks = grid_for(work, threads);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint8_t *k8 = static_cast<const uint8_t *>(key);
  const uint8_t *v8 = static_cast<const uint8_t *>(value);
  uint8_t *kc = static_cast<uint8_t *>(k_cache);
  uint8_t *vc = static_cast<uint8_t *>(v_cache);
#define PA_LAUNCH_RC(SRC, DST)                                                                    \
  reshape_and_cache_kernel<SRC, DST><<<blocks, threads, 0, s>>>(k8, v8, slot_mapping, num_tokens, \
                                                                H, D, bs, nslots, kc, vc,         \
                                                                cache->k_scale, cache->v_scale,   \
                                                                cache->k_head_scales,             \
                                                                cache->v_head_scales, device_error)
  if (dst == PA_F16) {
    PA_LAUNCH_RC(kF16, kF16);
  } else if (dst == PA_BF16) {
    PA_LAUNCH_RC(kBF16, kBF16);
  } else if (dst == PA_FP8_E4M3) {
    if (src_dtype == PA_F16) PA_LAUNCH_RC(kF16, kE4M3); else PA_LAUNCH_RC(kBF16, kE4M3);
  } else if (dst == PA_FP8_E5M2) {
    if (src_dtype == PA_F16) PA_LAUNCH_RC(kF16, kE5M2); else PA_LAUNCH_RC(kBF16, kE5M2);
  } else {
    if (src_dtype == PA_F16) PA_LAUNCH_RC(kF16, kI8); else PA_LAUNCH_RC(kBF16, kI8);
  }
#undef PA_LAUNCH_RC
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

extern "C" pa_status pa_copy_blocks(void *k_cache, void *v_cache, const pa_cache_desc *cache,
                                    const int64_t *block_mapping, int32_t num_pairs,
                                    int *device_error, pa_stream_t stream) {
  if (!valid_cache_desc(cache) || num_pairs < 0) return PA_ERR_INVALID;
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !block_mapping) return PA_ERR_INVALID;
  if (!aligned16(k_cache) || !aligned16(v_cache) || (reinterpret_cast<uintptr_t>(block_mapping) & 7u))
    return PA_ERR_INVALID;
  if (!supported_cache_shape(cache)) return PA_ERR_UNSUPPORTED;
  const long long block_bytes = static_cast<long long>(cache->kv_heads) * cache->block_size *
                                cache->head_dim * elt_bytes(cache->dtype);
  const long long work = static_cast<long long>(num_pairs) * 2 * (block_bytes / 16);
  const int threads = 256;
  const int blocks = grid_for(work, threads);
  copy_blocks_kernel<<<blocks, threads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache), block_mapping, num_pairs,
      block_bytes, cache->num_blocks, device_error);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

extern "C" pa_status pa_swap_blocks(void *k_cache, void *v_cache, const pa_cache_desc *cache, void *host_k,
                                    void *host_v, int64_t host_num_blocks, const int64_t *block_mapping,
                                    int32_t num_pairs, int32_t direction, int *device_error,
                                    pa_stream_t stream) {
  if (!valid_cache_desc(cache) || num_pairs < 0 || host_num_blocks < 0) return PA_ERR_INVALID;
  if (direction != PA_SWAP_OUT && direction != PA_SWAP_IN) return PA_ERR_INVALID;
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !host_k || !host_v || !block_mapping) return PA_ERR_INVALID;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(host_k) || !aligned16(host_v) ||
      (reinterpret_cast<uintptr_t>(block_mapping) & 7u))
    return PA_ERR_INVALID;
  if (!supported_cache_shape(cache)) return PA_ERR_UNSUPPORTED;
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return cuda_fail(e);
  uint8_t *hk = nullptr, *hv = nullptr;
  if (!device_view(host_k, device, &hk) || !device_view(host_v, device, &hv)) return PA_ERR_UNSUPPORTED;
  const long long block_bytes = static_cast<long long>(cache->kv_heads) * cache->block_size *
                                cache->head_dim * elt_bytes(cache->dtype);
  const long long work = static_cast<long long>(num_pairs) * 2 * (block_bytes / 16);
  const int threads = 256;
  const int blocks = grid_for((work + kSwapUnroll - 1) / kSwapUnroll, threads);
  uint8_t *dk = static_cast<uint8_t *>(k_cache), *dv = static_cast<uint8_t *>(v_cache);
  const bool out = direction == PA_SWAP_OUT;
  swap_blocks_kernel<<<blocks, threads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      out ? dk : hk, out ? dv : hv, out ? hk : dk, out ? hv : dv, block_mapping, num_pairs, block_bytes,
      out ? cache->num_blocks : host_num_blocks, out ? host_num_blocks : cache->num_blocks, device_error);
  e = cudaGetLastError();
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

extern "C" pa_status pa_selftest_wait_timeout(int *device_error, pa_stream_t stream) {
  if (device_error == nullptr) return PA_ERR_INVALID;
  selftest_wait_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(device_error);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

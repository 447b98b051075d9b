// pa_prefill: the C entry point, the tensor-map views it builds, and the
// instantiations for 16-bit caches (the kernel is in pa_prefill.cuh; the
// one-byte cache types have a translation unit each).
#include <limits.h>
#include <math.h>

#include "pa_decode_params.h"
#include "pa_prefill.cuh"

namespace pa {
namespace {

// [row groups, half, row, 64 elements] view of a 16-bit cache: a row group
// is 8 consecutive rows (token slots of one block and head), a half is a
// 128-byte column half of a row.  The box {64, 8, head_dim / 64,
// block_size / 8} is one whole (block, head) tile.  It lands group by group,
// each group half by half, as 8-row x 128-byte atoms with the 128-byte
// swizzle: the stage layout the prefill's tensor cores read.  The half
// stride (128 bytes) is smaller than the row stride; each box line is still
// 128 contiguous bytes.
bool encode_cache_view(CUtensorMap *map, const void *cache, const pa_cache_desc *c) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t row = static_cast<cuuint64_t>(c->head_dim) * 2;
  const cuuint64_t halves = static_cast<cuuint64_t>(c->head_dim / 64);
  const cuuint64_t groups = static_cast<cuuint64_t>(c->num_blocks) * c->kv_heads * (c->block_size / 8);
  const cuuint64_t dims[4] = {64, 8, halves, groups};
  const cuuint64_t strides[3] = {row, 128, row * 8};
  const cuuint32_t box[4] = {64, 8, static_cast<cuuint32_t>(halves), static_cast<cuuint32_t>(c->block_size / 8)};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void *>(cache), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [T, Hkv, G, head_dim] view of q, box {64 elements, G, 1, 128 / G}: one
// 128-byte half of the 128 (token, head) rows of a tile, token-major; rows
// past T read as zeros.
bool encode_q_view(CUtensorMap *map, const void *q, int num_tokens, int kv_heads, int G, int head_dim) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t row = static_cast<cuuint64_t>(head_dim) * 2;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(G),
                              static_cast<cuuint64_t>(kv_heads), static_cast<cuuint64_t>(num_tokens)};
  const cuuint64_t strides[3] = {row, row * G, row * G * kv_heads};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(G), 1, static_cast<cuuint32_t>(kPfTileRows / G)};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, const_cast<void *>(q), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// The decode's wide items on the tensor cores (16-bit caches, G = 2, 4, 8):
// the tile views of q and the caches, then the wide kernel over the wide
// item slots (those past the plan's count return at once).
pa_status launch_wide_items(const DecodeParams &d, int cache_dtype, int head_dim, cudaStream_t stream) {
  if ((cache_dtype != PA_F16 && cache_dtype != PA_BF16) || d.wide_seqs <= 0) return PA_ERR_UNSUPPORTED;
  const int G = d.num_q_heads / d.num_kv_heads;
  pa_cache_desc c{};
  c.num_blocks = d.num_blocks;
  c.kv_heads = d.num_kv_heads;
  c.block_size = d.block_size;
  c.head_dim = head_dim;
  c.dtype = cache_dtype;
  c.k_scale = c.v_scale = 1.f;
  PrefillParams p{};
  if (!encode_q_view(&p.tmap_q, d.q, d.num_seqs, d.num_kv_heads, G, head_dim) ||
      !encode_cache_view(&p.tmap_k, d.k_cache, &c) || !encode_cache_view(&p.tmap_v, d.v_cache, &c))
    return cuda_fail(cudaErrorInvalidValue);
  p.k_cache = d.k_cache;
  p.v_cache = d.v_cache;
  p.block_tables = d.block_tables;
  p.seq_lens = d.seq_lens;
  p.num_q_heads = d.num_q_heads;
  p.num_kv_heads = d.num_kv_heads;
  p.num_blocks = d.num_blocks;
  p.block_size = d.block_size;
  p.max_blocks = d.max_blocks;
  p.num_q_tokens = d.num_seqs;
  p.qk_scale_log2 = d.qk_scale_log2;
  p.v_scale = 1.f;
  p.err = d.err;
  p.wide_items = d.wide_items;
  p.wide_count = d.work + 2;
  p.part_ml = d.part_ml;
  p.part_o = d.part_o;
  p.max_parts = d.max_parts;
  p.partition_size = d.partition_size;
  const long long slots = static_cast<long long>((d.num_seqs + d.wide_seqs - 1) / d.wide_seqs) * d.max_parts;
  if (slots > 0x7fffffff) return PA_ERR_UNSUPPORTED;
  const int gx = static_cast<int>(slots);
  if (cache_dtype == PA_F16)
    return head_dim == 64 ? wide_by_group<kF16, 64>(G, p, gx, stream) : wide_by_group<kF16, 128>(G, p, gx, stream);
  return head_dim == 64 ? wide_by_group<kBF16, 64>(G, p, gx, stream) : wide_by_group<kBF16, 128>(G, p, gx, stream);
}

}  // namespace pa

using namespace pa;

extern "C" pa_status pa_prefill(void *out, const void *q, int32_t q_dtype, int32_t num_q_tokens,
                                const int32_t *cu_q_lens, int32_t num_seqs, int32_t num_q_heads,
                                int32_t max_q_len, const void *k_cache, const void *v_cache,
                                const pa_cache_desc *cache, const int32_t *block_tables,
                                int32_t max_blocks_per_seq, const int32_t *seq_lens, float scale,
                                int *device_error, pa_stream_t stream) {
  if (!valid_cache_desc(cache) || num_seqs < 0 || num_q_heads <= 0 || max_q_len < 0 || num_q_tokens < 0 ||
      max_blocks_per_seq <= 0 || !isfinite(scale))
    return PA_ERR_INVALID;
  if (num_seqs == 0 || max_q_len == 0 || num_q_tokens == 0) return PA_OK;
  if (!out || !q || !cu_q_lens || !k_cache || !v_cache || !block_tables || !seq_lens) return PA_ERR_INVALID;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(cu_q_lens) & 3u) || (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return PA_ERR_INVALID;
  if (num_q_heads % cache->kv_heads) return PA_ERR_INVALID;
  const int G = num_q_heads / cache->kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return PA_ERR_UNSUPPORTED;
  if (!supported_cache_shape(cache)) return PA_ERR_UNSUPPORTED;
  const bool byte_codes = cache->dtype >= PA_FP8_E4M3;  // FP8 or INT8, with scales
  if (byte_codes ? (q_dtype != PA_F16 && q_dtype != PA_BF16) : q_dtype != cache->dtype)
    return PA_ERR_UNSUPPORTED;
  if (num_seqs > 65535 || cache->kv_heads > 65535) return PA_ERR_UNSUPPORTED;      // grid limits
  if (static_cast<long long>(cache->num_blocks) * cache->kv_heads * cache->block_size > INT_MAX ||
      static_cast<long long>(max_blocks_per_seq) * cache->block_size > INT_MAX)
    return PA_ERR_UNSUPPORTED;  // TMA row coordinates are 32-bit

  PrefillParams p{};
  if (!encode_q_view(&p.tmap_q, q, num_q_tokens, cache->kv_heads, G, cache->head_dim) ||
      (!byte_codes && (!encode_cache_view(&p.tmap_k, k_cache, cache) || !encode_cache_view(&p.tmap_v, v_cache, cache))))
    return cuda_fail(cudaErrorInvalidValue);
  p.k_cache = static_cast<const uint8_t *>(k_cache);
  p.v_cache = static_cast<const uint8_t *>(v_cache);
  p.out = out;
  p.cu_q = cu_q_lens;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = cache->kv_heads;
  p.num_blocks = cache->num_blocks;
  p.block_size = cache->block_size;
  p.max_blocks = max_blocks_per_seq;
  p.num_q_tokens = num_q_tokens;
  p.max_q_len = max_q_len;
  const bool per_head = byte_codes && cache->k_head_scales != nullptr;
  p.qk_scale_log2 = scale * (byte_codes && !per_head ? cache->k_scale : 1.0f) * 1.4426950408889634f;
  p.v_scale = byte_codes && !per_head ? cache->v_scale : 1.0f;
  p.k_head_scale = per_head ? cache->k_head_scales : nullptr;
  p.v_head_scale = per_head ? cache->v_head_scales : nullptr;
  p.err = device_error;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int D = cache->head_dim;
  switch (cache->dtype) {
    case PA_F16: return dispatch_prefill<kF16>(q_dtype, D, G, p, num_seqs, max_q_len, s);
    case PA_BF16: return dispatch_prefill<kBF16>(q_dtype, D, G, p, num_seqs, max_q_len, s);
    case PA_FP8_E4M3: return dispatch_prefill_e4m3(q_dtype, D, G, p, num_seqs, max_q_len, s);
    case PA_FP8_E5M2: return dispatch_prefill_e5m2(q_dtype, D, G, p, num_seqs, max_q_len, s);
    case PA_INT8: return dispatch_prefill_i8(q_dtype, D, G, p, num_seqs, max_q_len, s);
  }
  return PA_ERR_UNSUPPORTED;
}

// Host entry points of the decode path: argument checks, partition choice,
// workspace layout, dispatch by cache dtype.
#include <cudaTypedefs.h>
#include <math.h>

#include <mutex>

#include "pa_decode_params.h"

namespace pa {
namespace {

// Tokens per work item.  512 unless that leaves fewer than ~1024 items
// (about 7 per SM), in which case it halves, down to one 64-token stage.
int choose_partition(int num_seqs, int kv_heads, int max_seq_len, int requested) {
  if (requested > 0) return requested;
  int P = 512;
  while (P > kStageTok &&
         static_cast<long long>(num_seqs) * kv_heads * ((max_seq_len + P - 1) / P) < 1024)
    P >>= 1;
  return P;
}

struct WorkspaceLayout {
  size_t pairs_off, wide_off, join_off, ml_off, o_off, total;
  int partition, max_parts;
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool layout_for(int num_seqs, int num_q_heads, int kv_heads, int head_dim, int max_seq_len,
                int partition_size, WorkspaceLayout *out) {
  if (num_seqs < 0 || num_q_heads <= 0 || kv_heads <= 0 || head_dim <= 0 || max_seq_len < 0)
    return false;
  if (partition_size < 0 || partition_size > kMaxPartition || partition_size % kStageTok) return false;
  WorkspaceLayout w;
  w.partition = choose_partition(num_seqs, kv_heads, max_seq_len, partition_size);
  w.max_parts = max_seq_len > 0 ? (max_seq_len + w.partition - 1) / w.partition : 1;
  const size_t units = static_cast<size_t>(num_seqs) * w.max_parts;
  w.pairs_off = 256;                                            // items (int4)
  // wide items: a chunk holds at least kWideRows / 8 sequences
  const size_t wide_units = static_cast<size_t>((num_seqs + kWideRows / 8 - 1) / (kWideRows / 8)) * w.max_parts;
  w.wide_off = align256(w.pairs_off + units * sizeof(int4));
  w.join_off = align256(w.wide_off + wide_units * sizeof(int4));  // row mismatch flags
  w.ml_off = align256(w.join_off + units);
  w.o_off = align256(w.ml_off + units * num_q_heads * sizeof(float2));
  w.total = align256(w.o_off + units * num_q_heads * head_dim * sizeof(float));
  *out = w;
  return true;
}

// Tiled view of a cache as rows of head_dim elements, one row per (block,
// head, token slot): 2-D [rows, 128 B] when a row is 128 bytes, 3-D
// [rows, 2, 128 B] when it is 256 bytes; the box is one (block, head) tile
// of block_size rows, written to shared memory with the 128-byte swizzle.
bool encode_cache_map(CUtensorMap *map, const void *cache, const pa_cache_desc *c) {
  const int elt = c->dtype >= PA_FP8_E4M3 ? 1 : 2;
  const int rowb = c->head_dim * elt;
  if (rowb < 128) return true;  // 64-byte rows use plain bulk copies
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const CUtensorMapDataType dt = elt == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
  const cuuint64_t rows = static_cast<cuuint64_t>(c->num_blocks) * c->kv_heads * c->block_size;
  const cuuint32_t inner = 128 / elt;  // elements in 128 bytes
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r;
  if (rowb == 128) {
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {inner, static_cast<cuuint32_t>(c->block_size)};
    r = enc(map, dt, 2, const_cast<void *>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const cuuint64_t dims[3] = {inner, 2, rows};
    const cuuint64_t strides[2] = {128, 256};
    const cuuint32_t box[3] = {inner, 2, static_cast<cuuint32_t>(c->block_size)};
    r = enc(map, dt, 3, const_cast<void *>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  return r == CUDA_SUCCESS;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" size_t pa_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                           int32_t num_kv_heads, int32_t head_dim,
                                           int32_t max_seq_len, int32_t partition_size) {
  WorkspaceLayout w;
  if (!layout_for(num_seqs, num_q_heads, num_kv_heads, head_dim, max_seq_len, partition_size, &w))
    return 0;
  return w.total;
}

extern "C" pa_status pa_decode(void *out, const void *q, int32_t q_dtype, int32_t num_seqs,
                               int32_t num_q_heads, const void *k_cache, const void *v_cache,
                               const pa_cache_desc *cache, const int32_t *block_tables,
                               int32_t max_blocks_per_seq, const int32_t *seq_lens,
                               int32_t max_seq_len, float scale, int32_t partition_size,
                               void *workspace, size_t workspace_bytes, int *device_error,
                               pa_stream_t stream) {
  if (!valid_cache_desc(cache) || num_seqs < 0 || num_q_heads <= 0 || max_seq_len < 0 ||
      max_blocks_per_seq <= 0 || !isfinite(scale))
    return PA_ERR_INVALID;
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens || !workspace)
    return PA_ERR_INVALID;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PA_ERR_INVALID;
  if (num_q_heads % cache->kv_heads) return PA_ERR_INVALID;
  const int G = num_q_heads / cache->kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return PA_ERR_UNSUPPORTED;
  if (!supported_cache_shape(cache)) return PA_ERR_UNSUPPORTED;
  if (q_dtype != PA_F16 && q_dtype != PA_BF16) return PA_ERR_UNSUPPORTED;
  const bool byte_codes = cache->dtype >= PA_FP8_E4M3;  // FP8 or INT8, with scales
  if (!byte_codes && q_dtype != cache->dtype) return PA_ERR_UNSUPPORTED;
  if (partition_size != 0 &&
      (partition_size < kStageTok || partition_size > kMaxPartition ||
       partition_size % kStageTok || partition_size % cache->block_size))
    return PA_ERR_INVALID;
  WorkspaceLayout w;
  if (!layout_for(num_seqs, num_q_heads, cache->kv_heads, cache->head_dim, max_seq_len,
                  partition_size, &w))
    return PA_ERR_INVALID;
  if (workspace_bytes < w.total) return PA_ERR_INVALID;
  DeviceInfo dev;
  if (!current_device_info(&dev)) return cuda_fail(cudaGetLastError());

  const long long cap_table = static_cast<long long>(max_blocks_per_seq) * cache->block_size;
  const long long cap_parts = static_cast<long long>(w.max_parts) * w.partition;
  const long long cap = cap_table < cap_parts ? cap_table : cap_parts;

  uint8_t *ws = static_cast<uint8_t *>(workspace);
  DecodeParams p{};
  p.out = out;
  p.q = static_cast<const uint8_t *>(q);
  p.k_cache = static_cast<const uint8_t *>(k_cache);
  p.v_cache = static_cast<const uint8_t *>(v_cache);
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = cache->kv_heads;
  p.num_blocks = cache->num_blocks;
  p.block_size = cache->block_size;
  p.max_blocks = max_blocks_per_seq;
  p.partition_size = w.partition;
  p.max_parts = w.max_parts;
  p.len_cap = static_cast<int>(cap > 0x7fffffff ? 0x7fffffff : cap);
  const bool per_head = byte_codes && cache->k_head_scales != nullptr;
  p.qk_scale_log2 = scale * (byte_codes && !per_head ? cache->k_scale : 1.0f) * 1.4426950408889634f;
  p.v_scale = byte_codes && !per_head ? cache->v_scale : 1.0f;
  p.k_head_scale = per_head ? cache->k_head_scales : nullptr;
  p.v_head_scale = per_head ? cache->v_head_scales : nullptr;
  p.work = reinterpret_cast<int *>(ws);
  p.items = reinterpret_cast<int4 *>(ws + w.pairs_off);
  p.wide_items = reinterpret_cast<int4 *>(ws + w.wide_off);
  p.plan_join = ws + w.join_off;
  p.part_ml = reinterpret_cast<float2 *>(ws + w.ml_off);
  p.part_o = reinterpret_cast<float *>(ws + w.o_off);
  p.err = device_error;

  if (!encode_cache_map(&p.tmap_k, k_cache, cache) ||
      !encode_cache_map(&p.tmap_v, v_cache, cache))  // tiled views for the swizzled (tensor-path) stages
    return cuda_fail(cudaErrorInvalidValue);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  switch (cache->dtype) {
    case PA_F16: return dispatch_decode_f16(q_dtype, cache->head_dim, G, p, dev, s);
    case PA_BF16: return dispatch_decode_bf16(q_dtype, cache->head_dim, G, p, dev, s);
    case PA_FP8_E4M3: return dispatch_decode_e4m3(q_dtype, cache->head_dim, G, p, dev, s);
    case PA_FP8_E5M2: return dispatch_decode_e5m2(q_dtype, cache->head_dim, G, p, dev, s);
    case PA_INT8: return dispatch_decode_i8(q_dtype, cache->head_dim, G, p, dev, s);
  }
  return PA_ERR_UNSUPPORTED;
}

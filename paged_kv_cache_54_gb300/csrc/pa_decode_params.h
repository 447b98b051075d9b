// Parameters shared by the decode kernels and the host entry point.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"
#include "pa_host.h"

namespace pa {

constexpr int kStageTok = 64;          // tokens per pipeline stage
constexpr int kConsumerWarps = 4;      // each owns 16 tokens of a stage
constexpr int kThreads = 32 * (1 + kConsumerWarps);
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr int kMaxStages = 12;
constexpr int kMaxPartition = 1024;
// Wide items (runs of sequences that share a partition's blocks, decoded on
// the tensor cores): the query rows of one, and the fewest worth taking.
constexpr int kWideRows = 256;
constexpr int kWideMinRows = 64;
#ifndef PA_DECODE_CTAS_PER_SM
#define PA_DECODE_CTAS_PER_SM 3
#endif
constexpr int kCtasPerSm = PA_DECODE_CTAS_PER_SM;  // resident decode CTAs per SM
// Registers per thread that still let kCtasPerSm CTAs of kThreads reside on
// one SM.  The 64K-entry register file is split between the SM's four
// sub-partitions and a warp takes all its registers from one of them, so the
// sub-partition holding the most warps, ceil(warps / 4), sets the limit
// (registers are allocated in units of 8 per thread).
__host__ __device__ constexpr int regs_for_ctas(int ctas) {
  return (16384 / (((ctas * (kThreads / 32) + 3) / 4) * 32)) / 8 * 8 > 255
             ? 255
             : (16384 / (((ctas * (kThreads / 32) + 3) / 4) * 32)) / 8 * 8;
}
constexpr int kMaxRegs = regs_for_ctas(kCtasPerSm);
// Shared memory of the GB300 (sm_103a) SM, used to plan each kernel's
// resident CTAs (and so its register budget) at compile time; the launch
// re-plans from the device's own figures.
constexpr int kSmemPerSm = 233472;
constexpr int kSmemOptin = 232448;

enum StageFlags : int { kFirst = 1, kLast = 2, kEnd = 4 };

struct StageInfo {
  int s, h, p;
  int tok0;   // sequence position of the stage's first token
  int ntok;   // valid tokens in the stage (0..64)
  int flags;
  int L;      // sequence length (clamped to the table capacity)
  int nP;     // number of partitions of the sequence
  int k;      // sequences sharing the item's blocks (s .. s+k-1)
};

struct SmemHeader {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t combine;
  StageInfo info[kMaxStages];
  // (m, l) of each consumer warp's query columns at an item's end, one
  // buffer per item parity (a warp may reach the next item's end while
  // another still reads this one's)
  float comb_m[2][kConsumerWarps][8];
  float comb_l[2][kConsumerWarps][8];
  int abort;
};

struct DecodeParams {
  // tiled views of the caches for the TMA (unused when a row is < 128 bytes)
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  void *out;
  const uint8_t *q;
  const uint8_t *k_cache;
  const uint8_t *v_cache;
  const int32_t *block_tables;
  const int32_t *seq_lens;
  int num_seqs, num_q_heads, num_kv_heads, num_blocks, block_size, max_blocks;
  int partition_size, max_parts, len_cap;
  float qk_scale_log2;  // softmax scale * log2(e) * k_scale (k_scale = 1 with per-head scales)
  float v_scale;        // v_scale (1 with per-head scales)
  const float *k_head_scale;  // [num_kv_heads] or null: per-head scales of a one-byte cache
  const float *v_head_scale;
  int num_stages, stage_bytes, k_off, v_off, q_off, stages_off;
  int kmax;   // most sequences one item may batch
  int item_major;  // claims take every KV head of an item in turn (else head by head)
  int longest_first;  // items listed by stage count, longest first (else in slot order)
  int *work;  // [0] claim counter, [1] number of items, [2] number of wide items
  int4 *items;  // (first sequence, partition, sequences, 0)
  int4 *wide_items;  // the same, for the wide kernel
  int wide_seqs;     // sequences of a wide chunk (0: no wide items)
  int wide_min;      // fewest sequences that make a wide item
  int after_wide;    // the decode kernel follows the wide kernel (see decode_body)
  uint8_t *plan_join;  // [S * max_parts] rows of (s, q) and (s-1, q) differ (a CTA's
                       // flags, when they do not fit its shared memory)
  int plan_tbl_bytes;  // shared memory for a plan CTA's block-table rows (0: read in place)
  float2 *part_ml;  // [S * max_parts * Hq] (max in log2 units, sum)
  float *part_o;    // [S * max_parts * Hq * D], normalised by its own sum
  int *err;
};


// The wide items (runs of sequences sharing a partition's blocks) on the
// tensor cores, after the decode kernel (pa_prefill.cu).
pa_status launch_wide_items(const DecodeParams &d, int cache_dtype, int head_dim, cudaStream_t stream);

// One instantiation family per cache dtype (separate translation units).
pa_status dispatch_decode_f16(int q_dtype, int head_dim, int group, DecodeParams p,
                              const DeviceInfo &dev, cudaStream_t stream);
pa_status dispatch_decode_bf16(int q_dtype, int head_dim, int group, DecodeParams p,
                               const DeviceInfo &dev, cudaStream_t stream);
pa_status dispatch_decode_e4m3(int q_dtype, int head_dim, int group, DecodeParams p,
                               const DeviceInfo &dev, cudaStream_t stream);
pa_status dispatch_decode_e5m2(int q_dtype, int head_dim, int group, DecodeParams p,
                               const DeviceInfo &dev, cudaStream_t stream);
pa_status dispatch_decode_i8(int q_dtype, int head_dim, int group, DecodeParams p,
                             const DeviceInfo &dev, cudaStream_t stream);

}  // namespace pa

#pragma once
// Paged causal prefill on the 5th-generation tensor cores: attention of each
// sequence's new tokens (the part a prefix-cache hit did not cover) over all
// of its tokens in the paged cache.
//
// One CTA = one KV head h and 256 query rows of one sequence, as two tiles
// of 128; a row is a (new token, query head of h's group) pair, token-major,
// so a CTA holds 256 / G new tokens.  Every K/V stage staged in shared memory
// serves both tiles.  Each tile is the M = 128 dimension of tcgen05.mma, and
// its row r lives in tensor-memory lane r (columns 256 * tile + ...):
//   S = Q K^T   M 128, N = 64 keys of a stage, K = head_dim   (S in TMEM)
//   O += P V    M 128, N = head_dim,  K = the stage's 64 keys  (O in TMEM)
// Warps:
//   0..7  softmax, one warpgroup per tile: thread r of a warpgroup owns row
//         r.  It reads its S row from TMEM, applies the causal mask (key
//         position <= the row's position) on the stages that reach past
//         some row of its warp, and an online softmax in base 2 (packed
//         f32x2 arithmetic, the scale folded into the exponent's fma),
//         writes P (16-bit pairs) back over the S buffer it just read, where
//         P V takes it as a tensor-memory A operand, and rescales its O row in
//         TMEM only when the row maximum has grown by more than 2^8 (lazy
//         rescaling: P entries stay below 256).  P has a buffer per stage
//         parity, so the next stage's softmax does not wait for this P V.
//   8     TMA: Q once (one 4-D box per tile and 128-byte half of a row),
//         then K and V in stages of 64 keys, one tensor copy per (block,
//         head) tile that lands it as 8-row x 128-byte swizzled atoms (the
//         stage layout is described at kv_row_off).  Lane j issues block j's
//         copies, so a stage's copies go out from several threads at once;
//         the block-table entries come from two 32-entry windows held one
//         entry per lane, the next fetched while the current one is in use.
//         This warp initialises the
//         barriers and issues Q and the first stage before the set-up
//         barrier.
//   9,10  MMA, one warp per tile (one thread of each issues): the tile's S of
//         the next stage is issued before waiting for this stage's P, so the
//         tensor cores work on it while the softmax warps work on P (S is
//         double-buffered in TMEM for that).  A thread issues a product
//         about every 30 ns, so one issuing thread for both tiles would hold
//         one tile's P V behind the other tile's S; with one per tile, each
//         answers its own tile's P at once.  tcgen05.commit signals
//         completions on mbarriers; a K/V stage is free once both tiles'
//         P V have completed.  Tile 0's rows end 64 tokens before tile 1's,
//         so it runs only the stages its rows reach and releases the others
//         once they are filled.
// Epilogue: each softmax thread scales its O row by 1 / l, and the tile's
// rows go through its q buffer (free once the tile's products are done) so
// that they leave as whole rows, two rows per warp store.
// TMEM: all 512 columns (per tile S / P: 2 x 64, O: head_dim); one CTA per
// SM, five K/V stages in flight.
//
// One-byte caches (FP8 e4m3 / e5m2, INT8): the products take fp16 operands.
// The TMA warp copies each (block, head) tile of codes whole (one bulk copy
// per block for K and for V) into a ring of four code slots; warps 12..15,
// one on each SM sub-partition, widen the codes exactly to fp16 into three
// 16-bit stages of the layout above and mark each stage full (warp 11 only
// completes the third warpgroup).  The softmax warpgroups take 168
// registers a thread and the others 88 (setmaxnreg), within the 512 x 128
// the block is launched with.  A bf16 query tile is rewritten in place as
// fp16 by its softmax warps, times a power of two that brings its largest
// entry within fp16's range; the factor, and the K scale, go into the score
// scale, the V scale into the output.
#include <limits.h>
#include <math.h>

#include "pa_common.cuh"
#include "pa_host.h"

namespace pa {

struct PrefillParams {
  CUtensorMap tmap_q;  // [T, Hkv, G, head_dim] view of q, box {64, G, 1, 128/G}
  CUtensorMap tmap_k;  // 16-bit caches: [row group, half, row, 64] view, box = one (block, head) tile
  CUtensorMap tmap_v;
  const uint8_t *k_cache;  // one-byte caches: the codes
  const uint8_t *v_cache;
  void *out;
  const int32_t *cu_q;
  const int32_t *block_tables;
  const int32_t *seq_lens;
  int num_q_heads, num_kv_heads, num_blocks, block_size, max_blocks;
  int num_q_tokens;     // rows of q and out: every sequence's rows must lie inside
  int max_q_len;        // the caller's bound on any sequence's new tokens
  float qk_scale_log2;  // softmax scale * log2(e) (* the per-tensor K scale of a one-byte cache)
  float v_scale;        // per-tensor V scale of a one-byte cache, else 1
  const float *k_head_scale;  // one-byte caches: [num_kv_heads] scales, or null
  const float *v_head_scale;
  int *err;
  // the decode's wide items (shared-prefix chunks), for wide_decode_kernel:
  // (first sequence, partition, sequences) each; their count on the device
  const int4 *wide_items;
  const int *wide_count;
  float2 *part_ml;  // the decode's split-K partials, [S * max_parts * Hq] (m, l)
  float *part_o;    // and [S * max_parts * Hq * D], normalised by l
  int max_parts, partition_size;
};

namespace {

constexpr int kPfTileRows = 128;     // rows per tile (M)
constexpr int kPfTiles = 2;          // tiles per CTA
constexpr int kPfRows = kPfTileRows * kPfTiles;
constexpr int kPfKeys = 64;          // keys per pipeline stage
constexpr int kPfTmaWarp = 8;
constexpr int kPfMmaWarp = 9;  // and 10: one issuing warp per tile
constexpr int kPfConvWarp0 = 12;  // one-byte caches: warps 12..15 widen the codes
constexpr int kPfConvWarps = 4;
// threads: softmax 8 warps, TMA, 2 MMA (one-byte caches: + an idle warp
// that completes the third warpgroup, + the widening warpgroup)
__host__ __device__ constexpr int pf_threads(bool kv8) { return 32 * (kv8 ? 16 : 11); }
constexpr int kPfHalf = kPfKeys * 128;  // bytes of one 128-byte column half of a 64-key stage
// A K or V stage holds its 64 keys as 8 groups of 8 rows.  Each group
// is stored as its 128-byte row halves, one after the other, and each
// half is an 8-row x 128-byte atom with the 128-byte swizzle.  A
// (block, head) tile is a whole number of groups, so one tensor copy lands
// it.  The tensor cores read K with the group stride as the 8-row stride
// (and step to the next half by one atom), and read V with the atom as the
// column-half stride and the group as the 8-key stride.
constexpr int kPfAtom = 1024;
template <int NH>
__device__ __forceinline__ int kv_row_off(int key, int hf) {  // byte offset of (key, half) in a stage
  return (key >> 3) * NH * kPfAtom + hf * kPfAtom + (key & 7) * 128;
}
constexpr int kPfStages = 5;      // 16-bit K/V stages (three with one-byte caches)
constexpr int kPfCodeSlots = 4;   // one-byte caches: stages of codes in flight
constexpr uint32_t kPfTmemCols = 512;
constexpr uint32_t kPfTileCols = 256;  // TMEM columns per tile
constexpr float kPfLazy = 8.f;  // rescale O only when the row maximum grows by more (base 2)



template <int D, bool KV8>
struct PfLayout {
  static constexpr int NH = D / 64;  // 128-byte halves of a 16-bit row
  static constexpr int NS = KV8 ? 3 : kPfStages;  // 16-bit K/V stages
  static constexpr int NC = KV8 ? kPfCodeSlots : 0;  // code slots
  static constexpr int Q_OFF = 1024;
  static constexpr int Q_HALF = kPfTileRows * 128;
  static constexpr int Q_TILE = NH * Q_HALF;
  static constexpr int STAGE_OFF = Q_OFF + kPfTiles * Q_TILE;
  static constexpr int STAGE_BYTES = 2 * NH * kPfHalf;  // K halves, then V halves
  static constexpr int CODE_OFF = STAGE_OFF + NS * STAGE_BYTES;
  static constexpr int CODE_BYTES = 2 * kPfKeys * D;    // K codes [key][d], then V codes
  static constexpr int SMEM = CODE_OFF + NC * CODE_BYTES;
};

struct PfHeader {
  uint64_t kv_full[kPfStages];
  uint64_t kv_empty[kPfStages];
  uint64_t s_full[kPfTiles][2];
  uint64_t p_full[kPfTiles][2];  // by stage parity: the softmax may run a stage ahead
  uint64_t pv_done[kPfTiles];
  uint64_t o_ready[kPfTiles];    // once: the tile's last P V has completed
  uint64_t q_full;
  uint64_t fin[kPfTiles];
  uint64_t code_full[kPfCodeSlots];  // one-byte caches: a stage's codes have landed
  uint64_t code_empty[kPfCodeSlots]; // and the slot has been widened
  uint64_t q_ready[kPfTiles];        // a bf16 query tile has been rewritten as fp16
  float qmax[kPfTiles][4];           // its warps' largest |q|
  uint32_t tmem_base;
  int abort;
};

// Widen the codes of a slot (K then V, the first `keys` keys of each) into a
// 16-bit stage: 8 codes make one 16-byte chunk, and chunk c of key row k of
// half hf lands in that row of the stage's atom layout at chunk c ^ (k mod
// 8).  A warp iteration converts 32 chunks, lane = (key, half, chunk), and
// the PARTS widening warps take interleaved iterations.  A warp's
// successive keys are then a multiple of 8 apart, so each lane keeps one
// swizzle phase and steps its source and destination by constants.  keys
// is a multiple of 8.
template <int KVT, int D, int PARTS>
__device__ __forceinline__ void widen_codes(const uint8_t *slot, uint8_t *stage, int keys, int lane, int part) {
  constexpr int NH = D / 64;
  constexpr int KPI = 32 / (NH * 8);     // keys per warp iteration
  constexpr int KSTEP = PARTS * KPI;     // keys between one warp's iterations
  static_assert(KSTEP % 8 == 0, "a lane's keys must keep their row in the atom");
  constexpr int SRC_STEP = KSTEP * D;
  constexpr int DST_STEP = KSTEP / 8 * NH * kPfAtom;
  const int kr = lane / (NH * 8), hf = (lane >> 3) % NH, c = lane & 7;
  const int k0 = part * KPI + kr;
  const int n = keys > k0 ? (keys - k0 + KSTEP - 1) / KSTEP : 0;  // this lane's keys of each tensor
  constexpr int B = 4;
#pragma unroll
  for (int tv = 0; tv < 2; ++tv) {
    const uint8_t *src = slot + tv * kPfKeys * D + k0 * D + hf * 64 + c * 8;
    uint8_t *dst = stage + tv * NH * kPfHalf + kv_row_off<NH>(k0, hf) + ((c ^ (k0 & 7)) << 4);
    // the loads of a batch go before its stores: the compiler cannot tell
    // that the stores do not alias them
    for (int m0 = 0; m0 < n; m0 += B) {
      uint2 w[B];
#pragma unroll
      for (int u = 0; u < B; ++u)
        if (m0 + u < n) w[u] = *reinterpret_cast<const uint2 *>(src + (m0 + u) * SRC_STEP);
#pragma unroll
      for (int u = 0; u < B; ++u) {
        if (m0 + u < n) {
          uint4 o;
          byte4_to_half2x2<KVT>(w[u].x, o.x, o.y);
          byte4_to_half2x2<KVT>(w[u].y, o.z, o.w);
          *reinterpret_cast<uint4 *>(dst + (m0 + u) * DST_STEP) = o;
        }
      }
    }
  }
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Two fp32 lanes in one 64-bit register pair, for the packed f32x2 arithmetic.
__device__ __forceinline__ uint64_t f2(float x, float y) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(x), "f"(y));
  return d;
}
__device__ __forceinline__ void f2_split(uint64_t v, float &x, float &y) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {  // a * b + c, both lanes
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// DT: the type of q and out; KVT: the cache's (DT itself for 16-bit caches).
// SD (shared decode): the CTA decodes one wide item of the paged decode
// instead of prefilling new tokens.  A wide item is a run of k sequences
// whose block tables agree over partition q (a shared prefix): their decode
// queries are the rows of the tiles (row r: sequence s0 + r / G, query head
// h * G + r % G, read from q [S, Hq, D] exactly as new tokens are read from
// a prefill's q), the keys are the partition's P tokens of the shared blocks
// (no mask: every row follows them all), and each row's (m, l) and O / l go
// to the decode's split-K partials of (sequence, partition q), which the
// decode's merge combines with the other partitions.
template <int DT, int KVT, int D, int G, bool SD>
__device__ __forceinline__ void prefill_body(const PrefillParams &p) {
  constexpr bool KV8 = is_byte(KVT);
  constexpr int MT = KV8 ? kF16 : DT;          // the products' operand type
  constexpr bool QCONV = KV8 && DT == kBF16;   // q is rewritten as fp16 first
  using Lay = PfLayout<D, KV8>;
  constexpr int NH = Lay::NH;
  constexpr int NS = Lay::NS;
  constexpr int NC = Lay::NC;
  constexpr int QT = kPfTileRows / G;  // new tokens per tile
  constexpr int QC = kPfRows / G;      // new tokens per CTA
  constexpr int KSTEPS = D / 16;
  constexpr int AB = MT == kF16 ? 0 : 1;
  constexpr uint32_t IDESC_QK = umma_idesc_f16(AB, kPfTileRows, kPfKeys, false);
  constexpr uint32_t IDESC_PV = umma_idesc_f16(AB, kPfTileRows, D, true);
  extern __shared__ __align__(1024) uint8_t smem[];
  PfHeader &hdr = *reinterpret_cast<PfHeader *>(smem);
  const int cta = SD ? 0 : gridDim.x - 1 - blockIdx.x;  // the longest (last) token ranges start first
  const int h = blockIdx.z;
  int s = blockIdx.y, qpart = 0, nseq = 0;
  if constexpr (SD) {  // the wide item: read from L2 (the plan wrote it in an earlier grid)
    if (static_cast<int>(blockIdx.x) >= __ldcg(p.wide_count)) return;
    const int4 it = __ldcg(p.wide_items + blockIdx.x);
    s = it.x;
    qpart = it.y;
    nseq = it.z;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the tensor-map descriptors are fetched while the lengths are read
  if (warp == kPfTmaWarp && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_q)) : "memory");
    if constexpr (!KV8) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_k)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_v)) : "memory");
    }
  }
  // and the TMA warp reads the sequence's first 64 block-table entries: a
  // window of 32 (lane j: entry 32 w + j) in use and the next one
  // (SD: the partition's entries, from its first)
  const int kofs = SD ? qpart * (p.partition_size / p.block_size) : 0;
  const int tbl_len = p.max_blocks - kofs;
  const int32_t *table = p.block_tables + static_cast<size_t>(s) * p.max_blocks + kofs;
  int win = 0, win_next = 0;
  if (warp == kPfTmaWarp) {
    if (lane < tbl_len) win = __ldg(table + lane);
    if (32 + lane < tbl_len) win_next = __ldg(table + 32 + lane);
  }

  int q0, n, L;
  if constexpr (SD) {
    q0 = s;                  // the sequences' query rows
    n = nseq;
    L = p.partition_size;    // the keys of the partition
    if (n < 1 || n > QC || s < 0 || n > p.num_q_tokens - s || qpart < 0 || qpart >= p.max_parts ||
        tbl_len < L / p.block_size) {
      if (threadIdx.x == 0) record_error(p.err, kErrSeqLen);
      return;
    }
  } else {
    q0 = __ldg(p.cu_q + s);
    n = __ldg(p.cu_q + s + 1) - q0;
    L = __ldg(p.seq_lens + s);
    // the rows [q0, q0 + n) of q and out must exist: out is written with plain
    // stores, so a bad cu_q_lens entry skips the sequence instead
    if (n < 0 || q0 < 0 || n > p.num_q_tokens - q0 || n > p.max_q_len || L < n ||
        L > p.max_blocks * p.block_size) {
      if (threadIdx.x == 0 && blockIdx.x == 0) record_error(p.err, kErrSeqLen);
      return;
    }
    if (cta * QC >= n) return;
  }
  if ((smem_addr(smem) & 1023u) != 0) {  // the swizzle needs 1024-byte atoms
    if (threadIdx.x == 0) record_error(p.err, kErrSmemAlign);
    return;
  }
  const int tiles = cta * QC + QT < n ? 2 : 1;          // the second tile may hold no new token
  // position of new token 0 (SD: past every key, so nothing is masked)
  const int pos0 = SD ? (1 << 29) : L - n;
  const int kv_end = SD ? L : pos0 + min(n, (cta + 1) * QC);  // keys 0..kv_end-1 are needed
  const int n_stages = (kv_end + kPfKeys - 1) / kPfKeys;
  // stages a tile needs: tile 0's rows end QT tokens before tile 1's, so its
  // products stop a stage earlier unless tile 1 is empty (SD: all of them)
  auto tile_stages = [&](int t) {
    return SD ? n_stages : (pos0 + min(n, cta * QC + (t + 1) * QT) + kPfKeys - 1) / kPfKeys;
  };
  uint8_t *qs = smem + Lay::Q_OFF;
  uint8_t *stages = smem + Lay::STAGE_OFF;
  uint8_t *codes = smem + Lay::CODE_OFF;
  volatile int *abort = &hdr.abort;
  const int bs = p.block_size;
  const int bpt = kPfKeys / bs;  // blocks per stage (<= 8)
  auto stage_blocks = [&](int i) { return min(bpt, (kv_end - i * kPfKeys + bs - 1) / bs); };
  // The producer's copies of stage i, issued by the whole TMA warp in stage
  // order: lane j copies block j of the stage, its table entry taken from
  // the window, and the windows move on (the next one fetched) once a
  // stage ends a window.
  // 16-bit caches: each (block, head) tile of K and V by one tensor copy
  // into stage i % NS.  One-byte caches: the codes of each block by one bulk
  // copy into slot i % NC, widened by the widening warps.
  auto issue_stage = [&](int i) {
    const int nblk = stage_blocks(i);
    const int e0 = i * bpt;  // the stage's first entry; bpt divides 32
    int phys = __shfl_sync(0xffffffffu, win, (e0 & 31) + (lane & (bpt - 1)));
    if (((e0 + bpt) & 31) == 0) {
      win = win_next;
      win_next = e0 + bpt + 32 + lane < tbl_len ? __ldg(table + e0 + bpt + 32 + lane) : 0;
    }
    if (lane < nblk && (phys < 0 || phys >= p.num_blocks)) {
      record_error(p.err, kErrBlockIndex);
      phys = 0;  // read a valid block; the result is void and flagged
    }
    if constexpr (KV8) {
      uint8_t *cb = codes + (i % NC) * Lay::CODE_BYTES;
      const uint32_t tile = static_cast<uint32_t>(bs) * D;
      if (lane == 0) mbar_arrive_expect_tx(&hdr.code_full[i % NC], 2u * nblk * tile);
      __syncwarp();
      if (lane < nblk) {
        const size_t off = (static_cast<size_t>(phys) * p.num_kv_heads + h) * tile;
        bulk_g2s(cb + lane * tile, p.k_cache + off, tile, &hdr.code_full[i % NC]);
        bulk_g2s(cb + kPfKeys * D + lane * tile, p.v_cache + off, tile, &hdr.code_full[i % NC]);
      }
    } else {
      const int st = i % NS;
      uint8_t *kb = stages + st * Lay::STAGE_BYTES;
      uint8_t *vb = kb + NH * kPfHalf;
      if (lane == 0) mbar_arrive_expect_tx(&hdr.kv_full[st], 2u * NH * static_cast<uint32_t>(nblk * bs) * 128u);
      __syncwarp();
      if (lane < nblk) {
        const int g0 = (phys * p.num_kv_heads + h) * (bs / 8);  // the tile's first row group
        tma_load_4d(kb + lane * bs * NH * 128, &p.tmap_k, 0, 0, 0, g0, &hdr.kv_full[st]);
        tma_load_4d(vb + lane * bs * NH * 128, &p.tmap_v, 0, 0, 0, g0, &hdr.kv_full[st]);
      }
    }
  };
  // The TMA warp initialises the barriers and issues q and the first stage
  // before the set-up barrier, so that those copies are in flight while
  // tensor memory is allocated.  (The copy engine takes one copy about every
  // 100 clocks, so issuing more here would only hold the barrier longer.)
  const int pre = 1;
  if (warp == kPfTmaWarp) {
    if (lane == 0) {
      for (int i = 0; i < NS; ++i) {
        mbar_init(&hdr.kv_full[i], KV8 ? kPfConvWarps : 1);  // one-byte caches: each widening warp
        mbar_init(&hdr.kv_empty[i], tiles);  // each tile's MMA warp frees the stage
      }
      for (int c = 0; c < NC; ++c) {
        mbar_init(&hdr.code_full[c], 1);
        mbar_init(&hdr.code_empty[c], kPfConvWarps);
      }
      for (int t = 0; t < kPfTiles; ++t) {
        mbar_init(&hdr.q_ready[t], 1);
        mbar_init(&hdr.s_full[t][0], 1);
        mbar_init(&hdr.s_full[t][1], 1);
        mbar_init(&hdr.p_full[t][0], kPfTileRows);
        mbar_init(&hdr.p_full[t][1], kPfTileRows);
        mbar_init(&hdr.pv_done[t], 1);
        mbar_init(&hdr.o_ready[t], 1);
      }
      mbar_init(&hdr.q_full, 1);
      mbar_init(&hdr.fin[0], 1);
      mbar_init(&hdr.fin[1], 1);
      hdr.abort = 0;
      fence_mbar_init();
      mbar_arrive_expect_tx(&hdr.q_full, tiles * NH * kPfTileRows * 128u);
      for (int t = 0; t < tiles; ++t)
  #pragma unroll
        for (int hf = 0; hf < NH; ++hf)
          tma_load_4d(qs + t * Lay::Q_TILE + hf * Lay::Q_HALF, &p.tmap_q, hf * 64, 0, h, q0 + cta * QC + t * QT,
                      &hdr.q_full);
    }
    __syncwarp();
    for (int i = 0; i < pre; ++i) issue_stage(i);
  }
  if (warp == kPfMmaWarp) tc_alloc(&hdr.tmem_base, kPfTmemCols);
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = hdr.tmem_base;

  // Roles.  With one-byte caches the softmax warpgroups take 168 registers
  // a thread and the other two (TMA, MMA, widening) 88: 256 x 168 +
  // 256 x 88 = 512 x 128, the registers the block is launched with.
  if (warp < 4 * kPfTiles) {
    if constexpr (KV8) asm volatile("setmaxnreg.inc.sync.aligned.u32 168;" ::: "memory");
    if (warp / 4 < tiles) {
      // ------------------------------------------------------------ softmax
      const int t = warp / 4;                  // tile
      const int r = threadIdx.x & 127;         // row = TMEM lane
      const int tok = cta * QC + t * QT + r / G;
      const int pos = pos0 + min(tok, n - 1);  // rows past the new tokens take the last one's (not stored)
      const uint32_t trow = tmem + t * kPfTileCols + (static_cast<uint32_t>(32 * (warp & 3)) << 16);
      float m = -INFINITY, l = 0.f;
      bool ok = true;
      // score scale (base 2) and output scale; one-byte caches fold in their
      // K and V scales, and a rewritten q its power-of-two factor
      float c = p.qk_scale_log2, vsc = 1.f;
      if constexpr (KV8) {
        vsc = p.v_scale;
        if (p.k_head_scale != nullptr) {
          c *= __ldg(p.k_head_scale + h);
          vsc = __ldg(p.v_head_scale + h);
        }
      }
      if constexpr (QCONV) {
        // the tile's q (bf16, swizzled in place; a pure elementwise rewrite
        // keeps the layout): scale by 2^e so that max |q| <= 2^15, round to fp16
        ok = __all_sync(0xffffffffu, mbar_wait(&hdr.q_full, 0, abort));
        uint4 *qt = reinterpret_cast<uint4 *>(qs + t * Lay::Q_TILE);
        constexpr int CH = Lay::Q_TILE / 16 / kPfTileRows;  // 16-byte chunks per thread
        float amax = 0.f;
        if (ok) {
  #pragma unroll
          for (int j = 0; j < CH; ++j) {
            const uint4 v = qt[j * kPfTileRows + r];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  #pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float2 x = half2_bits_to_float2<kBF16>(w[u]);
              amax = fmaxf(amax, fmaxf(fabsf(x.x), fabsf(x.y)));
            }
          }
        }
  #pragma unroll
        for (int o2 = 1; o2 < 32; o2 <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o2));
        if (lane == 0) hdr.qmax[t][warp & 3] = amax;
        named_bar_sync(1 + t, kPfTileRows);
        amax = fmaxf(fmaxf(hdr.qmax[t][0], hdr.qmax[t][1]), fmaxf(hdr.qmax[t][2], hdr.qmax[t][3]));
        float f = 1.f;
        if (amax > 16384.f && amax <= 3.0e38f) {
          int ex;
          frexpf(amax, &ex);
          f = ldexpf(1.f, 14 - ex);
        }
        if (ok) {
  #pragma unroll
          for (int j = 0; j < CH; ++j) {
            uint4 v = qt[j * kPfTileRows + r];
            uint32_t *w = reinterpret_cast<uint32_t *>(&v);
  #pragma unroll
            for (int u = 0; u < 4; ++u) {
              const float2 x = half2_bits_to_float2<kBF16>(w[u]);
              w[u] = pack2_rn<kF16>(x.x * f, x.y * f);
            }
            qt[j * kPfTileRows + r] = v;
          }
        }
        fence_proxy_async_smem();  // the rewritten q visible to the tensor cores
        named_bar_sync(1 + t, kPfTileRows);
        if (r == 0) mbar_arrive(&hdr.q_ready[t]);
        c /= f;
      }
      const int nst = tile_stages(t);
      for (int i = 0; i < nst && ok; ++i) {
        if (!__all_sync(0xffffffffu, mbar_wait(&hdr.s_full[t][i & 1], (i >> 1) & 1, abort))) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const int k0 = i * kPfKeys;
        float sv[kPfKeys];
        {
          uint32_t raw[32];
          tc_ld32(trow + (i & 1) * kPfKeys, raw);
  #pragma unroll
          for (int j = 0; j < 32; ++j) sv[j] = __uint_as_float(raw[j]);
          tc_ld32(trow + (i & 1) * kPfKeys + 32, raw);
  #pragma unroll
          for (int j = 0; j < 32; ++j) sv[32 + j] = __uint_as_float(raw[j]);
        }
        // Most stages lie wholly at or before every row of the warp: no mask,
        // and with a positive scale the maximum is taken on the raw scores and
        // the scale folded into the exponent's one fma.  Otherwise the scores
        // are scaled, then masked (key position > row position: -inf).
        const bool plain = c > 0.f && __all_sync(0xffffffffu, k0 + kPfKeys - 1 <= pos);
        float mx, cm;
        if (plain) {
          float a = sv[0], b = sv[32];  // two chains of 3-input maxima
  #pragma unroll
          for (int j = 1; j < 31; j += 2) {
            a = fmax3(a, sv[j], sv[j + 1]);
            b = fmax3(b, sv[32 + j], sv[33 + j]);
          }
          mx = fmax3(a, b, fmaxf(sv[31], sv[63])) * c;
          cm = c;
        } else {
          float mx0 = -INFINITY, mx1 = -INFINITY;
  #pragma unroll
          for (int j = 0; j < kPfKeys; j += 2) {
            sv[j] = (k0 + j <= pos) ? sv[j] * c : -INFINITY;
            sv[j + 1] = (k0 + j + 1 <= pos) ? sv[j + 1] * c : -INFINITY;
            mx0 = fmaxf(mx0, sv[j]);
            mx1 = fmaxf(mx1, sv[j + 1]);
          }
          mx = fmaxf(mx0, mx1);
          cm = 1.f;
        }
        const bool grow = mx > m + kPfLazy;
        if (__any_sync(0xffffffffu, grow && i > 0)) {  // tcgen05.ld / st are warp-wide
          // O holds the previous P V: wait for it, then rescale.  S of this
          // stage was issued after the P V before the previous one, and the
          // tensor pipe completes in order, so pv_done is at most one phase
          // behind here and the parity wait is exact.
          if (!__all_sync(0xffffffffu, mbar_wait(&hdr.pv_done[t], (i - 1) & 1, abort))) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const float alpha = grow ? fast_exp2(m - mx) : 1.f;
  #pragma unroll
          for (int c = 0; c < D; c += 32) {
            uint32_t ov[32];
            tc_ld32(trow + 2 * kPfKeys + c, ov);
  #pragma unroll
            for (int j = 0; j < 32; ++j) ov[j] = __float_as_uint(__uint_as_float(ov[j]) * alpha);
            tc_st32(trow + 2 * kPfKeys + c, ov);
          }
        }
        if (grow) {
          l *= fast_exp2(m - mx);  // 0 while m is -inf (l is 0 then)
          m = mx;
        }
        const float base = m == -INFINITY ? 0.f : m;
        // p = 2^(s * cm - base), two lanes per fma and per add of the row sum
        const uint64_t cm2 = f2(cm, cm), nb2 = f2(-base, -base);
        uint64_t sum0 = f2(0.f, 0.f), sum1 = sum0;
        uint32_t pw[kPfKeys / 2];
  #pragma unroll
        for (int j = 0; j < kPfKeys; j += 2) {
          float x, y;
          f2_split(ffma2(f2(sv[j], sv[j + 1]), cm2, nb2), x, y);
          const float a = fast_exp2(x), b = fast_exp2(y);
          pw[j / 2] = pack2_rn<MT>(a, b);
          if ((j & 2) == 0)
            sum0 = fadd2(sum0, f2(a, b));
          else
            sum1 = fadd2(sum1, f2(a, b));
        }
        {
          float l0, l1, l2, l3;
          f2_split(sum0, l0, l1);
          f2_split(sum1, l2, l3);
          l += (l0 + l1) + (l2 + l3);
        }
        tc_st32(trow + (i & 1) * kPfKeys, pw);  // P over the S buffer just read
        if (k0 + kPfKeys > kv_end) {
          // keys past kv_end hold stale (possibly NaN) values: zero their V rows,
          // since 0 * NaN would reach O.  Each tile does it before its own P V
          // (the tiles' products are issued independently); both write zeros.
          if (!__all_sync(0xffffffffu, mbar_wait(&hdr.kv_full[i % NS], (i / NS) & 1, abort))) {
            ok = false;
            break;
          }
          uint8_t *vb = stages + (i % NS) * Lay::STAGE_BYTES + NH * kPfHalf;
          const int z0 = kv_end - k0;
          for (int idx = r; idx < (kPfKeys - z0) * 8 * NH; idx += kPfTileRows) {
            const int hf = idx / ((kPfKeys - z0) * 8), rem = idx % ((kPfKeys - z0) * 8);
            *reinterpret_cast<uint4 *>(vb + kv_row_off<NH>(z0 + rem / 8, hf) + (rem % 8) * 16) =
                make_uint4(0u, 0u, 0u, 0u);
          }
          fence_proxy_async_smem();  // the zeroed V rows visible to the tensor cores
        }
        tc_fence_before_sync();  // P and O stores ordered before the arrive
        mbar_arrive(&hdr.p_full[t][i & 1]);
      }
      if (!ok) {
        record_error(p.err, kErrTimeout);
        *abort = 1;
      } else if (__all_sync(0xffffffffu, mbar_wait(&hdr.o_ready[t], 0, abort))) {
        // (pv_done cannot serve here: the softmax does not wait for every P V,
        // so the last two may both be pending and a parity wait would take the
        // older phase for the newer)
        tc_fence_after_sync();
        const float inv = vsc / l;
        if constexpr (SD) {
          // the row's split-K partial of partition qpart: O / l and (m, l),
          // kept in L2 for the merge (rows past the item's sequences skipped)
          const int rows = min(kPfTileRows, (n - t * QT) * G);
          const bool mine = r < rows;
          const int sr = q0 + t * QT + r / G;
          const size_t idx = (static_cast<size_t>(sr) * p.max_parts + qpart) * p.num_q_heads + h * G + r % G;
          float *po = p.part_o + idx * D;
          const uint64_t keep = l2_policy_evict_last();
  #pragma unroll
          for (int c = 0; c < D; c += 32) {
            uint32_t ov[32];
            tc_ld32(trow + 2 * kPfKeys + c, ov);
            if (mine) {
  #pragma unroll
              for (int j = 0; j < 32; j += 4)
                st_global_f4_hint(po + c + j,
                                  make_float4(__uint_as_float(ov[j]) * inv, __uint_as_float(ov[j + 1]) * inv,
                                              __uint_as_float(ov[j + 2]) * inv, __uint_as_float(ov[j + 3]) * inv),
                                  keep);
            }
          }
          if (mine) st_global_f2_hint(reinterpret_cast<float *>(p.part_ml + idx), m, l, keep);
        } else {
        // O / l goes through this tile's q buffer (its products have all
        // completed, so no product reads it any more): each thread writes
        // its row, 16-byte chunk ch at ch ^ (row mod 8), then the tile's
        // threads copy whole rows out, each warp instruction two rows of
        // 16-bit outputs (rows past the sequence's new tokens are skipped).
        constexpr int RB = D * 2;      // bytes of an output row
        constexpr int CPR = RB / 16;   // 16-byte chunks of a row
        uint8_t *stg = qs + t * Lay::Q_TILE;
  #pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t ov[32];
          tc_ld32(trow + 2 * kPfKeys + c, ov);
  #pragma unroll
          for (int j = 0; j < 32; j += 8) {
            uint4 v;
            v.x = pack2_rn<DT>(__uint_as_float(ov[j]) * inv, __uint_as_float(ov[j + 1]) * inv);
            v.y = pack2_rn<DT>(__uint_as_float(ov[j + 2]) * inv, __uint_as_float(ov[j + 3]) * inv);
            v.z = pack2_rn<DT>(__uint_as_float(ov[j + 4]) * inv, __uint_as_float(ov[j + 5]) * inv);
            v.w = pack2_rn<DT>(__uint_as_float(ov[j + 6]) * inv, __uint_as_float(ov[j + 7]) * inv);
            *reinterpret_cast<uint4 *>(stg + r * RB + ((((c + j) / 8) ^ (r & 7)) << 4)) = v;
          }
        }
        named_bar_sync(1 + t, kPfTileRows);
        const int tok0 = cta * QC + t * QT;                          // the tile's first token
        const int rows = min(kPfTileRows, (n - tok0) * G);           // rows with a new token
        uint8_t *obase = static_cast<uint8_t *>(p.out) + (static_cast<size_t>(q0 + tok0) * p.num_q_heads + h * G) * RB;
        const size_t tok_stride = static_cast<size_t>(p.num_q_heads) * RB;
  #pragma unroll 4
        for (int idx = r; idx < rows * CPR; idx += kPfTileRows) {
          const int rr = idx / CPR, ch = idx % CPR;
          const uint4 v = *reinterpret_cast<const uint4 *>(stg + rr * RB + ((ch ^ (rr & 7)) << 4));
          *reinterpret_cast<uint4 *>(obase + (rr / G) * tok_stride + (rr % G) * RB + ch * 16) = v;
        }
        }  // SD
      } else {
        record_error(p.err, kErrTimeout);
        *abort = 1;
      }
    }
  } else if (warp < 12) {
    if constexpr (KV8) asm volatile("setmaxnreg.dec.sync.aligned.u32 88;" ::: "memory");
    if (warp == kPfTmaWarp) {
      // ------------------------------------------------------------ TMA
      // The rest of the stages, each once its slot has been freed (16-bit
      // stages by both tiles' products, code slots by the widening warps).
      const int slots = KV8 ? NC : NS;
      int issued = pre;
      bool ok = true;
      for (int i = pre; i < n_stages; ++i) {
        bool freed = true;
        if (lane == 0 && i >= slots)
          freed = mbar_wait(KV8 ? &hdr.code_empty[i % NC] : &hdr.kv_empty[i % NS], ((i / slots) - 1) & 1, abort);
        if (!__shfl_sync(0xffffffffu, freed, 0)) {
          ok = false;
          break;
        }
        issue_stage(i);
        issued = i + 1;
      }
      if (lane == 0) {
        if (!ok) {
          record_error(p.err, kErrTimeout);
          *abort = 1;
          // wait, within the limit, for the copies still in flight
          for (int j = max(0, issued - slots); j < issued; ++j)
            mbar_wait(KV8 ? &hdr.code_full[j % NC] : &hdr.kv_full[j % NS], (j / slots) & 1, nullptr);
        }
        mbar_wait(&hdr.q_full, 0, nullptr);
      }
    } else if (warp == kPfMmaWarp || warp == kPfMmaWarp + 1) {
      // ------------------------------------------------------------ MMA (tile t)
      const int t = warp - kPfMmaWarp;
      if (lane == 0 && t < tiles) {
        bool ok = mbar_wait(QCONV ? &hdr.q_ready[t] : &hdr.q_full, 0, abort);
        const uint32_t qt = smem_addr(qs) + t * Lay::Q_TILE;
        const uint32_t saddr = smem_addr(stages);
        const uint32_t tt = tmem + t * kPfTileCols;
        auto issue_qk = [&](int i) -> bool {
          const int st = i % NS;
          if (!mbar_wait(&hdr.kv_full[st], (i / NS) & 1, abort)) return false;
          tc_fence_after_sync();
          // descriptors of the first k-step; a k-step advances the start
          // address field (16-byte units) by 32 bytes, a row half by a
          // region of q and by one atom of K
          const uint64_t a0 = umma_desc_sw128(qt, 16, 1024);
          const uint64_t b0 = umma_desc_sw128(saddr + st * Lay::STAGE_BYTES, 16, NH * kPfAtom);
          const uint32_t d = tt + (i & 1) * kPfKeys;
  #pragma unroll
          for (int kk = 0; kk < KSTEPS; ++kk) {
            const uint32_t off = (kk % 4) * 32;  // 16 elements = 32 bytes into the swizzled row
            tc_mma_f16(d, a0 + (((kk / 4) * Lay::Q_HALF + off) >> 4), b0 + (((kk / 4) * kPfAtom + off) >> 4),
                       IDESC_QK, kk > 0);
          }
          tc_commit(&hdr.s_full[t][i & 1]);
          return true;
        };
        const int nst = tile_stages(t);
        if (ok) ok = issue_qk(0);
        for (int i = 0; i < nst && ok; ++i) {
          if (i + 1 < nst && !issue_qk(i + 1)) {
            ok = false;
            break;
          }
          if (!mbar_wait(&hdr.p_full[t][i & 1], (i >> 1) & 1, abort)) {
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t b0 =
              umma_desc_sw128(saddr + (i % NS) * Lay::STAGE_BYTES + NH * kPfHalf, kPfAtom, NH * kPfAtom);
  #pragma unroll
          for (int kk = 0; kk < kPfKeys / 16; ++kk)  // 16 keys: 8 columns of P, two row groups of V
            tc_mma_f16_ta(tt + 2 * kPfKeys, tt + (i & 1) * kPfKeys + kk * 8, b0 + kk * (2 * NH * kPfAtom >> 4), IDESC_PV,
                          (i > 0 || kk > 0) ? 1u : 0u);
          tc_commit(&hdr.pv_done[t]);
          if (i + 1 == nst) tc_commit(&hdr.o_ready[t]);
          tc_commit(&hdr.kv_empty[i % NS]);
        }
        // stages wholly after this tile's rows: each is released once it has
        // been filled, so that its slot's phase still needs the other tile
        for (int i = nst; i < n_stages && ok; ++i) {
          if (!mbar_wait(&hdr.kv_full[i % NS], (i / NS) & 1, abort)) {
            ok = false;
            break;
          }
          tc_commit(&hdr.kv_empty[i % NS]);
        }
        if (!ok) {
          record_error(p.err, kErrTimeout);
          *abort = 1;
        }
        // every product this thread issued has completed before the memory is released
        tc_commit(&hdr.fin[t]);
        mbar_wait(&hdr.fin[t], 0, nullptr);
      }
    }
  } else {
    if constexpr (KV8) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 88;" ::: "memory");
      // ------------------------------------------------------------ widening
      // warp 12 + q widens warp-iterations q, q + 4, ... of every stage
      const int q = warp - kPfConvWarp0;
      bool ok = true;
      for (int i = 0; i < n_stages; ++i) {
        const int st = i % NS;
        if (!__all_sync(0xffffffffu, mbar_wait(&hdr.code_full[i % NC], (i / NC) & 1, abort))) {
          ok = false;
          break;
        }
        bool waited = true;
        if (lane == 0 && i >= NS) waited = mbar_wait(&hdr.kv_empty[st], ((i / NS) - 1) & 1, abort);
        if (!__shfl_sync(0xffffffffu, waited, 0)) {
          ok = false;
          break;
        }
        const int keys = min(bpt, (kv_end - i * kPfKeys + bs - 1) / bs) * bs;
        widen_codes<KVT, D, kPfConvWarps>(codes + (i % NC) * Lay::CODE_BYTES, stages + st * Lay::STAGE_BYTES, keys,
                                          lane, q);
        // the 16-bit stage visible to the tensor cores, and the code slot's
        // reads ordered before the bulk copy that refills it
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&hdr.kv_full[st]);
          mbar_arrive(&hdr.code_empty[i % NC]);
        }
      }
      if (!ok && lane == 0) {
        record_error(p.err, kErrTimeout);
        *abort = 1;
      }
    }
  }
  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kPfMmaWarp) {
    tc_fence_after_sync();
    tc_dealloc(tmem, kPfTmemCols);
  }
}

template <int DT, int KVT, int D, int G>
__global__ void __launch_bounds__(pf_threads(is_byte(KVT)), 1) prefill_kernel(const __grid_constant__ PrefillParams p) {
  prefill_body<DT, KVT, D, G, false>(p);
}

// The decode's wide items (16-bit caches).  Launched as a programmatic
// dependent of the decode's plan; once the plan has ended, it lets the decode
// kernel start beside it (their items are disjoint), and that kernel waits
// for this grid only before it ends.
template <int DT, int D, int G>
__global__ void __launch_bounds__(pf_threads(false), 1) wide_decode_kernel(const __grid_constant__ PrefillParams p) {
  grid_dependency_wait();  // the plan, and everything before it
  launch_dependents();
  prefill_body<DT, DT, D, G, true>(p);
}

template <int DT, int KVT, int D, int G>
pa_status launch_prefill(const PrefillParams &p, int num_seqs, int max_q_len, cudaStream_t stream) {
  using Lay = PfLayout<D, is_byte(KVT)>;
  constexpr int QC = kPfRows / G;
  static bool configured[64];  // per device: dynamic shared memory already allowed
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(prefill_kernel<DT, KVT, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Lay::SMEM);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  const dim3 grid((max_q_len + QC - 1) / QC, num_seqs, p.num_kv_heads);
  prefill_kernel<DT, KVT, D, G><<<grid, pf_threads(is_byte(KVT)), Lay::SMEM, stream>>>(p);
  e = cudaGetLastError();
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

// The wide kernel of one instantiation, as a programmatic dependent of the
// kernel before it (the plan).
template <int DT, int D, int G>
pa_status launch_wide(const PrefillParams &p, int grid_x, cudaStream_t stream) {
  using Lay = PfLayout<D, false>;
  static bool configured[64];  // per device: dynamic shared memory already allowed
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(wide_decode_kernel<DT, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::SMEM);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_x, 1, p.num_kv_heads);
  cfg.blockDim = dim3(pf_threads(false));
  cfg.dynamicSmemBytes = Lay::SMEM;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, wide_decode_kernel<DT, D, G>, p);
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

template <int DT, int D>
pa_status wide_by_group(int G, const PrefillParams &p, int grid_x, cudaStream_t stream) {
  switch (G) {
    case 2: return launch_wide<DT, D, 2>(p, grid_x, stream);
    case 4: return launch_wide<DT, D, 4>(p, grid_x, stream);
    case 8: return launch_wide<DT, D, 8>(p, grid_x, stream);
  }
  return PA_ERR_UNSUPPORTED;
}

template <int DT, int KVT, int D>
pa_status by_group(int G, const PrefillParams &p, int num_seqs, int max_q_len, cudaStream_t stream) {
  switch (G) {
    case 1: return launch_prefill<DT, KVT, D, 1>(p, num_seqs, max_q_len, stream);
    case 2: return launch_prefill<DT, KVT, D, 2>(p, num_seqs, max_q_len, stream);
    case 4: return launch_prefill<DT, KVT, D, 4>(p, num_seqs, max_q_len, stream);
    case 8: return launch_prefill<DT, KVT, D, 8>(p, num_seqs, max_q_len, stream);
  }
  return PA_ERR_UNSUPPORTED;
}

// The instantiations of one cache type: q / out of type q_dtype (the
// cache's own type for 16-bit caches; fp16 or bf16 for one-byte ones).
template <int KVT>
pa_status dispatch_prefill(int q_dtype, int head_dim, int G, const PrefillParams &p, int num_seqs,
                           int max_q_len, cudaStream_t s) {
  if constexpr (is_byte(KVT)) {
    if (q_dtype == kF16)
      return head_dim == 64 ? by_group<kF16, KVT, 64>(G, p, num_seqs, max_q_len, s)
                            : by_group<kF16, KVT, 128>(G, p, num_seqs, max_q_len, s);
    if (q_dtype == kBF16)
      return head_dim == 64 ? by_group<kBF16, KVT, 64>(G, p, num_seqs, max_q_len, s)
                            : by_group<kBF16, KVT, 128>(G, p, num_seqs, max_q_len, s);
    return PA_ERR_UNSUPPORTED;
  } else {
    if (q_dtype != KVT) return PA_ERR_UNSUPPORTED;
    return head_dim == 64 ? by_group<KVT, KVT, 64>(G, p, num_seqs, max_q_len, s)
                          : by_group<KVT, KVT, 128>(G, p, num_seqs, max_q_len, s);
  }
}

}  // namespace

pa_status dispatch_prefill_e4m3(int q_dtype, int head_dim, int G, const PrefillParams &p, int num_seqs,
                                int max_q_len, cudaStream_t s);
pa_status dispatch_prefill_e5m2(int q_dtype, int head_dim, int G, const PrefillParams &p, int num_seqs,
                                int max_q_len, cudaStream_t s);
pa_status dispatch_prefill_i8(int q_dtype, int head_dim, int G, const PrefillParams &p, int num_seqs,
                              int max_q_len, cudaStream_t s);

}  // namespace pa

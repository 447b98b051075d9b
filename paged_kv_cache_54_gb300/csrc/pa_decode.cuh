// Paged decode attention for sm_103a.
//
// Work decomposition.  A work item is one (KV head h, partition p, and a run
// of k >= 1 consecutive sequences s..s+k-1): the tokens [p*P, min((p+1)*P,
// L_s)) for the G query heads that share KV head h.  k > 1 when the
// sequences' block tables name the same physical blocks over the whole
// partition (a shared prefix, the beams of one prompt: blocks shared through
// reference counts and copy-on-write), so each shared tile is read once for
// all k * G queries.  A plan kernel lists the items in sequence order; a
// persistent kernel (several CTAs per SM) claims them from an atomic counter.
// With 16 or more KV heads the claims go item by item, every KV head of an
// item in turn, so CTAs running at the same time read the (block, head) tiles
// of one block, which lie next to each other in the cache; with fewer, head
// by head (each head's items in sequence order).  Sequences with more than one partition leave
// (m, l, o) partials that a merge kernel combines exactly (the
// flash-decoding reduction).
//
// CTA = 1 producer warp + 4 consumer warps.  The producer walks the block
// table and stages whole (block, head) tiles of K and V — contiguous
// block_size * head_dim runs in the [num_blocks, kv_heads, block_size,
// head_dim] layout — into shared memory with bulk asynchronous copies (TMA,
// cp.async.bulk) completing on a per-stage mbarrier.  A stage holds 64
// tokens; consumer warp c owns tokens [16c, 16c + 16) of each stage and keeps
// its own online-softmax state; the four states are combined at the end of
// each item.  Block-table entries, the next item's claim and its metadata
// are fetched one item ahead so the copy engine never waits on them.
//
// Consumers compute, per 16-token slice:
//   one query per tile (G == 1, nothing shared)  (SIMT): four lanes per
//                    token, warp-shuffle dot products in fp32; lanes own
//                    head_dim columns for the P*V accumulation.
//   several queries per tile (G >= 2, or sequences sharing the blocks)
//                    (MMA): S^T = K Q^T and O^T = V^T P^T are small dense
//                    contractions: mma.sync m16n8k16 with tokens and head_dim
//                    as M and the queries as N (padded to 8), fp32
//                    accumulation; FP8 codes are widened exactly to fp16 in
//                    registers.
// Softmax is kept in base-2 units (scores pre-multiplied by log2 e) with a
// lazily updated running maximum: the accumulators are rescaled only when
// the maximum grows by more than 2^8, which leaves o / l unchanged.
#pragma once

#include <type_traits>

#include "pa_common.cuh"
#include "pa_decode_params.h"

namespace pa {
namespace {  // kernels are private to each translation unit

constexpr float kLazyRescale = 8.0f;

// Stage buffers are written by tiled TMA with the 128-byte swizzle when a
// token row is at least 128 bytes: within every 1024-byte atom, the 16-byte
// chunk at byte offset `off` lands at off ^ (((off >> 7) & 7) << 4).  Every
// shared-memory read of K or V goes through swz<SW>() on the offset relative
// to the (1024-byte aligned) K or V region of the stage.
// Every item on the tensor-core path is staged this way (rows of at least
// 128 bytes): the swizzle makes its fragment reads conflict-free.  In the
// G == 1 kernels the items with one query per tile (SIMT path) keep the
// linear layout and 1-D bulk copies, on which their reads are already
// conflict-free; the items batching sequences that share blocks (beams)
// run on the tensor-core path and are staged swizzled, item by item.
template <int KV, int D>
__host__ __device__ constexpr bool tiled_rows() { return D * elt_bytes(KV) >= 128; }
template <int KV, int D, int G>
__host__ __device__ constexpr bool swizzled() { return tiled_rows<KV, D>() && G >= 2; }

template <bool SW>
__device__ __forceinline__ int swz(int off) {
  return SW ? (off ^ (((off >> 7) & 7) << 4)) : off;
}

// Combine scratch: row r (warp c, query j: r = c * QM + j) holds D floats in
// 16-byte units; unit u is stored at u ^ ((r >> 1) & 3) so that the end-of-item
// stores of the four lanes that share a unit index land in different banks.
template <int D>
__device__ __forceinline__ int scr(int row, int d) {
  return row * D + ((((d >> 2) ^ (row >> 1)) & 3) | ((d >> 2) & ~3)) * 4 + (d & 3);
}

// The combine scratch of consumer warp c is the part of the item's last
// stage that only warp c read: its 16 K rows, then its 16 V rows (each run
// contiguous in the linear and in the swizzled layout).  It holds QM rows of
// D floats, laid out by scr<D>.
template <int KV, int D>
struct WarpScratch {
  static constexpr int REG = 16 * D * elt_bytes(KV);  // bytes of a warp's 16 rows
  uint8_t *k, *v;
  __device__ __forceinline__ WarpScratch(uint8_t *stage, const DecodeParams &p, int c)
      : k(stage + p.k_off + c * REG), v(stage + p.v_off + c * REG) {}
  __device__ __forceinline__ float *at(int row, int d) const {
    const int off = scr<D>(row, d) * 4;
    return reinterpret_cast<float *>(off < REG ? k + off : v + (off - REG));
  }
};

__device__ __forceinline__ uint32_t w32(const uint4 &v, int i) {
  return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

__device__ __forceinline__ int clamp_len(int L, int cap, int *err) {
  if (L < 0 || L > cap) {
    record_error(err, kErrSeqLen);
    return L < 0 ? 0 : cap;
  }
  return L;
}

// Query rows one item can hold: 4 for G == 1 (a beam of four), 8 otherwise
// (one mma N tile).  Sequences per shared item: kmax = QM / G.
#ifndef PA_SHARE_G1
#define PA_SHARE_G1 1
#endif
__host__ __device__ constexpr int query_capacity(int G) { return G == 1 ? (PA_SHARE_G1 ? 4 : 1) : 8; }

// ----------------------------------------------------------------------------
// plan: list the work items; reset the claim counter
// ----------------------------------------------------------------------------
// Work is indexed by slot (s, q), which exists when q is below the
// sequence's partition count.  Partition q of sequence s is "full" when all
// its P tokens exist.  Slot (s, q) joins the item of (s-1, q) when s may join
// its predecessor, partition q is full in both and their block-table entries
// over it are equal; otherwise it leads an item of its own and takes the
// following slots (s+1, q), ... of its kmax group that join.
//
// The plan is one cluster of CTAs (its work is a few thousand small steps,
// and more SMs finish it sooner).  Each CTA owns a run of whole kmax groups,
// so its join decisions need only its own sequences' flags:
//  1) its rows of the block tables start towards shared memory; its lengths;
//     its flags cleared, and every wide flag set for chunks of enough
//     sequences;
//  2) the rows of s and s-1 (s inside the run; its first only when wide
//     chunks are looked for) compared in chunks of up to 4 entries (a chunk
//     never straddles two partitions), consecutive threads on consecutive
//     chunks of one row: a mismatch flags (s, q) and clears the wide flag of
//     its (chunk, partition); so does a sequence of the chunk whose
//     partition is not full, or that has one partition only.  A wide chunk
//     may span several runs: each CTA then stores the wide flags it cleared
//     into every CTA's copy before a cluster barrier;
//  3) each thread takes a run of consecutive slots and counts the items they
//     lead; a block scan places them within the CTA, and the CTAs' totals,
//     stored into every CTA's shared memory before one cluster barrier,
//     place the CTA; the items are written in slot order.  Longest first:
//     each CTA counts its items by stage count instead, and each item takes
//     a place in its count's range by a shared-memory atomic.

// Exclusive prefix sums of two counts over the NW warps of the block;
// *total = the block's sums.
template <int NW>
__device__ __forceinline__ int2 block_exclusive_scan2(int x, int y, int2 *warp_tot, int2 *total) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int vx = x, vy = y;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ax = __shfl_up_sync(0xffffffffu, vx, o), ay = __shfl_up_sync(0xffffffffu, vy, o);
    if (lane >= o) {
      vx += ax;
      vy += ay;
    }
  }
  if (lane == 31) warp_tot[warp] = make_int2(vx, vy);
  __syncthreads();
  if (warp == 0) {
    int2 t = lane < NW ? warp_tot[lane] : make_int2(0, 0);
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ax = __shfl_up_sync(0xffffffffu, t.x, o), ay = __shfl_up_sync(0xffffffffu, t.y, o);
      if (lane >= o) {
        t.x += ax;
        t.y += ay;
      }
    }
    if (lane < NW) warp_tot[lane] = t;  // inclusive over warps
  }
  __syncthreads();
  const int2 before = warp ? warp_tot[warp - 1] : make_int2(0, 0);
  *total = warp_tot[NW - 1];
  return make_int2(before.x + vx - x, before.y + vy - y);
}

constexpr int kPlanCluster = 16;            // CTAs of the plan's cluster (1 if a cluster cannot be had)
constexpr int kPlanThreads = 512;           // threads of a plan CTA
constexpr int kPlanBuckets = kMaxPartition / kStageTok;  // item lengths in stages
constexpr int kPlanSmemSeqs = 2048;         // a CTA's lengths in shared memory up to this many
constexpr int kPlanSmemSlots = 16384;       // a CTA's mismatch flags, one byte a slot
constexpr int kPlanWideFlags = 4096;        // most (wide chunk, partition) flags
constexpr int kPlanTableBytes = 96 * 1024;  // a CTA's block-table rows in shared memory up to this

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const __grid_constant__ DecodeParams p) {
  __shared__ int2 warp_tot[32];
  // each CTA's counts, stored there by that CTA: its items, its wide items
  // and (longest first) its items of each stage count
  __shared__ int s_tab[kPlanCluster][2 + kPlanBuckets];
  __shared__ int s_hist[kPlanBuckets], s_cur[kPlanBuckets];
  __shared__ int s_len[kPlanSmemSeqs];
  __shared__ __align__(4) uint8_t s_mis[kPlanSmemSlots];
  __shared__ uint8_t s_wide[kPlanWideFlags];
  extern __shared__ __align__(16) int4 s_tbl[];  // the run's table rows, when staged
  const int tid = threadIdx.x;
  const int rank = cluster_rank(), nranks = cluster_ctas();
  const int P = p.partition_size;
  const int bpp = P / p.block_size;
  const int S = p.num_seqs;
  const int MP = p.max_parts;
  // Items are listed in slot order, or longest first (by stage count, in
  // any order within a count; the decode's claims then run from the longest
  // items to the shortest, so its last ones are short).
  const bool lf = p.longest_first != 0;
  const int NB = P / kStageTok;
  if (tid < kPlanBuckets) s_hist[tid] = 0;
  launch_dependents();  // the decode grid may become resident; it waits for us
  // This kernel is a programmatic dependent of whatever precedes it on the
  // stream: it reads only the block tables and lengths (which the cache
  // writes before it never touch) and writes only this call's workspace, and
  // it waits for the preceding kernel before it ends, so the decode that
  // waits for it also follows every kernel before the call.
  //
  // Wide chunks: W = p.wide_seqs sequences from a multiple of W whose rows
  // all agree over a full partition become one wide item (decoded on the
  // tensor cores by the wide kernel) when there are at least p.wide_min of
  // them and each has more than one partition.
  const int W = p.wide_seqs;
  const int nchunks = W > 0 ? (S + W - 1) / W : 0;
  const bool use_wide = W > 0 && nchunks * MP <= kPlanWideFlags;
  // rows are compared when items batch sequences or wide chunks are looked for
  const bool compare = p.kmax > 1 || use_wide;
  // kmax, W and the slot strides below are powers of two: the indexing uses
  // shifts and masks (a division by a variable costs tens of instructions,
  // and this kernel is bound by the instructions it issues)
  const int kmask = p.kmax - 1;
  const int w_sh = W > 0 ? 31 - __clz(W) : 0;
  const int mp_sh = 32 - __clz(MP - 1);  // partitions per sequence, padded: 2^mp_sh
  // a sequence may join its predecessor: within a group of kmax (batched
  // items), or anywhere when wide chunks are looked for
  auto may_join = [&](int s) { return s > 0 && (use_wide || (s & kmask) != 0); };
  // this CTA's run of sequences [s_lo, s_hi): whole kmax groups
  const int U = p.kmax;
  const int nu = (S + U - 1) / U;
  const int s_lo = min(S, (rank * nu / nranks) * U);  // (nu is at most the sequence count)
  const int s_hi = min(S, ((rank + 1) * nu / nranks) * U);
  const int ns = s_hi - s_lo;
  // rows and lengths from r0: the run, and the sequence before it when its
  // first sequence is compared (wide chunks)
  const int r0 = (use_wide && s_lo > 0) ? s_lo - 1 : s_lo;
  const int nr = s_hi - r0;
  const bool len_smem = nr <= kPlanSmemSeqs;
  auto length = [&](int s) {
    return len_smem ? s_len[s - r0] : min(max(__ldg(p.seq_lens + s), 0), p.len_cap);
  };
  auto full = [&](int s, int q) { return length(s) >= (q + 1) * P; };
  const int nslots = ns * MP;
  uint8_t *mis = nslots <= kPlanSmemSlots ? s_mis : p.plan_join + static_cast<size_t>(s_lo) * MP;
  // 1) the table rows start towards shared memory (they are compared once
  //    the lengths are known); lengths; flags
  const long long tbl_words = static_cast<long long>(nr) * p.max_blocks;
  const bool tbl_smem = compare && p.plan_tbl_bytes > 0 && tbl_words * 4 <= p.plan_tbl_bytes;
  const int32_t *tbl = p.block_tables + static_cast<size_t>(r0) * p.max_blocks;  // row s at (s - r0)
  if (tbl_smem) {
    const int4 *src = reinterpret_cast<const int4 *>(tbl);
    for (int i = tid; i < tbl_words / 4; i += kPlanThreads) cp_async<16>(s_tbl + i, src + i);
    cp_async_commit();
    tbl = reinterpret_cast<const int32_t *>(s_tbl);
  }
  for (int s = r0 + tid; s < s_hi; s += kPlanThreads) {
    const int L = clamp_len(__ldg(p.seq_lens + s), p.len_cap, s >= s_lo ? p.err : nullptr);
    if (len_smem) s_len[s - r0] = L;
  }
  if (compare)  // (the workspace region is 256-byte aligned and padded: whole words)
    for (int i = tid * 4; i < nslots; i += 4 * kPlanThreads) *reinterpret_cast<uint32_t *>(mis + i) = 0u;
  if (use_wide) {  // every chunk's flags (a CTA's run may reach into a chunk another's starts)
    for (int i = tid; i < (nchunks << mp_sh); i += kPlanThreads) {
      const int c = i >> mp_sh, q = i & ((1 << mp_sh) - 1);
      const int n = min(W, S - c * W);
      if (q < MP) s_wide[c * MP + q] = (n >= p.wide_min && n >= 2) ? 1 : 0;
    }
  }
  if (tbl_smem) cp_async_wait<0>();
  __syncthreads();
  // This CTA's flags are set: the others may store into its shared memory
  // once they have waited on this arrival.
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  // 2) the rows compared
  if (compare) {
    const int cpp = (bpp + 3) >> 2;           // chunks per partition
    const int cpp_sh = 32 - __clz(cpp - 1);  // ... padded: 2^cpp_sh
    const int u_sh = mp_sh + cpp_sh;         // chunk slots per sequence: 2^u_sh
    const int nch = ns << u_sh;
    // 16-byte loads when every chunk is four aligned entries
    const bool vec = (bpp & 3) == 0 && (p.max_blocks & 3) == 0 &&
                     (reinterpret_cast<uintptr_t>(p.block_tables) & 15) == 0;
    // Each thread takes chunks tid, tid + kPlanThreads, ... four at a time
    // with all their loads in flight.
    for (int u0 = 0; u0 < nch; u0 += 4 * kPlanThreads) {
      int4 x[4], y[4];
      int js[4], jq[4], jn[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int u = u0 + i * kPlanThreads + tid;
        js[i] = -1;
        jq[i] = jn[i] = 0;
        x[i] = y[i] = make_int4(0, 0, 0, 0);
        if (u < nch) {
          const int sl = u >> u_sh;  // sequence s_lo + sl, partition q, its chunk j
          const int q = (u >> cpp_sh) & ((1 << mp_sh) - 1);
          const int j = u & ((1 << cpp_sh) - 1);
          const int sq = s_lo + sl;
          // (a run's first sequence leads its kmax group: compared only for
          // the wide chunks)
          if (q < MP && j < cpp && (sl > 0 || use_wide) && may_join(sq) && full(sq, q) && full(sq - 1, q)) {
            const int e0 = q * bpp + j * 4;              // first entry of the chunk
            const int nv = min(4, (q + 1) * bpp - e0);   // entries of the chunk (1..4)
            js[i] = sl;
            jq[i] = q;
            jn[i] = nv;
            const int32_t *ra = tbl + static_cast<size_t>(sq - r0) * p.max_blocks + e0;
            const int32_t *rb = ra - p.max_blocks;
            if (vec) {
              x[i] = *reinterpret_cast<const int4 *>(ra);
              y[i] = *reinterpret_cast<const int4 *>(rb);
            } else {
              x[i] = make_int4(ra[0], nv > 1 ? ra[1] : 0, nv > 2 ? ra[2] : 0, nv > 3 ? ra[3] : 0);
              y[i] = make_int4(rb[0], nv > 1 ? rb[1] : 0, nv > 2 ? rb[2] : 0, nv > 3 ? rb[3] : 0);
            }
          }
        }
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (js[i] < 0) continue;
        const bool differ = (x[i].x != y[i].x) || (jn[i] > 1 && x[i].y != y[i].y) ||
                            (jn[i] > 2 && x[i].z != y[i].z) || (jn[i] > 3 && x[i].w != y[i].w);
        if (differ) {  // several threads may write one flag, all the same value
          mis[js[i] * MP + jq[i]] = 1;
          if (use_wide && ((s_lo + js[i]) & (W - 1)) != 0) s_wide[((s_lo + js[i]) >> w_sh) * MP + jq[i]] = 0;
        }
      }
    }
    if (use_wide) {  // every sequence of a wide chunk: the partition full, more than one
      for (int i = tid; i < (ns << mp_sh); i += kPlanThreads) {
        const int sl = i >> mp_sh, q = i & ((1 << mp_sh) - 1);
        if (q < MP && !(length(s_lo + sl) > P && full(s_lo + sl, q))) s_wide[((s_lo + sl) >> w_sh) * MP + q] = 0;
      }
    }
    __syncthreads();
  }
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");  // every CTA's flags are set
  if (use_wide && ns > 0) {
    // the wide flags this CTA cleared, for the chunks its run reaches, into
    // every other CTA's copy (only zeros are stored, so the order of these
    // stores does not matter)
    const int c0 = s_lo >> w_sh, nc = ((s_hi - 1) >> w_sh) - c0 + 1;
    for (int t = tid; t < nc * MP * nranks; t += kPlanThreads) {
      const int f = c0 * MP + t / nranks, r = t % nranks;
      if (r != rank && s_wide[f] == 0) {
        uint32_t remote;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(&s_wide[f])), "r"(r));
        asm volatile("st.shared::cluster.u8 [%0], %1;" ::"r"(remote), "h"(static_cast<unsigned short>(0)) : "memory");
      }
    }
  }
  if (use_wide) cluster_sync();  // every CTA's wide flags are the cluster's
  // 3) items.  Slot (s, q) of the run joins (s-1, q):
  auto joins = [&](int sq, int q) {
    return compare && may_join(sq) && full(sq, q) && full(sq - 1, q) && mis[(sq - s_lo) * MP + q] == 0;
  };
  // (slots indexed with the padded stride; q >= MP holds nothing)
  const int nslots_p = ns << mp_sh;
  const int per = (nslots_p + kPlanThreads - 1) / kPlanThreads;  // a run of slots per thread
  const int i0 = min(nslots_p, tid * per), i1 = min(nslots_p, i0 + per);
  // the stage-count bucket of the item (s, q) leads: its partition's tokens
  auto bucket = [&](int sq, int q) {
    const int tok = min(P, length(sq) - q * P);
    return max(1, (tok + kStageTok - 1) / kStageTok) - 1;
  };
  // pass 0 counts the items the run leads, pass 1 writes them
  int nlead = 0, nwide = 0;
  int2 at = make_int2(0, 0), tot = make_int2(0, 0);
  for (int pass = 0; pass < 2; ++pass) {
    if (pass == 1) {
      int2 cta;
      at = block_exclusive_scan2<kPlanThreads / 32>(nlead, nwide, warp_tot, &cta);  // (and the histogram is done)
      if (tid < nranks) {  // this CTA's counts into row `rank` of CTA tid's table
        uint32_t remote;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(&s_tab[rank][0])), "r"(tid));
        for (int j = 0; j < (lf ? 2 + NB : 2); ++j) {
          const int v = j == 0 ? cta.x : j == 1 ? cta.y : s_hist[j - 2];
          asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(remote + 4 * j), "r"(v) : "memory");
        }
      }
      cluster_sync();  // every CTA's counts are here; no access to another CTA follows
      for (int r = 0; r < nranks; ++r) {
        const int tx = s_tab[r][0], ty = s_tab[r][1];
        if (r < rank) {
          at.x += tx;
          at.y += ty;
        }
        tot.x += tx;
        tot.y += ty;
      }
      if (lf) {
        // bucket b (b + 1 stages) starts after every longer bucket, and this
        // CTA's part of it after the lower ranks' parts (one warp: lane b)
        if (tid < 32) {
          int all = 0, below = 0;
          if (tid < NB) {
            for (int r = 0; r < nranks; ++r) {
              const int c = s_tab[r][2 + tid];
              all += c;
              if (r < rank) below += c;
            }
          }
          int suf = all;  // items of buckets tid, tid + 1, ...
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_down_sync(0xffffffffu, suf, o);
            if (tid + o < 32) suf += y;
          }
          if (tid < NB) s_cur[tid] = suf - all + below;
          tot.x = __shfl_sync(0xffffffffu, suf, 0);
        }
        __syncthreads();
      }
    }
    int sl = i0 >> mp_sh, q = i0 & ((1 << mp_sh) - 1);
    for (int i = i0; i < i1; ++i) {
      const int sq = s_lo + sl;
      if (q < MP && q * P < max(length(sq), 1)) {  // the slot exists
        if (use_wide && s_wide[(sq >> w_sh) * MP + q] != 0) {
          if ((sq & (W - 1)) == 0) {  // the chunk's first sequence leads its wide item
            if (pass == 0) ++nwide;
            else p.wide_items[at.y++] = make_int4(sq, q, min(W, S - sq), 0);
          }
        } else if (p.kmax == 1 || (sq & kmask) == 0 || !joins(sq, q)) {
          if (pass == 0) {
            if (lf) atomicAdd(&s_hist[bucket(sq, q)], 1);
            else ++nlead;
          } else {
            int ksz = 1;
            for (int j = 1; j < p.kmax && sq + j < S && ((sq + j) & kmask) != 0; ++j) {
              if (!joins(sq + j, q)) break;
              ++ksz;
            }
            const int pos = lf ? atomicAdd(&s_cur[bucket(sq, q)], 1) : at.x++;
            p.items[pos] = make_int4(sq, q, ksz, 0);
          }
        }
      }
      if (++q == (1 << mp_sh)) {
        q = 0;
        ++sl;
      }
    }
  }
  if (rank == 0 && tid == 0) {
    p.work[1] = tot.x;
    p.work[2] = tot.y;
    p.work[0] = 0;
  }
  grid_dependency_wait();
}

// ----------------------------------------------------------------------------
// merge: combine the partials of sequences split into several partitions
// ----------------------------------------------------------------------------
// One warp per (sequence, query head), kMergeWarps to a CTA:
//   out = sum_q w_q o_q / sum_q w_q,  w_q = exp2(m_q - M) l_q,  M = max_q m_q
// (the flash-decoding reduction; o_q is normalised by its own l_q).  Lane j
// holds the weights of partitions j and j + 32 (longer sequences take
// windows of 64) and owns D / 32 columns of every partial row.  The rows
// stream through a ring of R rows of shared memory per warp: each lane
// copies its own columns with cp.async, so R rows stay in flight with few
// registers live (16 rows a warp at 24 warps an SM; held in registers, 8
// rows took 75 registers for the same residency), and the first copies
// leave before the weights are read.  A lane reads back only what it copied
// itself.  R is 4 when no sequence has more than 4 partitions (room for
// more warps), else 16.
constexpr int kMergeWarps = 4;
constexpr int kMergeThreads = 32 * kMergeWarps;

template <int QT, int D, int kMergeRing>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const __grid_constant__ DecodeParams p) {
  constexpr int E = D / 32;  // columns per lane
  constexpr int CB = E * 4;  // bytes a lane copies from a row
  __shared__ __align__(16) float ring[kMergeWarps][kMergeRing][D];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long gw = blockIdx.x * static_cast<long long>(kMergeWarps) + warp;
  if (gw >= static_cast<long long>(p.num_seqs) * p.num_q_heads) return;
  const int s = static_cast<int>(gw / p.num_q_heads);
  const int hq = static_cast<int>(gw % p.num_q_heads);
  // the lengths are an input (no kernel of this call writes them): read
  // before waiting for the decode grid, whose partials come after
  const int L = min(max(__ldg(p.seq_lens + s), 0), p.len_cap);
  const int nP = max(1, (L + p.partition_size - 1) / p.partition_size);
  if (nP <= 1) return;  // the decode wrote this sequence's output itself
  grid_dependency_wait();
  const size_t qstride = static_cast<size_t>(p.num_q_heads);
  const size_t base = static_cast<size_t>(s) * p.max_parts * qstride + hq;
  const float2 *ml = p.part_ml + base;                  // partition q at ml[q * qstride]
  const float *po = p.part_o + base * D + lane * E;     // partition q at po + q * qstride * D
  float *slot = &ring[warp][0][lane * E];               // ring row r at slot + r * D
  // one commit group per row, empty past the last partition, so that the
  // group of row q is always the q-th committed
#pragma unroll
  for (int j = 0; j < kMergeRing; ++j) {
    if (j < nP) cp_async<CB>(slot + j * D, po + j * qstride * D);
    cp_async_commit();
  }
  float M = -INFINITY;
  float2 a0 = make_float2(-INFINITY, 0.f), a1 = make_float2(-INFINITY, 0.f);
  if (nP <= 64) {
    if (lane < nP) a0 = ml[lane * qstride];
    if (lane + 32 < nP) a1 = ml[(lane + 32) * qstride];
    M = fmaxf(a0.x, a1.x);
  } else {
    for (int q = lane; q < nP; q += 32) M = fmaxf(M, ml[q * qstride].x);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float den = 0.f;
  for (int w0 = 0; w0 < nP; w0 += 64) {
    if (w0 > 0) {
      a0 = w0 + lane < nP ? ml[(w0 + lane) * qstride] : make_float2(-INFINITY, 0.f);
      a1 = w0 + lane + 32 < nP ? ml[(w0 + lane + 32) * qstride] : make_float2(-INFINITY, 0.f);
    }
    const float wt0 = a0.y > 0.f ? exp2f(a0.x - M) * a0.y : 0.f;
    const float wt1 = a1.y > 0.f ? exp2f(a1.x - M) * a1.y : 0.f;
    float ws = wt0 + wt1;
#pragma unroll
    for (int o = 16; o; o >>= 1) ws += __shfl_xor_sync(0xffffffffu, ws, o);
    den += ws;
    const int cnt = min(64, nP - w0);
    for (int k = 0; k < cnt; ++k) {  // warp-uniform
      const int q = w0 + k;
      cp_async_wait<kMergeRing - 1>();  // row q has landed
      const float *src = slot + (q % kMergeRing) * D;
      float v[E];
      if constexpr (E == 4) {
        const float4 t = *reinterpret_cast<const float4 *>(src);
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
      } else {
        const float2 t = *reinterpret_cast<const float2 *>(src);
        v[0] = t.x; v[1] = t.y;
      }
      // the slot, read, takes row q + kMergeRing
      if (q + kMergeRing < nP) cp_async<CB>(slot + (q % kMergeRing) * D, po + (q + kMergeRing) * qstride * D);
      cp_async_commit();
      const float wk = __shfl_sync(0xffffffffu, k < 32 ? wt0 : wt1, k & 31);
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = fmaf(wk, v[e], acc[e]);
    }
  }
  cp_async_wait<0>();
  const float inv = den > 0.f ? 1.f / den : 0.f;
  uint16_t *out = static_cast<uint16_t *>(p.out) + (static_cast<size_t>(s) * p.num_q_heads + hq) * D + lane * E;
  if constexpr (E == 4) {
    *reinterpret_cast<uint2 *>(out) = make_uint2(pack2_rn<QT>(acc[0] * inv, acc[1] * inv),
                                                 pack2_rn<QT>(acc[2] * inv, acc[3] * inv));
  } else {
    *reinterpret_cast<uint32_t *>(out) = pack2_rn<QT>(acc[0] * inv, acc[1] * inv);
  }
}

// ----------------------------------------------------------------------------
// producer warp
// ----------------------------------------------------------------------------
template <int KV, int D, int G>
__device__ __forceinline__ void producer_warp(const DecodeParams &p, uint8_t *smem) {
  SmemHeader &hdr = *reinterpret_cast<SmemHeader *>(smem);
  uint8_t *stages = smem + p.stages_off;
  const volatile int *abort = &hdr.abort;
  const int lane = threadIdx.x & 31;
  constexpr int ROWB = D * elt_bytes(KV);
  const int bs = p.block_size;
  const uint32_t tile = static_cast<uint32_t>(bs) * ROWB;
  const int bps = kStageTok / bs;
  const int P = p.partition_size;
  const int bpp = P / bs;  // <= 128
  const int NS = p.num_stages;
  const int n_items = __ldcg(p.work + 1);  // the plan's outputs are read from L2
  const int total = n_items * p.num_kv_heads;
  constexpr uint32_t qbytes = G * D * 2;  // query rows of one sequence's group
  const uint64_t pol_kv = l2_policy_evict_first();  // each tile passes through L2 once

  auto load_table = [&](int w, int4 pr, int L, int (&ph)[4]) {
    const int nblk = (w < total) ? (min(max(L, 0), p.len_cap) + bs - 1) / bs : 0;
    const int32_t *row = p.block_tables + static_cast<size_t>(pr.x) * p.max_blocks;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int ib = lane + 32 * c;
      const int j = pr.y * bpp + ib;
      ph[c] = (ib < bpp && j < nblk) ? __ldg(row + j) : 0;
    }
  };

  // current item (loaded synchronously once)
  int w_c = 0;
  if (lane == 0) w_c = atomicAdd(p.work, 1);
  w_c = __shfl_sync(0xffffffffu, w_c, 0);
  // claim w -> (item, head): every head of an item in turn with many KV
  // heads (a block's tiles of all heads lie together), else head by head
  auto item_of = [&](int w) { return p.item_major ? w / p.num_kv_heads : w % n_items; };
  int4 pr_c = (w_c < total) ? __ldcg(p.items + item_of(w_c)) : make_int4(0, 0, 1, 0);
  int L_c = (w_c < total) ? __ldg(p.seq_lens + pr_c.x) : 0;
  int ph_c[4];
  load_table(w_c, pr_c, L_c, ph_c);
  // Next item, fetched one dependent step per issued stage: each step only
  // issues a load whose result the following step consumes, so the warp
  // never waits on a round trip while stages are being refilled.
  int w_raw = 0, w_n = 0, L_n = 0, pf = 0;
  int4 pr_n = make_int4(0, 0, 1, 0);
  int ph_n[4] = {0, 0, 0, 0};
  auto pf_step = [&]() {
    switch (pf) {
      case 0:
        if (lane == 0) w_raw = atomicAdd(p.work, 1);
        break;
      case 1:
        w_n = __shfl_sync(0xffffffffu, w_raw, 0);
        pr_n = (w_n < total) ? __ldcg(p.items + item_of(w_n)) : make_int4(0, 0, 1, 0);
        break;
      case 2:
        L_n = (w_n < total) ? __ldg(p.seq_lens + pr_n.x) : 0;
        break;
      default:
        load_table(w_n, pr_n, L_n, ph_n);
        break;
    }
    ++pf;
  };

  int it = 0;            // stages issued so far
  int stage = 0;         // it % NS
  uint32_t phase = 0;    // (it / NS) & 1
  bool ok = true;
  while (w_c < total) {
    const int h = p.item_major ? w_c % p.num_kv_heads : w_c / n_items;
    const int s = pr_c.x, pi = pr_c.y, kseq = pr_c.z;
    const int L = clamp_len(L_c, p.len_cap, lane == 0 ? p.err : nullptr);
    const int t_begin = pi * P;
    const int t_end = min(L, t_begin + P);
    const int ntok_item = max(0, t_end - t_begin);
    const int nstages = max(1, (ntok_item + kStageTok - 1) / kStageTok);
    const int nP = max(1, (L + P - 1) / P);
    for (int st = 0; st < nstages; ++st) {
      const int tok0 = t_begin + st * kStageTok;
      const int ntok = max(0, min(kStageTok, t_end - tok0));
      const int nb = (ntok + bs - 1) / bs;
      const int ib0 = st * bps;
      const int c = ib0 >> 5;
      const int reg = c == 0 ? ph_c[0] : c == 1 ? ph_c[1] : c == 2 ? ph_c[2] : ph_c[3];
      const int phys = __shfl_sync(0xffffffffu, reg, (ib0 & 31) + (lane < nb ? lane : 0));
      if (!mbar_wait(&hdr.empty[stage], phase ^ 1u, abort)) {
        ok = false;
        break;
      }
      uint8_t *sb = stages + static_cast<size_t>(stage) * p.stage_bytes;
      if (lane == 0) {
        StageInfo &inf = hdr.info[stage];
        inf.s = s;
        inf.h = h;
        inf.p = pi;
        inf.tok0 = tok0;
        inf.ntok = ntok;
        inf.L = L;
        inf.nP = nP;
        inf.k = kseq;
        inf.flags = (st == 0 ? kFirst : 0) | (st == nstages - 1 ? kLast : 0);
        mbar_arrive_expect_tx(&hdr.full[stage], nb * 2 * tile + (st == 0 ? kseq * qbytes : 0u));
      }
      __syncwarp();
      if (lane < nb) {
        int b = phys;
        if (static_cast<unsigned>(b) >= static_cast<unsigned>(p.num_blocks)) {
          record_error(p.err, kErrBlockIndex);
          b = 0;
        }
        bool tiled = swizzled<KV, D, G>();
        if constexpr (tiled_rows<KV, D>() && G == 1) tiled = kseq > 1;  // a shared item: tensor-core path
        if (tiled) {
          // tile rows [row0, row0 + bs) of the [num_blocks * kv_heads * bs, d] view
          const int row0 = (b * p.num_kv_heads + h) * bs;
          tma_load_tile<(D * elt_bytes(KV) > 128)>(sb + p.k_off + lane * tile, &p.tmap_k, row0, &hdr.full[stage],
                                                   pol_kv);
          tma_load_tile<(D * elt_bytes(KV) > 128)>(sb + p.v_off + lane * tile, &p.tmap_v, row0, &hdr.full[stage],
                                                   pol_kv);
        } else {
          const size_t off = (static_cast<size_t>(b) * p.num_kv_heads + h) * tile;
          bulk_g2s_hint(sb + p.k_off + lane * tile, p.k_cache + off, tile, &hdr.full[stage], pol_kv);
          bulk_g2s_hint(sb + p.v_off + lane * tile, p.v_cache + off, tile, &hdr.full[stage], pol_kv);
        }
      }
      if (st == 0 && lane >= 24 && lane - 24 < kseq) {  // one q copy per sequence of the item
        const int i = lane - 24;
        const uint8_t *qsrc =
            p.q + (static_cast<size_t>(s + i) * p.num_q_heads + static_cast<size_t>(h) * G) * D * 2;
        bulk_g2s(sb + p.q_off + i * qbytes, qsrc, qbytes, &hdr.full[stage]);
      }
      ++it;
      if (++stage == NS) {
        stage = 0;
        phase ^= 1u;
      }
      if (pf < 4) pf_step();
    }
    if (!ok) break;
    while (pf < 4) pf_step();
    w_c = w_n;
    pr_c = pr_n;
    L_c = L_n;
#pragma unroll
    for (int c = 0; c < 4; ++c) ph_c[c] = ph_n[c];
    pf = 0;
  }
  if (ok) {
    if (mbar_wait(&hdr.empty[stage], phase ^ 1u, abort)) {
      if (lane == 0) {
        hdr.info[stage].flags = kEnd;
        mbar_arrive(&hdr.full[stage]);
      }
    } else {
      ok = false;
    }
  }

  if (!ok) {
    if (lane == 0) {
      record_error(p.err, kErrTimeout);
      hdr.abort = 1;
    }
    // wait, within the limit, for the copies this warp started
    if (lane == 0) {
      for (int j = max(0, it - NS); j < it; ++j) mbar_wait(&hdr.full[j % NS], (j / NS) & 1, nullptr);
    }
    __syncwarp();
  }
}

// ----------------------------------------------------------------------------
// consumer state: SIMT (one query per KV head, nothing shared)
// ----------------------------------------------------------------------------
template <int KV, int QT, int D, int G, int QM>
struct SimtState {
  static constexpr bool SW = swizzled<KV, D, G>();
  // Lane = 4 * t8 + qd: four lanes per token, eight tokens per pass, two
  // passes per 16-token slice.  Lane qd of a token owns the 16-byte chunks
  // c == qd (mod 4) of the token's K row, visited in an order rotated by t8
  // so that the eight lanes of a shared-memory phase hit eight different
  // bank groups.  For P*V, lane l owns head_dim columns [l*EPL, l*EPL+EPL).
  static constexpr int ELT = elt_bytes(KV);
  static constexpr int ROWB = D * ELT;
  static constexpr int NCH = ROWB / 16;  // 16-byte chunks per token row
  static constexpr int NCHL = NCH / 4;   // chunks per lane
  static constexpr int EPC = 16 / ELT;   // elements per chunk
  static constexpr int EPL = D / 32;     // P*V columns per lane
  static constexpr int QS = QM;          // query rows per warp in the combine scratch

  float qf[G][NCHL][EPC];
  float o[G][EPL];
  float m[G], l[G];

  __device__ __forceinline__ static int chunk(int i, int qd, int t8) { return (4 * i + qd + 4 * t8) % NCH; }

  __device__ __forceinline__ void start(const uint8_t *qs, float qk_scale, int /*ncols*/) {
    const int lane = threadIdx.x & 31;
    const int t8 = lane >> 2, qd = lane & 3;
#pragma unroll
    for (int g = 0; g < G; ++g) {
#pragma unroll
      for (int i = 0; i < NCHL; ++i) {
        const uint8_t *src = qs + (static_cast<size_t>(g) * D + chunk(i, qd, t8) * EPC) * 2;
#pragma unroll
        for (int e = 0; e < EPC; e += 2) {
          const float2 f = half2_bits_to_float2<QT>(*reinterpret_cast<const uint32_t *>(src + e * 2));
          qf[g][i][e] = f.x * qk_scale;
          qf[g][i][e + 1] = f.y * qk_scale;
        }
      }
#pragma unroll
      for (int e = 0; e < EPL; ++e) o[g][e] = 0.f;
      m[g] = -INFINITY;
      l[g] = 0.f;
    }
  }

  __device__ __forceinline__ void chunk_to_float(const uint4 &v, float (&f)[EPC]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint32_t w = w32(v, k);
      if constexpr (ELT == 2) {
        const float2 a = half2_bits_to_float2<KV>(w);
        f[2 * k] = a.x;
        f[2 * k + 1] = a.y;
      } else {
        const float2 a = byte2_to_float2<KV>(w);
        const float2 b = byte2_to_float2<KV>(w >> 16);
        f[4 * k] = a.x;
        f[4 * k + 1] = a.y;
        f[4 * k + 2] = b.x;
        f[4 * k + 3] = b.y;
      }
    }
  }

  __device__ __forceinline__ void load_v(const uint8_t *Vb, int row, float (&f)[EPL]) {
    const int lane = threadIdx.x & 31;
    const uint8_t *src = Vb + swz<SW>(row * ROWB + lane * EPL * ELT);
    if constexpr (ELT == 2) {
#pragma unroll
      for (int e = 0; e < EPL; e += 2) {
        const float2 a = half2_bits_to_float2<KV>(*reinterpret_cast<const uint32_t *>(src + e * 2));
        f[e] = a.x;
        f[e + 1] = a.y;
      }
    } else {
#pragma unroll
      for (int e = 0; e < EPL; e += 2) {
        const float2 a = byte2_to_float2<KV>(*reinterpret_cast<const uint16_t *>(src + e));
        f[e] = a.x;
        f[e + 1] = a.y;
      }
    }
  }

  // one 16-token slice: rows row0..row0+15 of the stage's K and V regions
  // Kb, Vb; n valid tokens (1..16)
  __device__ __forceinline__ void slice(const uint8_t *Kb, const uint8_t *Vb, int row0, int n, float v_scale) {
    const int lane = threadIdx.x & 31;
    const int t8 = lane >> 2, qd = lane & 3;
    float acc[2][G][2];
#pragma unroll
    for (int ps = 0; ps < 2; ++ps)
#pragma unroll
      for (int g = 0; g < G; ++g) acc[ps][g][0] = acc[ps][g][1] = 0.f;
#pragma unroll
    for (int ps = 0; ps < 2; ++ps) {
      const int krow = (row0 + 8 * ps + t8) * ROWB;
#pragma unroll
      for (int i = 0; i < NCHL; ++i) {
        float kf[EPC];
        chunk_to_float(lds128(Kb + swz<SW>(krow + chunk(i, qd, t8) * 16)), kf);
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
          for (int e = 0; e < EPC; ++e)
            acc[ps][g][e & 1] = fmaf(qf[g][i][e], kf[e], acc[ps][g][e & 1]);
      }
    }
    float pr[2][G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float sc[2];
#pragma unroll
      for (int ps = 0; ps < 2; ++ps) {
        float x = acc[ps][g][0] + acc[ps][g][1];
        x += __shfl_xor_sync(0xffffffffu, x, 1);
        x += __shfl_xor_sync(0xffffffffu, x, 2);
        sc[ps] = (8 * ps + t8 < n) ? x : -INFINITY;
      }
      float mx = fmaxf(sc[0], sc[1]);
#pragma unroll
      for (int o2 = 4; o2 < 32; o2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
      if (mx > m[g] + kLazyRescale) {  // warp-uniform
        const float alpha = exp2f(m[g] - mx);
#pragma unroll
        for (int e = 0; e < EPL; ++e) o[g][e] *= alpha;
        l[g] *= alpha;
        m[g] = mx;
      }
      pr[0][g] = exp2f(sc[0] - m[g]);
      pr[1][g] = exp2f(sc[1] - m[g]);
      if (qd == 0) l[g] += pr[0][g] + pr[1][g];
    }
    // P * V: lane owns EPL columns; token tt's weight lives in lane 4*(tt%8)
#pragma unroll
    for (int tt = 0; tt < 16; ++tt) {
      if (tt < n) {
        float vf[EPL];
        load_v(Vb, row0 + tt, vf);
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float pt = __shfl_sync(0xffffffffu, pr[tt >> 3][g], 4 * (tt & 7)) * v_scale;
#pragma unroll
          for (int e = 0; e < EPL; ++e) o[g][e] = fmaf(pt, vf[e], o[g][e]);
        }
      }
    }
  }

  __device__ __forceinline__ void to_scratch(const WarpScratch<KV, D> &so, float *sm, float *sl, float /*v_scale*/,
                                             int /*ncols*/) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float ls = l[g];
#pragma unroll
      for (int o2 = 1; o2 < 32; o2 <<= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o2);
      if constexpr (EPL == 4) {
        *reinterpret_cast<float4 *>(so.at(g, lane * 4)) = make_float4(o[g][0], o[g][1], o[g][2], o[g][3]);
      } else {
#pragma unroll
        for (int e = 0; e < EPL; ++e) *so.at(g, lane * EPL + e) = o[g][e];
      }
      if (lane == 0) {
        sm[g] = m[g];
        sl[g] = ls;
      }
    }
  }
};

// ----------------------------------------------------------------------------
// consumer state: tensor-core mma.sync (several queries share the K/V tile)
// ----------------------------------------------------------------------------
// Fragment layout of m16n8k16 (lane = 4*gq + tq):
//   A regs: (row gq, cols 2tq..+1), (row gq+8, same), (row gq, cols 2tq+8..+9), (row gq+8, same)
//   B regs: (rows 2tq..+1, col gq), (rows 2tq+8..+9, col gq)
//   C regs: (row gq, cols 2tq, 2tq+1), (row gq+8, cols 2tq, 2tq+1)
// Scores S^T = K Q^T: M = slice token (row r is token r), N = query, K = head_dim.
//   The head_dim order is permuted so that lane tq reads whole 16-byte chunks
//   kchunk(tq, j) of a row: local element e of lane tq is column
//   kchunk(tq, e / CE) * CE + e % CE, and k-step kk uses local e = 4kk..4kk+3.
// Output O^T = V^T P^T: M = head_dim, N = query, K = slice token.
//   Token order of the K dimension: k = 2tq -> token 2tq, 2tq+1 -> 2tq+8,
//   2tq+8 -> 2tq+1, 2tq+9 -> 2tq+9, which makes each B register of P^T a pair
//   of scores one lane already holds (C rows gq and gq+8).
//   Head_dim order of the M dimension: lane gq owns DPL columns, read as the
//   16-byte chunks gq, gq+8, ... of a row (or 8 bytes at 8*gq when a row is
//   64 bytes); local column c maps to head_dim column vcol(gq, c); m-tile mi
//   uses local columns mi (row gq) and MTILES + mi (row gq+8).
//   These orders make every read of the swizzled stage conflict-free except
//   for 256-byte rows, where the V reads are 2-way.
template <int KV, int QT, int D, int G, int QM>
struct MmaState {
  static constexpr bool SW = tiled_rows<KV, D>();  // always staged swizzled when rows allow
  static constexpr bool KV8 = is_byte(KV);
  static constexpr int MT = KV8 ? kF16 : KV;  // mma input type
  static constexpr int ELT = elt_bytes(KV);
  static constexpr int ROWB = D * ELT;
  static constexpr int KSTEPS = D / 16;
  static constexpr int MTILES = D / 16;
  static constexpr int CE = 16 / ELT;       // elements per 16-byte chunk
  static constexpr int LCH = (D / 4) / CE;  // chunks of a K row per lane
  static constexpr int DPL = D / 8;         // output columns per lane group
  static constexpr int QS = QM;  // query rows per warp in the combine scratch
  // INT8 codes enter the products as 1152 + c (two instructions fewer per
  // four codes); the offset comes off the scores as 1152 * sum(q) and off
  // the output as 1152 * l, with l summed from the rounded weights the
  // products used
  static constexpr bool I8OFF = KV == kI8;

  uint32_t qb[KSTEPS][2];
  float oacc[MTILES][4];
  float m2[2], l2[2];
  float qk_mult;
  float kcorr[2];  // (INT8) -1152 * sum(q) * qk_mult of query columns 2tq, 2tq+1

  __device__ __forceinline__ static void widen4(uint32_t w, uint32_t &lo, uint32_t &hi) {
    if constexpr (I8OFF) {
      i8x4_to_half2x2_offset(w, lo, hi);
    } else {
      byte4_to_half2x2<KV>(w, lo, hi);
    }
  }

  // 16-byte chunk j of a K row read by lane tq: contiguous chunks on the
  // swizzled layout, chunks tq, tq+4, ... on the linear one (fewest bank
  // conflicts for each)
  __device__ __forceinline__ static int kchunk(int tq, int j) { return SW ? LCH * tq + j : tq + 4 * j; }
  __device__ __forceinline__ static int kcol(int tq, int e) { return kchunk(tq, e / CE) * CE + e % CE; }
  // head_dim column of the lane's local V column c
  __device__ __forceinline__ static int vcol(int gq, int c) {
    if constexpr (DPL * ELT >= 16) {
      return (gq + 8 * (c / CE)) * CE + c % CE;
    } else {
      return gq * DPL + c;
    }
  }

  // q rows [ncols][D] in shared memory: the query heads of the group, for
  // each sequence that shares the item's blocks; columns >= ncols are zero.
  // Lane (gq, tq) needs row gq's local elements 0..D/4-1: chunk j of them
  // is the CE columns at kchunk(tq, j) * CE, read with 16-byte loads.
  __device__ __forceinline__ void start(const uint8_t *qs, float qk_scale, int ncols) {
    const int lane = threadIdx.x & 31;
    const int gq = lane >> 2, tq = lane & 3;
    const bool real = gq < ncols;
    constexpr int QW = D / 8;  // 32-bit words of q the lane holds (two elements each)
    uint32_t qw[QW];
    const uint8_t *qrow = qs + static_cast<size_t>(real ? gq : 0) * D * 2;
#pragma unroll
    for (int j = 0; j < LCH; ++j) {
#pragma unroll
      for (int h = 0; h < CE / 8; ++h) {  // CE q elements = CE * 2 bytes
        const uint4 v = real ? lds128(qrow + kchunk(tq, j) * CE * 2 + 16 * h) : make_uint4(0u, 0u, 0u, 0u);
        const int w0 = j * (CE / 2) + 4 * h;
        qw[w0] = v.x;
        qw[w0 + 1] = v.y;
        qw[w0 + 2] = v.z;
        qw[w0 + 3] = v.w;
      }
    }
    float f = 1.f;
    if constexpr (KV8 && QT == kBF16) {
      // fp16 operands: scale q by a power of two so the group's largest
      // entry fits fp16's range; the factor is undone on the scores.
      float amax = 0.f;
#pragma unroll
      for (int w = 0; w < QW; ++w) {
        const float2 x = half2_bits_to_float2<kBF16>(qw[w]);
        amax = fmaxf(amax, fmaxf(fabsf(x.x), fabsf(x.y)));
      }
#pragma unroll
      for (int o2 = 1; o2 < 32; o2 <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o2));
      if (amax > 16384.f) {
        int ex;
        frexpf(amax, &ex);
        f = ldexpf(1.f, 14 - ex);
      }
#pragma unroll
      for (int w = 0; w < QW; ++w) {
        const float2 x = half2_bits_to_float2<kBF16>(qw[w]);
        qw[w] = pack2_rn<kF16>(x.x * f, x.y * f);
      }
    }
    // k-step kk uses local elements 4kk..4kk+3: words 2kk (cols 2tq, 2tq+1)
    // and 2kk + 1 (cols 2tq+8, 2tq+9)
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      qb[kk][0] = qw[2 * kk];
      qb[kk][1] = qw[2 * kk + 1];
    }
    qk_mult = qk_scale / f;
    if constexpr (I8OFF) {
      // sum of the fp16 q the products use, row gq, then columns 2tq, 2tq+1
      float qs = 0.f;
#pragma unroll
      for (int w = 0; w < QW; ++w) {
        const float2 x = half2_bits_to_float2<kF16>(qw[w]);
        qs += x.x + x.y;
      }
      qs += __shfl_xor_sync(0xffffffffu, qs, 1);
      qs += __shfl_xor_sync(0xffffffffu, qs, 2);
      const float qs0 = __shfl_sync(0xffffffffu, qs, (2 * tq) * 4);
      const float qs1 = __shfl_sync(0xffffffffu, qs, (2 * tq + 1) * 4);
      kcorr[0] = -kI8Offset * qs0 * qk_mult;
      kcorr[1] = -kI8Offset * qs1 * qk_mult;
    }
#pragma unroll
    for (int mi = 0; mi < MTILES; ++mi)
#pragma unroll
      for (int k = 0; k < 4; ++k) oacc[mi][k] = 0.f;
    m2[0] = m2[1] = -INFINITY;
    l2[0] = l2[1] = 0.f;
  }

  // A register of K for k-step kk from the row's LCH chunks; r = 0 (cols
  // 2tq..+1) or 1 (cols 2tq+8..+9)
  __device__ __forceinline__ static uint32_t k_reg(const uint4 (&ch)[LCH], int kk, int r) {
    if constexpr (ELT == 2) {
      const int e = 4 * kk + 2 * r;  // local element (even)
      return w32(ch[e / CE], (e % CE) / 2);
    } else {
      const int e = 4 * kk;
      const uint32_t w = w32(ch[e / CE], (e % CE) / 4);
      return byte2_to_half2_bits<KV>(r ? (w >> 16) : w);
    }
  }

  // A register of V^T: pair (row ra, row rb) of output column index `col`
  // within the lane's DPL columns
  __device__ __forceinline__ static uint32_t v_pair(const uint32_t *ra, const uint32_t *rb, int col) {
    if constexpr (ELT == 2) {
      const uint32_t a = ra[col / 2], b = rb[col / 2];
      return prmt(a, b, (col & 1) ? 0x7632u : 0x5410u);
    } else {
      const int byte = col & 3;
      const uint32_t a = ra[col / 4], b = rb[col / 4];
      const uint32_t two = prmt(a, b, static_cast<uint32_t>(byte | ((4 + byte) << 4)));
      return byte2_to_half2_bits<KV>(two);
    }
  }

  // FP8 V^T: (row ra, row rb) pairs of output columns col and col+1 (col even)
  __device__ __forceinline__ static void v_pair2(const uint32_t *ra, const uint32_t *rb, int col,
                                                 uint32_t &lo, uint32_t &hi) {
    const uint32_t b = col & 3;
    const uint32_t two = prmt(ra[col / 4], rb[col / 4], b | ((4 + b) << 4) | ((b + 1) << 8) | ((5 + b) << 12));
    widen4(two, lo, hi);
  }

  __device__ __forceinline__ void slice(const uint8_t *Kb, const uint8_t *Vb, int row0, int n, float v_scale) {
    const int lane = threadIdx.x & 31;
    const int gq = lane >> 2, tq = lane & 3;
    // ---- S^T = K Q^T ----
    uint4 k0[LCH], k1[LCH];
#pragma unroll
    for (int j = 0; j < LCH; ++j) {
      k0[j] = lds128(Kb + swz<SW>((row0 + gq) * ROWB + kchunk(tq, j) * 16));
      k1[j] = lds128(Kb + swz<SW>((row0 + gq + 8) * ROWB + kchunk(tq, j) * 16));
    }
    // four independent accumulators so the k-steps do not form one chain
    float sacc[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int k = 0; k < 4; ++k) sacc[a][k] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      uint32_t a0, a1, a2, a3;
      if constexpr (ELT == 2) {
        a0 = k_reg(k0, kk, 0);
        a1 = k_reg(k1, kk, 0);
        a2 = k_reg(k0, kk, 1);
        a3 = k_reg(k1, kk, 1);
      } else {  // local elements 4kk..4kk+3 are one word of the row's chunk
        const int e = 4 * kk;
        widen4(w32(k0[e / CE], (e % CE) / 4), a0, a2);
        widen4(w32(k1[e / CE], (e % CE) / 4), a1, a3);
      }
      mma16816<MT>(sacc[kk & 3], a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
    }
    float sc[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float sum = (sacc[0][k] + sacc[1][k]) + (sacc[2][k] + sacc[3][k]);
      if constexpr (I8OFF) {
        sc[k] = fmaf(sum, qk_mult, kcorr[k & 1]);
      } else {
        sc[k] = sum * qk_mult;
      }
    }
    // rows gq (regs 0,1) and gq+8 (regs 2,3); columns 2tq, 2tq+1
    if (gq >= n) sc[0] = sc[1] = -INFINITY;
    if (gq + 8 >= n) sc[2] = sc[3] = -INFINITY;
    float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
#pragma unroll
    for (int o2 = 4; o2 < 32; o2 <<= 1) {
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
    }
    const bool up0 = mx0 > m2[0] + kLazyRescale, up1 = mx1 > m2[1] + kLazyRescale;
    if (__any_sync(0xffffffffu, up0 || up1)) {
      const float al0 = up0 ? exp2f(m2[0] - mx0) : 1.f;
      const float al1 = up1 ? exp2f(m2[1] - mx1) : 1.f;
      if (up0) m2[0] = mx0;
      if (up1) m2[1] = mx1;
#pragma unroll
      for (int mi = 0; mi < MTILES; ++mi) {
        oacc[mi][0] *= al0;
        oacc[mi][2] *= al0;
        oacc[mi][1] *= al1;
        oacc[mi][3] *= al1;
      }
      l2[0] *= al0;
      l2[1] *= al1;
    }
    const float p0 = exp2f(sc[0] - m2[0]), p1 = exp2f(sc[1] - m2[1]);
    const float p2 = exp2f(sc[2] - m2[0]), p3 = exp2f(sc[3] - m2[1]);
    // P^T as the B operand: query gq, tokens (2tq, 2tq+8) and (2tq+1, 2tq+9)
    const uint32_t packA = pack2_rn<MT>(p0, p2);  // query 2tq
    const uint32_t packB = pack2_rn<MT>(p1, p3);  // query 2tq+1
    if constexpr (I8OFF) {  // the weights as rounded for the products
      const float2 ra = half2_bits_to_float2<kF16>(packA), rb = half2_bits_to_float2<kF16>(packB);
      l2[0] += ra.x + ra.y;
      l2[1] += rb.x + rb.y;
    } else {
      l2[0] += p0 + p2;
      l2[1] += p1 + p3;
    }
    const int src0 = (2 * tq) * 4 + (gq >> 1), src1 = (2 * tq + 1) * 4 + (gq >> 1);
    const uint32_t xA0 = __shfl_sync(0xffffffffu, packA, src0), xB0 = __shfl_sync(0xffffffffu, packB, src0);
    const uint32_t xA1 = __shfl_sync(0xffffffffu, packA, src1), xB1 = __shfl_sync(0xffffffffu, packB, src1);
    const uint32_t b0 = (gq & 1) ? xB0 : xA0;
    const uint32_t b1 = (gq & 1) ? xB1 : xA1;
    // ---- O^T += V^T P^T ----
    constexpr int VW = DPL * ELT / 4;  // 32-bit words of a row the lane reads
    uint32_t r0[VW], r1[VW], r2[VW], r3[VW];
    const int t0 = 2 * tq, t1 = 2 * tq + 8, t2 = 2 * tq + 1, t3 = 2 * tq + 9;
    if constexpr (VW >= 4) {  // whole 16-byte chunks gq, gq + 8, ...
#pragma unroll
      for (int j = 0; j < VW / 4; ++j) {
        const int cb = (gq + 8 * j) * 16;
        const uint4 a = lds128(Vb + swz<SW>((row0 + t0) * ROWB + cb));
        const uint4 b = lds128(Vb + swz<SW>((row0 + t1) * ROWB + cb));
        const uint4 c = lds128(Vb + swz<SW>((row0 + t2) * ROWB + cb));
        const uint4 d = lds128(Vb + swz<SW>((row0 + t3) * ROWB + cb));
        r0[4 * j] = a.x; r0[4 * j + 1] = a.y; r0[4 * j + 2] = a.z; r0[4 * j + 3] = a.w;
        r1[4 * j] = b.x; r1[4 * j + 1] = b.y; r1[4 * j + 2] = b.z; r1[4 * j + 3] = b.w;
        r2[4 * j] = c.x; r2[4 * j + 1] = c.y; r2[4 * j + 2] = c.z; r2[4 * j + 3] = c.w;
        r3[4 * j] = d.x; r3[4 * j + 1] = d.y; r3[4 * j + 2] = d.z; r3[4 * j + 3] = d.w;
      }
    } else {  // 64-byte rows: 8 bytes at 8 * gq
      const int cb = gq * 8;
      const uint2 a = *reinterpret_cast<const uint2 *>(Vb + swz<SW>((row0 + t0) * ROWB + cb));
      const uint2 b = *reinterpret_cast<const uint2 *>(Vb + swz<SW>((row0 + t1) * ROWB + cb));
      const uint2 c = *reinterpret_cast<const uint2 *>(Vb + swz<SW>((row0 + t2) * ROWB + cb));
      const uint2 d = *reinterpret_cast<const uint2 *>(Vb + swz<SW>((row0 + t3) * ROWB + cb));
      r0[0] = a.x; r0[1] = a.y;
      r1[0] = b.x; r1[1] = b.y;
      r2[0] = c.x; r2[1] = c.y;
      r3[0] = d.x; r3[1] = d.y;
    }
    if (n < 16) {  // stale rows may hold NaN: zero them so 0 * NaN never reaches the sum
#pragma unroll
      for (int w = 0; w < VW; ++w) {
        if (t0 >= n) r0[w] = 0u;
        if (t1 >= n) r1[w] = 0u;
        if (t2 >= n) r2[w] = 0u;
        if (t3 >= n) r3[w] = 0u;
      }
    }
    if constexpr (ELT == 2) {
#pragma unroll
      for (int mi = 0; mi < MTILES; ++mi) {
        const uint32_t a0 = v_pair(r0, r1, mi);
        const uint32_t a1 = v_pair(r0, r1, MTILES + mi);
        const uint32_t a2 = v_pair(r2, r3, mi);
        const uint32_t a3 = v_pair(r2, r3, MTILES + mi);
        mma16816<MT>(oacc[mi], a0, a1, a2, a3, b0, b1);
      }
    } else {
      // bytes (c, c+1) of rows (ra, rb) -> pairs for m-tiles c and c+1
#pragma unroll
      for (int mi = 0; mi < MTILES; mi += 2) {
        uint32_t x0[2], x1[2], x2[2], x3[2];
        v_pair2(r0, r1, mi, x0[0], x0[1]);
        v_pair2(r0, r1, MTILES + mi, x1[0], x1[1]);
        v_pair2(r2, r3, mi, x2[0], x2[1]);
        v_pair2(r2, r3, MTILES + mi, x3[0], x3[1]);
        mma16816<MT>(oacc[mi], x0[0], x1[0], x2[0], x3[0], b0, b1);
        mma16816<MT>(oacc[mi + 1], x0[1], x1[1], x2[1], x3[1], b0, b1);
      }
    }
    (void)v_scale;
  }

  __device__ __forceinline__ void to_scratch(const WarpScratch<KV, D> &so, float *sm, float *sl, float v_scale,
                                             int ncols) {
    const int lane = threadIdx.x & 31;
    const int gq = lane >> 2, tq = lane & 3;
    float ls0 = l2[0], ls1 = l2[1];
#pragma unroll
    for (int o2 = 4; o2 < 32; o2 <<= 1) {
      ls0 += __shfl_xor_sync(0xffffffffu, ls0, o2);
      ls1 += __shfl_xor_sync(0xffffffffu, ls1, o2);
    }
    const int qa = 2 * tq, qb2 = 2 * tq + 1;
    // local column c holds oacc[c][0|1] (c < MTILES) or oacc[c - MTILES][2|3];
    // runs of four local columns are four consecutive head_dim columns
#pragma unroll
    for (int c0 = 0; c0 < DPL; c0 += 4) {
      float va[4], vb[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + u;
        va[u] = (c < MTILES ? oacc[c % MTILES][0] : oacc[c % MTILES][2]);
        vb[u] = (c < MTILES ? oacc[c % MTILES][1] : oacc[c % MTILES][3]);
        if constexpr (I8OFF) {
          va[u] = fmaf(-kI8Offset, ls0, va[u]);
          vb[u] = fmaf(-kI8Offset, ls1, vb[u]);
        }
        va[u] *= v_scale;
        vb[u] *= v_scale;
      }
      const int d = vcol(gq, c0);
      if (qa < ncols) *reinterpret_cast<float4 *>(so.at(qa, d)) = make_float4(va[0], va[1], va[2], va[3]);
      if (qb2 < ncols) *reinterpret_cast<float4 *>(so.at(qb2, d)) = make_float4(vb[0], vb[1], vb[2], vb[3]);
    }
    if (gq == 0) {
      if (qa < ncols) {
        sm[qa] = m2[0];
        sl[qa] = ls0;
      }
      if (qb2 < ncols) {
        sm[qb2] = m2[1];
        sl[qb2] = ls1;
      }
    }
  }
};

// ----------------------------------------------------------------------------
// combine the four consumer warps' states and write the item's result
// ----------------------------------------------------------------------------
// Query column j of an item is head h*G + j%G of sequence s + j/G.
// Consumer warp c takes the columns c, c + 4, ...; lanes 0..3 weigh the
// four warps' states, w_c = exp2(m_c - M) / sum_c exp2(m_c - M) l_c, and
// every lane then sums its D / 32 columns of the four states.
template <int KV, int QT, int D, int G, int QM>
__device__ __forceinline__ void combine_item(const DecodeParams &p, const StageInfo &inf, int ncols, uint8_t *last,
                                             const float (*sm)[8], const float (*sl)[8]) {
  constexpr int E = D / 32;  // columns per lane
  const int cw = (threadIdx.x >> 5) - 1, lane = threadIdx.x & 31;
  const int P = p.partition_size;
  for (int j = cw; j < ncols; j += kConsumerWarps) {
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < kConsumerWarps; ++c) M = fmaxf(M, sm[c][j]);
    float w = 0.f, wl = 0.f;
    if (lane < kConsumerWarps) {
      const float mc = sm[lane][j];
      w = (mc == -INFINITY) ? 0.f : exp2f(mc - M);
      wl = w * sl[lane][j];
    }
    wl += __shfl_xor_sync(0xffffffffu, wl, 1);
    wl += __shfl_xor_sync(0xffffffffu, wl, 2);
    const float wsum = __shfl_sync(0xffffffffu, wl, 0);
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    float acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll
    for (int c = 0; c < kConsumerWarps; ++c) {
      const float wc = __shfl_sync(0xffffffffu, w, c) * inv;
      const float *src = WarpScratch<KV, D>(last, p, c).at(j, lane * E);
      if constexpr (E == 4) {
        const float4 v = *reinterpret_cast<const float4 *>(src);
        acc[0] = fmaf(wc, v.x, acc[0]);
        acc[1] = fmaf(wc, v.y, acc[1]);
        acc[2] = fmaf(wc, v.z, acc[2]);
        acc[3] = fmaf(wc, v.w, acc[3]);
      } else {
        const float2 v = *reinterpret_cast<const float2 *>(src);
        acc[0] = fmaf(wc, v.x, acc[0]);
        acc[1] = fmaf(wc, v.y, acc[1]);
      }
    }
    const int sj = inf.s + j / G;
    const int hq = inf.h * G + j % G;
    const int Lj = (G == 1 && inf.k == 1) ? inf.L : min(max(__ldg(p.seq_lens + sj), 0), p.len_cap);
    if ((Lj + P - 1) / P <= 1) {
      uint16_t *out = static_cast<uint16_t *>(p.out) + (static_cast<size_t>(sj) * p.num_q_heads + hq) * D + lane * E;
      if constexpr (E == 4) {
        *reinterpret_cast<uint2 *>(out) = make_uint2(pack2_rn<QT>(acc[0], acc[1]), pack2_rn<QT>(acc[2], acc[3]));
      } else {
        *reinterpret_cast<uint32_t *>(out) = pack2_rn<QT>(acc[0], acc[1]);
      }
    } else {
      const size_t idx = (static_cast<size_t>(sj) * p.max_parts + inf.p) * p.num_q_heads + hq;
      const uint64_t keep = l2_policy_evict_last();  // the merge reads the partials next
      float *po = p.part_o + idx * D + lane * E;
      if constexpr (E == 4) {
        st_global_f4_hint(po, make_float4(acc[0], acc[1], acc[2], acc[3]), keep);
      } else {
        st_global_f2_hint(po, acc[0], acc[1], keep);
      }
      if (lane == 0) st_global_f2_hint(reinterpret_cast<float *>(p.part_ml + idx), M, wsum, keep);
    }
  }
}

// ----------------------------------------------------------------------------
// one work item, from its first (already waited) stage to its combine
// ----------------------------------------------------------------------------
template <int KV, int QT, int D, int G, int QM, class State>
__device__ __forceinline__ bool run_item(const DecodeParams &p, SmemHeader &hdr, uint8_t *stages, int cw,
                                         int &stage, uint32_t &phase, uint32_t &cpar, StageInfo inf,
                                         const volatile int *abort) {
  const int lane = threadIdx.x & 31;
  const int ncols = inf.k * G;
  // scales of the item's KV head: per tensor (folded in by the host) or per head
  float qk_scale = p.qk_scale_log2, v_scale = p.v_scale;
  if constexpr (is_byte(KV)) {
    if (p.k_head_scale != nullptr) {
      qk_scale *= __ldg(p.k_head_scale + inf.h);
      v_scale = __ldg(p.v_head_scale + inf.h);
    }
  }
  State st;
  st.start(stages + static_cast<size_t>(stage) * p.stage_bytes + p.q_off, qk_scale, ncols);
  while (true) {
    const uint8_t *sb = stages + static_cast<size_t>(stage) * p.stage_bytes;
    const int n = min(16, inf.ntok - 16 * cw);
    if (n > 0) st.slice(sb + p.k_off, sb + p.v_off, 16 * cw, n, v_scale);
    __syncwarp();
    if (inf.flags & kLast) break;  // the last stage is kept: it becomes the combine scratch
    if (lane == 0) mbar_arrive(&hdr.empty[stage]);
    if (++stage == p.num_stages) {
      stage = 0;
      phase ^= 1u;
    }
    if (!mbar_wait(&hdr.full[stage], phase, abort)) return false;
    const StageInfo nxt = hdr.info[stage];
    inf.ntok = nxt.ntok;
    inf.flags = nxt.flags;
  }
  // The four warps' states meet in the item's last stage: each warp writes
  // its state over the rows only it read (no wait for the others), and
  // (m, l) into the header's buffer of this item's parity.  One
  // consumer-wide barrier (its phase parity alternates with the items), then
  // every warp reads all four states and hands the stage back by itself.
  uint8_t *last = stages + static_cast<size_t>(stage) * p.stage_bytes;
  st.to_scratch(WarpScratch<KV, D>(last, p, cw), hdr.comb_m[cpar][cw], hdr.comb_l[cpar][cw], v_scale, ncols);
  mbar_arrive(&hdr.combine);
  if (!mbar_wait(&hdr.combine, cpar, abort)) return false;
  combine_item<KV, QT, D, G, QM>(p, inf, ncols, last, hdr.comb_m[cpar], hdr.comb_l[cpar]);
  cpar ^= 1u;
  __syncwarp();
  if (lane == 0) mbar_arrive(&hdr.empty[stage]);
  if (++stage == p.num_stages) {
    stage = 0;
    phase ^= 1u;
  }
  return true;
}

// ----------------------------------------------------------------------------
// the persistent decode kernel
// ----------------------------------------------------------------------------
// MMA: every item runs on the tensor-core path; otherwise items whose tile
// serves a single query run on the SIMT path and shared items on the MMA one.
template <int KV, int QT, int D, int G, bool MMA>
__device__ __forceinline__ void decode_body(const DecodeParams &p) {
  constexpr int QM = query_capacity(G);
  static_assert(QM * D * 4 <= 2 * WarpScratch<KV, D>::REG && QM <= 8,
                "a warp's combine state must fit in the stage rows it read");
  extern __shared__ __align__(128) uint8_t smem[];
  SmemHeader &hdr = *reinterpret_cast<SmemHeader *>(smem);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int i = 0; i < p.num_stages; ++i) {
      mbar_init(&hdr.full[i], 1);
      mbar_init(&hdr.empty[i], kConsumerWarps);
    }
    mbar_init(&hdr.combine, kConsumerThreads);
    hdr.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if ((smem_addr(smem + p.stages_off) & 1023u) != 0) {  // the swizzle needs 1024-byte atoms
    if (threadIdx.x == 0) record_error(p.err, kErrSmemAlign);
    return;
  }
  // The plan (and every kernel before it: the cache writes) must be
  // complete.  After the wide kernel, this grid starts only once every wide
  // CTA has seen the plan end, so it does not wait here: it waits for the
  // wide grid before it ends (its first CTA, below), so that the merge,
  // which waits for this grid, follows both.
  if (!p.after_wide) grid_dependency_wait();
  // Only the merge of this call may start early.  Without one the next
  // kernel on the stream waits for this grid to end: a later call's plan
  // rewrites the workspace this grid reads.
  if (p.max_parts > 1) launch_dependents();
  if (warp == 0) {
    producer_warp<KV, D, G>(p, smem);
    if (p.after_wide && blockIdx.x == 0 && threadIdx.x == 0) grid_dependency_wait();
    return;
  }
  const int cw = warp - 1;
  const int lane = threadIdx.x & 31;
  const volatile int *abort = &hdr.abort;
  uint8_t *stages = smem + p.stages_off;
  using Mma = MmaState<KV, QT, D, G, QM>;
  int stage = 0;
  uint32_t phase = 0, cpar = 0;
  bool failed = false;
  while (true) {
    if (!mbar_wait(&hdr.full[stage], phase, abort)) {
      failed = true;
      break;
    }
    const StageInfo inf = hdr.info[stage];
    if (inf.flags & kEnd) break;
    bool ok;
    if constexpr (MMA) {
      ok = run_item<KV, QT, D, G, QM, Mma>(p, hdr, stages, cw, stage, phase, cpar, inf, abort);
    } else {
      using Simt = SimtState<KV, QT, D, G, QM>;
      if (QM > G && inf.k > 1)
        ok = run_item<KV, QT, D, G, QM, Mma>(p, hdr, stages, cw, stage, phase, cpar, inf, abort);
      else
        ok = run_item<KV, QT, D, G, QM, Simt>(p, hdr, stages, cw, stage, phase, cpar, inf, abort);
    }
    if (!ok) {
      failed = true;
      break;
    }
  }
  if (failed && lane == 0) {
    record_error(p.err, kErrTimeout);
    hdr.abort = 1;
  }
}

// Shared-memory plan of one decode instantiation.
struct DecodeSmemPlan {
  int stage_bytes, k_off, v_off, q_off, stages_off, num_stages, total;
};

template <int KV, int D, int G>
__host__ __device__ constexpr DecodeSmemPlan plan_smem(int max_smem) {
  constexpr int ROWB = D * elt_bytes(KV);
  constexpr int QM = query_capacity(G);
  DecodeSmemPlan s{0, 0, 0, 0, 0, 0, 0};
  s.k_off = 0;
  s.v_off = kStageTok * ROWB;
  s.q_off = 2 * kStageTok * ROWB;
  // stages and their K / V regions start on 1024-byte boundaries (the
  // swizzle atom of the tensor copies)
  s.stage_bytes = (s.q_off + QM * D * 2 + 1023) / 1024 * 1024;
  s.stages_off = (static_cast<int>(sizeof(SmemHeader)) + 1023) / 1024 * 1024;
  int ns = (max_smem - s.stages_off) / s.stage_bytes;
  if (ns > kMaxStages) ns = kMaxStages;
  s.num_stages = ns;
  s.total = s.stages_off + ns * s.stage_bytes;
  return s;
}

// Resident CTAs per SM for a shared-memory budget: as many (up to kCtasPerSm)
// as leave each at least two pipeline stages; the hardware reserves 1 KB per
// resident CTA.
template <int KV, int D, int G>
__host__ __device__ constexpr int resident_ctas(int smem_per_sm, int smem_optin) {
  for (int ctas = kCtasPerSm; ctas >= 1; --ctas) {
    int budget = smem_optin;
    if (ctas > 1 && smem_per_sm / ctas - 1024 < budget) budget = smem_per_sm / ctas - 1024;
    if (plan_smem<KV, D, G>(budget).num_stages >= 2) return ctas;
  }
  return 0;
}

template <int KV, int D, int G>
__host__ __device__ constexpr int kernel_regs() {
  return regs_for_ctas(resident_ctas<KV, D, G>(kSmemPerSm, kSmemOptin) > 0
                           ? resident_ctas<KV, D, G>(kSmemPerSm, kSmemOptin)
                           : 1);
}

// The tiled TMA reads the tensor maps from the kernel's parameter space, so
// the kernels that may stage swizzled tiles (rows of 128 bytes or more) take
// their parameters as grid constants; the others take them by value.
template <int KV, int QT, int D, int G, bool MMA>
__global__ void __maxnreg__((kernel_regs<KV, D, G>())) decode_kernel_tma(const __grid_constant__ DecodeParams p) {
  decode_body<KV, QT, D, G, MMA>(p);
}

template <int KV, int QT, int D, int G, bool MMA>
__global__ void __maxnreg__((kernel_regs<KV, D, G>())) decode_kernel(const DecodeParams p) {
  decode_body<KV, QT, D, G, MMA>(p);
}




// ----------------------------------------------------------------------------
// host launch of one instantiation: plan, persistent decode, merge
// ----------------------------------------------------------------------------
template <int KV, int QT, int D, int G, bool MMA>
pa_status launch_decode(DecodeParams p, const DeviceInfo &dev, cudaStream_t stream) {
  const int ctas = resident_ctas<KV, D, G>(dev.smem_per_sm, dev.max_smem_optin);
  int budget = dev.max_smem_optin;
  if (ctas > 1) budget = min(budget, dev.smem_per_sm / ctas - 1024);
  const DecodeSmemPlan sp = plan_smem<KV, D, G>(budget);
  if (ctas < 1 || sp.num_stages < 2) return PA_ERR_UNSUPPORTED;
  p.num_stages = sp.num_stages;
  p.stage_bytes = sp.stage_bytes;
  p.k_off = sp.k_off;
  p.v_off = sp.v_off;
  p.q_off = sp.q_off;
  p.stages_off = sp.stages_off;
  p.kmax = query_capacity(G) / G;
  // runs of sequences sharing a whole partition's blocks go to the tensor
  // cores (16-bit caches, query groups of 2 or more, split sequences)
  const bool wide = !is_byte(KV) && G >= 2 && p.max_parts > 1;
  // Claims take every KV head of an item in turn with 16 or more KV heads
  // (neighbouring tiles of one block at a time), else head by head.  With
  // wide items, the decode keeps the sequences' own tails, of varied
  // lengths: those are listed longest first and claimed item by item, so
  // that the last claims are short.
  p.item_major = p.num_kv_heads >= 16 || wide;
  p.longest_first = wide;
  p.wide_seqs = wide ? kWideRows / G : 0;
  p.wide_min = kWideMinRows / G;
  void (*kern)(DecodeParams);
  if constexpr (tiled_rows<KV, D>()) {
    kern = decode_kernel_tma<KV, QT, D, G, MMA>;
  } else {
    kern = decode_kernel<KV, QT, D, G, MMA>;
  }
  static int configured_bytes[64];  // per device: dynamic smem already allowed
  int dev_id = 0;
  cudaError_t e = cudaGetDevice(&dev_id);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev_id < 0 || dev_id >= 64 || configured_bytes[dev_id] < sp.total) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, sp.total);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev_id >= 0 && dev_id < 64) configured_bytes[dev_id] = sp.total;
  }
  // the plan, the decode and the merge are launched as programmatic
  // dependents: each may start before the kernel ahead of it ends (each
  // waits on the device for what it needs)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kPlanThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  // the plan: one cluster of up to kPlanCluster CTAs (no more than there
  // are kmax groups), or a cluster of one CTA where no such cluster can be
  // placed; each
  // stages its run's block-table rows in shared memory when they are
  // 16-byte aligned and fit
  p.plan_tbl_bytes = ((p.kmax > 1 || wide) && (p.max_blocks & 3) == 0 &&
                      (reinterpret_cast<uintptr_t>(p.block_tables) & 15) == 0)
                         ? kPlanTableBytes
                         : 0;
  static bool plan_configured[64];  // per device: the plan's dynamic shared memory and cluster size allowed
  if (dev_id < 0 || dev_id >= 64 || !plan_configured[dev_id]) {
    e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPlanTableBytes);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev_id >= 0 && dev_id < 64) plan_configured[dev_id] = true;
  }
  cfg.dynamicSmemBytes = p.plan_tbl_bytes;
  {
    const int groups = (p.num_seqs + p.kmax - 1) / p.kmax;
    const int nc = groups < kPlanCluster ? groups : kPlanCluster;
    cudaLaunchAttribute pattr[2];
    pattr[0] = attr[0];
    pattr[1].id = cudaLaunchAttributeClusterDimension;
    pattr[1].val.clusterDim.x = nc;
    pattr[1].val.clusterDim.y = 1;
    pattr[1].val.clusterDim.z = 1;
    cfg.gridDim = dim3(nc);
    cfg.attrs = pattr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, plan_kernel, p);
    for (int smaller = nc > 8 ? 8 : 1; e != cudaSuccess && smaller >= 1 && smaller < static_cast<int>(cfg.gridDim.x);
         smaller = smaller > 1 ? 1 : 0) {  // a smaller cluster: 8 CTAs, then one
      (void)cudaGetLastError();
      pattr[1].val.clusterDim.x = smaller;
      cfg.gridDim = dim3(smaller);
      e = cudaLaunchKernelEx(&cfg, plan_kernel, p);
    }
    if (e != cudaSuccess) return cuda_fail(e);
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // the wide items first, on their own SMs; the decode kernel fills the rest
  p.after_wide = wide ? 1 : 0;
  if (wide) {
    const pa_status st = launch_wide_items(p, KV, D, stream);
    if (st != PA_OK) return st;
  }
  const long long items = static_cast<long long>(p.num_seqs) * p.max_parts * p.num_kv_heads;
  const long long slots = static_cast<long long>(dev.sm_count) * ctas;
  const int grid = static_cast<int>(items < slots ? items : slots);
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sp.total;
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return cuda_fail(e);
  if (p.max_parts > 1) {
    const long long warps = static_cast<long long>(p.num_seqs) * p.num_q_heads;
    cfg.gridDim = dim3(static_cast<unsigned>((warps + kMergeWarps - 1) / kMergeWarps));
    cfg.blockDim = dim3(kMergeThreads);
    cfg.dynamicSmemBytes = 0;
    e = cudaLaunchKernelEx(&cfg, p.max_parts <= 4 ? merge_kernel<QT, D, 4> : merge_kernel<QT, D, 16>, p);
    if (e != cudaSuccess) return cuda_fail(e);
  }
  e = cudaGetLastError();
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

#ifndef PA_MMA_MIN_GROUP
#define PA_MMA_MIN_GROUP 2
#endif

template <int KV, int QT, int D>
pa_status launch_by_group(int group, const DecodeParams &p, const DeviceInfo &dev, cudaStream_t s) {
  switch (group) {
    case 1: return launch_decode<KV, QT, D, 1, (PA_MMA_MIN_GROUP <= 1)>(p, dev, s);
    case 2: return launch_decode<KV, QT, D, 2, (PA_MMA_MIN_GROUP <= 2)>(p, dev, s);
    case 4: return launch_decode<KV, QT, D, 4, true>(p, dev, s);
    case 8: return launch_decode<KV, QT, D, 8, true>(p, dev, s);
  }
  return PA_ERR_UNSUPPORTED;
}

template <int KV, int QT>
pa_status launch_by_dim(int head_dim, int group, const DecodeParams &p, const DeviceInfo &dev,
                        cudaStream_t s) {
  if (head_dim == 64) return launch_by_group<KV, QT, 64>(group, p, dev, s);
  if (head_dim == 128) return launch_by_group<KV, QT, 128>(group, p, dev, s);
  return PA_ERR_UNSUPPORTED;
}

}  // namespace
}  // namespace pa

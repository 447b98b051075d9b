// Paged causal prefill: attention of each sequence's new tokens (the part a
// prefix-cache hit did not cover) over all of its tokens in the paged cache.
//
// One CTA = one KV head h, one tile of 64 query rows of one sequence; a row
// is a (new token, query head of h's group) pair, token-major, so a tile
// holds 64 / G new tokens.  Warp w of the four consumer warps owns rows
// 16w..16w+15 as the M dimension of m16n8k16 tensor-core products:
//   S = Q K^T   (N = 64 keys of the stage, K = head_dim)
//   O += P V    (N = head_dim,            K = the stage's 64 keys)
// with an online softmax in base 2 between them and the causal mask (key
// position <= the row's position).  The fifth warp stages the K and V tiles
// of 64 keys with tiled TMA, one box per (block, 128-byte half of a row),
// written with the 128-byte swizzle; Q, K (both operands read row-wise) and
// V (read transposed) come out of the swizzled tiles with ldmatrix without
// bank conflicts.  P never leaves registers: the accumulator fragment of S
// is the A-operand fragment of P V.
#include <limits.h>
#include <math.h>

#include "pa_common.cuh"
#include "pa_host.h"

namespace pa {
namespace {

constexpr int kPfWarps = 4;                  // consumer warps
constexpr int kPfRows = 16 * kPfWarps;       // query rows per CTA
constexpr int kPfKeys = 64;                  // keys per pipeline stage
constexpr int kPfStages = 3;
constexpr int kPfThreads = 32 * (kPfWarps + 1);
constexpr int kPfHalf = kPfKeys * 128;       // one 128-byte column half of a 64-key tile

struct PrefillParams {
  CUtensorMap tmap_k;  // [rows, head_dim] 16-bit view of each cache, box {64, block_size}
  CUtensorMap tmap_v;
  void *out;
  const uint8_t *q;
  const int32_t *cu_q;
  const int32_t *block_tables;
  const int32_t *seq_lens;
  int num_q_heads, num_kv_heads, num_blocks, block_size, max_blocks;
  float qk_scale_log2;  // softmax scale * log2(e)
  int *err;
};

struct PfHeader {
  uint64_t full[kPfStages];
  uint64_t empty[kPfStages];
  int abort;
};

template <int D>
struct PfLayout {
  static constexpr int NH = D / 64;  // 128-byte halves of a 16-bit row
  static constexpr int Q_OFF = 1024;
  static constexpr int Q_HALF = kPfRows * 128;
  static constexpr int STAGE_OFF = Q_OFF + NH * Q_HALF;
  static constexpr int STAGE_BYTES = 2 * NH * kPfHalf;  // K halves, then V halves
  static constexpr int SMEM = STAGE_OFF + kPfStages * STAGE_BYTES;
};

// chunk c (16 bytes) of row r in a region of 128-byte rows written with the
// 128-byte swizzle (region 1024-byte aligned)
__device__ __forceinline__ uint32_t swz128(int r, int c) {
  return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

template <int DT, int D, int G>
__global__ void __launch_bounds__(kPfThreads, 2) prefill_kernel(const __grid_constant__ PrefillParams p) {
  using Lay = PfLayout<D>;
  constexpr int NH = Lay::NH;
  constexpr int QT = kPfRows / G;  // new tokens per CTA
  constexpr int KSTEPS = D / 16;
  constexpr int NTD = D / 8;  // n-tiles of the output
  extern __shared__ __align__(1024) uint8_t smem[];
  PfHeader &hdr = *reinterpret_cast<PfHeader *>(smem);
  const int tile = gridDim.x - 1 - blockIdx.x;  // the longest (last) tiles start first
  const int s = blockIdx.y, h = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int q0 = __ldg(p.cu_q + s);
  const int n = __ldg(p.cu_q + s + 1) - q0;
  const int L = __ldg(p.seq_lens + s);
  if (n < 0 || L < n || L > p.max_blocks * p.block_size || n > static_cast<int>(gridDim.x) * QT) {
    if (threadIdx.x == 0 && blockIdx.x == 0) record_error(p.err, kErrSeqLen);
    return;
  }
  if (tile * QT >= n) return;
  if ((smem_addr(smem) & 1023u) != 0) {  // the swizzle needs 1024-byte atoms
    if (threadIdx.x == 0) record_error(p.err, kErrSmemAlign);
    return;
  }
  const int pos0 = L - n;                        // position of new token 0
  const int kv_end = pos0 + min(n, (tile + 1) * QT);  // keys 0..kv_end-1 are needed
  const int n_tiles = (kv_end + kPfKeys - 1) / kPfKeys;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kPfStages; ++i) {
      mbar_init(&hdr.full[i], 1);
      mbar_init(&hdr.empty[i], kPfWarps);
    }
    hdr.abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  uint8_t *qs = smem + Lay::Q_OFF;
  uint8_t *stages = smem + Lay::STAGE_OFF;

  // ---------------------------------------------------------------- producer
  if (warp == kPfWarps) {
    if (lane != 0) return;
    const int bs = p.block_size;
    const int bpt = kPfKeys / bs;  // blocks per stage
    int issued = 0;
    bool ok = true;
    for (int i = 0; i < n_tiles; ++i) {
      const int st = i % kPfStages;
      if (i >= kPfStages && !mbar_wait(&hdr.empty[st], ((i / kPfStages) - 1) & 1, &hdr.abort)) {
        ok = false;
        break;
      }
      const int k0 = i * kPfKeys;
      const int nblk = min(bpt, (kv_end - k0 + bs - 1) / bs);
      mbar_arrive_expect_tx(&hdr.full[st], 2u * NH * static_cast<uint32_t>(nblk * bs) * 128u);
      uint8_t *kb = stages + st * Lay::STAGE_BYTES;
      uint8_t *vb = kb + NH * kPfHalf;
      const int32_t *row = p.block_tables + static_cast<size_t>(s) * p.max_blocks + k0 / bs;
      for (int j = 0; j < nblk; ++j) {
        int phys = __ldg(row + j);
        if (phys < 0 || phys >= p.num_blocks) {
          record_error(p.err, kErrBlockIndex);
          phys = 0;  // read a valid block; the result is void and flagged
        }
        const int r0 = (phys * p.num_kv_heads + h) * bs;
#pragma unroll
        for (int hf = 0; hf < NH; ++hf) {
          tma_load_2d(kb + hf * kPfHalf + j * bs * 128, &p.tmap_k, hf * 64, r0, &hdr.full[st]);
          tma_load_2d(vb + hf * kPfHalf + j * bs * 128, &p.tmap_v, hf * 64, r0, &hdr.full[st]);
        }
      }
      issued = i + 1;
    }
    if (!ok) {
      record_error(p.err, kErrTimeout);
      hdr.abort = 1;
      // wait, within the limit, for the copies still in flight
      for (int j = max(0, issued - kPfStages); j < issued; ++j)
        mbar_wait(&hdr.full[j % kPfStages], (j / kPfStages) & 1, nullptr);
    }
    return;
  }

  // ---------------------------------------------------------------- consumers
  const int gq = lane >> 2, tq = lane & 3;
  // Q rows of the tile into shared memory (zeros past the new tokens)
  for (int idx = threadIdx.x; idx < kPfRows * (D / 8); idx += kPfWarps * 32) {
    const int r = idx / (D / 8), c = idx % (D / 8);
    const int t = tile * QT + r / G;
    const int hq = h * G + r % G;
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    if (t < n)
      v = __ldg(reinterpret_cast<const uint4 *>(
          p.q + ((static_cast<size_t>(q0 + t) * p.num_q_heads + hq) * D + c * 8) * 2));
    *reinterpret_cast<uint4 *>(qs + (c / 8) * Lay::Q_HALF + swz128(r, c % 8)) = v;
  }
  named_bar_sync(1, kPfWarps * 32);
  uint32_t qa[KSTEPS][4];
#pragma unroll
  for (int kk = 0; kk < KSTEPS; ++kk) {
    const int r = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;
    const int c = 2 * kk + (lane >> 4);
    ldsm_x4(smem_addr(qs + (c / 8) * Lay::Q_HALF + swz128(r, c % 8)), qa[kk][0], qa[kk][1], qa[kk][2],
            qa[kk][3]);
  }
  // positions of the lane's two rows (rows past the new tokens take the last
  // one's, and are not stored)
  const int ra = 16 * warp + gq, rb = ra + 8;
  const int ta = tile * QT + ra / G, tb = tile * QT + rb / G;
  const int pa_ = pos0 + min(ta, n - 1), pb_ = pos0 + min(tb, n - 1);
  const int pmax = pos0 + min(tile * QT + (16 * warp + 15) / G, n - 1);

  float o[NTD][4];
#pragma unroll
  for (int j = 0; j < NTD; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;
  const volatile int *abort = &hdr.abort;
  bool ok = true;
  for (int i = 0; i < n_tiles; ++i) {
    const int st = i % kPfStages;
    if (!mbar_wait(&hdr.full[st], (i / kPfStages) & 1, abort)) {
      ok = false;
      break;
    }
    const int k0 = i * kPfKeys;
    if (k0 <= pmax) {  // else every key of the stage is past all the warp's rows
      const uint8_t *kb = stages + st * Lay::STAGE_BYTES;
      const uint8_t *vb = kb + NH * kPfHalf;
      // ---- S = Q K^T ----
      float sc[8][4];
#pragma unroll
      for (int j = 0; j < 8; ++j) sc[j][0] = sc[j][1] = sc[j][2] = sc[j][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) {
        const int c = 2 * kk + ((lane >> 3) & 1);
#pragma unroll
        for (int jp = 0; jp < 4; ++jp) {
          const int key = 16 * jp + (lane & 7) + (lane >> 4) * 8;
          uint32_t b0, b1, b2, b3;
          ldsm_x4(smem_addr(kb + (c / 8) * kPfHalf + swz128(key, c % 8)), b0, b1, b2, b3);
          mma16816<DT>(sc[2 * jp], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
          mma16816<DT>(sc[2 * jp + 1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b2, b3);
        }
      }
      // ---- scale, causal mask, online softmax (rows ra: regs 0,1; rb: regs 2,3) ----
      float xa = -INFINITY, xb = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = k0 + 8 * j + 2 * tq + e;
          sc[j][e] = key <= pa_ ? sc[j][e] * p.qk_scale_log2 : -INFINITY;
          sc[j][2 + e] = key <= pb_ ? sc[j][2 + e] * p.qk_scale_log2 : -INFINITY;
          xa = fmaxf(xa, sc[j][e]);
          xb = fmaxf(xb, sc[j][2 + e]);
        }
      }
      xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, 1));
      xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, 2));
      xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, 1));
      xb = fmaxf(xb, __shfl_xor_sync(0xffffffffu, xb, 2));
      const float na = fmaxf(ma, xa), nb = fmaxf(mb, xb);
      const float ba = na == -INFINITY ? 0.f : na, bb = nb == -INFINITY ? 0.f : nb;
      const float aa = exp2f(ma - ba), ab = exp2f(mb - bb);
      ma = na;
      mb = nb;
      la *= aa;
      lb *= ab;
#pragma unroll
      for (int j = 0; j < NTD; ++j) {
        o[j][0] *= aa;
        o[j][1] *= aa;
        o[j][2] *= ab;
        o[j][3] *= ab;
      }
      uint32_t pf[4][4];  // P as the A operand, k-step kk2 = keys 16kk2..16kk2+15
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float p0 = exp2f(sc[j][0] - ba), p1 = exp2f(sc[j][1] - ba);
        const float p2 = exp2f(sc[j][2] - bb), p3 = exp2f(sc[j][3] - bb);
        la += p0 + p1;
        lb += p2 + p3;
        pf[j >> 1][(j & 1) * 2] = pack2_rn<DT>(p0, p1);
        pf[j >> 1][(j & 1) * 2 + 1] = pack2_rn<DT>(p2, p3);
      }
      // ---- O += P V ----
      const bool tail = k0 + kPfKeys > kv_end;  // keys >= kv_end hold stale data: zero their V
#pragma unroll
      for (int kk2 = 0; kk2 < 4; ++kk2) {
        const int key = 16 * kk2 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int ndp = 0; ndp < NTD / 2; ++ndp) {
          const int c = 2 * ndp + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_trans(smem_addr(vb + (c / 8) * kPfHalf + swz128(key, c % 8)), b0, b1, b2, b3);
          if (tail) {
            const int ka = k0 + 16 * kk2 + 2 * tq, kb2 = ka + 8;
            const uint32_t ma0 = (ka < kv_end ? 0x0000FFFFu : 0u) | (ka + 1 < kv_end ? 0xFFFF0000u : 0u);
            const uint32_t mb0 = (kb2 < kv_end ? 0x0000FFFFu : 0u) | (kb2 + 1 < kv_end ? 0xFFFF0000u : 0u);
            b0 &= ma0;
            b2 &= ma0;
            b1 &= mb0;
            b3 &= mb0;
          }
          mma16816<DT>(o[2 * ndp], pf[kk2][0], pf[kk2][1], pf[kk2][2], pf[kk2][3], b0, b1);
          mma16816<DT>(o[2 * ndp + 1], pf[kk2][0], pf[kk2][1], pf[kk2][2], pf[kk2][3], b2, b3);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&hdr.empty[st]);
  }
  if (!ok) {
    if (lane == 0) {
      record_error(p.err, kErrTimeout);
      hdr.abort = 1;
    }
    return;
  }
  // ---- normalise and store ----
  la += __shfl_xor_sync(0xffffffffu, la, 1);
  la += __shfl_xor_sync(0xffffffffu, la, 2);
  lb += __shfl_xor_sync(0xffffffffu, lb, 1);
  lb += __shfl_xor_sync(0xffffffffu, lb, 2);
  const float ia = 1.f / la, ib = 1.f / lb;
  uint8_t *out = static_cast<uint8_t *>(p.out);
  if (ta < n) {
    uint8_t *row = out + (static_cast<size_t>(q0 + ta) * p.num_q_heads + h * G + ra % G) * D * 2;
#pragma unroll
    for (int j = 0; j < NTD; ++j)
      *reinterpret_cast<uint32_t *>(row + (8 * j + 2 * tq) * 2) = pack2_rn<DT>(o[j][0] * ia, o[j][1] * ia);
  }
  if (tb < n) {
    uint8_t *row = out + (static_cast<size_t>(q0 + tb) * p.num_q_heads + h * G + rb % G) * D * 2;
#pragma unroll
    for (int j = 0; j < NTD; ++j)
      *reinterpret_cast<uint32_t *>(row + (8 * j + 2 * tq) * 2) = pack2_rn<DT>(o[j][2] * ib, o[j][3] * ib);
  }
}

template <int DT, int D, int G>
pa_status launch_prefill(const PrefillParams &p, int num_seqs, int max_q_len, cudaStream_t stream) {
  constexpr int QT = kPfRows / G;
  static bool configured[64];  // per device: dynamic shared memory already allowed
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    e = cudaFuncSetAttribute(prefill_kernel<DT, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             PfLayout<D>::SMEM);
    if (e != cudaSuccess) return cuda_fail(e);
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  const dim3 grid((max_q_len + QT - 1) / QT, num_seqs, p.num_kv_heads);
  prefill_kernel<DT, D, G><<<grid, kPfThreads, PfLayout<D>::SMEM, stream>>>(p);
  e = cudaGetLastError();
  return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

template <int DT, int D>
pa_status by_group(int G, const PrefillParams &p, int num_seqs, int max_q_len, cudaStream_t stream) {
  switch (G) {
    case 1: return launch_prefill<DT, D, 1>(p, num_seqs, max_q_len, stream);
    case 2: return launch_prefill<DT, D, 2>(p, num_seqs, max_q_len, stream);
    case 4: return launch_prefill<DT, D, 4>(p, num_seqs, max_q_len, stream);
    case 8: return launch_prefill<DT, D, 8>(p, num_seqs, max_q_len, stream);
  }
  return PA_ERR_UNSUPPORTED;
}

// [rows, head_dim] view of a 16-bit cache, box {64 elements, block_size rows}
// (one 128-byte half of one (block, head) tile), 128-byte swizzle.
bool encode_prefill_map(CUtensorMap *map, const void *cache, const pa_cache_desc *c) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t rows = static_cast<cuuint64_t>(c->num_blocks) * c->kv_heads * c->block_size;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(c->head_dim), rows};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(c->head_dim) * 2};
  const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(c->block_size)};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void *>(cache), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" pa_status pa_prefill(void *out, const void *q, int32_t q_dtype, const int32_t *cu_q_lens,
                                int32_t num_seqs, int32_t num_q_heads, int32_t max_q_len, const void *k_cache,
                                const void *v_cache, const pa_cache_desc *cache, const int32_t *block_tables,
                                int32_t max_blocks_per_seq, const int32_t *seq_lens, float scale,
                                int *device_error, pa_stream_t stream) {
  if (!valid_cache_desc(cache) || num_seqs < 0 || num_q_heads <= 0 || max_q_len < 0 ||
      max_blocks_per_seq <= 0 || !isfinite(scale))
    return PA_ERR_INVALID;
  if (num_seqs == 0 || max_q_len == 0) return PA_OK;
  if (!out || !q || !cu_q_lens || !k_cache || !v_cache || !block_tables || !seq_lens) return PA_ERR_INVALID;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(cu_q_lens) & 3u) || (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return PA_ERR_INVALID;
  if (num_q_heads % cache->kv_heads) return PA_ERR_INVALID;
  const int G = num_q_heads / cache->kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return PA_ERR_UNSUPPORTED;
  if (!supported_cache_shape(cache)) return PA_ERR_UNSUPPORTED;
  if (cache->dtype != PA_F16 && cache->dtype != PA_BF16) return PA_ERR_UNSUPPORTED;  // 16-bit caches only
  if (q_dtype != cache->dtype) return PA_ERR_UNSUPPORTED;
  if (num_seqs > 65535 || cache->kv_heads > 65535) return PA_ERR_UNSUPPORTED;      // grid limits
  if (static_cast<long long>(cache->num_blocks) * cache->kv_heads * cache->block_size > INT_MAX ||
      static_cast<long long>(max_blocks_per_seq) * cache->block_size > INT_MAX)
    return PA_ERR_UNSUPPORTED;  // TMA row coordinates are 32-bit

  PrefillParams p{};
  if (!encode_prefill_map(&p.tmap_k, k_cache, cache) || !encode_prefill_map(&p.tmap_v, v_cache, cache))
    return cuda_fail(cudaErrorInvalidValue);
  p.out = out;
  p.q = static_cast<const uint8_t *>(q);
  p.cu_q = cu_q_lens;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = cache->kv_heads;
  p.num_blocks = cache->num_blocks;
  p.block_size = cache->block_size;
  p.max_blocks = max_blocks_per_seq;
  p.qk_scale_log2 = scale * 1.4426950408889634f;
  p.err = device_error;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cache->dtype == PA_F16)
    return cache->head_dim == 64 ? by_group<kF16, 64>(G, p, num_seqs, max_q_len, s)
                                 : by_group<kF16, 128>(G, p, num_seqs, max_q_len, s);
  return cache->head_dim == 64 ? by_group<kBF16, 64>(G, p, num_seqs, max_q_len, s)
                               : by_group<kBF16, 128>(G, p, num_seqs, max_q_len, s);
}

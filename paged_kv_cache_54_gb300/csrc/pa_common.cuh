// Shared device helpers for libpa: dtype tags, conversions, mbarrier and
// bulk-copy PTX wrappers, bounded waits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

enum DType : int { kF16 = 0, kBF16 = 1, kE4M3 = 2, kE5M2 = 3, kI8 = 4 };

enum DevErr : int {
  kErrNone = 0,
  kErrBlockIndex = 1,
  kErrSlot = 2,
  kErrSeqLen = 3,
  kErrTimeout = 4,
  kErrCopyIndex = 5,
  kErrSmemAlign = 6,
};

// Wait limit for every spin on an mbarrier: 2 s of %globaltimer.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

__host__ __device__ constexpr bool is_fp8(int dt) { return dt == kE4M3 || dt == kE5M2; }
// one-byte KV codes: FP8 or INT8, each stored as value / scale
__host__ __device__ constexpr bool is_byte(int dt) { return is_fp8(dt) || dt == kI8; }
__host__ __device__ constexpr int elt_bytes(int dt) { return is_byte(dt) ? 1 : 2; }

__device__ __forceinline__ void record_error(int *err, int code) {
  if (err != nullptr) atomicCAS(err, 0, code);
}

// ----------------------------------------------------------------------------
// conversions
// ----------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ float2 half2_bits_to_float2(uint32_t w) {
  if constexpr (DT == kF16) {
    __half2 h = *reinterpret_cast<const __half2 *>(&w);
    return __half22float2(h);
  } else {
    __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(&w);
    return __bfloat1622float2(h);
  }
}

// Four INT8 codes in one word -> two __half2 (codes 0,1 -> lo; 2,3 -> hi),
// exact.  Flipping the sign bit turns code c into the unsigned u = c + 128;
// the half with bit pattern 0x6400 | u is 1024 + u (exponent 10, so the ten
// mantissa bits count units), and subtracting 1152 = 1024 + 128 leaves c.
__device__ __forceinline__ void i8x4_to_half2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
  const uint32_t u = w ^ 0x80808080u;
  uint32_t a, b;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(a) : "r"(u), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(b) : "r"(u), "r"(0x64646464u));
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  const __half2 x = __hsub2(*reinterpret_cast<const __half2 *>(&a), bias);
  const __half2 y = __hsub2(*reinterpret_cast<const __half2 *>(&b), bias);
  lo = *reinterpret_cast<const uint32_t *>(&x);
  hi = *reinterpret_cast<const uint32_t *>(&y);
}

// Four INT8 codes -> two __half2 of 1152 + c (exact integers in
// [1024, 1279]): the widening above without its subtraction.  For a sum
// over codes, sum_i (1152 + c_i) x_i = sum_i c_i x_i + 1152 sum_i x_i, so a
// caller that removes 1152 sum_i x_i once saves the subtraction per pair.
__device__ __forceinline__ void i8x4_to_half2x2_offset(uint32_t w, uint32_t &lo, uint32_t &hi) {
  const uint32_t u = w ^ 0x80808080u;
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(lo) : "r"(u), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(hi) : "r"(u), "r"(0x64646464u));
}
constexpr float kI8Offset = 1152.f;

// two one-byte codes (low byte = first element) -> __half2 bits (exact:
// every e4m3 / e5m2 value and every int8 is an fp16 value)
template <int DT>
__device__ __forceinline__ uint32_t byte2_to_half2_bits(uint32_t two_codes) {
  if constexpr (DT == kI8) {
    uint32_t lo, hi;
    i8x4_to_half2x2(two_codes, lo, hi);
    return lo;
  } else {
    __half2_raw r = __nv_cvt_fp8x2_to_halfraw2(
        static_cast<__nv_fp8x2_storage_t>(two_codes & 0xFFFFu),
        DT == kE4M3 ? __NV_E4M3 : __NV_E5M2);
    return static_cast<uint32_t>(r.x) | (static_cast<uint32_t>(r.y) << 16);
  }
}

// four one-byte codes in one word -> two __half2 (codes 0,1 -> lo; codes
// 2,3 -> hi), exact
template <int DT>
__device__ __forceinline__ void byte4_to_half2x2(uint32_t w, uint32_t &lo, uint32_t &hi) {
  if constexpr (DT == kE4M3) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, a;\n\tcvt.rn.f16x2.e4m3x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
  } else if constexpr (DT == kE5M2) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\t"
        "cvt.rn.f16x2.e5m2x2 %0, a;\n\tcvt.rn.f16x2.e5m2x2 %1, b;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
  } else {
    i8x4_to_half2x2(w, lo, hi);
  }
}

template <int DT>
__device__ __forceinline__ float2 byte2_to_float2(uint32_t two_codes) {
  uint32_t h = byte2_to_half2_bits<DT>(two_codes);
  return __half22float2(*reinterpret_cast<const __half2 *>(&h));
}

template <int DT>
__device__ __forceinline__ uint16_t float_to_storage16(float x) {
  if constexpr (DT == kF16) {
    return __half_as_ushort(__float2half_rn(x));
  } else {
    return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  }
}

template <int DT>
__device__ __forceinline__ uint32_t pack2_rn(float lo, float hi) {
  if constexpr (DT == kF16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  }
}

// ----------------------------------------------------------------------------
// shared-memory addressing, mbarriers, bulk copies
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

#ifndef PA_WAIT_HINT_NS
#define PA_WAIT_HINT_NS 0
#endif

// One test of an mbarrier phase.  The instruction may suspend the thread
// until the phase completes or a time limit passes; with PA_WAIT_HINT_NS > 0
// that limit is raised to the given number of nanoseconds, so a waiting warp
// sleeps instead of re-issuing the test.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
#if PA_WAIT_HINT_NS > 0
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "n"(PA_WAIT_HINT_NS)
      : "memory");
#else
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
#endif
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for the phase of `bar` with the given parity to complete.  Returns
// false if it did not within kWaitLimitNs, or if *abort became nonzero.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, const volatile int *abort) {
  const uint32_t a = smem_addr(bar);
  if (mbar_try_wait(a, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(a, parity)) return true;
    if ((i & 63u) == 0) {
      if (abort != nullptr && *abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
  }
}

// Bulk (TMA) copy global -> shared of `bytes` (multiple of 16, both addresses
// 16-byte aligned), completing on the mbarrier's transaction count.
__device__ __forceinline__ void bulk_g2s(void *smem_dst, const void *gmem_src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Tiled TMA load of one tile of a 2-D ([rows, 128 B]) or 3-D ([rows, 2, 128 B])
// tensor view, rows [row0, row0 + box rows), completing on the mbarrier's
// transaction count.  The tensor map lives in the kernel's parameter space.
// L2 eviction priorities.  The decode streams each K/V tile through L2 once
// (evict first), so the split-K partials it writes stay in L2 until the
// merge reads them (evict last).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// One (block, head) tile of a cache by tiled TMA: rows [row0, row0 + box)
// of the [rows, 128 B] (2-D) or [rows, 2, 128 B] (3-D) view, with an L2
// cache policy.
template <bool kThreeD>
__device__ __forceinline__ void tma_load_tile(void *smem_dst, const CUtensorMap *map, int row0, uint64_t *bar,
                                              uint64_t policy) {
  if constexpr (kThreeD) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_addr(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(0), "r"(row0), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
  } else {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row0), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
  }
}

// bulk_g2s with an L2 cache policy
__device__ __forceinline__ void bulk_g2s_hint(void *smem_dst, const void *gmem_src, uint32_t bytes, uint64_t *bar,
                                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// four floats to global memory with an L2 cache policy (16-byte aligned)
__device__ __forceinline__ void st_global_f4_hint(float *addr, float4 v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(addr), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w), "l"(policy)
               : "memory");
}

// two floats to global memory with an L2 cache policy (8-byte aligned)
__device__ __forceinline__ void st_global_f2_hint(float *addr, float a, float b, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.v2.f32 [%0], {%1, %2}, %3;" ::"l"(addr), "f"(a), "f"(b), "l"(policy)
               : "memory");
}

// Tiled TMA load of the 2-D box at (x, y) (x in elements, a multiple of 16
// bytes), completing on the mbarrier's transaction count.
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
      : "memory");
}

// D += A * B on the legacy tensor-core path, m16n8k16, fp32 accumulators;
// A and B both fp16 (MT == kF16) or both bf16.
template <int MT>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  if constexpr (MT == kF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

// ----------------------------------------------------------------------------
// 5th-generation tensor cores (tcgen05) and tensor memory
// ----------------------------------------------------------------------------
// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets (all in 16-byte units), the fixed version field (bits 46-48 =
// 0b001) and the 128-byte swizzle (layout type 2, bits 61-63).  For a
// K-major operand in 128-byte-swizzled rows the stride offset is the 1024
// bytes between groups of 8 rows; for an MN-major one the leading offset
// is the distance between 64-element column blocks and the stride offset
// the 1024 bytes between groups of 8 K-rows.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) |
         (static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor of tcgen05.mma kind::f16 with an fp32 accumulator:
// A and B fp16 (ab = 0) or bf16 (ab = 1), B K-major or MN-major, M x N.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int ab, int M, int N, bool b_mn_major) {
  return (1u << 4) | (static_cast<uint32_t>(ab) << 7) | (static_cast<uint32_t>(ab) << 10) |
         ((b_mn_major ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// D (tensor memory) = A * B (+ D when accumulate != 0); issued by one thread.
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D (tensor memory) = A * B (+ D), A read from tensor memory (row r of A in
// lane r, two 16-bit elements per 32-bit column, element 2c in the low half
// of column c) and B from shared memory; issued by one thread.
__device__ __forceinline__ void tc_mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on the mbarrier when every tcgen05 operation this thread has
// issued so far has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Tensor-memory allocation (one whole warp): the base address is written to
// *dst in shared memory.
__device__ __forceinline__ void tc_alloc(uint32_t *dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tc_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// 32 consecutive 32-bit columns of the warp's 32 lanes (lane = thread), and
// the wait for them, in one statement so no use can move above the wait.
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {"
      "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tc_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {"
      "%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
      "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Tiled TMA load of the 4-D box at (x, y, z, w), completing on the mbarrier.
__device__ __forceinline__ void tma_load_4d(void *smem_dst, const CUtensorMap *map, int x, int y, int z, int w,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_addr(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_addr(bar))
      : "memory");
}


// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start before the previous kernel in the stream ends;
// grid_dependency_wait() blocks until that kernel has completed and its
// memory is visible.  launch_dependents() lets the next such kernel start.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// Thread-block clusters: this CTA's rank, the cluster's CTA count, and a
// barrier over every thread of the cluster that orders their memory
// accesses before it (release) with those after it (acquire).
__device__ __forceinline__ int cluster_rank() {
  unsigned r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return static_cast<int>(r);
}
__device__ __forceinline__ int cluster_ctas() {
  unsigned n;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(n));
  return static_cast<int>(n);
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint4 lds128(const void *p) {
  return *reinterpret_cast<const uint4 *>(p);
}

// Per-thread asynchronous copy of BYTES (8 or 16, both addresses aligned to
// it) from global to shared memory, bypassing L1 for 16.  Copies are grouped
// by commit; cp_async_wait<N>() returns once at most N of the thread's most
// recent groups are still in flight.
template <int BYTES>
__device__ __forceinline__ void cp_async(void *smem_dst, const void *gmem_src) {
  static_assert(BYTES == 8 || BYTES == 16, "cp.async of 8 or 16 bytes");
  if constexpr (BYTES == 16)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem_dst)), "l"(gmem_src) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(smem_dst)), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

}  // namespace pa

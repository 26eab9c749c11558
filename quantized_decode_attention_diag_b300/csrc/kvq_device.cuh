// Device helpers shared by the append and decode kernels (sm_103a).
//
// Only hand-written inline PTX for data movement (cp.async.bulk + mbarrier),
// the legacy warp-level tensor-core MMA, packed fp32 pairs and bit tricks;
// all math library functions (exp2f, fp16 conversions with explicit rounding
// modes) are called, not re-implemented.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "kvq_internal.h"

namespace kvq {

constexpr unsigned kFullMask = 0xffffffffu;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void flag_status(int* status, int bit) {
  if (status) atomicOr(status, bit);
}

// ---------------------------------------------------------------- bf16 -----
// Two bf16 values packed in a 32-bit word -> exact fp32 values.
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// ----------------------------------------------------- packed fp32 pairs ---
// add/sub of two fp32 pairs with round-to-nearest per element (sm_100+).
__device__ __forceinline__ void addsub2(float& a0, float& a1, float& b0, float& b1) {
  // (a, b) <- (a + b, a - b), elementwise on the pairs (a0, a1), (b0, b1)
  float s0, s1, d0, d1;
  asm("{\n\t.reg .b64 ra, rb, rs, rd;\n\t"
      "mov.b64 ra, {%4, %5};\n\t"
      "mov.b64 rb, {%6, %7};\n\t"
      "add.rn.f32x2 rs, ra, rb;\n\t"
      "sub.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rs;\n\t"
      "mov.b64 {%2, %3}, rd;\n\t}"
      : "=f"(s0), "=f"(s1), "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
  a0 = s0; a1 = s1; b0 = d0; b1 = d1;
}

// f = fma(x - z, inv, c) on a pair of fp32 values, round-to-nearest per
// element (packed f32x2, sm_100+); returns the raw bits of both results.
__device__ __forceinline__ void subfma2(float x0, float x1, float z, float inv, float c,
                                        uint32_t& r0, uint32_t& r1) {
  asm("{\n\t.reg .b64 rx, rz, rd, ri, rc, rr;\n\t"
      "mov.b64 rx, {%2, %3};\n\t"
      "mov.b64 rz, {%4, %4};\n\t"
      "mov.b64 ri, {%5, %5};\n\t"
      "mov.b64 rc, {%6, %6};\n\t"
      "sub.rn.f32x2 rd, rx, rz;\n\t"
      "fma.rn.f32x2 rr, rd, ri, rc;\n\t"
      "mov.b64 {%0, %1}, rr;\n\t}"
      : "=r"(r0), "=r"(r1)
      : "f"(x0), "f"(x1), "f"(z), "f"(inv), "f"(c));
}

// (r0, r1) = (a0 b0, a1 b1) and (a0 - b0, a1 - b1): packed fp32 pairs,
// round-to-nearest per element (sm_100+).
__device__ __forceinline__ void mul2(float a0, float a1, float b0, float b1, float& r0, float& r1) {
  asm("{\n\t.reg .b64 ra, rb, rr;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rr, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rr;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ void sub2(float a0, float a1, float b0, float b1, float& r0, float& r1) {
  asm("{\n\t.reg .b64 ra, rb, rr;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "sub.rn.f32x2 rr, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rr;\n\t}"
      : "=f"(r0), "=f"(r1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}

// Three-input minimum and maximum (sm_100+).
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Prefetch of `bytes` (a multiple of 16; 16-byte aligned address) into L2 by
// the bulk-copy engine; a hint, nothing waits for it.
__device__ __forceinline__ void l2_prefetch_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// ------------------------------------------------------ mbarrier + bulk ----
__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Global -> shared bulk copy (TMA engine, no tensor map); completes `bytes`
// transactions on `bar`.  dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// mbar_expect_tx + bulk_g2s by the lanes with `pred` set, as predicated
// instructions (no branch, no reconvergence point in the caller's loop).
__device__ __forceinline__ void bulk_g2s_if(bool pred, uint32_t dst, const void* src,
                                            unsigned bytes, uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.u32 p, %0, 0;\n\t"
      "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%1], %2;\n\t"
      "@p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%3], [%4], %2, [%1];\n\t"
      "}" ::"r"(static_cast<unsigned>(pred)),
      "r"(bar), "r"(bytes), "r"(dst), "l"(src)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar`, giving up after ~2^limit_log2 SM cycles
// (2^31: about a second).  Returns false on timeout; the caller records it and
// drains its copies with the full limit.
// A shorter limit (a debugging aid) also polls with test_wait, which never
// suspends the thread: try_wait may sleep until the phase completes, so a short
// limit could never run out.
constexpr int kWaitLimitLog2 = 31;
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, unsigned parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, unsigned parity,
                                                  int limit_log2 = kWaitLimitLog2) {
  if (limit_log2 < kWaitLimitLog2) {
    const long long t0 = clock64();
    while (!mbar_test_wait(bar, parity)) {
      if (clock64() - t0 > (1ll << limit_log2)) return false;
    }
    return true;
  }
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > (1ll << limit_log2)) return false;
  }
  return true;
}

// Both of two consecutive barriers (bar, bar + 1) at phase `parity`, for the
// whole warp (every lane calls it; the result is warp-uniform): one combined
// non-blocking test and a vote on the fast path; when a copy is late, bounded
// waits on each barrier with the limit read from shared memory (*limit_log2, a
// volatile load, so that no register holds it across the caller's loop).
__device__ __forceinline__ bool mbar_wait2_warp(uint64_t* bar, unsigned parity,
                                                const int* limit_log2) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 q, [%1 + 8], %2;\n\t"
      "and.pred p, p, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  if (__all_sync(0xffffffffu, ok != 0)) return true;
  int lim;
  asm volatile("ld.volatile.shared.s32 %0, [%1];" : "=r"(lim) : "r"(smem_u32(limit_log2)));
  const bool a = mbar_wait_bounded(bar, parity, lim);
  const bool b = mbar_wait_bounded(bar + 1, parity, lim);
  return __all_sync(0xffffffffu, a && b);
}

// ------------------------------------------------------ tensor-core MMA ----
// D[16x8] += A[16x16] * B[16x8], fp16 inputs, fp32 accumulate (warp-wide).
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
  asm(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// ------------------------------------------- code -> fp16 pair conversion --
// fp16 1024.0 is 0x6400; OR-ing a small integer c (< 1024) into the low
// mantissa bits gives exactly 1024 + c.  Scaled fields (c << k) give
// 1024 + c * 2^k and are brought back with an exact fma.
__device__ __forceinline__ uint32_t lop_or_magic(uint32_t x, uint32_t mask) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(r) : "r"(x), "r"(mask), "r"(0x64006400u));
  return r;  // (x & mask) | 0x64006400
}

__device__ __forceinline__ uint32_t h2_sub1024(uint32_t x) {
  __half2 r = __hsub2(*reinterpret_cast<__half2*>(&x), __half2(__half(1024.f), __half(1024.f)));
  return *reinterpret_cast<uint32_t*>(&r);
}

// (1024 + c * 2^k) * 2^-k - 1024 * 2^-k = c, exact in fp16
template <int K>
__device__ __forceinline__ uint32_t h2_unscale(uint32_t x) {
  constexpr float inv = 1.0f / float(1 << K);
  constexpr float off = -1024.0f / float(1 << K);
  __half2 r = __hfma2(*reinterpret_cast<__half2*>(&x), __half2(__half(inv), __half(inv)),
                      __half2(__half(off), __half(off)));
  return *reinterpret_cast<uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t pack_half2(__half lo, __half hi) {
  return static_cast<uint32_t>(__half_as_ushort(lo)) |
         (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
}

}  // namespace kvq

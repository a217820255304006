// Device helpers for the NVFP4 GEMV kernels (sm_103a): format conversions, packed-half math and
// streaming loads, as inline PTX.
//
// Format facts used here (the C header states them with their sources): an E2M1 byte holds the
// element with even k in its low nibble; an E4M3FN block scale covers 16 consecutive k.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace nvfp4 {

// Four packed E2M1 bytes (8 elements, byte j = elements 2j, 2j+1) -> four f16x2 words; word j
// holds byte j's two elements in the same nibble -> half order the conversion uses for every
// operand, so lane-wise products of two such words pair equal k.  Exact: every E2M1 value is an
// f16 value.
__device__ __forceinline__ void e2m1x8_to_f16x2x4(uint32_t w, uint32_t& h0, uint32_t& h1,
                                                  uint32_t& h2, uint32_t& h3) {
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "mov.b32 {q0, q1, q2, q3}, %4;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, q0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, q1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, q2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, q3;\n\t}"
      : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
      : "r"(w));
}

// One packed E2M1 byte (low 8 bits of v) -> f16x2.
__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t v) {
  uint32_t h;
  asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
      "mov.b32 {q0, q1, q2, q3}, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, q0;\n\t}"
      : "=r"(h)
      : "r"(v));
  return h;
}

// Two E4M3FN bytes (low byte = first scale) -> f16x2 (low half = first scale).  Exact: every
// E4M3FN value, subnormals and NaN included, is an f16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(v));
  return h;
}

// acc += a * b on both halves (f16x2, round-to-nearest).
__device__ __forceinline__ void hfma2(uint32_t& acc, uint32_t a, uint32_t b) {
  asm("fma.rn.f16x2 %0, %1, %2, %0;" : "+r"(acc) : "r"(a), "r"(b));
}

// Both halves of an f16x2 widened to f32 (exact).
__device__ __forceinline__ float2 f16x2_to_f32x2(uint32_t h) {
  float lo, hi;
  asm("{\n\t.reg .b16 l, u;\n\t"
      "mov.b32 {l, u}, %2;\n\t"
      "cvt.f32.f16 %0, l;\n\t"
      "cvt.f32.f16 %1, u;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h));
  return make_float2(lo, hi);
}

// Two exact block partials scaled by their block scales, in fp32: for p0 (block A) and p1 (block
// B) as f16x2 half sums and sa2 = (scale A, scale B) as f16x2, returns
// ((p0.lo + p0.hi) * sa.A, (p1.lo + p1.hi) * sa.B) by four mixed-precision FMAs (f16 operands,
// f32 accumulation).  Exact: each half sum is a multiple of 1/4 below 2^9 and a scale has 4
// significant bits, so every product and both sums fit fp32's 24 bits.
__device__ __forceinline__ float2 scaled_block_pair(uint32_t p0, uint32_t p1, uint32_t sa2) {
  float a, b;
  asm("{\n\t.reg .b16 a0, a1, b0, b1, s0, s1;\n\t"
      "mov.b32 {a0, a1}, %2;\n\t"
      "mov.b32 {b0, b1}, %3;\n\t"
      "mov.b32 {s0, s1}, %4;\n\t"
      "fma.rn.f32.f16 %0, a0, s0, 0f00000000;\n\t"
      "fma.rn.f32.f16 %0, a1, s0, %0;\n\t"
      "fma.rn.f32.f16 %1, b0, s1, 0f00000000;\n\t"
      "fma.rn.f32.f16 %1, b1, s1, %1;\n\t}"
      : "=f"(a), "=f"(b)
      : "r"(p0), "r"(p1), "r"(sa2));
  return make_float2(a, b);
}

// acc += a * b on both lanes of an fp32 pair (one packed fp32x2 FMA, round-to-nearest each).
__device__ __forceinline__ void ffma2(float2& acc, float2 a, float2 b) {
  asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%0, %1};\n\t"
      "fma.rn.f32x2 rc, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rc;\n\t}"
      : "+f"(acc.x), "+f"(acc.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
}

// 16-byte read-only streaming load: not allocated in L1 (each byte of A is read once).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint16_t ld_stream_u16(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// Loads of the vector (and of the activation) read through L2 only (.cg), never from an L1 line:
// under programmatic dependent launch the data may have been written by a grid that was still
// running when this one started, after another grid on this SM had cached the old bytes.
__device__ __forceinline__ uint4 ld_l2_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t ld_l2_u32(const void* p) {
  uint32_t v;
  asm volatile("ld.global.cg.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint16_t ld_l2_u16(const void* p) {
  uint16_t v;
  asm volatile("ld.global.cg.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// fp32 -> IEEE binary16 bits, round-to-nearest-even, overflow to +-inf.
__device__ __forceinline__ uint16_t f32_to_f16_bits(float x) {
  return __half_as_ushort(__float2half_rn(x));
}

// fp32 -> bfloat16 bits, round-to-nearest-even.
__device__ __forceinline__ uint16_t f32_to_bf16_bits(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ uint16_t f32_to_out_bits(float x, bool bf16) {
  return bf16 ? f32_to_bf16_bits(x) : f32_to_f16_bits(x);
}

}  // namespace nvfp4

// ------------------------------------------------------------------ async-copy and barrier PTX
namespace nvfp4 {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for the phase of `bar` with the given parity to complete, for at most `limit_ns`
// nanoseconds of wall time.  Returns false on timeout (the caller then stops and reports).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
  }
}

// As mbar_wait_bounded, for waiters off the critical path (an epilogue waiting for a whole
// mainloop): they sleep between polls instead of taking issue slots from the warps that work.
__device__ __forceinline__ bool mbar_wait_sleepy(uint32_t bar, uint32_t parity,
                                                 uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    __nanosleep(200);
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
  }
}

// L2 policy for data read exactly once.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk (non-tensor) async copy global -> shared, completing `bytes` of transaction count on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1], %2, [%3], %4;" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(policy)
      : "memory");
}

// Bulk prefetch of global bytes into L2 (a hint: no value read by anyone changes).  src 16-byte
// aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Barrier over a subset of the CTA's warps (id 1..15; `threads` a multiple of 32).
__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

}  // namespace nvfp4

// NVFP4 activation quantizer with a fixed global scale (GB300, sm_103a).
//
// cutedsl/bridge.py (nvfp4-megamoe-kernel), section "Quantization", quantize_activation_nvfp4:
// with the global scale given, every 16-element block is quantized on its own, so one thread (or
// one lane) owns whole blocks and the step needs no reduction across threads or kernels.  All
// arithmetic is fp32 with IEEE round-to-nearest divisions, as the page's torch operations are:
//   x_norm = x / gs;  amax = max(max |x_norm|, 1e-8);  scale = e4m3(amax / 6);
//   x_scaled = x_norm / max(scale, 1e-8);  magnitude = min(|x_scaled|, 6);
//   code = table[rint(2 * magnitude)] (the page's half-step table) or the nearest E2M1 grid point
//   with ties to the even code;  nibble = code | 8 if x_scaled < 0.
// The scale conversion is the page's float8_e4m3fn cast: nearest, ties to even, and NaN (0x7F)
// for a value past 464 (it would round beyond 448, the largest finite E4M3).  The block's codes
// are then 0.  Inputs are finite bf16 values (a NaN input gives unspecified bytes for its block).
#pragma once

#include <stdint.h>

#include "nvfp4_device.cuh"

namespace nvfp4 {

enum : int { kRoundHalfStepTable = 0, kRoundNearestEven = 1 };

// half-step table [0, 1, 2, 3, 4, 4, 5, 5, 6, 6, 6, 7, 7], entry i in bits 4i .. 4i+3
constexpr uint64_t kHalfStepTable = 0x7766655443210ull;

// Two non-negative fp32 values -> two E4M3FN bytes, low byte from `lo`: round to nearest even;
// a value past 464 has no finite encoding and gives NaN (0x7F), as a float8_e4m3fn cast does.
// (The hardware conversion saturates instead, so those two cases are patched after it.)
constexpr uint32_t kE4m3Nan = 0x7Fu;

__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  if (lo > 464.0f) r = (uint16_t)((r & 0xFF00u) | kE4m3Nan);
  if (hi > 464.0f) r = (uint16_t)((r & 0x00FFu) | (kE4m3Nan << 8));
  return r;
}

__device__ __forceinline__ uint32_t e2m1_code(float mag, int rounding) {
  if (rounding == kRoundHalfStepTable) {
    const int hs = min(max(__float2int_rn(2.0f * mag), 0), 12);
    return (uint32_t)((kHalfStepTable >> (4 * hs)) & 0xFu);
  }
  // midpoints 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5: a value on a midpoint goes to the even code
  return (uint32_t)(mag > 0.25f) + (uint32_t)(mag >= 0.75f) + (uint32_t)(mag > 1.25f) +
         (uint32_t)(mag >= 1.75f) + (uint32_t)(mag > 2.5f) + (uint32_t)(mag >= 3.5f) +
         (uint32_t)(mag > 5.0f);
}

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// Quantizes two 16-element blocks held as 32 bf16 values in xv (64 bytes, element 2i in the low
// half of word i).  Returns the 16 packed bytes (element 2j in the low nibble of byte j) and the
// two scale bytes (block 0 in the low byte).
__device__ __forceinline__ void quantize_blocks2(const uint32_t (&xv)[16], float gs, int rounding,
                                                 uint32_t (&packed)[4], uint16_t& sf2) {
  float xn[32];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    xn[2 * i] = __fdiv_rn(bf16_bits_to_f32(xv[i] & 0xFFFFu), gs);
    xn[2 * i + 1] = __fdiv_rn(bf16_bits_to_f32(xv[i] >> 16), gs);
  }
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    a0 = fmaxf(a0, fabsf(xn[i]));
    a1 = fmaxf(a1, fabsf(xn[16 + i]));
  }
  a0 = fmaxf(a0, 1e-8f);
  a1 = fmaxf(a1, 1e-8f);
  sf2 = f32x2_to_e4m3x2(__fdiv_rn(a0, 6.0f), __fdiv_rn(a1, 6.0f));
  const float2 sv = f16x2_to_f32x2(e4m3x2_to_f16x2(sf2));
  const float d0 = fmaxf(sv.x, 1e-8f), d1 = fmaxf(sv.y, 1e-8f);
  const bool nan0 = (sf2 & 0xFFu) == kE4m3Nan, nan1 = (sf2 >> 8) == kE4m3Nan;
#pragma unroll
  for (int w = 0; w < 4; ++w) packed[w] = 0u;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float xs = __fdiv_rn(xn[i], i < 16 ? d0 : d1);
    const uint32_t nib = e2m1_code(fminf(fabsf(xs), 6.0f), rounding) | (xs < 0.f ? 8u : 0u);
    if (!(i < 16 ? nan0 : nan1)) packed[i >> 3] |= nib << (4 * (i & 7));
  }
}

// Standalone quantizer: eight consecutive threads own one 16-element block, two elements each
// (x 16-byte aligned, K % 16 == 0, so a block never straddles two warps).  The block maximum is a
// shuffle reduction over the eight lanes; each lane then writes the byte of its element pair and
// the block's first lane the scale byte (a warp writes 32 consecutive packed bytes).  The kernel
// releases its dependents at once (they only read what it writes after their own grid wait) and
// waits for the preceding work before touching memory.
__global__ void __launch_bounds__(256) quantize_activation_kernel(
    const uint16_t* __restrict__ x, float gs, int rounding, uint8_t* __restrict__ b,
    uint8_t* __restrict__ sfb, int64_t n_pairs) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const bool valid = t < n_pairs;  // n_pairs % 8 == 0: a block's eight lanes agree
  const uint32_t w = ld_l2_u32(x + 2 * (valid ? t : 0));
  const float xn0 = __fdiv_rn(bf16_bits_to_f32(w & 0xFFFFu), gs);
  const float xn1 = __fdiv_rn(bf16_bits_to_f32(w >> 16), gs);
  float a = fmaxf(fabsf(xn0), fabsf(xn1));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
  a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 4));
  a = fmaxf(a, 1e-8f);
  const uint16_t s2 = f32x2_to_e4m3x2(__fdiv_rn(a, 6.0f), 0.f);
  const float d = fmaxf(f16x2_to_f32x2(e4m3x2_to_f16x2(s2)).x, 1e-8f);
  const float xs0 = __fdiv_rn(xn0, d), xs1 = __fdiv_rn(xn1, d);
  const uint32_t nib0 = e2m1_code(fminf(fabsf(xs0), 6.0f), rounding) | (xs0 < 0.f ? 8u : 0u);
  const uint32_t nib1 = e2m1_code(fminf(fabsf(xs1), 6.0f), rounding) | (xs1 < 0.f ? 8u : 0u);
  const bool nan_scale = (s2 & 0xFFu) == kE4m3Nan;  // the block's codes are 0
  if (valid) {
    b[t] = nan_scale ? (uint8_t)0 : (uint8_t)(nib0 | (nib1 << 4));
    if ((t & 7) == 0) sfb[t >> 3] = (uint8_t)(s2 & 0xFFu);
  }
}

}  // namespace nvfp4

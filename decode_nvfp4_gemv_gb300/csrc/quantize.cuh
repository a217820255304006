// NVFP4 activation quantizer with a fixed global scale (GB300, sm_103a).
//
// cutedsl/bridge.py (nvfp4-megamoe-kernel), section "Quantization", quantize_activation_nvfp4:
// with the global scale given, every 16-element block is quantized on its own, so one thread (or
// one lane) owns whole blocks and the step needs no reduction across threads or kernels.  All
// arithmetic is fp32 in the page's order, with IEEE round-to-nearest divisions:
//   x_norm = x / gs;  amax = max(max |x_norm|, 1e-8);  scale = e4m3_rn_sat(amax / 6);
//   x_scaled = x_norm / max(scale, 1e-8);  magnitude = min(|x_scaled|, 6);
//   code = table[rint(2 * magnitude)] (the page's half-step table) or the nearest E2M1 grid point
//   with ties to the even code;  nibble = code | 8 if x_scaled < 0.
// A block scale that rounds above 448 saturates to 448 (the conversion is `satfinite`).  Inputs
// are finite bf16 values (a NaN input gives unspecified bytes for its block).
#pragma once

#include <stdint.h>

#include "nvfp4_device.cuh"

namespace nvfp4 {

enum : int { kRoundHalfStepTable = 0, kRoundNearestEven = 1 };

// half-step table [0, 1, 2, 3, 4, 4, 5, 5, 6, 6, 6, 7, 7], entry i in bits 4i .. 4i+3
constexpr uint64_t kHalfStepTable = 0x7766655443210ull;

// Two fp32 values -> two E4M3FN bytes (round to nearest even, saturating): low byte from `lo`.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2_sat(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
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
  sf2 = f32x2_to_e4m3x2_sat(__fdiv_rn(a0, 6.0f), __fdiv_rn(a1, 6.0f));
  const float2 sv = f16x2_to_f32x2(e4m3x2_to_f16x2(sf2));
  const float d0 = fmaxf(sv.x, 1e-8f), d1 = fmaxf(sv.y, 1e-8f);
#pragma unroll
  for (int w = 0; w < 4; ++w) packed[w] = 0u;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float xs = __fdiv_rn(xn[i], i < 16 ? d0 : d1);
    const uint32_t nib = e2m1_code(fminf(fabsf(xs), 6.0f), rounding) | (xs < 0.f ? 8u : 0u);
    packed[i >> 3] |= nib << (4 * (i & 7));
  }
}

// One 16-element block (the standalone kernel's unit; K need only be a multiple of 16).
__device__ __forceinline__ void quantize_block1(const uint32_t (&xv)[8], float gs, int rounding,
                                                uint32_t (&packed)[2], uint8_t& sf) {
  float xn[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    xn[2 * i] = __fdiv_rn(bf16_bits_to_f32(xv[i] & 0xFFFFu), gs);
    xn[2 * i + 1] = __fdiv_rn(bf16_bits_to_f32(xv[i] >> 16), gs);
  }
  float a = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(xn[i]));
  a = fmaxf(a, 1e-8f);
  const uint16_t s2 = f32x2_to_e4m3x2_sat(__fdiv_rn(a, 6.0f), 0.f);
  sf = (uint8_t)(s2 & 0xFFu);
  const float d = fmaxf(f16x2_to_f32x2(e4m3x2_to_f16x2(s2)).x, 1e-8f);
  packed[0] = packed[1] = 0u;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float xs = __fdiv_rn(xn[i], d);
    const uint32_t nib = e2m1_code(fminf(fabsf(xs), 6.0f), rounding) | (xs < 0.f ? 8u : 0u);
    packed[i >> 3] |= nib << (4 * (i & 7));
  }
}

// Standalone quantizer: thread t quantizes block t of the [L][K/16] blocks (x 16-byte aligned, K %
// 16 == 0): 32 bytes of bf16 in, 8 packed bytes and 1 scale byte out (coalesced across the warp).
__global__ void __launch_bounds__(256) quantize_activation_kernel(
    const uint16_t* __restrict__ x, float gs, int rounding, uint8_t* __restrict__ b,
    uint8_t* __restrict__ sfb, int64_t n_blocks) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t >= n_blocks) return;
  const uint4 v0 = ld_ro_v4(x + 16 * t);
  const uint4 v1 = ld_ro_v4(x + 16 * t + 8);
  const uint32_t xv[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  uint32_t packed[2];
  uint8_t sf;
  quantize_block1(xv, gs, rounding, packed, sf);
  *reinterpret_cast<uint2*>(b + 8 * t) = make_uint2(packed[0], packed[1]);
  sfb[t] = sf;
}

}  // namespace nvfp4

// General-alignment NVFP4 GEMV for GB300 (sm_103a): any K % 16 == 0, any byte alignment of A,
// sfa, b and sfb.
//
// Why: the TMA and vector-load kernels need 16-byte aligned operands (and K % 256 or K % 32);
// the byte-load kernel takes anything but moves one byte per load.  This kernel keeps wide loads
// for misaligned rows: a lane's 16 bytes of a row that starts d bytes past a 16-byte boundary are
// the last 16 - d bytes of one aligned 16-byte chunk and the first d bytes of the next, so the lane
// loads both chunks and funnel-shifts them by d bytes.  All lanes of a warp read the same row at
// offsets that differ by multiples of 16, so d (and the branch on it) is the same for the whole
// warp.  A lane's second chunk is the next lane's first, so it is read through L1: DRAM sees
// each byte once.
//
// Decomposition.  CTA (l, p), p < P, owns q or q + 1 contiguous rows of batch l (M = P q + r; the
// first r CTAs take q + 1).  The CTA stages its vector b[l] in shared memory (one f16x2 word per
// packed byte, chunk-swizzled; fp32 block scales; both zero-padded to a whole 32-element step).
// Warp w takes the row groups (4 rows) w, w + W, ... and walks K in 1024-element steps: lane t
// takes the 32 elements at 1024 s + 32 t of each of the 4 rows, exactly the item of the TMA kernels
// (exact f16x2 block partials, mixed-precision scaling, fp32 accumulation).  A lane whose 32
// elements straddle K (K % 32 == 16) zeroes its second block's scale byte.  Every load stays inside
// the caller's buffers: a chunk that would begin before the first or end past the last byte of A
// (or of the batch's vector) is assembled from byte loads instead.  All loads of a step are issued
// before the first use, so the four rows' DRAM round trips overlap.
//
// Measured on GB300 (7168 x 16384, every operand 1 byte off): 27.9 us per call against 35.1 us for
// the byte-load kernel.  It is latency-bound: a warp owns whole rows, so the 7168 rows keep at
// most ~12 warps per SM busy with one step each in flight.  Taking the next lane's chunk by shuffle
// and pipelining two steps measured slower (36.7 us), and three CTAs per SM spilled registers.
#pragma once

#include <stdint.h>

#include "gemv_kernels.cuh"
#include "gemv_tma.cuh"
#include "nvfp4_device.cuh"

namespace nvfp4 {

struct ShiftArgs {
  const uint8_t* A;
  const uint8_t* sfa;
  const uint8_t* b;
  const uint8_t* sfb;
  uint16_t* c;
  float g_a, g_b;
  int64_t M, K, L;
  int64_t a_bytes;   // readable bytes of A from A (every matrix), for the end-of-buffer guard
  int32_t P;         // CTAs per batch
  int32_t rows_q, rows_r;  // M = P rows_q + rows_r: the first rows_r CTAs of a batch take one more
  Groups G;
  int32_t out_bf16;
};

// Shared memory of a CTA for K: the vector words and fp32 block scales, K rounded up to 32.
__host__ __device__ constexpr int64_t shift_smem_bytes(int64_t K) {
  return ((K + 31) / 32) * 32 * 2 + ((K + 31) / 32) * 2 * 4;
}

__global__ void __launch_bounds__(256, 2) gemv_shift_kernel(const ShiftArgs p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int64_t K = p.K, K2 = p.K >> 1, K16 = p.K >> 4;
  const int64_t Kp = ((K + 31) / 32) * 32;  // K padded to whole 32-element lane slices
  uint32_t* bq = reinterpret_cast<uint32_t*>(smem);             // Kp/2 words, chunk-swizzled
  float* sbf = reinterpret_cast<float*>(smem + Kp * 2);         // Kp/16 block scales
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, W = blockDim.x >> 5;
  // the batch and the CTA's rows in 32-bit arithmetic, as in the TMA kernels
  const uint32_t P32 = (uint32_t)p.P, l32 = blockIdx.x / P32, pi32 = blockIdx.x - l32 * P32;
  const uint32_t q = (uint32_t)p.rows_q, r = (uint32_t)p.rows_r;
  const int64_t l = l32;
  const int64_t m0 = (int64_t)pi32 * q + (pi32 < r ? pi32 : r);
  const int64_t n = q + (pi32 < r ? 1u : 0u);

  pdl_launch_dependents();
  pdl_wait();
  int64_t a_first = p.G.shared_a ? m0 : l * p.M + m0;  // first row of A this CTA reads
  float ga = p.g_a, gb = p.g_b;
  if (p.G.E > 0) {
    const int e = group_of_batch(p.G, l, lane);
    if (e < 0) {  // a token without an expert: zero outputs (every warp agrees on e)
      for (int64_t t = threadIdx.x; t < n; t += blockDim.x) p.c[l * p.M + m0 + t] = 0;
      return;
    }
    a_first = (int64_t)e * p.M + m0;
    ga = __ldcg(p.G.g_a + e);
    gb = __ldcg(p.G.g_b + e);
  }

  // stage b[l] as f16x2 words and sfb[l] as fp32, 16 bytes per load through L2 (shifted into place
  // as for A; bytes past the batch's vector are zero)
  const uint8_t* b_l = p.b + l * K2;
  const uint32_t db = (uint32_t)((uintptr_t)b_l & 15u);
  for (int64_t i = threadIdx.x; i < Kp / 32; i += blockDim.x) {
    const uint4 v = ld16_shifted<true>(b_l + 16 * i, db, b_l, b_l + K2);
    uint4 w0, w1, w2, w3;
    e2m1x8_to_f16x2x4(v.x, w0.x, w0.y, w0.z, w0.w);
    e2m1x8_to_f16x2x4(v.y, w1.x, w1.y, w1.z, w1.w);
    e2m1x8_to_f16x2x4(v.z, w2.x, w2.y, w2.z, w2.w);
    e2m1x8_to_f16x2x4(v.w, w3.x, w3.y, w3.z, w3.w);
    uint4* dst = reinterpret_cast<uint4*>(bq);
    const uint32_t q = (uint32_t)(4 * i);
    dst[swz_chunk(q + 0)] = w0;
    dst[swz_chunk(q + 1)] = w1;
    dst[swz_chunk(q + 2)] = w2;
    dst[swz_chunk(q + 3)] = w3;
  }
  const uint8_t* sfb_l = p.sfb + l * K16;
  const uint32_t dsb = (uint32_t)((uintptr_t)sfb_l & 15u);
  for (int64_t i = threadIdx.x; i < (Kp / 16 + 15) / 16; i += blockDim.x) {
    const uint4 v = ld16_shifted<true>(sfb_l + 16 * i, dsb, sfb_l, sfb_l + K16);
    const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int64_t blk = 16 * i + j;
      if (blk < Kp / 16)
        sbf[blk] = f16x2_to_f32x2(e4m3x2_to_f16x2((uint16_t)((wv[j >> 2] >> (8 * (j & 3))) & 0xFFu))).x;
    }
  }
  __syncthreads();

  const uint8_t* A_end = p.A + p.a_bytes;
  const uint32_t bq32 = smem_addr(bq), sb32 = smem_addr(sbf);
  const uint32_t x = ((uint32_t)lane >> 1) & 3u;
  const uint32_t bsw[4] = {16u * (0u ^ x), 16u * (1u ^ x), 16u * (2u ^ x), 16u * (3u ^ x)};
  const int64_t nsteps = (K + kStep - 1) / kStep;
  const int64_t rgs = (n + 3) >> 2;
  for (int64_t rg = warp; rg < rgs; rg += W) {
    const uint8_t* arow[4];
    const uint8_t* srow[4];
    uint32_t d[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int64_t r = min(4 * rg + i, n - 1);  // re-read the last row
      arow[i] = p.A + (a_first + r) * K2;
      srow[i] = p.sfa + (a_first + r) * K16;
      d[i] = (uint32_t)((uintptr_t)arow[i] & 15u);
    }
    float2 acc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
    for (int64_t s = 0; s < nsteps; ++s) {
      const int64_t k = s * kStep + 32 * lane;  // this lane's first element
      if (k < K) {
        const bool second = k + 16 < K;          // the lane's second block lies inside K
        // every load of the step is issued before the first use, so the four rows' DRAM round
        // trips overlap
        uint4 lo[4], hi[4];
        bool fast[4];
        uint32_t s0[4], s1[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint8_t* a = arow[i] + (k >> 1) - d[i];
          fast[i] = a >= p.A && a + 32 <= A_end;
          lo[i] = hi[i] = make_uint4(0u, 0u, 0u, 0u);
          if (fast[i]) {
            lo[i] = ld_l1_v4(a);
            if (d[i]) hi[i] = ld_l1_v4(a + 16);  // mostly the next lane's chunk: an L1 hit
          }
          const uint8_t* sp = srow[i] + (k >> 4);
          s0[i] = __ldg(sp);
          s1[i] = second ? (uint32_t)__ldg(sp + 1) : 0u;
        }
        uint4 av[4];
        uint16_t sv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          av[i] = fast[i] ? (d[i] ? shift16(lo[i], hi[i], d[i]) : lo[i])
                          : ld16_bytes(arow[i] + (k >> 1), p.A, A_end);
          sv[i] = (uint16_t)(s0[i] | (s1[i] << 8));
        }
        const uint32_t so = (uint32_t)s;
        const uint32_t bb = bq32 + so * 2048u + 64u * lane;
        uint32_t bw[16];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 t = lds_v4(bb + bsw[j]);
          bw[4 * j] = t.x;
          bw[4 * j + 1] = t.y;
          bw[4 * j + 2] = t.z;
          bw[4 * j + 3] = t.w;
        }
        const float2 sb = lds_f2(sb32 + so * 256u + 8u * lane);
        item_compute4(av, sv, bw, sb, acc);
      }
    }
    float r4[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) r4[i] = acc[i].x + acc[i].y;
    const float v = warp_reduce_rows<4>(r4, lane);
    const int64_t row = 4 * rg + (lane >> 3);  // lanes 8j .. 8j+7 hold row j of the group
    if ((lane & 7) == 0 && row < n)
      p.c[l * p.M + m0 + row] = f32_to_out_bits((v * ga) * gb, p.out_bf16 != 0);
  }
}

}  // namespace nvfp4

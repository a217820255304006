// NVFP4 block-scaled batched GEMV kernels for GB300 (sm_103a).
//
//   c[l][m] = fp16(g_a * g_b * sum_k e2m1(A[l][m][k]) e2m1(b[l][k]) e4m3(sfa[l][m][k/16]) e4m3(sfb[l][k/16]))
//
// ("nvFP4 Batch GEMV算子系列(下)", section "NVFP4 Batched GEMV 概念阐述".)  The work is a pure
// stream over A and sfa (8/9 and 1/9 of the bytes); b and sfb are tiny and reused by every row.
//
// Arithmetic shared by both kernels: each 16-element block partial sum is exact (products of two
// E2M1 values are multiples of 0.25 and at most 36 in magnitude), the block scale product
// sfa * sfb is exact in fp32 (at most 8 significant bits), so the only roundings are the fp32
// additions across blocks and the final fp16 conversion.
#pragma once

#include <stdint.h>

#include "nvfp4_device.cuh"

namespace nvfp4 {

constexpr unsigned kFullMask = 0xffffffffu;

// ------------------------------------------------------------------------------------------------
// Grouped (mixture-of-experts) form.  A and sfa hold E expert matrices ([E][M][K/2], [E][M][K/16]);
// batch l is a token (b[l], c[l]) that uses expert e(l) and the global scales g_a[e], g_b[e]
// (cutedsl/bridge.py, "Kernel Launch": per-expert global scales; "compute_expert_offsets": tokens
// sorted by expert, offsets[e] = tokens of experts 0..e).  e(l) comes from the inclusive offsets
// (e(l) = the first e with l < offsets[e], which for non-decreasing offsets is the number of
// offsets <= l) or from a per-token expert index.  A token with no expert (past the last offset,
// or an index outside [0, E)) gets an output row of zeros.  E == 0 is the plain batched form.
// ------------------------------------------------------------------------------------------------
struct Groups {
  const int32_t* offsets;    // [E], or null
  const int32_t* expert_of;  // [L], or null
  const float* g_a;          // [E]
  const float* g_b;          // [E]
  int32_t E;
  int32_t shared_a;          // 1: every batch reads the one matrix A (the batches are N tokens
                             // sharing the weights), with the call's g_a and g_b
};

// Expert of batch l, or -1; called by all 32 lanes of a warp (the counts are a warp reduction).
// Every index read is in range whatever the offsets hold.
__device__ __forceinline__ int group_of_batch(const Groups& G, int64_t l, int lane) {
  if (G.expert_of) {
    const int e = __ldcg(G.expert_of + l);
    return (e >= 0 && e < G.E) ? e : -1;
  }
  int cnt = 0;
  for (int e = lane; e < G.E; e += 32) cnt += (int64_t)__ldcg(G.offsets + e) <= l ? 1 : 0;
  const int e = __reduce_add_sync(0xffffffffu, cnt);
  return e < G.E ? e : -1;
}

// ------------------------------------------------------------------------------------------------
// SIMPLE: one warp per output row (l, m), lane j handles whole 16-element blocks j, j+32, ...
// All arithmetic in fp32, byte loads, so any K % 16 == 0 and any byte alignment works.  Used when
// the streaming kernel's shape or alignment conditions do not hold, and as a cross-check.
// ------------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) gemv_simple_kernel(
    const uint8_t* __restrict__ A, const uint8_t* __restrict__ sfa,
    const uint8_t* __restrict__ b, const uint8_t* __restrict__ sfb, float g_a, float g_b,
    uint16_t* __restrict__ c, int64_t M, int64_t K, int64_t L, const Groups G, int out_bf16) {
  const int lane = threadIdx.x & 31;
  const int64_t warps_per_cta = blockDim.x >> 5;
  const int64_t n_rows = M * L;
  const int64_t K2 = K >> 1, K16 = K >> 4;
  for (int64_t row = blockIdx.x * warps_per_cta + (threadIdx.x >> 5); row < n_rows;
       row += (int64_t)gridDim.x * warps_per_cta) {
    const int64_t l = row / M;
    int64_t a_index = G.shared_a ? row - l * M : row;  // row of A (and of sfa) this row reads
    float ga = g_a, gb = g_b;
    if (G.E > 0) {
      const int e = group_of_batch(G, l, lane);
      if (e < 0) {
        if (lane == 0) c[row] = 0;
        continue;
      }
      a_index = (int64_t)e * M + (row - l * M);
      ga = __ldcg(G.g_a + e);
      gb = __ldcg(G.g_b + e);
    }
    const uint8_t* a_row = A + a_index * K2;
    const uint8_t* sa_row = sfa + a_index * K16;
    const uint8_t* b_l = b + l * K2;
    const uint8_t* sb_l = sfb + l * K16;
    float acc = 0.f;
    for (int64_t j = lane; j < K16; j += 32) {
      float block = 0.f;  // exact: a multiple of 0.25, at most 576 in magnitude
#pragma unroll
      for (int t = 0; t < 8; ++t) {
        const float2 av = f16x2_to_f32x2(e2m1x2_to_f16x2(a_row[8 * j + t]));
        const float2 bv = f16x2_to_f32x2(e2m1x2_to_f16x2(b_l[8 * j + t]));
        block = fmaf(av.x, bv.x, block);
        block = fmaf(av.y, bv.y, block);
      }
      const uint16_t pair = (uint16_t)sa_row[j] | ((uint16_t)sb_l[j] << 8);
      const float2 s = f16x2_to_f32x2(e4m3x2_to_f16x2(pair));
      acc = fmaf(block, s.x * s.y, acc);
    }
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) acc += __shfl_xor_sync(kFullMask, acc, w);
    if (lane == 0) c[row] = f32_to_out_bits((acc * ga) * gb, out_bf16 != 0);
  }
}

// ------------------------------------------------------------------------------------------------
// STREAM: the bandwidth kernel.
//
// Decomposition.  CTA (l, p), p < P, owns q or q + 1 contiguous rows of batch l, M = P q + r, the
// first r CTAs taking q + 1 (so P * L CTAs, sized by the host to one wave: a multiple of the SM
// count).  It first decodes b[l] into shared memory as one f16x2 word per packed byte and sfb[l] as
// fp32.  Its rows are cut into groups of R rows and K into S slices of whole 1024-element steps;
// each (group, slice) is a unit, and warp w takes units w, w + W, ...  Within a unit, lane t of a
// step reads 16 bytes (32 elements, two scale blocks) of each of its R rows at k = k0 + 32 t: one
// warp-wide request covers 512 contiguous bytes of a row.  The step after next is loaded before the
// current one is computed (across unit boundaries too), so each warp keeps up to 2 * R 16-byte
// loads per lane in flight.
//
// Per row and step the lane decodes 16 bytes with cvt.rn.f16x2.e2m1x2, multiplies them by the
// staged vector words with packed f16 FMAs (two chains of 8, one per block: each half-lane sum is
// at most 8 * 36 = 288 in quarter units, so exact in f16), multiplies each half sum by the f16
// block scale sfa with mixed-precision FMAs (f16 operands, exact f32 result) and adds the block
// term times sfb into the row's pair of fp32 accumulators (one per block position, one packed
// fp32x2 FMA for both), which the unit's end adds.  At the end of a unit the R row sums
// are reduced across the warp (a transposing butterfly: R - 1 exchange shuffles, then
// 5 - log2(R) plain ones) and stored to a shared array partial[slice][row].  After the CTA
// barrier, thread t sums partial[0..S)[t] in slice order (deterministic), applies g_a and g_b in
// fp32 and stores fp16.  The output stores are coalesced.
//
// Shared-memory vector layout.  A lane reads its 16 vector words for a step as four 16-byte
// chunks; chunk q of the decoded vector (words 4q .. 4q+3) is stored at chunk q ^ ((q >> 3) & 3),
// which puts the eight lanes of each 128-byte shared-memory wavefront on eight different bank
// groups (without it, lanes 2 apart collide: a 4-way conflict).
// ------------------------------------------------------------------------------------------------
struct StreamArgs {
  const uint8_t* A;
  const uint8_t* sfa;
  const uint8_t* b;
  const uint8_t* sfb;
  uint16_t* c;
  float g_a, g_b;
  int64_t M, K, L;
  int32_t P;            // CTAs per batch
  int32_t S;            // K slices per row
  int32_t slice_steps;  // 1024-element steps per slice (the last slice may be shorter)
  int32_t rows_cap;     // ceil(M / P): row capacity of the shared partial array
  int32_t rows_q, rows_r;  // M = P rows_q + rows_r: the first rows_r CTAs of a batch take one more
  Groups G;             // grouped form (G.E > 0)
  int32_t out_bf16;     // 1: bfloat16 output instead of fp16
};

constexpr int kStep = 1024;  // elements one warp covers per step (32 lanes x 32)

__device__ __forceinline__ uint32_t swz_chunk(uint32_t q) { return q ^ ((q >> 3) & 3u); }

template <int R>
__device__ __forceinline__ float warp_reduce_rows(float (&v)[R], int lane) {
  // exchange phase: halve the set of row values each lane carries, pairing lanes `width` apart
#pragma unroll
  for (int cnt = R, width = 16; cnt > 1; cnt >>= 1, width >>= 1) {
    const bool upper = (lane & width) != 0;
#pragma unroll
    for (int i = 0; i < cnt / 2; ++i) {
      const float keep = upper ? v[i + cnt / 2] : v[i];
      const float send = upper ? v[i] : v[i + cnt / 2];
      v[i] = keep + __shfl_xor_sync(kFullMask, send, width);
    }
  }
  // plain butterfly inside each group of 32 / R lanes; lane t then holds row t / (32 / R)
#pragma unroll
  for (int width = 16 / R; width >= 1; width >>= 1) v[0] += __shfl_xor_sync(kFullMask, v[0], width);
  return v[0];
}

// Loads one step of a unit: 16 bytes of A and 2 scale bytes for each of the R rows at element k.
// Rows past the CTA's last row re-read that row (their sums are discarded); lanes at or past the
// slice end load nothing.
template <int R>
__device__ __forceinline__ void stream_load(const uint8_t* __restrict__ A_c,
                                            const uint8_t* __restrict__ sfa_c, int64_t K2,
                                            int64_t K16, int row0, int n, int64_t k, int64_t k_end,
                                            uint4 (&av)[R], uint16_t (&sv)[R]) {
  if (k >= k_end) return;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int64_t r = min(row0 + i, n - 1);
    av[i] = ld_stream_v4(A_c + r * K2 + (k >> 1));
    sv[i] = ld_stream_u16(sfa_c + r * K16 + (k >> 4));
  }
}

template <int R>
__device__ __forceinline__ void stream_compute(const uint32_t* __restrict__ bq,
                                               const float* __restrict__ sbf, int64_t k,
                                               const uint4 (&av)[R], const uint16_t (&sv)[R],
                                               float2 (&acc)[R]) {
  // vector words for bytes k/2 .. k/2 + 15 (chunks q .. q+3, swizzled) and the two block scales
  const uint32_t q = (uint32_t)(k >> 3);
  uint4 bw[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) bw[j] = reinterpret_cast<const uint4*>(bq)[swz_chunk(q + j)];
  const float2 sb = *reinterpret_cast<const float2*>(sbf + (k >> 4));
#pragma unroll
  for (int i = 0; i < R; ++i) {
    uint32_t h[16];
    e2m1x8_to_f16x2x4(av[i].x, h[0], h[1], h[2], h[3]);
    e2m1x8_to_f16x2x4(av[i].y, h[4], h[5], h[6], h[7]);
    e2m1x8_to_f16x2x4(av[i].z, h[8], h[9], h[10], h[11]);
    e2m1x8_to_f16x2x4(av[i].w, h[12], h[13], h[14], h[15]);
    uint32_t p0 = 0u, p1 = 0u;  // f16x2 zeros
    hfma2(p0, h[0], bw[0].x);
    hfma2(p0, h[1], bw[0].y);
    hfma2(p0, h[2], bw[0].z);
    hfma2(p0, h[3], bw[0].w);
    hfma2(p0, h[4], bw[1].x);
    hfma2(p0, h[5], bw[1].y);
    hfma2(p0, h[6], bw[1].z);
    hfma2(p0, h[7], bw[1].w);
    hfma2(p1, h[8], bw[2].x);
    hfma2(p1, h[9], bw[2].y);
    hfma2(p1, h[10], bw[2].z);
    hfma2(p1, h[11], bw[2].w);
    hfma2(p1, h[12], bw[3].x);
    hfma2(p1, h[13], bw[3].y);
    hfma2(p1, h[14], bw[3].z);
    hfma2(p1, h[15], bw[3].w);
    ffma2(acc[i], scaled_block_pair(p0, p1, e4m3x2_to_f16x2(sv[i])), sb);
  }
}

template <int R>
__global__ void __launch_bounds__(512) gemv_stream_kernel(const StreamArgs p) {
  extern __shared__ __align__(16) uint8_t smem[];
  const int64_t K = p.K, K2 = p.K >> 1, K16 = p.K >> 4;
  uint32_t* bq = reinterpret_cast<uint32_t*>(smem);                   // K/2 words (swizzled)
  float* sbf = reinterpret_cast<float*>(smem + 4 * K2);                // K/16 floats
  float* part = reinterpret_cast<float*>(smem + 4 * K2 + 4 * K16);     // S x rows_cap floats

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, W = blockDim.x >> 5;
  // the batch and the CTA's rows in 32-bit arithmetic, as in the TMA kernels
  const uint32_t P32 = (uint32_t)p.P, l32 = blockIdx.x / P32, pi32 = blockIdx.x - l32 * P32;
  const uint32_t q = (uint32_t)p.rows_q, r = (uint32_t)p.rows_r;
  const int64_t l = l32;
  const int64_t m0 = (int64_t)pi32 * q + (pi32 < r ? pi32 : r);
  const int n = (int)(q + (pi32 < r ? 1u : 0u));
  int64_t ea = p.G.shared_a ? 0 : l;  // which matrix of A this CTA reads
  float ga = p.g_a, gb = p.g_b;
  if (p.G.E > 0) {  // grouped: every warp finds the same expert (the offsets do not change)
    const int e = group_of_batch(p.G, l, lane);
    if (e < 0) {
      for (int t = tid; t < n; t += blockDim.x) p.c[l * p.M + m0 + t] = 0;
      return;
    }
    ea = e;
    ga = __ldcg(p.G.g_a + e);
    gb = __ldcg(p.G.g_b + e);
  }
  const uint8_t* A_c = p.A + (ea * p.M + m0) * K2;
  const uint8_t* sfa_c = p.sfa + (ea * p.M + m0) * K16;
  const int G = (n + R - 1) / R;
  const int U = G * p.S;
  const int64_t slice_elems = (int64_t)p.slice_steps * kStep;

  // A warp walks the positions (unit u, step j) of its units u = warp, warp + W, ... in order.
  // Positions and unit geometry are warp-uniform, so the walk never diverges; only the lanes past
  // a slice's end sit out its last step.  The data of the next position is loaded before the
  // current one is computed, across unit boundaries too.
  auto unit_geometry = [&](int unit, int& g_, int64_t& kb_, int64_t& ke_, int& nsteps_) {
    g_ = unit / p.S;
    kb_ = (int64_t)(unit - g_ * p.S) * slice_elems;
    ke_ = min(K, kb_ + slice_elems);
    nsteps_ = (int)((ke_ - kb_ + kStep - 1) / kStep);
  };
  int u = warp, j = 0;
  int g = 0, nsteps = 0;
  int64_t kb = 0, ke = 0;
  uint4 av[R];
  uint16_t sv[R];
  if (u < U) {
    unit_geometry(u, g, kb, ke, nsteps);
    stream_load<R>(A_c, sfa_c, K2, K16, g * R, n, kb + 32 * lane, ke, av, sv);
  }

  // Stage the vector while those loads are in flight: 16 packed bytes -> 16 f16x2 words, stored
  // as four swizzled chunks; the block scales as fp32.
  const uint8_t* b_l = p.b + l * K2;
  for (int64_t i = tid; i < K2 / 16; i += blockDim.x) {
    const uint4 v = ld_l2_v4(b_l + 16 * i);
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
  for (int64_t i = tid; i < K16 / 2; i += blockDim.x) {
    const float2 sc = f16x2_to_f32x2(e4m3x2_to_f16x2(ld_l2_u16(sfb_l + 2 * i)));
    sbf[2 * i] = sc.x;
    sbf[2 * i + 1] = sc.y;
  }
  __syncthreads();

  float2 acc[R];  // per row: running sums of the lane's first and second blocks of a step
#pragma unroll
  for (int i = 0; i < R; ++i) acc[i] = make_float2(0.f, 0.f);
  while (u < U) {
    // the next position and, when it starts a new unit, that unit's geometry
    int un = u, jn = j + 1, gn = g, nsn = nsteps;
    int64_t kbn = kb, ken = ke;
    if (jn >= nsteps) {
      un = u + W;
      jn = 0;
      if (un < U) unit_geometry(un, gn, kbn, ken, nsn);
    }
    uint4 an[R];
    uint16_t sn[R];
    if (un < U)
      stream_load<R>(A_c, sfa_c, K2, K16, gn * R, n, kbn + (int64_t)jn * kStep + 32 * lane, ken,
                     an, sn);
    const int64_t k = kb + (int64_t)j * kStep + 32 * lane;
    if (k < ke) stream_compute<R>(bq, sbf, k, av, sv, acc);
    if (un != u) {
      float r[R];
#pragma unroll
      for (int i = 0; i < R; ++i) r[i] = acc[i].x + acc[i].y;
      const float row_sum = warp_reduce_rows<R>(r, lane);
      const int s = u - g * p.S;
      const int jr = lane / (32 / R);
      if ((lane & (32 / R - 1)) == 0 && g * R + jr < n) part[s * p.rows_cap + g * R + jr] = row_sum;
#pragma unroll
      for (int i = 0; i < R; ++i) acc[i] = make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int i = 0; i < R; ++i) {
      av[i] = an[i];
      sv[i] = sn[i];
    }
    u = un;
    j = jn;
    g = gn;
    kb = kbn;
    ke = ken;
    nsteps = nsn;
  }
  __syncthreads();

  uint16_t* c_c = p.c + l * p.M + m0;
  for (int t = tid; t < n; t += blockDim.x) {
    float v = part[t];
    for (int s = 1; s < p.S; ++s) v += part[s * p.rows_cap + t];
    c_c[t] = f32_to_out_bits((v * ga) * gb, p.out_bf16 != 0);
  }
}

}  // namespace nvfp4

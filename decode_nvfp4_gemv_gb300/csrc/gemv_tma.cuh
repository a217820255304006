// TMA-ring NVFP4 GEMV kernels for GB300 (sm_103a): the bandwidth path for K % 256 == 0.
//
// Why: the work is a read-once stream of A (8/9 of the bytes) and sfa (1/9).  Holding enough bytes
// in flight to cover HBM latency with per-thread loads costs registers and occupancy; the Tensor
// Memory Accelerator's bulk copies move whole row tiles into shared memory with one instruction
// each and need no registers to keep them in flight.  (Measured on GB300: many small bulk copies
// are slow, so tiles are whole rows and one copy each.)
//
// Decomposition.  CTA (l, p), p < P, owns q or q + 1 contiguous rows of batch l (M = P q + r; the
// first r CTAs take q + 1), starting at row p q + min(p, r).
// Because rows are contiguous in memory, the CTA's A bytes (and its sfa bytes) form one
// contiguous run, cut into tiles of TR whole rows.  Warp W_c (the last) is the producer: one lane
// walks the tiles and, for each, waits until ring stage s = T mod NS is free, then issues two
// cp.async.bulk copies (the tile's A rows and sfa rows) that complete the stage's `full` mbarrier
// by transaction count.  Warps 0 .. W_c-1 consume: for each tile they wait on `full`, process
// their items and release the stage by arriving on its `empty` mbarrier (one arrival per warp).
//
// Items.  A tile is cut into groups of 4 rows x 1024-element segments.  For an item, lane t takes
// 16 bytes (32 elements, two scale blocks) of each of the 4 rows at k = 1024 * seg + 32 t,
// multiplies them with the vector's f16x2 words by packed f16 FMAs (exact block partials), scales
// each block partial by sfa (mixed-precision FMAs, exact) and by sfb (one packed fp32x2 FMA into
// the row's two accumulators) and accumulates per row.  A warp reduces its 4 row sums
// across lanes and writes them to partial[row][slot] in shared memory; after the last tile,
// thread t sums partial[t][0 .. slots) in slot order (deterministic), applies g_a and g_b in fp32
// and stores fp16.
//
// Two variants differ in where the vector lives:
//   gemv_tma_kernel        b[l] decoded into shared memory (one f16x2 word per packed byte,
//                          swizzled as in the stream kernel) and sfb[l] as fp32; item i goes to
//                          warp i mod W_c.  Any K % 256 == 0 within the shared-memory budget.
//   gemv_tma_rv_kernel<NSW> when W_c NSW >= nseg > W_c (NSW = 1 or 2 segments per warp, for every
//                          row group; a warp's segments are warp + j W_c, and one that starts past
//                          K is idle) or nseg divides W_c (each warp owns one segment and every
//                          (W_c/nseg)-th row group): a warp touches the same segments in every
//                          tile, so it decodes its slice of b into registers once.  No vector reads
//                          in the inner loop, and the ring gets the shared memory.
//
// Split K over a cluster (register-vector kernel, `CL`).  When the rows of a call are too few to
// give every CTA slot of one wave enough work, K is cut into S slices of whole 1024-element
// segments and a thread-block cluster of S CTAs shares each row range: cluster CTA z streams
// slice z of its rows (one bulk copy per row and operand, since a slice of consecutive rows is not
// contiguous), holds slice z of the vector in registers and sums its rows' partials over its own
// warps as above.  Each row is owned by one CTA of the cluster (rows [o n / S, (o+1) n / S) by
// CTA o); every CTA stores its partial of a row into the owner's shared memory (distributed shared
// memory), and after one cluster barrier the owner adds the S partials in slice order and stores
// the row.  Deterministic, and no global workspace: the second pass of the reduction never leaves
// the cluster.
//
// Programmatic dependent launch.  The host launches with programmatic stream serialization, so the
// next kernel in the stream may be scheduled while this one drains.  Every thread executes
// griddepcontrol.wait before its first access to memory a preceding kernel may write; with the
// `early_weights` flag (the caller guarantees that no kernel still running writes A or sfa) the
// producer requests the first NS - 1 tiles of A and sfa before that wait (all but the tail of the
// last of them), and only the vector, its scales, the outputs and the rest of the ring wait.  griddepcontrol.wait returns at once for a
// launch without the attribute.
//
// Bounded waits.  Every mbarrier wait gives up after one second of wall time (%globaltimer).  A
// consumer that gives up sets a shared abort flag; a producer that gives up waits (again bounded)
// for the copies it already issued before its warp exits, so no copy outlives the CTA.  An aborted
// CTA writes fp16 NaN to all of its outputs, which is how the host sees the failure.
#pragma once

#include <stdint.h>

#include "gemv_kernels.cuh"
#include "nvfp4_device.cuh"
#include "quantize.cuh"

namespace nvfp4 {

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // one second
constexpr int kTmaMaxStages = 8;
constexpr int kTmaMaxClusterK = 8;                // K slices (cluster CTAs) of a split-K launch
constexpr uint32_t kTmaHeaderBytes = 256;         // barriers (16 B per stage) + abort flag

struct TmaArgs {
  const uint8_t* A;
  const uint8_t* sfa;
  const uint8_t* b;
  const uint8_t* sfb;
  uint16_t* c;
  float g_a, g_b;
  int64_t M, K, L;
  int32_t P;             // CTAs per batch
  int32_t tile_rows;     // TR: rows per ring stage
  int32_t stages;        // NS <= kTmaMaxStages
  int32_t rows_cap;      // ceil(M / P)
  int32_t rows_q, rows_r; // M = P rows_q + rows_r: the first rows_r CTAs of a batch take one row more
  int32_t slots;         // partial sums per row (consumer warps, or segments for the rv kernel)
  int32_t early_weights; // 1: stream A and sfa before the programmatic-launch wait
  uint32_t stage_bytes;  // bytes per ring stage (A rows, then sfa rows at sfa_off)
  uint32_t sfa_off;      // offset of the sfa rows inside a stage (16-byte aligned)
  uint32_t b_off, sb_off, part_off, ring_off;  // shared-memory layout (bytes); b/sb unused by rv
  // fused activation quantization (rv kernel with QX): the vector arrives as bf16 x [L][K] with
  // global scale x_gs and is quantized in the staging step; the first CTA of each batch writes the
  // packed bytes and scale bytes to b_out / sfb_out ([L][K/2], [L][K/16])
  const uint16_t* x;
  float x_gs;
  int32_t rounding;
  uint8_t* b_out;
  uint8_t* sfb_out;
  Groups G;              // grouped form (G.E > 0; never with early_weights: e(l) is read after
                         // the programmatic-launch wait)
  int32_t out_bf16;      // 1: bfloat16 output instead of fp16
  // operands not 16-byte aligned: the 16-byte aligned interiors [lo, hi) of the A and sfa buffers,
  // and the ends of the b and sfb buffers (unused when aligned)
  const uint8_t *A_lo, *A_hi, *S_lo, *S_hi, *b_end, *sfb_end;
  int32_t test_stall;    // tests of the failure path: the producer issues nothing
  // split K over a cluster (CL): S slices of slice_segs 1024-element segments each (the last
  // slice may end short of that at K); a stage holds a tile's rows rs_a (A) and rs_s (sfa) bytes
  // apart (K/2 and K/16 when unsplit); red_off: the owner's S x red_rows partial sums
  int32_t k_slices;
  int32_t slice_segs;
  uint32_t rs_a, rs_s;
  uint32_t red_off;
  int32_t red_rows;
  // rows [pf_row0, pf_row0 + pf_rows) of the CTA's rows are prefetched into L2 before the launch
  // wait (pf_rows = 0: none); the host sets the first ring fill in strict stream order
  int32_t pf_row0, pf_rows;
};

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a));
  return v;
}
__device__ __forceinline__ uint32_t lds_u8(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ uint16_t lds_u16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
  return v;
}
__device__ __forceinline__ float2 lds_f2(uint32_t a) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
  return v;
}

// ------------------------------------------------------------------------------------------------
// Reading 16 bytes at any alignment (the operands' rows need not start on 16-byte boundaries).
// ------------------------------------------------------------------------------------------------
// 16-byte read-only load kept in L1, for data a neighbouring lane reads again.
__device__ __forceinline__ uint4 ld_l1_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// The 16 bytes that start d bytes into the 32 bytes lo:hi (d < 16, the same for the whole warp).
__device__ __forceinline__ uint4 shift16(const uint4& lo, const uint4& hi, uint32_t d) {
  const uint32_t v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  const uint32_t r = 8u * (d & 3u);
  uint32_t o[4];
  switch (d >> 2) {  // the word part of the shift: warp-uniform, so no divergence
#define NVFP4_SHIFT_CASE(Q)                               \
    case Q:                                               \
      _Pragma("unroll") for (int i = 0; i < 4; ++i)       \
        o[i] = __funnelshift_r(v[i + Q], v[i + Q + 1], r); \
      break;
    NVFP4_SHIFT_CASE(0)
    NVFP4_SHIFT_CASE(1)
    NVFP4_SHIFT_CASE(2)
    default:
      NVFP4_SHIFT_CASE(3)
#undef NVFP4_SHIFT_CASE
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// The 16 bytes at p read one by one, those outside [start, end) taken as zero (the first and the
// last chunk of a buffer).  All sixteen loads are issued before the first is used, so the bytes
// cost one memory round trip, not sixteen.  L2 = true reads through L2 only (.cg).
template <bool L2 = false>
__device__ __forceinline__ uint4 ld16_bytes(const uint8_t* p, const uint8_t* start,
                                            const uint8_t* end) {
  uint32_t v[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const uint8_t* q = p + j;
    v[j] = (q >= start && q < end) ? (uint32_t)(L2 ? __ldcg(q) : *q) : 0u;
  }
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = v[4 * i] | (v[4 * i + 1] << 8) | (v[4 * i + 2] << 16) | (v[4 * i + 3] << 24);
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// The 16 bytes at p (any alignment); d = p mod 16, the same for every lane of the warp.  Only
// bytes in [start, end) are read: when the two aligned chunks around p do not both lie inside it,
// the bytes are loaded one by one and those outside are zero.  L2 = true reads through L2 only
// (.cg), as every load of the vector must (a preceding grid may have written it).
template <bool L2 = false>
__device__ __forceinline__ uint4 ld16_shifted(const uint8_t* p, uint32_t d, const uint8_t* start,
                                              const uint8_t* end) {
  const uint8_t* a = p - d;
  if (a >= start && a + (d ? 32 : 16) <= end) {  // one aligned chunk when p is aligned
    const uint4 lo = L2 ? ld_l2_v4(a) : ld_l1_v4(a);
    if (d == 0) return lo;
    return shift16(lo, L2 ? ld_l2_v4(a + 16) : ld_l1_v4(a + 16), d);
  }
  return ld16_bytes<L2>(p, start, end);
}

// One row times one 32-element lane slice: decode, exact block partials, scale.  bw: the 16
// vector words for this lane's 32 elements; sb: the two vector block scales.  acc holds the row's
// running sums of the lane's first and second blocks (added at the flush).
__device__ __forceinline__ void row_compute(const uint4& av, uint16_t sv, const uint32_t (&bw)[16],
                                            float2 sb, float2& acc) {
  uint32_t h[16];
  e2m1x8_to_f16x2x4(av.x, h[0], h[1], h[2], h[3]);
  e2m1x8_to_f16x2x4(av.y, h[4], h[5], h[6], h[7]);
  e2m1x8_to_f16x2x4(av.z, h[8], h[9], h[10], h[11]);
  e2m1x8_to_f16x2x4(av.w, h[12], h[13], h[14], h[15]);
  uint32_t p0 = 0u, p1 = 0u;  // f16x2 zeros
#pragma unroll
  for (int q = 0; q < 8; ++q) hfma2(p0, h[q], bw[q]);
#pragma unroll
  for (int q = 8; q < 16; ++q) hfma2(p1, h[q], bw[q]);
  ffma2(acc, scaled_block_pair(p0, p1, e4m3x2_to_f16x2(sv)), sb);
}

// One row group (4 rows) times one 32-element lane slice.
__device__ __forceinline__ void item_compute4(const uint4 (&av)[4], const uint16_t (&sv)[4],
                                              const uint32_t (&bw)[16], float2 sb,
                                              float2 (&acc)[4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i) row_compute(av[i], sv[i], bw, sb, acc[i]);
}

// Reduces the 4 row sums of a group across the warp and stores them to partial[row][slot].
__device__ __forceinline__ void tma_flush(float2 (&acc)[4], int lane, int row0, int rows_t,
                                          float* part_tile, int slots, int slot) {
  float r[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) r[i] = acc[i].x + acc[i].y;
  const float v = warp_reduce_rows<4>(r, lane);
  const int j = lane >> 3;  // lanes 8j .. 8j+7 hold row j of the group
  if ((lane & 7) == 0 && row0 + j < rows_t) part_tile[(row0 + j) * slots + slot] = v;
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = make_float2(0.f, 0.f);
}

// Shared prologue: CTA geometry, barrier initialisation, dependent-launch trigger.
struct TmaCta {
  int64_t l, pi, m0;
  int n, NT, Wc;
  int64_t ea;     // the matrix of A this CTA streams: l, or the expert of token l
  float ga, gb;   // global scales
  bool skip;      // grouped form: token l has no expert, its outputs are zeros
  int z;          // split K: this CTA's slice (its rank in the cluster); 0 unsplit
  int64_t k0;     // first element of the slice
  int kz;         // elements in the slice (K unsplit)
};

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}

__device__ __forceinline__ TmaCta tma_setup(const TmaArgs& p, uint64_t* bars,
                                            volatile int* abort_flag) {
  TmaCta g;
  // The batch and the CTA's rows, in 32-bit arithmetic and without a 64-bit division: this runs
  // before the CTA's first copy.  Measured on GB300 against floor(M pi / P) in 64-bit arithmetic:
  // c2 11.58 -> 11.42 us, c3 -0.6%, c4 and c5 unchanged (32-bit floor(M pi / P) alone: 11.50 us).
  // split K: a cluster of S CTAs shares one row range, CTA z taking slice z (a launch without
  // clusters is one-CTA clusters: rank 0, cluster index = CTA index)
  const uint32_t bid = p.k_slices > 1 ? cluster_id_x() : blockIdx.x, P = (uint32_t)p.P;
  const uint32_t l = bid / P, pi = bid - l * P;
  g.z = p.k_slices > 1 ? (int)cluster_ctarank() : 0;
  g.k0 = (int64_t)g.z * p.slice_segs * kStep;
  g.kz = p.k_slices > 1 ? (int)min(p.K - g.k0, (int64_t)p.slice_segs * kStep) : (int)p.K;
  const uint32_t q = (uint32_t)p.rows_q, r = (uint32_t)p.rows_r;
  g.l = l;
  g.pi = pi;
  g.m0 = (int64_t)pi * q + (pi < r ? pi : r);
  g.n = (int)(q + (pi < r ? 1u : 0u));
  g.NT = (g.n + p.tile_rows - 1) / p.tile_rows;
  g.Wc = (blockDim.x >> 5) - 1;
  g.ea = p.G.shared_a ? 0 : g.l;
  g.ga = p.g_a;
  g.gb = p.g_b;
  g.skip = false;
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(smem_addr(&bars[s]), 1);                          // producer's arrive + bytes
      mbar_init(smem_addr(&bars[p.stages + s]), (uint32_t)g.Wc);  // one arrival per consumer
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();
  pdl_launch_dependents();
  return g;
}

// Grouped form, after the programmatic-launch wait: each warp finds token l's expert itself (all
// warps read the same offsets, so they agree).  A token without an expert gets zero outputs.
__device__ __forceinline__ void tma_resolve_group(const TmaArgs& p, TmaCta& g, int lane) {
  if (p.G.E <= 0) return;
  const int e = group_of_batch(p.G, g.l, lane);
  // one decision for the whole CTA (called by every thread), so no warp can be left waiting at a
  // barrier for warps that skipped, even if the routing changed under a misbehaving writer
  g.skip = __syncthreads_or(e < 0) != 0;
  if (g.skip) {
    for (int t = threadIdx.x; t < g.n; t += blockDim.x) p.c[g.l * p.M + g.m0 + t] = 0;
    return;
  }
  g.ea = e;
}

// Grouped form: the expert's global scales, for the consumer warps only.  The producer streams as
// soon as the expert is known; the consumers' loads are in flight while their first tile arrives
// and are first used by the epilogue.  Measured on GB300 against loading them in every thread
// before the producer started (experts of 3584 x 6144): 16 tokens on 16 experts 34.2 -> 33.5 us,
// the decode workload g1 (16 token rows, 13-15 experts) 31.6 -> 30.9 us.
__device__ __forceinline__ void tma_group_scales(const TmaArgs& p, TmaCta& g) {
  if (p.G.E <= 0) return;
  g.ga = __ldcg(p.G.g_a + g.ea);
  g.gb = __ldcg(p.G.g_b + g.ea);
}

// Ring position of tile T: stage T mod NS and the parity (T / NS) mod 2 of that stage's use,
// advanced one tile at a time (no division in the loops).
struct RingPos {
  int s = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void advance(int stages) {
    if (++s == stages) {
      s = 0;
      phase ^= 1u;
    }
  }
};

// Unaligned operands: a tile's bytes [g0, g1) go to the stage at offset g - floor16(g0).  The part
// of the aligned superset [floor16(g0), ceil16(g1)) that lies inside the 16-byte aligned interior
// [lo, hi) of the operand's buffer, [c0, c1), arrives by one bulk copy; bytes of [g0, g1) outside
// it (only in the buffer's first and last partial chunk, at most 15 bytes each) are stored by the
// producer one by one, so nothing outside the buffer is read.
struct USpan {
  const uint8_t *u0, *c0, *c1;
  uint32_t n;  // bytes of the bulk copy (0: none)
};

__device__ __forceinline__ USpan unaligned_span(const uint8_t* g0, const uint8_t* g1,
                                                const uint8_t* lo, const uint8_t* hi) {
  USpan sp;
  sp.u0 = reinterpret_cast<const uint8_t*>((uintptr_t)g0 & ~(uintptr_t)15);
  const uint8_t* u1 = reinterpret_cast<const uint8_t*>(((uintptr_t)g1 + 15) & ~(uintptr_t)15);
  sp.c0 = sp.u0 > lo ? sp.u0 : lo;
  sp.c1 = u1 < hi ? u1 : hi;
  sp.n = sp.c1 > sp.c0 ? (uint32_t)(sp.c1 - sp.c0) : 0u;
  return sp;
}

// The producer lane prefetches rows [pf_row0, pf_row0 + pf_rows) of the CTA's A and sfa rows
// (contiguous, so one prefetch each; 16-byte aligned operands only) into L2 before the launch wait.  A prefetch is a hint that
// changes no value: every read of A still follows the wait (strict stream order) and sees what
// the preceding work wrote; the copies after the wait then find the bytes in L2.
__device__ __forceinline__ void tma_prefetch_rows(const TmaArgs& p, const TmaCta& g) {
  const int64_t K2 = p.K >> 1, K16 = p.K >> 4;
  const int r0 = min(g.n, p.pf_row0), r1 = min(g.n, p.pf_row0 + p.pf_rows);
  if (r1 <= r0) return;
  const int64_t row = g.ea * p.M + g.m0 + r0;
  bulk_prefetch_l2(p.A + row * K2, (uint32_t)((r1 - r0) * K2));
  bulk_prefetch_l2(p.sfa + row * K16, (uint32_t)((r1 - r0) * K16));
}

__device__ __forceinline__ void stage_unaligned(uint8_t* st, const uint8_t* g0, const uint8_t* g1,
                                                const USpan& sp, uint32_t full, uint64_t pol) {
  if (sp.c0 > g0 || sp.c1 < g1) {  // edge bytes: all loads issued before the stores
    uint32_t head[4] = {0u, 0u, 0u, 0u}, tail[4] = {0u, 0u, 0u, 0u};  // 16 bytes each, packed
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint8_t* x = g0 + j;
      if (x < g1 && x < sp.c0) head[j >> 2] |= (uint32_t)*x << (8 * (j & 3));
      const uint8_t* y = g1 - 16 + j;
      if (y >= g0 && y >= sp.c1) tail[j >> 2] |= (uint32_t)*y << (8 * (j & 3));
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const uint8_t* x = g0 + j;
      if (x < g1 && x < sp.c0) st[x - sp.u0] = (uint8_t)(head[j >> 2] >> (8 * (j & 3)));
      const uint8_t* y = g1 - 16 + j;
      if (y >= g0 && y >= sp.c1) st[y - sp.u0] = (uint8_t)(tail[j >> 2] >> (8 * (j & 3)));
    }
  }
  if (sp.n) bulk_copy_g2s(smem_addr(st + (sp.c0 - sp.u0)), sp.c0, sp.n, full, pol);
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// The producer lane: streams the CTA's row tiles into the ring.  UA: operands not 16-byte aligned
// (stage_unaligned above); the stage then holds each tile's bytes from the 16-byte boundary at or
// below its first byte.  CL: split K, one copy per row of the slice's bytes (A, then sfa).
template <bool UA, bool CL = false>
__device__ __forceinline__ void tma_produce(const TmaArgs& p, const TmaCta& g, uint64_t* bars,
                                            volatile int* abort_flag, uint8_t* ring) {
  const int64_t K2 = p.K >> 1, K16 = p.K >> 4;
  const int NS = p.stages, TR = p.tile_rows;
  const uint64_t pol = l2_evict_first_policy();
  const uint8_t* A_c = p.A + (g.ea * p.M + g.m0) * K2;
  const uint8_t* S_c = p.sfa + (g.ea * p.M + g.m0) * K16;
  int issued = 0;
  bool ok = true;
  if (p.test_stall) return;  // every consumer wait then runs out at its limit
  // Early weights: the producer's first launch wait comes after its early copies; rows to
  // prefetch into L2 (pf_rows) are requested just before it.
  bool waited = false;
  auto launch_wait = [&]() {
    if (!waited && p.pf_rows) tma_prefetch_rows(p, g);
    waited = true;
    pdl_wait();
  };
  RingPos rp;
  for (int T = 0; T < g.NT; ++T, rp.advance(NS)) {
    const int s = rp.s;
    // Early weights: the first NS - 1 tiles are requested before the preceding work has finished,
    // the last tile of the first fill only once it has.  Requested early, that tile's bytes would
    // compete for HBM with the preceding call's last tiles: measured on GB300 against requesting
    // the whole ring early, c2 12.34 -> 11.50 us, c3 -3.6%, c4 -1.2%, c5 -1.3%.
    if (p.early_weights && T == NS - 1) launch_wait();
    // stage s was last filled in the previous round: wait until its consumers released it
    if (T >= NS && !mbar_wait_bounded(smem_addr(&bars[NS + s]), rp.phase ^ 1u, kWaitLimitNs)) {
      ok = false;
      break;
    }
    if (*abort_flag) {
      ok = false;
      break;
    }
    const int rows_t = min(TR, g.n - T * TR);
    const uint32_t bytesA = (uint32_t)(rows_t * K2), bytesS = (uint32_t)(rows_t * K16);
    const uint32_t full = smem_addr(&bars[s]);
    uint8_t* st = ring + (size_t)s * p.stage_bytes;
    if constexpr (CL) {
      // the slice [k0, k0 + kz) of each row: kz / 2 bytes of A at K/2-byte row steps, kz / 16 of
      // sfa at K/16 (every address and size a multiple of 16: K % 256 == 0 and whole segments).
      // Early weights: the last row's A copy of the last tile requested before the wait follows
      // the wait, as the unsplit tail does.
      const uint32_t ra = (uint32_t)(g.kz >> 1), rs = (uint32_t)(g.kz >> 4);
      const uint8_t* ga = A_c + (int64_t)T * TR * K2 + (g.k0 >> 1);
      const uint8_t* gs = S_c + (int64_t)T * TR * K16 + (g.k0 >> 4);
      const bool hold = p.early_weights && T == NS - 2;
      mbar_arrive_expect_tx(full, (uint32_t)rows_t * (ra + rs));
      for (int r = 0; r < rows_t; ++r) {
        bulk_copy_g2s(smem_addr(st + p.sfa_off + r * p.rs_s), gs + (int64_t)r * K16, rs, full, pol);
        if (!(hold && r == rows_t - 1))
          bulk_copy_g2s(smem_addr(st + r * p.rs_a), ga + (int64_t)r * K2, ra, full, pol);
      }
      if (hold) {
        launch_wait();
        bulk_copy_g2s(smem_addr(st + (rows_t - 1) * p.rs_a), ga + (int64_t)(rows_t - 1) * K2, ra,
                      full, pol);
      }
    } else if constexpr (UA) {
      // the copies' bytes are expected first; the arrival comes after the edge stores, so the
      // consumers that see the phase complete see those bytes too
      const uint8_t* ga = A_c + (int64_t)T * TR * K2;
      const uint8_t* gs = S_c + (int64_t)T * TR * K16;
      const USpan sa = unaligned_span(ga, ga + bytesA, p.A_lo, p.A_hi);
      const USpan ss = unaligned_span(gs, gs + bytesS, p.S_lo, p.S_hi);
      mbar_expect_tx(full, sa.n + ss.n);
      stage_unaligned(st, ga, ga + bytesA, sa, full, pol);
      stage_unaligned(st + p.sfa_off, gs, gs + bytesS, ss, full, pol);
      mbar_arrive(full);
    } else {
      // Early weights: the last tile requested before the wait keeps the tail of its A bytes (one
      // row of a tile of more than 4 rows, else 16 bytes) until after the wait, so that tile
      // completes only once the preceding work has.  Measured on GB300 against requesting the
      // whole tile early: c2 -0.5%, c3 -0.5%, c4 7.64 -> 7.34 us, c5 -1%; holding back one row of
      // c2's 4-row tile measured 1% slower than 16 bytes.
      const uint8_t* ga = A_c + (int64_t)T * TR * K2;
      uint32_t hold = 0;
      if (p.early_weights && T == NS - 2) hold = rows_t > 4 ? (uint32_t)K2 : 16u;
      if (hold >= bytesA) hold = 0;
      mbar_arrive_expect_tx(full, bytesA + bytesS);
      bulk_copy_g2s(smem_addr(st), ga, bytesA - hold, full, pol);
      bulk_copy_g2s(smem_addr(st + p.sfa_off), S_c + (int64_t)T * TR * K16, bytesS, full, pol);
      if (hold) {
        launch_wait();
        bulk_copy_g2s(smem_addr(st) + bytesA - hold, ga + (bytesA - hold), hold, full, pol);
      }
    }
    issued = T + 1;
  }
  if (!ok) {
    *abort_flag = 1;
    // let every copy already issued land before this warp (and so the CTA) can exit
    for (int T = max(0, issued - NS); T < issued; ++T)
      mbar_wait_bounded(smem_addr(&bars[T % NS]), (T / NS) & 1, kWaitLimitNs);
  }
}

// Consumer wait for the tile at ring position r; the outcome is voted so the whole warp leaves
// together.
__device__ __forceinline__ bool tma_consume_wait(const TmaArgs& p, uint64_t* bars,
                                                 volatile int* abort_flag, const RingPos& r,
                                                 int lane) {
  const bool ready = mbar_wait_bounded(smem_addr(&bars[r.s]), r.phase, kWaitLimitNs);
  if (!__all_sync(kFullMask, ready && *abort_flag == 0)) {
    if (lane == 0) *abort_flag = 1;
    return false;
  }
  return true;
}

__device__ __forceinline__ void tma_release(const TmaArgs& p, uint64_t* bars, const RingPos& r,
                                            int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(smem_addr(&bars[p.stages + r.s]));
}

__device__ __forceinline__ void tma_epilogue(const TmaArgs& p, const TmaCta& g, const float* part,
                                             volatile int* abort_flag) {
  const bool failed = *abort_flag != 0;
  uint16_t* c_c = p.c + g.l * p.M + g.m0;
  for (int t = threadIdx.x; t < g.n; t += 32 * g.Wc) {
    float v = 0.f;
    for (int q = 0; q < p.slots; ++q) v += part[t * p.slots + q];
    const uint16_t nan_bits = p.out_bf16 ? (uint16_t)0x7FC0 : (uint16_t)0x7E00;
    c_c[t] = failed ? nan_bits : f32_to_out_bits((v * g.ga) * g.gb, p.out_bf16 != 0);
  }
}

// ------------------------------------------------------------------------------------------------
// Vector in shared memory (general K).
// ------------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(544, 1) gemv_tma_kernel(const TmaArgs p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);  // full[0..NS), empty[NS..2NS)
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 16 * kTmaMaxStages);
  uint32_t* bq = reinterpret_cast<uint32_t*>(smem + p.b_off);
  float* sbf = reinterpret_cast<float*>(smem + p.sb_off);
  float* part = reinterpret_cast<float*>(smem + p.part_off);
  uint8_t* ring = smem + p.ring_off;
  const int64_t K = p.K, K2 = p.K >> 1, K16 = p.K >> 4;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  TmaCta g = tma_setup(p, bars, abort_flag);
  if (!p.early_weights) {
    if (p.pf_rows && warp == g.Wc && lane == 0) tma_prefetch_rows(p, g);
    pdl_wait();
  }
  tma_resolve_group(p, g, lane);
  if (g.skip) return;
  if (warp == g.Wc) {
    if (lane == 0) tma_produce<false>(p, g, bars, abort_flag, ring);
    return;
  }
  tma_group_scales(p, g);
  if (p.early_weights) pdl_wait();

  const int Wc = g.Wc, cw = warp, cthreads = 32 * Wc;
  const uint8_t* b_l = p.b + g.l * K2;
  for (int64_t i = threadIdx.x; i < K2 / 16; i += cthreads) {
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
  const uint8_t* sfb_l = p.sfb + g.l * K16;
  for (int64_t i = threadIdx.x; i < K16 / 2; i += cthreads) {
    const float2 sc = f16x2_to_f32x2(e4m3x2_to_f16x2(ld_l2_u16(sfb_l + 2 * i)));
    sbf[2 * i] = sc.x;
    sbf[2 * i + 1] = sc.y;
  }
  for (int i = threadIdx.x; i < p.rows_cap * p.slots; i += cthreads) part[i] = 0.f;
  named_barrier(1, (uint32_t)cthreads);

  // Per-thread constants: a lane's chunk swizzle term is (lane >> 1) & 3 for every segment.
  const int nseg = (int)((K + kStep - 1) / kStep);
  const uint32_t K2u = (uint32_t)K2, K16u = (uint32_t)K16, Ku = (uint32_t)K;
  const uint32_t ring32 = smem_addr(ring), bq32 = smem_addr(bq), sb32 = smem_addr(sbf);
  const uint32_t x = ((uint32_t)lane >> 1) & 3u;
  const uint32_t bsw[4] = {16u * (0u ^ x), 16u * (1u ^ x), 16u * (2u ^ x), 16u * (3u ^ x)};
  const int rg0 = cw / nseg, sg0 = cw - rg0 * nseg;
  float2 acc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
  RingPos rp;
  for (int T = 0; T < g.NT; ++T, rp.advance(p.stages)) {
    if (!tma_consume_wait(p, bars, abort_flag, rp, lane)) break;
    const int rows_t = min(p.tile_rows, g.n - T * p.tile_rows);
    const uint32_t stA = ring32 + (uint32_t)rp.s * p.stage_bytes;
    const uint32_t stS = stA + p.sfa_off;
    float* part_tile = part + (size_t)T * p.tile_rows * p.slots;
    const int rgs = (rows_t + 3) >> 2;
    int rg = rg0, sg = sg0, cur = -1;
    uint32_t aoff[4], soff[4];
    while (rg < rgs) {  // this warp's items it = cw, cw + Wc, ... as (row group, segment)
      if (rg != cur) {
        if (cur >= 0) tma_flush(acc, lane, 4 * cur, rows_t, part_tile, p.slots, cw);
        cur = rg;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t r = (uint32_t)min(4 * rg + i, rows_t - 1);  // re-read the last row
          aoff[i] = stA + r * K2u + 16u * lane;
          soff[i] = stS + r * K16u + 2u * lane;
        }
      }
      if ((uint32_t)sg * 1024u + 32u * lane < Ku) {
        const uint32_t so = (uint32_t)sg;
        uint4 av[4];
        uint16_t sv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          av[i] = lds_v4(aoff[i] + so * 512u);
          sv[i] = lds_u16(soff[i] + so * 64u);
        }
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
      sg += Wc;
      while (sg >= nseg) {
        sg -= nseg;
        ++rg;
      }
    }
    if (cur >= 0) tma_flush(acc, lane, 4 * cur, rows_t, part_tile, p.slots, cw);
    tma_release(p, bars, rp, lane);
  }
  named_barrier(1, (uint32_t)cthreads);
  tma_epilogue(p, g, part, abort_flag);
}

// Cluster barrier over every thread of every CTA of the cluster: the release orders this thread's
// distributed-shared-memory stores before the barrier, the acquire makes the other CTAs' stores
// visible after it.  Every thread of the cluster reaches it once, after bounded work, so it ends.
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// Stores one float into the shared memory of cluster CTA `rank` at the offset of local_addr.
__device__ __forceinline__ void st_cluster_f32(uint32_t local_addr, uint32_t rank, float v) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(remote), "f"(v) : "memory");
}

// Split K: the second pass of the reduction, inside the cluster.  Every consumer thread sends this
// CTA's partial of its rows (the sum over its slots, or NaN if the CTA gave up) to the row's owner
// CTA; after the cluster barrier the owner adds the S partials in slice order and stores the row.
__device__ __forceinline__ void tma_cluster_reduce(const TmaArgs& p, const TmaCta& g,
                                                   const float* part, float* red,
                                                   volatile int* abort_flag) {
  const int S = p.k_slices, n = g.n, rr = p.red_rows, cthreads = 32 * g.Wc;
  const bool failed = *abort_flag != 0;
  const uint32_t red32 = smem_addr(red);
  for (int t = threadIdx.x; t < n; t += cthreads) {  // rows n <= rows_cap: no divergence at exit
    float v = 0.f;
    for (int q = 0; q < p.slots; ++q) v += part[t * p.slots + q];
    const int o = (t * S + S - 1) / n;       // rows [o n / S, (o+1) n / S) belong to CTA o
    const int idx = t - (o * n) / S;
    st_cluster_f32(red32 + 4u * (uint32_t)(g.z * rr + idx), (uint32_t)o,
                   failed ? __int_as_float(0x7fc00000) : v);
  }
  __syncwarp();
  cluster_barrier();
  const int r0 = (g.z * n) / S, r1 = ((g.z + 1) * n) / S;
  uint16_t* c_c = p.c + g.l * p.M + g.m0 + r0;
  for (int t = threadIdx.x; t < r1 - r0; t += cthreads) {
    float v = red[t];
    for (int z = 1; z < S; ++z) v += red[z * rr + t];
    c_c[t] = f32_to_out_bits((v * g.ga) * g.gb, p.out_bf16 != 0);
  }
}

// ------------------------------------------------------------------------------------------------
// Vector slice in registers (W_c NSW segment slots cover the segment count, or the segment count
// divides W_c).
// QX: the vector is bf16 and is quantized to NVFP4 here (see quantize.cuh); its bytes feed the same
// decode as packed input would.  CL: split K over a cluster (the CTA's segments are those of its
// slice; rows of a stage lie rs_a / rs_s bytes apart).  VA: A and sfa aligned, b or sfb not: the
// vector is staged by shifted loads (a separate instantiation; a run-time switch there slowed
// the aligned kernels' main loop by 0.5-1.3%).
// ------------------------------------------------------------------------------------------------
template <int NSW, bool QX, bool UA, bool CL = false, bool VA = false>
__global__ void __launch_bounds__(UA ? 288 : 544, UA ? 2 : 1) gemv_tma_rv_kernel(const TmaArgs p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 16 * kTmaMaxStages);
  float* part = reinterpret_cast<float*>(smem + p.part_off);
  uint8_t* ring = smem + p.ring_off;
  const int64_t K = p.K, K2 = p.K >> 1, K16 = p.K >> 4;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  TmaCta g = tma_setup(p, bars, abort_flag);
  if (!p.early_weights) {
    if (p.pf_rows && warp == g.Wc && lane == 0) tma_prefetch_rows(p, g);
    pdl_wait();
  }
  tma_resolve_group(p, g, lane);
  if (g.skip) {
    if constexpr (CL) cluster_barrier();  // the one cluster barrier every CTA takes part in
    return;
  }
  if (warp == g.Wc) {
    if (lane == 0) tma_produce<UA, CL>(p, g, bars, abort_flag, ring);
    if constexpr (CL) {  // the producer warp takes part in the cluster barrier of the reduction
      __syncwarp();
      cluster_barrier();
    }
    return;
  }
  tma_group_scales(p, g);
  if (p.early_weights) pdl_wait();

  const int Wc = g.Wc, cthreads = 32 * Wc;
  const int nseg = CL ? p.slice_segs : (int)((K + kStep - 1) / kStep);
  const bool many = nseg >= Wc;                     // Wc | nseg: all row groups, NSW segments
  const int rg_first = many ? 0 : warp / nseg;      // nseg | Wc: one segment, every rg_step-th
  const int rg_step = many ? 1 : Wc / nseg;         //   row group
  const int slot = many ? warp : warp % nseg;
  int seg[NSW];
  bool live[NSW];
  uint32_t bw[NSW][16];
  float2 sb[NSW];
#pragma unroll
  // the vector slice: every segment's loads go out before the first is decoded (one L2 round
  // trip, not NSW; with a branch between them they went out one after another: c2 11.3 ->
  // 12.3 us)
  int64_t kks[NSW];
  uint4 vv[NSW];
  uint16_t ss[NSW];
#pragma unroll
  for (int j = 0; j < NSW; ++j) {
    seg[j] = many ? warp + j * Wc : warp % nseg;
    const int64_t k = (int64_t)seg[j] * kStep + 32 * lane;  // inside the slice
    live[j] = k < g.kz;
    // lanes past the slice's end read its first element and never use it
    kks[j] = g.k0 + (live[j] ? k : 0);
  }
  if constexpr (QX) {
#pragma unroll
    for (int j = 0; j < NSW; ++j) {
      const int64_t kk = kks[j];
      const uint16_t* xs = p.x + g.l * K + kk;
      uint32_t xv[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 t = ld_l2_v4(xs + 8 * q);
        xv[4 * q] = t.x;
        xv[4 * q + 1] = t.y;
        xv[4 * q + 2] = t.z;
        xv[4 * q + 3] = t.w;
      }
      uint32_t pk[4];
      quantize_blocks2(xv, p.x_gs, p.rounding, pk, ss[j]);
      vv[j] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      // one writer per segment: the first CTA of the batch, and (when several warps share a
      // segment) the warps of the first row-group round
      if (live[j] && g.pi == 0 && rg_first == 0) {
        *reinterpret_cast<uint4*>(p.b_out + g.l * K2 + (kk >> 1)) = vv[j];
        *reinterpret_cast<uint16_t*>(p.sfb_out + g.l * K16 + (kk >> 4)) = ss[j];
      }
    }
  } else if constexpr (UA || VA) {  // any alignment, through L2
    // A lane reads the two aligned 16-byte chunks around its 16 bytes and shifts them; only at the
    // buffer's first and last bytes (nothing outside [b, b_end) is read) does it read byte by byte.
    // The usual case is one warp-uniform block with all the loads in flight at once.
    const uint8_t* bps[NSW];
    uint32_t dd[NSW];
    bool fast = true;
#pragma unroll
    for (int j = 0; j < NSW; ++j) {
      bps[j] = p.b + g.l * K2 + (kks[j] >> 1);
      dd[j] = (uint32_t)((uintptr_t)bps[j] & 15u);
      const uint8_t* a = bps[j] - dd[j];
      fast = fast && a >= p.b && a + (dd[j] ? 32 : 16) <= p.b_end;
    }
    const bool sfb_even = (((uintptr_t)p.sfb) & 1u) == 0;  // K/16 is even: the grid's parity
    if (__all_sync(0xffffffffu, fast)) {
      // consecutive live lanes hold consecutive 16-byte chunks: a lane's second chunk is the
      // next lane's first; lane 31, and a lane whose neighbour does not hold the next chunk (the
      // last live lane of a partial segment), loads its own
      uint4 lo[NSW], hi[NSW];
      bool own[NSW];
#pragma unroll
      for (int j = 0; j < NSW; ++j) {
        const unsigned long long nxt =
            __shfl_down_sync(0xffffffffu, reinterpret_cast<unsigned long long>(bps[j]), 1);
        own[j] = lane == 31 || nxt != reinterpret_cast<unsigned long long>(bps[j] + 16);
        lo[j] = ld_l2_v4(bps[j] - dd[j]);
        hi[j] = (own[j] && dd[j]) ? ld_l2_v4(bps[j] - dd[j] + 16) : make_uint4(0u, 0u, 0u, 0u);
      }
      // the scale bytes go out before the shuffles below wait for the chunks
      if (sfb_even) {
#pragma unroll
        for (int j = 0; j < NSW; ++j) ss[j] = ld_l2_u16(p.sfb + g.l * K16 + (kks[j] >> 4));
      } else {
#pragma unroll
        for (int j = 0; j < NSW; ++j) {
          const uint8_t* sp = p.sfb + g.l * K16 + (kks[j] >> 4);
          ss[j] = (uint16_t)((uint32_t)__ldcg(sp) | ((uint32_t)__ldcg(sp + 1) << 8));
        }
      }
#pragma unroll
      for (int j = 0; j < NSW; ++j) {
        const uint4 nx = make_uint4(__shfl_down_sync(0xffffffffu, lo[j].x, 1),
                                    __shfl_down_sync(0xffffffffu, lo[j].y, 1),
                                    __shfl_down_sync(0xffffffffu, lo[j].z, 1),
                                    __shfl_down_sync(0xffffffffu, lo[j].w, 1));
        if (!own[j]) hi[j] = nx;
      }
#pragma unroll
      for (int j = 0; j < NSW; ++j) vv[j] = dd[j] ? shift16(lo[j], hi[j], dd[j]) : lo[j];
    } else {  // a warp holding the buffer's first or last bytes
#pragma unroll
      for (int j = 0; j < NSW; ++j) {
        const uint8_t* a = bps[j] - dd[j];
        const bool ok = a >= p.b && a + (dd[j] ? 32 : 16) <= p.b_end;
        uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
        if (ok) {
          lo = ld_l2_v4(a);
          if (dd[j]) hi = ld_l2_v4(a + 16);
        }
        const uint8_t* sp = p.sfb + g.l * K16 + (kks[j] >> 4);
        ss[j] = (uint16_t)((uint32_t)__ldcg(sp) | ((uint32_t)__ldcg(sp + 1) << 8));
        // the lanes whose chunks reach past the buffer: lanes 0..15 of the warp load one byte each
        // of such a lane's 16 bytes (one request), which then collects them by shuffles
        uint4 vb = make_uint4(0u, 0u, 0u, 0u);
        for (uint32_t need = __ballot_sync(0xffffffffu, !ok); need; need &= need - 1u) {
          const int e = __ffs((int)need) - 1;
          const uint8_t* base = reinterpret_cast<const uint8_t*>(
              __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(bps[j]), e));
          const uint8_t* q = base + (lane & 15);
          const uint32_t byte = (lane < 16 && q >= p.b && q < p.b_end) ? (uint32_t)__ldcg(q) : 0u;
          uint32_t w4[4] = {0u, 0u, 0u, 0u};
#pragma unroll
          for (int t = 0; t < 16; ++t) w4[t >> 2] |= __shfl_sync(0xffffffffu, byte, t) << (8 * (t & 3));
          if (lane == e) vb = make_uint4(w4[0], w4[1], w4[2], w4[3]);
        }
        vv[j] = !ok ? vb : dd[j] ? shift16(lo, hi, dd[j]) : lo;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < NSW; ++j) {
      vv[j] = ld_l2_v4(p.b + g.l * K2 + (kks[j] >> 1));
      ss[j] = ld_l2_u16(p.sfb + g.l * K16 + (kks[j] >> 4));
    }
  }
#pragma unroll
  for (int j = 0; j < NSW; ++j) {
    e2m1x8_to_f16x2x4(vv[j].x, bw[j][0], bw[j][1], bw[j][2], bw[j][3]);
    e2m1x8_to_f16x2x4(vv[j].y, bw[j][4], bw[j][5], bw[j][6], bw[j][7]);
    e2m1x8_to_f16x2x4(vv[j].z, bw[j][8], bw[j][9], bw[j][10], bw[j][11]);
    e2m1x8_to_f16x2x4(vv[j].w, bw[j][12], bw[j][13], bw[j][14], bw[j][15]);
    sb[j] = f16x2_to_f32x2(e4m3x2_to_f16x2(ss[j]));
  }
  for (int i = threadIdx.x; i < p.rows_cap * p.slots; i += cthreads) part[i] = 0.f;
  named_barrier(1, (uint32_t)cthreads);

  const uint32_t ring32 = smem_addr(ring);
  const uint32_t rsA = p.rs_a, rsS = p.rs_s;  // K/2 and K/16 unsplit
  uint32_t lane_a[NSW], lane_s[NSW];  // this lane's byte offsets inside a row, per segment
#pragma unroll
  for (int j = 0; j < NSW; ++j) {
    lane_a[j] = (uint32_t)seg[j] * 512u + 16u * lane;
    lane_s[j] = (uint32_t)seg[j] * 64u + 2u * lane;
  }
  // UA: a tile's A (sfa) bytes sit in the stage from the 16-byte boundary at or below their first
  // byte, so row r starts dA + r K/2 (dS + r K/16) bytes in.  K/2 and K/16 are multiples of 16
  // here, so every row of a tile has the same residue dA (dS): a lane reads the aligned 16-byte
  // words at and after its row offset and shifts them by dA, the same for the whole CTA.
  const uint8_t* A_c = p.A + (g.ea * p.M + g.m0) * K2;
  const uint8_t* S_c = p.sfa + (g.ea * p.M + g.m0) * K16;
  RingPos rp;
  for (int T = 0; T < g.NT; ++T, rp.advance(p.stages)) {
    if (!tma_consume_wait(p, bars, abort_flag, rp, lane)) break;
    const int rows_t = min(p.tile_rows, g.n - T * p.tile_rows);
    const int rgs = (rows_t + 3) >> 2;
    const uint32_t stA = ring32 + (uint32_t)rp.s * p.stage_bytes;
    const uint32_t stS = stA + p.sfa_off;
    const uint32_t dA = UA ? (uint32_t)((uintptr_t)(A_c + (int64_t)T * p.tile_rows * K2) & 15u) : 0u;
    const uint32_t dS = UA ? (uint32_t)((uintptr_t)(S_c + (int64_t)T * p.tile_rows * K16) & 15u) : 0u;
    float* part_tile = part + (size_t)T * p.tile_rows * p.slots;
    for (int rg = rg_first; rg < rgs; rg += rg_step) {
      uint32_t aoff[4], soff[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t r = (uint32_t)min(4 * rg + i, rows_t - 1);  // re-read the last row
        aoff[i] = stA + r * rsA;
        soff[i] = stS + dS + r * rsS;
      }
      float2 acc[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
      for (int j = 0; j < NSW; ++j) {
        if (live[j]) {
          if constexpr (UA) {
            // one row at a time: the shift needs two 16-byte words a row, and holding all four
            // rows' words at once spilled registers in the two-segment form
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const uint32_t o = aoff[i] + lane_a[j];
              const uint4 lo = lds_v4(o);
              const uint4 a = dA ? shift16(lo, lds_v4(o + 16), dA) : lo;
              const uint32_t so = soff[i] + lane_s[j];
              const uint16_t sv =
                  (dS & 1u) ? (uint16_t)(lds_u8(so) | (lds_u8(so + 1) << 8)) : lds_u16(so);
              row_compute(a, sv, bw[j], sb[j], acc[i]);
            }
          } else {
            uint4 av[4];
            uint16_t sv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              av[i] = lds_v4(aoff[i] + lane_a[j]);
              sv[i] = lds_u16(soff[i] + lane_s[j]);
            }
            item_compute4(av, sv, bw[j], sb[j], acc);
          }
        }
      }
      tma_flush(acc, lane, 4 * rg, rows_t, part_tile, p.slots, slot);
    }
    tma_release(p, bars, rp, lane);
  }
  named_barrier(1, (uint32_t)cthreads);
  if constexpr (CL)
    tma_cluster_reduce(p, g, part, reinterpret_cast<float*>(smem + p.red_off), abort_flag);
  else
    tma_epilogue(p, g, part, abort_flag);
}

}  // namespace nvfp4

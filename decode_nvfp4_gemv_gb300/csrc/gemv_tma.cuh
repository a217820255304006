// TMA-ring NVFP4 GEMV kernel for GB300 (sm_103a): the bandwidth path for K % 256 == 0.
//
// Why: the work is a read-once stream of A (8/9 of the bytes) and sfa (1/9).  Holding enough
// bytes in flight to cover HBM latency with per-thread loads costs registers and occupancy; the
// Tensor Memory Accelerator's bulk copies instead move whole row tiles into shared memory with one
// instruction each and need no registers to keep them in flight.
//
// Decomposition.  CTA (l, p), p < P, owns the contiguous rows [M*p/P, M*(p+1)/P) of batch l.
// Because rows are contiguous in memory, the CTA's A bytes (and its sfa bytes) form one
// contiguous run, cut into tiles of TR whole rows.  Warp W_c (the last) is the producer: one lane
// walks the tiles and, for each, waits until ring stage s = T mod NS is free, then issues two
// cp.async.bulk copies (the tile's A rows and sfa rows) that complete the stage's `full` mbarrier
// by transaction count.  Warps 0 .. W_c-1 are consumers: while the first copies are in flight they
// decode b[l] into shared memory (one f16x2 word per packed byte, swizzled as in the stream
// kernel) and sfb[l] into fp32; then, for each tile, they wait on `full`, process their items, and
// release the stage by arriving on its `empty` mbarrier (one arrival per consumer warp).
//
// Items.  A tile of TR rows and K columns is cut into groups of 4 rows x 1024-element segments;
// item i goes to consumer warp i mod W_c.  For an item, lane t takes 16 bytes (32 elements, two
// scale blocks) of each of the 4 rows at k = 1024 * seg + 32 t, multiplies them with the staged
// vector words by packed f16 FMAs (exact block partials, as in the stream kernel), scales each
// block partial by sfa * sfb in fp32 and accumulates per row.  A warp's items within a tile come in
// increasing order, so its row group changes monotonically; when it changes (and at the tile end)
// the 4 row sums are reduced across the warp and written to partial[row][warp] in shared memory
// (each slot is written at most once; slots a warp never touches stay zero).  After the last
// tile, thread t sums partial[t][0 .. W_c) in warp order (deterministic), applies g_a and g_b in
// fp32 and stores fp16.
//
// Bounded waits.  Every mbarrier wait gives up after one second of wall time (%globaltimer).  A
// consumer that gives up sets a shared abort flag; a producer that gives up waits (again bounded)
// for the copies it already issued before its warp exits, so no copy outlives the CTA.  An aborted
// CTA writes fp16 NaN to all of its outputs, which is how the host sees the failure.
#pragma once

#include <stdint.h>

#include "gemv_kernels.cuh"
#include "nvfp4_device.cuh"

namespace nvfp4 {

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // one second
constexpr int kTmaMaxStages = 8;

struct TmaArgs {
  const uint8_t* A;
  const uint8_t* sfa;
  const uint8_t* b;
  const uint8_t* sfb;
  uint16_t* c;
  float g_a, g_b;
  int64_t M, K, L;
  int32_t P;           // CTAs per batch
  int32_t tile_rows;   // TR: rows per ring stage (a multiple of 4, or less than 4 only if M is)
  int32_t stages;      // NS <= kTmaMaxStages
  int32_t rows_cap;    // ceil(M / P)
  uint32_t stage_bytes;  // bytes per ring stage (A rows, then sfa rows at sfa_off)
  uint32_t sfa_off;      // offset of the sfa rows inside a stage (16-byte aligned)
  uint32_t b_off, sb_off, part_off, ring_off;  // shared-memory layout (bytes)
};

__device__ __forceinline__ void tma_flush(float (&acc)[4], int lane, int rg, int rows_t,
                                          float* part_tile, int Wc, int cw) {
  const float v = warp_reduce_rows<4>(acc, lane);
  const int j = lane >> 3;  // lanes 8j .. 8j+7 hold row j of the group
  if ((lane & 7) == 0 && 4 * rg + j < rows_t) part_tile[(4 * rg + j) * Wc + cw] = v;
#pragma unroll
  for (int i = 0; i < 4; ++i) acc[i] = 0.f;
}

__global__ void __launch_bounds__(544, 1) gemv_tma_kernel(const TmaArgs p) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int64_t K = p.K, K2 = p.K >> 1, K16 = p.K >> 4;
  const int NS = p.stages;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);  // full[0..NS), empty[NS..2NS)
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 16 * kTmaMaxStages);
  uint32_t* bq = reinterpret_cast<uint32_t*>(smem + p.b_off);
  float* sbf = reinterpret_cast<float*>(smem + p.sb_off);
  float* part = reinterpret_cast<float*>(smem + p.part_off);
  uint8_t* ring = smem + p.ring_off;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int Wc = (blockDim.x >> 5) - 1;  // consumer warps; warp Wc produces
  const int64_t l = blockIdx.x / p.P;
  const int64_t pi = blockIdx.x - l * p.P;
  const int64_t m0 = (p.M * pi) / p.P, m1 = (p.M * (pi + 1)) / p.P;
  const int n = (int)(m1 - m0);
  const int TR = p.tile_rows;
  const int NT = (n + TR - 1) / TR;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_addr(&bars[s]), 1);            // producer's arrive + copy bytes
      mbar_init(smem_addr(&bars[NS + s]), (uint32_t)Wc);  // one arrival per consumer warp
    }
    *abort_flag = 0;
    mbar_init_fence();
  }
  __syncthreads();

  if (warp == Wc) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      const uint8_t* A_c = p.A + (l * p.M + m0) * K2;
      const uint8_t* S_c = p.sfa + (l * p.M + m0) * K16;
      int issued = 0;
      bool ok = true;
      for (int T = 0; T < NT; ++T) {
        const int s = T % NS;
        if (T >= NS && !mbar_wait_bounded(smem_addr(&bars[NS + s]), ((T / NS) - 1) & 1,
                                          kWaitLimitNs)) {
          ok = false;
          break;
        }
        if (*abort_flag) {
          ok = false;
          break;
        }
        const int rows_t = min(TR, n - T * TR);
        const uint32_t bytesA = (uint32_t)(rows_t * K2), bytesS = (uint32_t)(rows_t * K16);
        const uint32_t full = smem_addr(&bars[s]);
        uint8_t* st = ring + (size_t)s * p.stage_bytes;
        mbar_arrive_expect_tx(full, bytesA + bytesS);
        bulk_copy_g2s(smem_addr(st), A_c + (int64_t)T * TR * K2, bytesA, full, pol);
        bulk_copy_g2s(smem_addr(st + p.sfa_off), S_c + (int64_t)T * TR * K16, bytesS, full, pol);
        issued = T + 1;
      }
      if (!ok) {
        *abort_flag = 1;
        // let every copy already issued land before this warp (and so the CTA) can exit
        for (int T = max(0, issued - NS); T < issued; ++T)
          mbar_wait_bounded(smem_addr(&bars[T % NS]), (T / NS) & 1, kWaitLimitNs);
      }
    }
    return;
  }

  // -------------------------------------------------------------------- consumers
  const int cw = warp;
  const int ctid = tid;  // 0 .. 32*Wc - 1
  const int cthreads = 32 * Wc;

  const uint8_t* b_l = p.b + l * K2;
  for (int64_t i = ctid; i < K2 / 16; i += cthreads) {
    const uint4 v = ld_ro_v4(b_l + 16 * i);
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
  for (int64_t i = ctid; i < K16 / 2; i += cthreads) {
    const float2 sc = f16x2_to_f32x2(e4m3x2_to_f16x2(ld_ro_u16(sfb_l + 2 * i)));
    sbf[2 * i] = sc.x;
    sbf[2 * i + 1] = sc.y;
  }
  for (int i = ctid; i < p.rows_cap * Wc; i += cthreads) part[i] = 0.f;
  named_barrier(1, (uint32_t)cthreads);

  const int nseg = (int)((K + kStep - 1) / kStep);
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  bool aborted = false;
  for (int T = 0; T < NT; ++T) {
    const int s = T % NS;
    // the verdict is voted so the whole warp leaves together (shuffles follow)
    const bool ready = mbar_wait_bounded(smem_addr(&bars[s]), (T / NS) & 1, kWaitLimitNs);
    if (!__all_sync(kFullMask, ready && *abort_flag == 0)) {
      if (lane == 0) *abort_flag = 1;
      aborted = true;
      break;
    }
    const int rows_t = min(TR, n - T * TR);
    const uint8_t* stA = ring + (size_t)s * p.stage_bytes;
    const uint8_t* stS = stA + p.sfa_off;
    float* part_tile = part + (size_t)T * TR * Wc;
    const int items = ((rows_t + 3) >> 2) * nseg;
    int cur_rg = -1;
    for (int it = cw; it < items; it += Wc) {
      const int rg = it / nseg, sg = it - rg * nseg;
      if (rg != cur_rg) {
        if (cur_rg >= 0) tma_flush(acc, lane, cur_rg, rows_t, part_tile, Wc, cw);
        cur_rg = rg;
      }
      const int64_t k = (int64_t)sg * kStep + 32 * lane;
      if (k < K) {
        uint4 av[4];
        uint16_t sv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = min(4 * rg + i, rows_t - 1);  // rows past the tile re-read its last row
          av[i] = *reinterpret_cast<const uint4*>(stA + (int64_t)r * K2 + (k >> 1));
          sv[i] = *reinterpret_cast<const uint16_t*>(stS + (int64_t)r * K16 + (k >> 4));
        }
        stream_compute<4>(bq, sbf, k, av, sv, acc);
      }
    }
    if (cur_rg >= 0) tma_flush(acc, lane, cur_rg, rows_t, part_tile, Wc, cw);
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(&bars[NS + s]));
  }
  (void)aborted;
  named_barrier(1, (uint32_t)cthreads);

  const bool failed = *abort_flag != 0;
  uint16_t* c_c = p.c + l * p.M + m0;
  for (int t = ctid; t < n; t += cthreads) {
    float v = 0.f;
    for (int w = 0; w < Wc; ++w) v += part[t * Wc + w];
    c_c[t] = failed ? (uint16_t)0x7E00 : f32_to_f16_bits((v * p.g_a) * p.g_b);
  }
}

}  // namespace nvfp4

// Small-N NVFP4 GEMM / GEMV on the 5th-generation tensor cores (tcgen05, sm_103a).
//
//   c[l][n][m] = fp16(g_a * g_b * sum_k e2m1(A_l[m][k]) e2m1(b_l[n][k]) e4m3(sfa_l[m][k/16]) e4m3(sfb_l[n][k/16]))
//
// "nvFP4 Batch GEMV算子系列(下)", sections on torch._scaled_mm and the Blackwell tensor memory:
// the tensor cores take E2M1 operands with one E4M3 scale per 16 elements (block_scale,
// scale_vec::4X) and apply the scales inside the MMA, accumulating in fp32 in tensor memory
// (TMEM).  Here one instruction multiplies a 128-row x 64-element tile of A by a 16-column x 64-
// element tile of tokens; the tokens are the N <= 16 vectors that share A (a decode batch), or a
// single vector per batch (the batched GEMV, N = 1, columns 1..15 are zeros).
//
// Decomposition.  Output tiles of 128 rows; K is cut into S slices (a cluster of S CTAs along K)
// so that tiles x S CTAs fill the GPU.  CTA (l, tile, s) streams its rows' K slice in chunks of
// 256 elements (128 bytes per row) through an NS-stage shared-memory ring:
//   warp 0      producer: per chunk, four TMA tensor copies (A rows 128 B wide with the 128-byte
//               swizzle the MMA reads, the tokens' 128 B, and both tiles' 16 scale bytes per row)
//               completing the stage's `full` mbarrier;
//   warp 1      allocates TMEM and issues, per chunk, four tcgen05.mma (K = 64 each) whose
//               completion (tcgen05.commit) frees the stage;
//   warps 2..5  copy each stage's scale bytes from shared memory into TMEM (tcgen05.st; each warp
//               owns its TMEM lane quadrant);
//   warps 6..9  epilogue: read the accumulator (tcgen05.ld) and store, while the MMAs of the next
//               tile go to the other of two accumulator buffers.
// With S == 1 a CTA is persistent over tiles u = blockIdx.x, blockIdx.x + gridDim.x, ... and its
// ring streams across tile boundaries.  With S > 1 (one tile per cluster) every CTA sends each
// row's fp32 partial to the CTA of the cluster that owns the row (distributed shared memory);
// after one cluster barrier the owner sums the S partials in rank order, so the result is
// deterministic and no global workspace is used.
//
// Tensor memory layout (32-bit columns; row m of a tile lives in TMEM lane m):
//   columns 16 b .. 16 b + 15     accumulator buffer b (b = tile index mod 2), D[m][n]
//   columns 32 + 32 s + 4 j + q   stage s, MMA step j: A's four block scales (one byte each) of
//                                 row 32 q + r at lane r of quadrant 0, of the lane's own row at
//                                 q = 0 and at q = the lane's quadrant elsewhere (the arrangement
//                                 that the blocked 32 x 4 scale layout and a lane-per-row reading
//                                 both describe)
//   columns 48 + 32 s + 4 j + q   stage s, step j: the tokens' block scales, token r at lane r of
//                                 every quadrant, all four q
//
// Signed block scales: the MMA reads scales as unsigned E4M3; the scale warps negate in place each
// 16-element block whose scale is negative (its E2M1 sign bits flipped) and pass the magnitude, so
// every E4M3FN scale, negative ones included, gives the definition's result.
//
// Bounded waits: every mbarrier wait gives up after one second; a CTA that gives up writes NaN for
// its outputs (its partial, under split K).  Programmatic dependent launch as in the TMA kernels.
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "gemv_tma.cuh"
#include "nvfp4_device.cuh"

namespace nvfp4 {

constexpr int kTcRows = 128;          // MMA M
constexpr int kTcCols = 16;           // MMA N (tokens, zero-padded)
constexpr int kTcChunkBytes = 128;    // bytes of a row per ring stage (256 elements)
constexpr int kTcMaxStages = 6;
constexpr int kTcThreads = 320;       // producer, MMA, 4 scale warps, 4 epilogue warps
constexpr uint32_t kTcTmemCols = 256;
// stage layout (bytes, every part 1024-aligned): A 128 x 128, tokens 16 x 128, sfa 128 x 16.
// The tokens' scales (16 x 16 bytes a stage) sit in a small array after the ring: inside a stage
// they would round it up to the next 1024 bytes, and five stages of 21504 bytes leave no room for
// a second CTA on the SM under split K.
constexpr uint32_t kTcOffB = 16384, kTcOffSA = 18432, kTcStageBytes = 20480;
constexpr uint32_t kTcSbBytes = 256;
constexpr uint32_t kTcHeaderBytes = 1024;  // barriers, TMEM address, abort flag
constexpr uint32_t kTcRedBytes = 9216;     // split-K partials: S x ceil(128 / S) rows x 16 fp32

struct TcArgs {
  uint16_t* c;
  float g_a, g_b;
  int64_t M;          // rows per batch
  int32_t K;          // elements (K % 256 == 0)
  int32_t L;          // batches
  int32_t N;          // tokens per batch (1 .. 16)
  int32_t tiles;      // ceil(M / 128)
  int32_t S;          // K slices = cluster size
  int32_t chunks;     // K / 256
  int32_t stages;     // NS
  int32_t a_rows_per_batch;   // M for the batched GEMV (A_l = rows l*M ..), 0 when A is shared
  int32_t early_weights;
  int32_t total_tiles;        // L * tiles
  uint32_t red_off;           // split-K partial buffer (bytes from the aligned window), S > 1
  int32_t test_stall;  // tests of the failure path: the producer issues nothing
};

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile stored with the 128-byte swizzle
// (rows of 128 bytes, 8-row atoms 1024 bytes apart; tcgen05 descriptor version 1).
__device__ __forceinline__ uint64_t tc_desc_sw128(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) |
         ((uint64_t)(1024u >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor: E2M1 x E2M1, E4M3 scales, K-major operands, N = 16, M = 128.
constexpr uint32_t kTcIdesc =
    (1u << 7) | (1u << 10) | ((uint32_t)(kTcCols >> 3) << 17) | ((uint32_t)(kTcRows >> 4) << 24);

__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t sfa,
                                       uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X"
      " [%0], %1, %2, %6, [%3], [%4], p;\n\t}"
      ::"r"(d), "l"(a), "l"(b), "r"(sfa), "r"(sfb), "r"(accumulate), "r"(kTcIdesc)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};"
      ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]),
        "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]),
        "r"(v[14]), "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// Stores four floats into the shared memory of cluster CTA `rank` at the offset of local_addr.
__device__ __forceinline__ void st_cluster_v4(uint32_t local_addr, uint32_t rank, float a, float b,
                                              float c, float d) {
  uint32_t remote;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_addr), "r"(rank));
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "f"(a), "f"(b),
               "f"(c), "f"(d)
               : "memory");
}

// Negates, in a stage tile of 128-byte rows stored with the 128-byte swizzle (16-byte chunk c of
// row r at chunk c ^ (r mod 8) of its 1024-byte atom), every 16-element block of row r whose
// scale byte (sign bit 7 of byte j of the scale words) is negative: its 8 bytes XOR 0x88 flip
// the sign bit of each E2M1 element.
__device__ __forceinline__ void tc_negate_blocks(uint8_t* tile, int r, const uint32_t (&sc)[4]) {
  uint8_t* row = tile + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
  for (int j = 0; j < 16; ++j)
    if ((sc[j >> 2] >> (8 * (j & 3) + 7)) & 1u) {
      uint64_t* blk = reinterpret_cast<uint64_t*>(row + (((j >> 1) ^ (r & 7)) << 4) + ((j & 1) << 3));
      *blk ^= 0x8888888888888888ull;
    }
}

// ---------------------------------------------------------------- the kernel
// Header (start of the 1024-aligned window): per stage full / ready / empty, the two accumulator
// buffers' full / empty, the TMEM base address and the abort flag.
struct TcHeader {
  uint64_t full[kTcMaxStages];
  uint64_t ready[kTcMaxStages];
  uint64_t empty[kTcMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint32_t tmem;
  int32_t abort;
};

// Work of one CTA: with S == 1 the tiles blockIdx.x, blockIdx.x + gridDim.x, ... (persistent,
// the ring streams across tile boundaries and the accumulator is double-buffered); with S > 1
// one tile, K slice blockIdx.x mod S.
struct TcWork {
  int slice, c0, nloc, u0, ustep, ntiles;
};

__device__ __forceinline__ TcWork tc_work(const TcArgs& p) {
  TcWork w;
  w.slice = p.S > 1 ? (int)(blockIdx.x % p.S) : 0;
  const int per = (p.chunks + p.S - 1) / p.S;
  w.c0 = w.slice * per;
  w.nloc = min(p.chunks, w.c0 + per) - w.c0;
  if (p.S > 1) {
    w.u0 = (int)(blockIdx.x / p.S);
    w.ustep = p.total_tiles;
    w.ntiles = 1;
  } else {
    w.u0 = (int)blockIdx.x;
    w.ustep = (int)gridDim.x;
    w.ntiles = (p.total_tiles - w.u0 + w.ustep - 1) / w.ustep;
  }
  return w;
}

// First rows of tile u in the A and token tensors.
__device__ __forceinline__ void tc_rows(const TcArgs& p, int u, int& l, int& tile, int& a_row0,
                                        int& b_row0) {
  l = u / p.tiles;
  tile = u - l * p.tiles;
  a_row0 = l * p.a_rows_per_batch + tile * kTcRows;
  b_row0 = l * p.N;
}

__global__ void __launch_bounds__(kTcThreads, 1) gemv_tc_kernel(
    const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mB,
    const __grid_constant__ CUtensorMap mSA, const __grid_constant__ CUtensorMap mSB,
    const TcArgs p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-aligned window (the 128-byte swizzle atoms and the MMA descriptors assume it)
  const uint32_t raw32 = smem_addr(smem_raw);
  const uint32_t base32 = (raw32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base32 - raw32);
  TcHeader* h = reinterpret_cast<TcHeader*>(base);
  const uint32_t ring32 = base32 + kTcHeaderBytes;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NS = p.stages;
  const uint32_t sb_off = kTcHeaderBytes + (uint32_t)NS * kTcStageBytes;  // stage s: + 256 s
  const TcWork w = tc_work(p);
  const int npairs = w.ntiles * w.nloc;  // (tile, chunk) pairs this CTA streams
  const uint32_t stage_tx = kTcRows * kTcChunkBytes + (uint32_t)p.N * kTcChunkBytes +
                            kTcRows * 16u + (uint32_t)p.N * 16u;  // bytes of one stage's copies
  const bool early_in_setup = p.early_weights && !p.test_stall && p.S > 1;
  // With static weights the first stages' A and sfa copies go out before the launch wait: stage g
  // expects all of its bytes, the vectors' copies follow after the wait.
  auto request_early_weights = [&](int g) {
    const int k = g / w.nloc, i = g - k * w.nloc;
    int l, tile, ar, br;
    tc_rows(p, w.u0 + k * w.ustep, l, tile, ar, br);
    const uint32_t st = ring32 + g * kTcStageBytes, full = smem_addr(&h->full[g]);
    mbar_arrive_expect_tx(full, stage_tx);
    tma_load_2d(st, &mA, (w.c0 + i) * kTcChunkBytes, ar, full);
    tma_load_2d(st + kTcOffSA, &mSA, (w.c0 + i) * 16, ar, full);
  };

  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_addr(&h->tmem)), "n"(kTcTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  if (tid == 0) {
    // fetch the four tensor-map descriptors while the CTA sets up
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mB)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mSA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&mSB)) : "memory");
    for (int s = 0; s < NS; ++s) {
      mbar_init(smem_addr(&h->full[s]), 1);
      mbar_init(smem_addr(&h->ready[s]), 128);
      mbar_init(smem_addr(&h->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_addr(&h->acc_full[b]), 1);
      mbar_init(smem_addr(&h->acc_empty[b]), 128);
    }
    h->abort = 0;
    mbar_init_fence();
    // Static weights under split K (one tile per CTA): this thread, the producer, requests the
    // first stages' A and sfa as soon as the barriers exist, ahead of the TMEM allocation, the
    // zeroing below and the CTA barrier.  Measured on GB300 (M = 7168, K = 16384): N = 2 / 8 / 16
    // from 14.00 / 13.92 / 14.35 to 13.38 / 13.56 / 14.16 us; persistent CTAs (S = 1) measured 2%
    // slower with it, so they request them after the CTA barrier.
    if (early_in_setup)
      for (int g = 0; g < min(NS, npairs); ++g) request_early_weights(g);
  }
  // token rows N .. 15 of every stage are never written by the copies: zero them once
  const int zero_words = (kTcCols - p.N) * 32;
  for (int i = tid; i < NS * zero_words; i += kTcThreads) {
    const int s = i / zero_words;
    reinterpret_cast<uint32_t*>(base + kTcHeaderBytes + s * kTcStageBytes + kTcOffB +
                                p.N * kTcChunkBytes)[i - s * zero_words] = 0u;
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  pdl_launch_dependents();
  const uint32_t tmem = h->tmem;
  volatile int32_t* abort_flag = &h->abort;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && !p.test_stall) {  // stalled: every wait for its copies runs out
      // static weights: the first stages' A and sfa copies before the launch wait (under split K
      // they already went out during the set-up above)
      const int pre = p.early_weights ? min(NS, npairs) : 0;
      if (!early_in_setup)
        for (int g = 0; g < pre; ++g) request_early_weights(g);
      pdl_wait();
      for (int g = 0; g < pre; ++g) {
        const int k = g / w.nloc, i = g - k * w.nloc;
        int l, tile, ar, br;
        tc_rows(p, w.u0 + k * w.ustep, l, tile, ar, br);
        const uint32_t st = ring32 + g * kTcStageBytes, full = smem_addr(&h->full[g]);
        tma_load_2d(st + kTcOffB, &mB, (w.c0 + i) * kTcChunkBytes, br, full);
        tma_load_2d(base32 + sb_off + g * kTcSbBytes, &mSB, (w.c0 + i) * 16, br, full);
      }
      RingPos rp;
      int issued = 0;
      for (int g = 0, k = 0, i = 0; g < npairs; ++g, rp.advance(NS)) {
        if (g >= pre) {
          if (g >= NS &&
              !mbar_wait_bounded(smem_addr(&h->empty[rp.s]), rp.phase ^ 1u, kWaitLimitNs)) {
            *abort_flag = 1;
            break;
          }
          if (*abort_flag) break;
          int l, tile, ar, br;
          tc_rows(p, w.u0 + k * w.ustep, l, tile, ar, br);
          const uint32_t st = ring32 + rp.s * kTcStageBytes, full = smem_addr(&h->full[rp.s]);
          const int x = (w.c0 + i) * kTcChunkBytes, xs = (w.c0 + i) * 16;
          mbar_arrive_expect_tx(full, stage_tx);
          tma_load_2d(st, &mA, x, ar, full);
          tma_load_2d(st + kTcOffB, &mB, x, br, full);
          tma_load_2d(st + kTcOffSA, &mSA, xs, ar, full);
          tma_load_2d(base32 + sb_off + rp.s * kTcSbBytes, &mSB, xs, br, full);
        }
        issued = g + 1;
        if (++i == w.nloc) {
          i = 0;
          ++k;
        }
      }
      // every copy issued lands before the CTA may exit
      for (int g = max(0, issued - NS); g < issued; ++g)
        mbar_wait_bounded(smem_addr(&h->full[g % NS]), (uint32_t)(g / NS) & 1u, kWaitLimitNs);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      RingPos rp;
      for (int k = 0; k < w.ntiles; ++k) {
        const uint32_t ab = (uint32_t)k & 1u;
        bool ok = k < 2 || mbar_wait_bounded(smem_addr(&h->acc_empty[ab]),
                                              (uint32_t)((k >> 1) - 1) & 1u, kWaitLimitNs);
        tc_fence_after();
        for (int i = 0; ok && i < w.nloc; ++i, rp.advance(NS)) {
          if (!mbar_wait_bounded(smem_addr(&h->ready[rp.s]), rp.phase, kWaitLimitNs) ||
              *abort_flag) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = ring32 + rp.s * kTcStageBytes;
          const uint32_t sfa_col = tmem + 32u + 32u * rp.s, sfb_col = sfa_col + 16u;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tc_mma(tmem + 16u * ab, tc_desc_sw128(st + 32u * j),
                   tc_desc_sw128(st + kTcOffB + 32u * j), sfa_col + 4u * j, sfb_col + 4u * j,
                   (i > 0 || j > 0) ? 1u : 0u);
          tc_commit(smem_addr(&h->empty[rp.s]));
        }
        if (!ok) {  // the flag first: an epilogue warp that sees this commit reads it after
          *abort_flag = 1;
          __threadfence_block();
        }
        tc_commit(smem_addr(&h->acc_full[ab]));  // also on failure, so the epilogue goes on
        if (!ok) break;
      }
    }
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------------ scales into TMEM
    const uint32_t q = (uint32_t)warp & 3u;  // this warp's TMEM lane quadrant
    const uint32_t lane_addr = (32u * q) << 16;
    RingPos rp;
    for (int g = 0; g < npairs; ++g, rp.advance(NS)) {
      const bool ok = mbar_wait_bounded(smem_addr(&h->full[rp.s]), rp.phase, kWaitLimitNs);
      if (!__all_sync(0xffffffffu, ok && *abort_flag == 0)) {
        if (lane == 0) *abort_flag = 1;
        break;
      }
      uint8_t* st = base + kTcHeaderBytes + rp.s * kTcStageBytes;
      uint4 rows[4];  // the 16 scale bytes of rows 32 c + lane, c = 0..3 (word j = MMA step j)
#pragma unroll
      for (int c = 0; c < 4; ++c)
        rows[c] = *reinterpret_cast<const uint4*>(st + kTcOffSA + (32 * c + lane) * 16);
      uint4 tb = make_uint4(0u, 0u, 0u, 0u);
      if (lane < p.N)
        tb = *reinterpret_cast<const uint4*>(base + sb_off + rp.s * kTcSbBytes + lane * 16);
      // Signed scales.  The MMA reads block scales as unsigned E4M3, so a block whose scale is
      // negative enters negated instead: XOR 0x88 on its 8 bytes flips the sign of each of its
      // 16 elements (exact), and its scale enters as the magnitude (the sign bit cleared below;
      // a NaN byte stays NaN).  Row 32 q + lane of A is this lane's to patch, the vectors' rows
      // belong to the lanes of quadrant 0's warp.  Then the generic-proxy stores are made visible
      // to the MMA's reads before the stage is handed over.
      {
        const uint4 own = q == 0 ? rows[0] : q == 1 ? rows[1] : q == 2 ? rows[2] : rows[3];
        const uint32_t sa[4] = {own.x, own.y, own.z, own.w};
        const uint32_t sb4[4] = {tb.x, tb.y, tb.z, tb.w};
        const bool neg_a = ((own.x | own.y | own.z | own.w) & 0x80808080u) != 0;
        const bool neg_b = q == 0 && ((tb.x | tb.y | tb.z | tb.w) & 0x80808080u) != 0;
        if (__any_sync(0xffffffffu, neg_a || neg_b)) {
          if (neg_a) tc_negate_blocks(st, 32 * q + lane, sa);
          if (neg_b) tc_negate_blocks(st + kTcOffB, lane, sb4);
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        rows[c].x &= 0x7F7F7F7Fu;
        rows[c].y &= 0x7F7F7F7Fu;
        rows[c].z &= 0x7F7F7F7Fu;
        rows[c].w &= 0x7F7F7F7Fu;
      }
      tb.x &= 0x7F7F7F7Fu;
      tb.y &= 0x7F7F7F7Fu;
      tb.z &= 0x7F7F7F7Fu;
      tb.w &= 0x7F7F7F7Fu;
      const uint4 own = q == 0 ? rows[0] : q == 1 ? rows[1] : q == 2 ? rows[2] : rows[3];
      uint32_t v[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t ow = j == 0 ? own.x : j == 1 ? own.y : j == 2 ? own.z : own.w;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 r = rows[c];
          const uint32_t rw = j == 0 ? r.x : j == 1 ? r.y : j == 2 ? r.z : r.w;
          v[4 * j + c] = c == 0 ? ow : rw;
        }
      }
      tc_st16(tmem + lane_addr + 32u + 32u * rp.s, v);
      uint32_t u[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t x = j == 0 ? tb.x : j == 1 ? tb.y : j == 2 ? tb.z : tb.w;
#pragma unroll
        for (int c = 0; c < 4; ++c) u[4 * j + c] = x;
      }
      tc_st16(tmem + lane_addr + 48u + 32u * rp.s, u);
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      tc_fence_before();
      mbar_arrive(smem_addr(&h->ready[rp.s]));
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const uint32_t q = (uint32_t)warp & 3u;
    const int rr = (int)(32u * q) + lane;  // row of the tile (TMEM lane)
    const int rmax = (kTcRows + p.S - 1) / p.S;
    for (int k = 0; k < w.ntiles; ++k) {
      const uint32_t ab = (uint32_t)k & 1u;
      bool fin = *abort_flag == 0 &&
                 mbar_wait_sleepy(smem_addr(&h->acc_full[ab]), (uint32_t)(k >> 1) & 1u,
                                  kWaitLimitNs);
      fin = __all_sync(0xffffffffu, fin);
      tc_fence_after();
      uint32_t d[16];
      tc_ld16(tmem + ((32u * q) << 16) + 16u * ab, d);
      tc_fence_before();
      mbar_arrive(smem_addr(&h->acc_empty[ab]));
      const bool failed = !fin || *abort_flag != 0;
      int l, tile, ar, br;
      tc_rows(p, w.u0 + k * w.ustep, l, tile, ar, br);
      if (k == 0) pdl_wait();  // c may be read or written by the preceding work
      if (p.S == 1) {
        const int64_t m = (int64_t)tile * kTcRows + rr;
        if (m < p.M) {
#pragma unroll
          for (int n = 0; n < kTcCols; ++n)
            if (n < p.N)
              p.c[(int64_t)(l * p.N + n) * p.M + m] =
                  failed ? (uint16_t)0x7E00
                         : f32_to_f16_bits((__uint_as_float(d[n]) * p.g_a) * p.g_b);
        }
      } else {
        // this row's partial goes to the CTA of the cluster that owns the row
        int o = 0;
        while (o + 1 < p.S && (o + 1) * kTcRows / p.S <= rr) ++o;
        const int idx = rr - o * kTcRows / p.S;
        const uint32_t dst = base32 + p.red_off + (uint32_t)((w.slice * rmax + idx) * 16) * 4u;
        const float nan = __int_as_float(0x7fc00000);
#pragma unroll
        for (int n = 0; n < 16; n += 4)
          st_cluster_v4(dst + 4u * n, (uint32_t)o,
                        failed ? nan : __uint_as_float(d[n]), failed ? nan : __uint_as_float(d[n + 1]),
                        failed ? nan : __uint_as_float(d[n + 2]),
                        failed ? nan : __uint_as_float(d[n + 3]));
      }
    }
  }

  // ------------------------------------------------------------ split-K reduction, teardown
  tc_fence_before();
  __syncthreads();
  if (p.S > 1) {
    cluster_sync_all();  // every partial of the cluster has landed in its owner
    pdl_wait();
    const int rmax = (kTcRows + p.S - 1) / p.S;
    const int r0 = w.slice * kTcRows / p.S, r1 = (w.slice + 1) * kTcRows / p.S;
    int l, tile, ar, br;
    tc_rows(p, w.u0, l, tile, ar, br);
    const float* red = reinterpret_cast<const float*>(base + p.red_off);
    const int nr = r1 - r0;
    for (int it = tid; it < nr * p.N; it += kTcThreads) {  // consecutive threads: consecutive rows
      const int n = it / nr, idx = it - n * nr;
      const int64_t m = (int64_t)tile * kTcRows + r0 + idx;
      float v = 0.f;
      for (int src = 0; src < p.S; ++src) v += red[(src * rmax + idx) * 16 + n];
      if (m < p.M) p.c[(int64_t)(l * p.N + n) * p.M + m] = f32_to_f16_bits((v * p.g_a) * p.g_b);
    }
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "n"(kTcTmemCols) : "memory");
  }
}

}  // namespace nvfp4

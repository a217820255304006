/*
 * nvfp4_gemv.h -- C ABI of the GB300 (sm_103a) NVFP4 block-scaled batched GEMV library
 * (libnvfp4_gemv.so).
 *
 * The operation ("nvFP4 Batch GEMV算子系列(下)", section "NVFP4 Batched GEMV 概念阐述": blocks of
 * 16 K-elements share one FP8 scale, a single fp32 global scale per operand multiplies the result,
 * floor(k/16) is the block id; the page's formula image is lost and this is its written form):
 *
 *   c[l][m] = fp16( g_a * g_b * sum_{k<K} e2m1(A[l][m][k]) * e2m1(b[l][k])
 *                                        * e4m3(sfa[l][m][k/16]) * e4m3(sfb[l][k/16]) )
 *
 * for l < L, m < M.  This is the blog's per-batch matrix-vector product (section
 * "pytorch实现NVFP4 batch gemv": one (m x k) by (k x 1) product per batch l, fp16 out), without its
 * N = 128 padding of the vector and its 128x4 scale tiles, which served a tensor-core GEMM.
 *
 * Element formats:
 *   e2m1  4-bit float: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0; magnitudes
 *         0, 0.5, 1, 1.5, 2, 3, 4, 6 (cutedsl/bridge.py, "Constants": E2M1_MAGNITUDES).
 *         Two per byte: element 2j in the low nibble of byte j, element 2j+1 in the high nibble
 *         (bridge.py, "Quantization": packed = (odd << 4) | even).
 *   e4m3  float8_e4m3fn block scale (blog, "准备数据"): sign, 4 exponent bits (bias 7), 3 mantissa
 *         bits; no infinity; 0x7F / 0xFF are NaN and make the outputs that use them NaN.
 *   c     IEEE binary16 bits; fp32 accumulation, one fp32 multiply by g_a and one by g_b, then
 *         round-to-nearest-even, overflow to +-inf.
 *
 * Layouts (dense, row-major, K contiguous; all sizes in elements unless stated):
 *   A   uint8 [L][M][K/2]    sfa uint8 [L][M][K/16]
 *   b   uint8 [L][K/2]       sfb uint8 [L][K/16]
 *   c   uint16 [L][M]        (fp16 bits; written, never read)
 *
 * Memory and ownership: every pointer is memory the device can read (c: write) -- device memory of
 * the calling thread's current CUDA device, or host memory the device can access.  The caller owns
 * every buffer; the library keeps no pointer after a call returns and allocates no memory in any
 * call.  c must not overlap any input.
 *
 * Execution: the call validates its arguments on the host, then enqueues its kernel(s) on `stream`
 * (a cudaStream_t; NULL = the legacy default stream) and returns without synchronizing.  Errors of
 * the launched kernels surface at the caller's next synchronization.  TMA kernels are launched with
 * programmatic dependent launch: they may be scheduled while the preceding kernel drains, but every
 * thread waits for the preceding work before touching memory it may write (unless
 * NVFP4_FLAG_EARLY_WEIGHTS says A and sfa are safe to read early), so stream order is kept.  Calls are deterministic:
 * the same inputs give the same output bits.  No call synchronizes, allocates or reads device
 * memory on the host, so calls can be captured in a CUDA graph once the device has been used by
 * one uncaptured call (which caches its properties).
 *
 * Errors (checked in this order, before anything is enqueued; nothing is written on error):
 *   NVFP4_ERR_INVALID_VALUE   M < 0, L < 0, K <= 0, K % 16 != 0, a NULL pointer when M*L > 0,
 *                             c overlapping an input, or an inaccessible pointer
 *   NVFP4_ERR_UNSUPPORTED_SHAPE  M, L or K/2 above 2^31 - 1, or an invalid forced plan
 *   NVFP4_ERR_MISALIGNED      c not 2-byte aligned, or a forced plan other than TMA_RV, SHIFT or
 *                             SIMPLE while A, sfa, b or sfb is not 16-byte aligned
 *   Any alignment of A, sfa, b and sfb is accepted.  When only b or sfb is not 16-byte aligned,
 *   TMA_RV keeps the plan aligned operands get and loads the vector with shifted loads.  When A or
 *   sfa is not, the automatic plan is TMA_RV's unaligned form if K % 256 == 0 and every CTA gets 8
 *   rows; else (and for aligned operands with K % 32 != 0) the SHIFT kernel (aligned 16-byte
 *   loads shifted into place), or the SIMPLE kernel (byte loads) when the vector does not fit
 *   shared memory.
 *   NVFP4_ERR_ARCH            the current device is not compute capability 10.3 (GB300)
 *   NVFP4_ERR_CUDA            a CUDA runtime call or the launch failed (nvfp4_last_error() has
 *                             the runtime's message)
 *   M * L == 0 with valid K is a successful no-op.
 */
#ifndef NVFP4_GEMV_H_
#define NVFP4_GEMV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define NVFP4_ABI_VERSION 7

typedef enum nvfp4_status {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_VALUE = 1,
  NVFP4_ERR_MISALIGNED = 2,
  NVFP4_ERR_UNSUPPORTED_SHAPE = 3,
  NVFP4_ERR_ARCH = 4,
  NVFP4_ERR_CUDA = 5
} nvfp4_status;

/* Kernel families a plan may force. */
typedef enum nvfp4_kernel {
  NVFP4_KERNEL_AUTO = 0,    /* the planner's choice */
  NVFP4_KERNEL_SIMPLE = 1,  /* one warp per output row, byte loads; any K % 16 == 0 */
  NVFP4_KERNEL_STREAM = 2,  /* 128-bit streaming loads, vector staged in shared memory, intra-CTA
                               split-K; needs K % 32 == 0 and K <= nvfp4_max_stream_k() */
  NVFP4_KERNEL_TMA = 3,     /* row tiles streamed into a shared-memory ring by bulk async copies
                               (TMA) and mbarriers, vector in shared memory; needs K % 256 == 0 */
  NVFP4_KERNEL_TMA_RV = 4,  /* as TMA with each consumer warp's vector slice held in registers;
                               needs K % 256 == 0 and a forced warp count to divide the number of
                               1024-element K segments (or be a multiple of it); the automatic
                               count for an odd number past 16 takes warps of two segments with
                               one idle.  A vector (b,
                               sfb) not 16-byte aligned is loaded with shifted loads; A or sfa not
                               16-byte aligned take its unaligned form (bulk copies of each
                               tile's aligned interior, the buffers' first and last partial
                               16 bytes copied one by one, shifted out of shared memory; at most
                               8 consumer warps).  With k_slices = S > 1 (A and sfa aligned,
                               S <= 8; slices of ceil(segments / S) 1024-element segments, the
                               last one the rest and not empty) K is split over a
                               thread-block cluster of S CTAs that reduce their partial sums in
                               distributed shared memory, in slice order (no workspace) */
  NVFP4_KERNEL_TC = 5,      /* tensor cores (tcgen05.mma kind::mxf4nvf4, block scales applied by
                               the MMA, fp32 accumulator in tensor memory): 128-row tiles x up to
                               16 vectors, K split over a cluster of k_split (<= 8) CTAs with a
                               deterministic on-chip reduction; needs K % 256 == 0.  The MMA
                               reads block scales as unsigned E4M3: a block whose scale is negative
                               is negated in shared memory and enters with the scale's magnitude */
  NVFP4_KERNEL_SHIFT = 6    /* any K % 16 == 0 and any byte alignment of A, sfa, b, sfb: 16-byte
                               aligned loads around each lane's bytes, funnel-shifted into place,
                               vector staged in shared memory; needs the vector to fit there
                               (about 2.25 bytes per element of K) */
} nvfp4_kernel;

/* Plan flags. */
enum {
  /* The caller guarantees that no kernel that may still be running when this call's kernel starts
     (the preceding work in the stream) writes A or sfa -- as for static weights.  The kernel then
     starts streaming A and sfa before it waits for that work to finish. */
  NVFP4_FLAG_EARLY_WEIGHTS = 1,
  /* Launch without programmatic dependent launch (plain stream order). */
  NVFP4_FLAG_NO_PDL = 2,
  /* nvfp4_gemv_batched_bf16 only (INVALID_VALUE elsewhere): quantize the bf16 vector inside the
     register-vector TMA kernel (one launch; every CTA quantizes the part of the vector it reads)
     instead of a quantizer launch ahead of the GEMV.  The plan's kernel must be TMA_RV, and A and
     sfa 16-byte aligned (NVFP4_ERR_MISALIGNED otherwise). */
  NVFP4_FLAG_QUANTIZE_IN_GEMV = 4,
  /* For tests of the failure path only: the producer of the TMA and tensor-core kernels issues no
     copies, so every wait for them gives up at its one-second limit and the launch writes NaN
     (0x7E00) to all of its outputs; nothing faults and the context stays usable.  The other
     kernels ignore it.  Never set in normal use. */
  NVFP4_FLAG_TEST_STALL = 8,
  /* Without NVFP4_FLAG_EARLY_WEIGHTS, the TMA kernels prefetch the first ring fill of A and sfa into
     L2 before they wait for the preceding work (a hint: every read still follows the wait and sees
     that work's writes).  This flag turns the prefetch off; the results are the same bits. */
  NVFP4_FLAG_NO_L2_PREFETCH = 16
};

/*
 * Launch plan.  Zero in any field means "planner's choice" for that field.  Used by
 * nvfp4_gemv_batched_ex to force a decomposition (tests cover every plan on the same inputs; the
 * output must not depend on it beyond fp32 summation order) and returned by nvfp4_gemv_plan.
 */
typedef struct nvfp4_plan {
  int32_t kernel;          /* nvfp4_kernel */
  int32_t rows_per_warp;   /* STREAM: rows a warp processes together (1, 2 or 4); TMA*: 4 */
  int32_t k_split;         /* STREAM: K slices per row inside a CTA (1 .. ceil(K/1024));
                              TMA_RV: 1024-element segments per warp (filled in by the planner);
                              TC: K slices = cluster size (1 .. 8, at most K/256) */
  int32_t ctas_per_batch;  /* SIMPLE, STREAM, TMA*, SHIFT: CTAs sharing one batch's rows (1 .. M);
                              TC with k_split 1: persistent CTAs for the whole launch (0 = as many
                              as fit); TC with k_split > 1: filled in (tiles x k_split) */
  int32_t warps_per_cta;   /* SIMPLE, SHIFT: 1 .. 8; STREAM: 1 .. 16; TMA*: consumer warps 1 .. 16
                              (one producer warp is added); TC: 4 (fixed) */
  int32_t tile_rows;       /* TMA*: rows per ring stage (1 .. 256); TC: 128 (fixed) */
  int32_t stages;          /* TMA*: ring stages (2 .. 8); TC: 2 .. 6 stages of 256 elements */
  int32_t flags;           /* NVFP4_FLAG_* (honoured by the automatic plan too) */
  int32_t k_slices;        /* TMA_RV: K slices over a thread-block cluster (0 or 1: no split;
                              2 .. 8, each slice at least one 1024-element segment).  The
                              automatic plan splits K when one wave of CTA slots would give each
                              CTA fewer than 8 rows, when K is too long for one CTA's registers
                              (past 32 segments) and for 27-32 segments; ctas_per_batch then
                              counts row ranges (the grid is ctas_per_batch x L x k_slices CTAs,
                              at most the clusters the GPU holds at once per wave) */
} nvfp4_plan;

/*
 * c = fp16(g_a * g_b * A (x) b) per batch, as described above.  A, sfa, g_a: the matrix operand and
 * its block and global scales; b, sfb, g_b: the vector operand and its scales; c: the output;
 * M, K, L: rows, reduction length, batches; stream: cudaStream_t to enqueue on.
 * Returns an nvfp4_status.
 */
int nvfp4_gemv_batched(const uint8_t* A, const uint8_t* sfa, float g_a,
                       const uint8_t* b, const uint8_t* sfb, float g_b,
                       uint16_t* c, int64_t M, int64_t K, int64_t L, void* stream);

/* As nvfp4_gemv_batched, with a plan (NULL = automatic).  Fields of `plan` the planner cannot
 * honour (e.g. the STREAM kernel when K % 32 != 0) give NVFP4_ERR_UNSUPPORTED_SHAPE. */
int nvfp4_gemv_batched_ex(const uint8_t* A, const uint8_t* sfa, float g_a,
                          const uint8_t* b, const uint8_t* sfb, float g_b,
                          uint16_t* c, int64_t M, int64_t K, int64_t L, void* stream,
                          const nvfp4_plan* plan);

/* The plan nvfp4_gemv_batched would use for (M, K, L) on the current device, with every field
 * filled in.  Touches no memory other than *out.  Returns an nvfp4_status. */
int nvfp4_gemv_plan(int64_t M, int64_t K, int64_t L, nvfp4_plan* out);

/* The device limits the planner reads. */
typedef struct nvfp4_device_limits {
  int32_t sms;             /* streaming multiprocessors (152 on GB300) */
  int32_t max_smem_optin;  /* bytes of shared memory one CTA may opt into (232448 on GB300) */
  int32_t max_smem_sm;     /* bytes of shared memory per SM (233472 on GB300) */
} nvfp4_device_limits;

/* The plan nvfp4_gemv_batched_ex would use for (M, K, L) and `forced` (NULL = automatic), or the
 * status it would return for an unsupported forced plan, computed for a device with the given
 * limits and without touching any device.  For host-side tests and capacity planning.
 *
 * Arguments: lim and out non-NULL; lim plausible (sms >= 1, max_smem_optin >= 1024,
 * max_smem_sm >= max_smem_optin), else NVFP4_ERR_INVALID_VALUE; M, L >= 1 and K a positive
 * multiple of 16, each below 2^31 (K/2 for K), else NVFP4_ERR_INVALID_VALUE or
 * NVFP4_ERR_UNSUPPORTED_SHAPE as for the launching entry points.  Inputs are taken as 16-byte
 * aligned.  The STREAM kernel's CTAs per SM come from the driver's occupancy query when a device
 * is present, else 1; every other choice depends on the limits alone, so a plan computed here
 * with a device's own limits equals the one that device's launches use.  No counterpart in the
 * pages: it exposes this library's planner. */
int nvfp4_plan_for_limits(const nvfp4_device_limits* lim, int64_t M, int64_t K, int64_t L,
                          const nvfp4_plan* forced, nvfp4_plan* out);

/* Largest K the STREAM kernel accepts on the current device (its shared-memory bound), or 0 if the
 * device cannot be queried. */
int64_t nvfp4_max_stream_k(void);

/* Static English name of a status code ("unknown status" for other values). */
const char* nvfp4_status_string(int status);

/* Detail text of the last non-OK status returned to the calling thread ("" if none).  The pointer
 * stays valid until that thread's next call into the library. */
const char* nvfp4_last_error(void);

/* ------------------------------------------------------------------------------------------
 * Activation quantization (cutedsl/bridge.py, "Quantization", quantize_activation_nvfp4): bf16
 * x [L][K] -> packed E2M1 b [L][K/2] and E4M3FN block scales sfb [L][K/16], with a fixed fp32
 * global scale (x ~= global_scale * e4m3(sfb) * e2m1(b)).  Per 16-element block, in fp32 with IEEE
 * round-to-nearest divisions: x_norm = x / global_scale; scale = e4m3(max(max|x_norm|, 1e-8) / 6)
 * rounded to nearest even, as the page's float8_e4m3fn cast does: a value past 464 has no finite
 * encoding and gives the NaN byte 0x7F, and that block's codes are 0 (so every output that uses
 * the block is NaN); x_scaled = x_norm / max(scale, 1e-8); magnitude min(|x_scaled|, 6) rounded
 * to E2M1 by `rounding`; the sign of x_scaled.  Each block is independent, so the step needs no
 * reduction and no workspace.  x must hold finite values.
 * ------------------------------------------------------------------------------------------ */
enum {
  NVFP4_ROUND_HALF_STEP_TABLE = 0,  /* the page's rule: table[rint(2 * magnitude)], table =
                                       0,1,2,3,4,4,5,5,6,6,6,7,7 (codes) */
  NVFP4_ROUND_NEAREST_EVEN = 1      /* nearest E2M1 value, ties to the even code */
};

/* Quantizes x (uint16 bf16 bits, [L][K], 16-byte aligned) into b and sfb (16-byte aligned, caller
 * owned, not overlapping x).  K % 16 == 0; global_scale finite and > 0 (else INVALID_VALUE).
 * L == 0 enqueues nothing.  Enqueued on `stream`; returns an nvfp4_status. */
int nvfp4_quantize_activation(const uint16_t* x, float global_scale, int rounding, uint8_t* b,
                              uint8_t* sfb, int64_t K, int64_t L, void* stream);

/* The GEMV with a bf16 vector: quantizes x as nvfp4_quantize_activation does (global scale
 * x_global_scale, which becomes g_b) and computes c as nvfp4_gemv_batched with that vector.  The
 * quantized vector is also written to b_out [L][K/2] and sfb_out [L][K/16] (caller owned, 16-byte
 * aligned, required: they hold the vector whichever kernel runs).  The quantizer runs first on
 * the same stream and releases the GEMV at once (programmatic dependent launch; the GEMV waits for
 * it before reading the vector), or, with NVFP4_FLAG_QUANTIZE_IN_GEMV, the register-vector TMA
 * kernel quantizes inside its vector staging.  plan: as for nvfp4_gemv_batched_ex (NULL =
 * automatic).  Checks are
 * those of both calls; M == 0 or L == 0 enqueues nothing (b_out and sfb_out are not written). */
int nvfp4_gemv_batched_bf16(const uint8_t* A, const uint8_t* sfa, float g_a, const uint16_t* x,
                            float x_global_scale, int rounding, uint8_t* b_out, uint8_t* sfb_out,
                            uint16_t* c, int64_t M, int64_t K, int64_t L, void* stream,
                            const nvfp4_plan* plan);

/* ------------------------------------------------------------------------------------------
 * Grouped (mixture-of-experts) decode GEMV.  cutedsl/bridge.py, "Kernel Launch"
 * (run_nvfp4_grouped_gemm: a 2-D token operand times a 3-D expert operand, per-expert fp32 global
 * scales, bf16 output) and "compute_expert_offsets" (tokens sorted by expert; offsets[e] = the
 * number of tokens of experts 0..e); the per-token expert index is the row-to-group map of the
 * grouped-GEMM API in the flashinfer docs (group_deepgemm_fp8_nt_groupwise, m_indices).
 *
 *   c[t][m] = out( g_a[e] * g_b[e] * sum_k e2m1(A[e][m][k]) e2m1(b[t][k]) e4m3(sfa[e][m][k/16])
 *                                          e4m3(sfb[t][k/16]) ),   e = e(t)
 *
 * A [E][M][K/2], sfa [E][M][K/16]: the experts' weights (layout of nvfp4_gemv_batched with L = E).
 * b [T][K/2], sfb [T][K/16]: one packed vector per token.  c [T][M]: 16-bit outputs, fp16
 * (NVFP4_OUT_F16) or bfloat16 (NVFP4_OUT_BF16), round to nearest even.  g_a, g_b: [E] fp32 device
 * arrays.  Exactly one of:
 *   expert_offsets [E] int32: inclusive cumulative token counts, non-decreasing; token t belongs
 *     to the first e with t < expert_offsets[e];
 *   expert_of_token [T] int32: the expert of each token.
 * A token without an expert (t >= expert_offsets[E-1], or an index outside [0, E)) gets an output
 * row of zeros.  Offsets that decrease give an unspecified (but in-bounds) assignment.
 * The expert indices and global scales are read on the device after the preceding work in the
 * stream, so they may be produced by it (a router); NVFP4_FLAG_EARLY_WEIGHTS and
 * NVFP4_FLAG_QUANTIZE_IN_GEMV are rejected (INVALID_VALUE).  1 <= E <= 65536.  Other checks,
 * alignment (16 bytes for A, sfa, b, sfb; 4 for g_a, g_b and the indices), plans and status
 * codes: as for nvfp4_gemv_batched_ex with L = T; M == 0 or T == 0 enqueues nothing.
 * ------------------------------------------------------------------------------------------ */
typedef enum { NVFP4_OUT_F16 = 0, NVFP4_OUT_BF16 = 1 } nvfp4_out_dtype;

int nvfp4_gemv_grouped(const uint8_t* A, const uint8_t* sfa, const float* g_a, const uint8_t* b,
                       const uint8_t* sfb, const float* g_b, const int32_t* expert_offsets,
                       const int32_t* expert_of_token, uint16_t* c, int out_dtype, int64_t M,
                       int64_t K, int64_t E, int64_t T, void* stream, const nvfp4_plan* plan);

/* ------------------------------------------------------------------------------------------
 * Small-N GEMM: N vectors (a decode batch of tokens) that share one weight matrix.
 * "nvFP4 Batch GEMV算子系列(下)", section pytorch实现: (m, k) @ (n, k)^T -> (m, n) with block
 * scales, here for small n and without padding n to 128.
 *
 *   c[n][m] = fp16( g_a * g_b * sum_k e2m1(A[m][k]) e2m1(b[n][k]) e4m3(sfa[m][k/16]) e4m3(sfb[n][k/16]) )
 *
 * A [M][K/2], sfa [M][K/16] (one matrix), b [N][K/2], sfb [N][K/16], c [N][M] (fp16 bits).
 * The automatic plan is the tensor-core kernel (NVFP4_KERNEL_TC, groups of up to 16 vectors per
 * launch) when K % 256 == 0 and A, sfa, b, sfb are 16-byte aligned; otherwise, or with a forced
 * CUDA-core plan, the batched kernels run one vector per batch, all batches reading A (L2 serves
 * the repeats).  Every E4M3FN scale byte is taken as the format defines it on both paths (the TC
 * kernel negates the blocks whose scales are negative, since its MMA reads scale magnitudes).
 * Checks, statuses and ownership as for nvfp4_gemv_batched_ex with L = N (A holds
 * one matrix); M == 0 or N == 0 enqueues nothing.
 * ------------------------------------------------------------------------------------------ */
int nvfp4_gemm_small_n(const uint8_t* A, const uint8_t* sfa, float g_a, const uint8_t* b,
                       const uint8_t* sfb, float g_b, uint16_t* c, int64_t M, int64_t K, int64_t N,
                       void* stream, const nvfp4_plan* plan);

/* NVFP4_ABI_VERSION of the built library. */
int nvfp4_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_GEMV_H_ */

// C ABI of the NVFP4 batched GEMV (declared in include/nvfp4_gemv.h): argument validation, the
// launch planner and the launches.  Nothing here allocates, synchronizes or reads device memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "../../include/nvfp4_gemv.h"
#include "gemv_kernels.cuh"
#include "gemv_shift.cuh"
#include "gemv_tc.cuh"
#include "gemv_tma.cuh"

namespace {

thread_local char g_last_error[512] = "";

int fail(int status, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
  va_end(ap);
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(NVFP4_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// ---------------------------------------------------------------- per-device properties (cached)
constexpr int kMaxDevices = 64;

struct DeviceInfo {
  cudaError_t err = cudaSuccess;
  int major = 0, minor = 0;
  int sms = 0;
  int max_smem_optin = 0;   // bytes of shared memory one CTA may opt into
  int max_smem_sm = 0;      // bytes of shared memory per SM
  int pageable_access = 0;  // the device can read pageable host memory
  // registers a thread of the one-segment register-vector kernel takes (its three-CTA plans
  // assume at most kRv1RegsForThreeCtas); the design value when no device is queried
  int rv1_regs = 65;
  int rv2_regs = 90;  // the same for the two-segment kernel
  // thread-block clusters of S CTAs resident at once at occ CTAs per SM ([occ - 1][S]), from the
  // occupancy query; 0 where not queried
  int cluster_cap[2][9] = {};
  PFN_cuTensorMapEncodeTiled_v12000 encode_tiled = nullptr;  // driver's tensor-map encoder
};

// Three CTAs of at most 8 warps (7 consumers and the producer) fit an SM's 64 K registers at up to
// 72 registers a thread, also within each of the four schedulers' 16 K (6 warps x 72 x 32).
constexpr int kRv1RegsForThreeCtas = 72;

// CTAs of the aligned register-vector kernel (Wc consumer warps and the producer) that an SM's
// registers hold: each of the four schedulers owns a quarter (16 K) of the register file, and a
// warp takes its registers in units of 8 a thread.
int64_t rv_ctas_by_regs(const DeviceInfo& d, int64_t Wc, int64_t nsw) {
  const int64_t regs = ((nsw == 2 ? d.rv2_regs : d.rv1_regs) + 7) / 8 * 8;
  const int64_t warps_per_scheduler = 16384 / (regs * 32);
  return std::max<int64_t>(1, 4 * warps_per_scheduler / (Wc + 1));
}

// The same counts on GB300 (152 SMs), for planning without a device.  A cluster's CTAs share one
// GPC, so past two CTAs a cluster the GPCs' SM counts leave CTA slots empty: 36 clusters of 4 at
// one CTA per SM hold 144 of the 152 slots, 36 of 8 at two per SM 288 of 304.
constexpr int kClusterCapGb300[2][9] = {{0, 152, 76, 46, 36, 28, 23, 15, 15},
                                        {0, 304, 152, 97, 74, 58, 46, 38, 36}};

// Clusters of S CTAs (2 <= S <= 8) the device holds at once at occ (1 or 2) CTAs per SM.
int64_t clusters_resident(const DeviceInfo& d, int occ, int64_t S) {
  occ = std::min(std::max(occ, 1), 2);
  if (d.cluster_cap[occ - 1][S] > 0) return d.cluster_cap[occ - 1][S];
  return std::max<int64_t>(1, (int64_t)kClusterCapGb300[occ - 1][S] * d.sms / 152);
}

std::once_flag g_dev_once[kMaxDevices];
DeviceInfo g_dev[kMaxDevices];

template <int R>
cudaError_t prepare_stream_kernel(int max_smem) {
  return cudaFuncSetAttribute(nvfp4::gemv_stream_kernel<R>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

// Shared memory up to the opt-in limit and the largest carveout, so two ~110 KiB CTAs fit per SM.
cudaError_t prepare_tma_kernel(void (*k)(const nvfp4::TmaArgs), int max_smem) {
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout,
                              (int)cudaSharedmemCarveoutMaxShared);
}

void init_device(int dev) {
  DeviceInfo& d = g_dev[dev];
  cudaError_t e;
  if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) ||
      (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) ||
      (e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) ||
      (e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                  dev)) ||
      (e = cudaDeviceGetAttribute(&d.max_smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor,
                                  dev)) ||
      (e = cudaDeviceGetAttribute(&d.pageable_access, cudaDevAttrPageableMemoryAccess, dev))) {
    d.err = e;
    return;
  }
  if (d.major != 10 || d.minor != 3) return;  // no kernels for other architectures
  if ((e = prepare_stream_kernel<1>(d.max_smem_optin)) ||
      (e = prepare_stream_kernel<2>(d.max_smem_optin)) ||
      (e = prepare_stream_kernel<4>(d.max_smem_optin)) ||
      (e = prepare_tma_kernel(nvfp4::gemv_tma_kernel, d.max_smem_optin)) ||
      (e = prepare_tma_kernel(nvfp4::gemv_tma_rv_kernel<1, false, false>, d.max_smem_optin)) ||
      (e = prepare_tma_kernel(nvfp4::gemv_tma_rv_kernel<2, false, false>, d.max_smem_optin)) ||
      (e = prepare_tma_kernel(nvfp4::gemv_tma_rv_kernel<1, true, false>, d.max_smem_optin)) ||
      (e = prepare_tma_kernel(nvfp4::gemv_tma_rv_kernel<2, true, false>, d.max_smem_optin)) ||
      (e = prepare_tma_kernel(nvfp4::gemv_tma_rv_kernel<1, false, true>, d.max_smem_optin)) ||
      (e = prepare_tma_kernel(nvfp4::gemv_tma_rv_kernel<2, false, true>, d.max_smem_optin)) ||
      (e = prepare_tma_kernel(nvfp4::gemv_tma_rv_kernel<1, false, false, true>,
                              d.max_smem_optin)) ||
      (e = prepare_tma_kernel(nvfp4::gemv_tma_rv_kernel<2, false, false, true>,
                              d.max_smem_optin)) ||
      (e = prepare_tma_kernel(nvfp4::gemv_tma_rv_kernel<1, true, false, true>,
                              d.max_smem_optin)) ||
      (e = prepare_tma_kernel(nvfp4::gemv_tma_rv_kernel<2, true, false, true>,
                              d.max_smem_optin)) ||
      (e = prepare_tma_kernel(nvfp4::gemv_tma_rv_kernel<1, false, false, false, true>,
                              d.max_smem_optin)) ||
      (e = prepare_tma_kernel(nvfp4::gemv_tma_rv_kernel<2, false, false, false, true>,
                              d.max_smem_optin)) ||
      (e = prepare_tma_kernel(nvfp4::gemv_tma_rv_kernel<1, false, false, true, true>,
                              d.max_smem_optin)) ||
      (e = prepare_tma_kernel(nvfp4::gemv_tma_rv_kernel<2, false, false, true, true>,
                              d.max_smem_optin)) ||
      (e = cudaFuncSetAttribute(nvfp4::gemv_shift_kernel,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, d.max_smem_optin)) ||
      (e = cudaFuncSetAttribute(nvfp4::gemv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                d.max_smem_optin)) ||
      (e = cudaFuncSetAttribute(nvfp4::gemv_tc_kernel,
                                cudaFuncAttributePreferredSharedMemoryCarveout,
                                (int)cudaSharedmemCarveoutMaxShared))) {
    d.err = e;
    return;
  }
  {
    cudaFuncAttributes fa;
    if (cudaFuncGetAttributes(&fa, nvfp4::gemv_tma_rv_kernel<1, false, false>) == cudaSuccess)
      d.rv1_regs = fa.numRegs;
    else
      cudaGetLastError();
    if (cudaFuncGetAttributes(&fa, nvfp4::gemv_tma_rv_kernel<2, false, false>) == cudaSuccess)
      d.rv2_regs = fa.numRegs;
    else
      cudaGetLastError();
  }
  // clusters resident at once, for one and two CTAs per SM (shared memory sized to allow exactly
  // that many; 128 threads keep the registers out of the answer)
  for (int occ = 1; occ <= 2; ++occ)
    for (int S = 2; S <= nvfp4::kTmaMaxClusterK; ++S) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3((unsigned)S);
      cfg.blockDim = dim3(128);
      cfg.dynamicSmemBytes = (size_t)std::min(d.max_smem_optin, d.max_smem_sm / occ - 1024);
      cudaLaunchAttribute a[1];
      a[0].id = cudaLaunchAttributeClusterDimension;
      a[0].val.clusterDim.x = (unsigned)S;
      a[0].val.clusterDim.y = 1;
      a[0].val.clusterDim.z = 1;
      cfg.attrs = a;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, nvfp4::gemv_tma_rv_kernel<1, false, false, true>,
                                         &cfg) == cudaSuccess &&
          n > 0)
        d.cluster_cap[occ - 1][S] = n;
      else
        cudaGetLastError();
    }
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                       &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    d.encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  else
    cudaGetLastError();
}

int current_device(const DeviceInfo** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(NVFP4_ERR_CUDA, "device ordinal %d", dev);
  std::call_once(g_dev_once[dev], init_device, dev);
  const DeviceInfo& d = g_dev[dev];
  if (d.err != cudaSuccess) return cuda_fail(d.err, "device query");
  if (d.major != 10 || d.minor != 3)
    return fail(NVFP4_ERR_ARCH, "device %d is sm_%d%d; this library is built for sm_103a only",
                dev, d.major, d.minor);
  *out = &d;
  return NVFP4_OK;
}

// ---------------------------------------------------------------- argument checks
bool overlaps(const void* a, int64_t na, const void* b, int64_t nb) {
  const uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return x < y + (uintptr_t)nb && y < x + (uintptr_t)na;
}

bool matrix_aligned16(const void* A, const void* sfa) {
  return (((uintptr_t)A | (uintptr_t)sfa) & 15u) == 0;
}

// n_mats: matrices in A and sfa (L for the batched form, E for the grouped form).
// *aligned16: A, sfa, b and sfb all 16-byte aligned (the vector-load and TMA kernels need it; the
// simple kernel's byte loads take any alignment).
int check_args(const uint8_t* A, const uint8_t* sfa, const uint8_t* b, const uint8_t* sfb,
               const uint16_t* c, int64_t M, int64_t K, int64_t L, bool* noop,
               bool* aligned16, int64_t n_mats = -1) {
  if (n_mats < 0) n_mats = L;
  *noop = false;
  *aligned16 = true;
  if (M < 0 || L < 0 || K <= 0)
    return fail(NVFP4_ERR_INVALID_VALUE, "need M >= 0, L >= 0, K > 0 (M=%lld K=%lld L=%lld)",
                (long long)M, (long long)K, (long long)L);
  if (K % 16 != 0)
    return fail(NVFP4_ERR_INVALID_VALUE, "K=%lld is not a multiple of 16", (long long)K);
  const int64_t kMax = (int64_t(1) << 31) - 1;
  if (M > kMax || L > kMax || K / 2 > kMax)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "M, L and K/2 must be below 2^31");
  if (M == 0 || L == 0) {
    *noop = true;
    return NVFP4_OK;
  }
  if (!A || !sfa || !b || !sfb || !c) return fail(NVFP4_ERR_INVALID_VALUE, "NULL pointer");
  *aligned16 = (((uintptr_t)A | (uintptr_t)sfa | (uintptr_t)b | (uintptr_t)sfb) & 15u) == 0;
  if ((uintptr_t)c & 1u) return fail(NVFP4_ERR_MISALIGNED, "c must be 2-byte aligned");
  // products fit easily: M, L < 2^31 and K/2 < 2^31 would overflow int64 only beyond 2^62
  const int64_t nA = M * n_mats * (K / 2), nSA = M * n_mats * (K / 16), nB = L * (K / 2),
                nSB = L * (K / 16), nC = 2 * M * L;
  if (overlaps(c, nC, A, nA) || overlaps(c, nC, sfa, nSA) || overlaps(c, nC, b, nB) ||
      overlaps(c, nC, sfb, nSB))
    return fail(NVFP4_ERR_INVALID_VALUE, "c overlaps an input");
  return NVFP4_OK;
}

// Rejects host pointers the device cannot dereference and device pointers of another device.
int check_access(const DeviceInfo& d, const void* p, const char* name) {
  cudaPointerAttributes at;
  cudaError_t e = cudaPointerGetAttributes(&at, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return cuda_fail(e, "cudaPointerGetAttributes");
  }
  if (at.type == cudaMemoryTypeUnregistered && !d.pageable_access)
    return fail(NVFP4_ERR_INVALID_VALUE, "%s is host memory the device cannot access", name);
  if (at.type == cudaMemoryTypeDevice) {
    int dev = -1;
    cudaGetDevice(&dev);
    if (at.device != dev)
      return fail(NVFP4_ERR_INVALID_VALUE, "%s lives on device %d, current device is %d", name,
                  at.device, dev);
  }
  return NVFP4_OK;
}

// ---------------------------------------------------------------- planner
constexpr int64_t kStreamThreads = 256;

int64_t stream_smem_bytes(int64_t K, int64_t S, int64_t rows_cap) {
  return 2 * K + K / 4 + 4 * S * rows_cap;
}

int64_t max_stream_k(const DeviceInfo& d) {
  // vector words + scales for K, plus a small partial array (keep 8 KiB for it)
  const int64_t budget = d.max_smem_optin - 8192;
  int64_t k = (budget * 4) / 9;  // 2.25 bytes per element
  return k - k % 32;
}

int stream_occupancy(const DeviceInfo& d, int R, int threads, int64_t smem) {
  int n = 0;
  cudaError_t e = cudaErrorInvalidValue;
  if (R == 1)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, nvfp4::gemv_stream_kernel<1>, threads,
                                                      (size_t)smem);
  else if (R == 2)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, nvfp4::gemv_stream_kernel<2>, threads,
                                                      (size_t)smem);
  else
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, nvfp4::gemv_stream_kernel<4>, threads,
                                                      (size_t)smem);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return 1;
  }
  return std::max(n, 1);
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int64_t align_up(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

bool stream_ok(const DeviceInfo& d, int64_t K) { return K % 32 == 0 && K <= max_stream_k(d); }

int plan_simple(const DeviceInfo& d, int64_t M, int64_t L, const nvfp4_plan& f, nvfp4_plan* pl) {
  if (f.warps_per_cta > 8)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "simple kernel: at most 8 warps per CTA");
  const int W = f.warps_per_cta ? f.warps_per_cta : 8;
  const int64_t rows = M * L;
  int64_t ctas = f.ctas_per_batch ? (int64_t)f.ctas_per_batch * L
                                  : std::min<int64_t>(ceil_div(rows, W), (int64_t)d.sms * 8);
  if (ctas > (int64_t(1) << 31) - 1) ctas = (int64_t(1) << 31) - 1;
  pl->kernel = NVFP4_KERNEL_SIMPLE;
  pl->warps_per_cta = W;
  pl->ctas_per_batch = (int32_t)std::max<int64_t>(1, ceil_div(ctas, L));
  pl->rows_per_warp = 1;
  pl->k_split = 1;
  return NVFP4_OK;
}

// CTAs per batch for a grid of whole waves where L allows: from one wave of `slots` CTA slots,
// the smallest P up to 8 P0 + 8 whose last wave is at least 1% fuller than the best so far.
int64_t wave_filling_ctas(int64_t M, int64_t L, int64_t slots) {
  const int64_t P0 = std::min<int64_t>(M, std::max<int64_t>(1, slots / L));
  int64_t best = P0;
  double best_fill = -1.0;
  for (int64_t p = P0; p <= std::min<int64_t>(M, 8 * P0 + 8); ++p) {
    const int64_t grid = p * L;
    const double fill = (double)grid / (double)(ceil_div(grid, slots) * slots);
    if (fill <= best_fill + 0.01) continue;
    best = p;
    best_fill = fill;
    if (fill >= 0.999) break;
  }
  return best;
}

// General-alignment kernel: CTAs of 8 warps over contiguous rows, two per SM when the staged
// vector leaves room for two.
int plan_shift(const DeviceInfo& d, int64_t M, int64_t K, int64_t L, const nvfp4_plan& f,
               nvfp4_plan* pl) {
  const int64_t smem = nvfp4::shift_smem_bytes(K);
  if (smem > d.max_smem_optin)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE,
                "shift kernel: the vector for K=%lld needs %lld bytes of shared memory",
                (long long)K, (long long)smem);
  if (f.warps_per_cta > 8)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "shift kernel: at most 8 warps per CTA");
  if (f.rows_per_warp && f.rows_per_warp != 4)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "shift kernel processes 4 rows per warp");
  const int W = f.warps_per_cta ? f.warps_per_cta : 8;
  const int64_t occ = smem + 1024 <= d.max_smem_sm / 2 ? 2 : 1;
  int64_t P = f.ctas_per_batch ? std::min<int64_t>(f.ctas_per_batch, M)
                               : wave_filling_ctas(M, L, (int64_t)d.sms * occ);
  if (P * L > (int64_t(1) << 31) - 1) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "grid too large");
  pl->kernel = NVFP4_KERNEL_SHIFT;
  pl->warps_per_cta = W;
  pl->ctas_per_batch = (int32_t)P;
  pl->rows_per_warp = 4;
  pl->k_split = 1;
  return NVFP4_OK;
}

int plan_stream(const DeviceInfo& d, int64_t M, int64_t K, int64_t L, const nvfp4_plan& f,
                nvfp4_plan* pl) {
  if (!stream_ok(d, K))
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE,
                "stream kernel needs K %% 32 == 0 and K <= %lld (K=%lld)",
                (long long)max_stream_k(d), (long long)K);
  if (f.warps_per_cta > 16)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "stream kernel: at most 16 warps per CTA");
  const int W = f.warps_per_cta ? f.warps_per_cta : (int)(kStreamThreads / 32);
  const int64_t steps = ceil_div(K, nvfp4::kStep);
  // One wave: as many CTAs as fit on the device at once, split evenly over the batches, each
  // owning a contiguous run of rows.
  const int occ = stream_occupancy(d, 4, W * 32, stream_smem_bytes(K, 1, 1024));
  const int64_t slots = (int64_t)d.sms * occ;
  int64_t P = f.ctas_per_batch ? f.ctas_per_batch : std::max<int64_t>(1, slots / L);
  P = std::min(P, M);
  int64_t rows_cap = ceil_div(M, P);
  while (!f.ctas_per_batch && stream_smem_bytes(K, 1, rows_cap) > d.max_smem_optin && P < M) {
    P = std::min(M, 2 * P);  // very tall matrices: more, shorter CTAs
    rows_cap = ceil_div(M, P);
  }
  if (P * L > (int64_t(1) << 31) - 1) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "grid too large");
  const int R = f.rows_per_warp ? f.rows_per_warp : (rows_cap >= 8 ? 4 : rows_cap >= 2 ? 2 : 1);
  if (R != 1 && R != 2 && R != 4)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "rows_per_warp must be 1, 2 or 4");
  const int64_t G = ceil_div(rows_cap, R);
  // K slices: the fewest that minimise the busiest warp's step count, ceil(units / W) * steps per
  // slice (units = row groups x slices), within the shared-memory budget.
  int64_t S = f.k_split;
  if (S == 0) {
    int64_t best = -1;
    for (int64_t s = 1; s <= steps; ++s) {
      const int64_t ss = ceil_div(steps, s), se = ceil_div(steps, ss);
      if (se != s) continue;
      if (stream_smem_bytes(K, se, rows_cap) > d.max_smem_optin) break;
      const int64_t crit = ceil_div(G * se, W) * ss;
      if (best < 0 || crit < best) {
        best = crit;
        S = se;
      }
    }
    if (S == 0) S = 1;
  }
  if (S < 1 || S > steps) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "k_split out of range");
  const int64_t slice_steps = ceil_div(steps, S);
  S = ceil_div(steps, slice_steps);
  if (stream_smem_bytes(K, S, rows_cap) > d.max_smem_optin)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "plan needs %lld bytes of shared memory",
                (long long)stream_smem_bytes(K, S, rows_cap));
  pl->kernel = NVFP4_KERNEL_STREAM;
  pl->rows_per_warp = R;
  pl->k_split = (int32_t)S;
  pl->ctas_per_batch = (int32_t)P;
  pl->warps_per_cta = W;
  return NVFP4_OK;
}

// Shared-memory layout of the TMA kernels: barriers and abort flag, the decoded vector and its fp32
// block scales (shared-memory-vector variant only), the per-(row, slot) partial sums, then NS ring
// stages of TR rows (A rows, then sfa rows).  Every region starts 16-byte aligned, ring stages
// 128-byte aligned.
struct TmaLayout {
  int64_t b_off, sb_off, part_off, red_off, red_rows, ring_off, sfa_off, stage_bytes, total;
  int64_t rs_a, rs_s;  // bytes between the rows of a stage (A, sfa)
};

// Split K into S slices of whole 1024-element segments: ceil(nseg / S) each, the last slice the
// rest (shorter when S does not divide nseg); every slice must hold at least one segment.
int64_t slice_segs(int64_t nseg, int64_t S) { return S > 1 ? ceil_div(nseg, S) : nseg; }
bool slices_valid(int64_t nseg, int64_t S) {
  return S >= 2 && S <= nvfp4::kTmaMaxClusterK && (S - 1) * ceil_div(nseg, S) < nseg;
}

// ua: operands not 16-byte aligned; a stage then holds each tile's A and sfa bytes from the
// 16-byte boundary at or below their first byte, plus the 16 bytes a lane's second aligned read
// may reach past them: 32 bytes more for each.  S > 1: K split over a cluster of S CTAs; a stage
// holds one slice of each row (slice_segs segments), and the owner's partial sums of the cluster
// (S x ceil(rows_cap / S) floats) follow the per-slot partials.
TmaLayout tma_layout(bool rv, int64_t K, int64_t TR, int64_t NS, int64_t rows_cap, int64_t slots,
                     bool ua = false, int64_t S = 1) {
  TmaLayout t;
  const int64_t seg_s = S > 1 ? slice_segs(ceil_div(K, nvfp4::kStep), S) : 0;
  t.rs_a = S > 1 ? seg_s * (nvfp4::kStep / 2) : K / 2;
  t.rs_s = S > 1 ? seg_s * (nvfp4::kStep / 16) : K / 16;
  t.b_off = nvfp4::kTmaHeaderBytes;
  t.sb_off = t.b_off + (rv ? 0 : 2 * K);
  t.part_off = align_up(t.sb_off + (rv ? 0 : K / 4), 16);
  t.red_off = align_up(t.part_off + 4 * rows_cap * slots, 16);
  t.red_rows = S > 1 ? ceil_div(rows_cap, S) : 0;
  t.ring_off = align_up(t.red_off + 4 * S * t.red_rows, 128);
  const int64_t slack = ua ? 32 : 0;
  t.sfa_off = align_up(TR * t.rs_a + slack, 128);
  t.stage_bytes = align_up(t.sfa_off + TR * t.rs_s + slack, 128);
  t.total = t.ring_off + NS * t.stage_bytes;
  return t;
}

// Consumer warps for the register-vector variant: they divide the K-segment count (NSW = 1 or 2
// segments per warp) or are a multiple of it; an automatic choice for a count with no such
// divisor (an odd count past 16) takes warps of two segments with the last warp's second segment
// past the end (idle: the kernel skips segments that start at or past K).  Returns 0 if nothing
// fits.
int64_t rv_warps(int64_t nseg, int64_t forced, int64_t* nsw, int64_t max_warps = 16) {
  auto ok = [&](int64_t w) -> bool {
    if (w < 1 || w > max_warps) return false;
    if (nseg >= w) {
      if (nseg % w || nseg / w > 2) return false;
      *nsw = nseg / w;
      return true;
    }
    if (w % nseg) return false;
    *nsw = 1;
    return true;
  };
  if (forced) return ok(forced) ? forced : 0;
  // preference from sweeps: 12 warps when the mapping allows, else 8, then the nearest counts
  // (16 would need <= 60 registers per thread for two CTAs per SM)
  for (int64_t w : {12, 8, 7, 6, 14, 10, 9, 5, 4, 11, 13, 3, 2, 1, 15, 16})
    if (ok(w)) return w;
  const int64_t w = (nseg + 1) / 2;
  if (nseg > 2 && w <= max_warps) {
    *nsw = 2;
    return w;
  }
  return 0;
}

// Small calls: the register-vector ring on a grid sized by the bytes of the call, with K split
// over a cluster only when a CTA would otherwise hold more than 32 segments.  Sweeps on GB300 of
// K = 256 .. 65536 and M x L = 16 .. 2400 (us per call, early weights, graphs of 1000 calls):
//   - the ring beats the stream kernel on every such shape, by 1.3-3x (512 x 16384: 2.31 us on
//     152 CTAs against 5.5; 128 x 256 (18.8 KB): 1.95 against 2.82);
//   - the best grid follows the bytes B of the call, not the rows: about 1.9 us + B / 2.5 TB/s
//     on 76 CTAs, 2.1 us + B / 5.3 TB/s on 152 and 2.7 us + B / 7 TB/s on 304, so 76 CTAs below
//     about 1.5 MB (2400 x 1024: 2.12 us, against 2.35 on 152 and 3.03 on 304), 152 up to about
//     13 MB (2000 x 4096: 2.98; 400 x 7168: 1.75 against 2.29 on 76), 304 beyond (700 x 16384 x 3:
//     5.19 against 6.50 on 152);
//   - K = 32768 runs unsplit on at most 152 CTAs (1000 rows: 6.26 us, 8.05 on 304 CTAs, 6.60
//     split in two); at K = 65536
//     four slices of 16384 win (512 rows: 6.99 us on 57 x 4 CTAs, 7.32 with two slices);
//   - clusters of 4 and 8 CTAs fit only 74 x 4 and 36 x 8 of the 304 CTA slots at once (57 x 4
//     and 28 x 8 run in one wave, 76 x 4 and 38 x 8 take twice as long), so split grids stop at
//     3/4 of the slots and at the clusters resident at the slice's CTAs per SM.
// The byte thresholds scale with the SM count (10 KB and 85 KB per SM).  Sets *S (1: unsplit) and
// *P (CTAs per batch); *S = 0 when no split fits the segment count.
constexpr int64_t kSmallCallBytesPerSm = 10 * 1024;
constexpr int64_t kMidCallBytesPerSm = 85 * 1024;

int64_t call_bytes(int64_t M, int64_t K, int64_t L) { return M * L * (K / 2 + K / 16); }

bool small_call(const DeviceInfo& d, int64_t M, int64_t K, int64_t L) {
  return call_bytes(M, K, L) < kMidCallBytesPerSm * d.sms;
}

void small_call_plan(const DeviceInfo& d, int64_t M, int64_t K, int64_t L, int64_t* S_out,
                     int64_t* P_out) {
  const int64_t nseg = ceil_div(K, nvfp4::kStep), slots = 2 * (int64_t)d.sms;
  const int64_t B = call_bytes(M, K, L);
  int64_t S = 1;
  if (nseg > 32) {
    S = 0;
    for (bool exact : {true, false})  // slices that divide the segments first
      for (int64_t s = 2; s <= nvfp4::kTmaMaxClusterK && !S; ++s)
        if (slices_valid(nseg, s) && (!exact || nseg % s == 0) && slice_segs(nseg, s) <= 16)
          S = s;
  }
  *S_out = S;
  *P_out = 0;
  if (!S) return;
  int64_t G = B < kSmallCallBytesPerSm * d.sms ? slots / 4
              : B < kMidCallBytesPerSm * d.sms ? slots / 2
                                                : slots;  // CTAs of the launch
  if (S > 1) {
    // no more clusters than the GPU holds at once, at the CTAs per SM the slice's warps allow
    int64_t nsw = 1;
    const int64_t W = rv_warps(slice_segs(nseg, S), 0, &nsw);
    const int occ = W ? (int)std::min<int64_t>(2, rv_ctas_by_regs(d, W, nsw)) : 1;
    G = std::min<int64_t>({G, slots * 3 / 4, clusters_resident(d, occ, S) * S});
  }
  // more than 16 segments unsplit (K up to 32768): one CTA per SM (1000 x 32768: 6.26 us on 152
  // CTAs, 8.05 on 304)
  if (S == 1 && nseg > 16) G = std::min<int64_t>(G, slots / 2);
  *P_out = std::min<int64_t>(M, std::max<int64_t>(1, G / (L * S)));
}

// Ring sizing, from sweeps on GB300 over the four large decode shapes: two stages of up to ~56 KiB
// (A and sfa rows) per CTA and two CTAs per SM; deeper rings of smaller stages were slower, and a
// ring that leaves room for only one CTA per SM was much slower.
constexpr int64_t kTmaStageTarget = 57344;  // stage bytes (A + sfa rows) the planner aims for
// ... and for an unsplit CTA alone on its SM (by registers) on 19-22 segments with early
// weights: two stages of about 120 KB in place of four of 56.  Measured on GB300 (10-11 warps of
// two segments, 152 CTAs; us per call, 4-row tiles x 4 stages against 8-row tiles x 2): 2048 x
// 18944 7.70 -> 6.98, 3584 x 18944 9.89 -> 9.43, 14336 x 18944 28.71 -> 27.55, 3584 x 20480
// 10.11 -> 9.58, 3584 x 22528 10.31 -> 9.91; at 24 segments it lost up to 1.4%, and in strict
// order 2-3% on 2048-3584 rows.
constexpr int64_t kTmaStageTargetOneCta = 122880;
constexpr int64_t kTmaSmallStage = 24576;   // stages below this get up to 4 ring slots
constexpr int64_t kTmaSmallStageLarge = 20480;  // the same on large calls
constexpr int64_t kTmaLargeStage = 32768;   // from this on: 3 slots if a CTA holds <= 4 stages

// ua: operands not 16-byte aligned (register-vector kernel only; stages carry 32 bytes of slack).
// S: K slices over a cluster of S CTAs (register-vector kernel, aligned operands, at most
// kTmaMaxClusterK slices, each with at least one 1024-element segment).
int plan_tma(const DeviceInfo& d, int64_t M, int64_t K, int64_t L, const nvfp4_plan& f, bool rv,
             nvfp4_plan* pl, bool ua = false, int64_t S = 1) {
  if (ua && !rv)
    return fail(NVFP4_ERR_MISALIGNED,
                "the shared-memory-vector TMA kernel needs 16-byte aligned A, sfa, b and sfb");
  if (K % 256 != 0)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "TMA kernels need K %% 256 == 0 (K=%lld)",
                (long long)K);
  if (S > 1) {
    if (ua)
      return fail(NVFP4_ERR_MISALIGNED, "split K over a cluster needs 16-byte aligned A and sfa");
    if (!rv || !slices_valid(ceil_div(K, nvfp4::kStep), S))
      return fail(NVFP4_ERR_UNSUPPORTED_SHAPE,
                  "split K: the register-vector kernel, k_slices <= %d, each slice at least one "
                  "of the %lld 1024-element segments (k_slices=%lld)",
                  nvfp4::kTmaMaxClusterK, (long long)ceil_div(K, nvfp4::kStep), (long long)S);
  }
  if (f.warps_per_cta > 16)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "TMA kernels: at most 16 consumer warps");
  if (f.rows_per_warp && f.rows_per_warp != 4)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "TMA kernels process 4 rows per warp");
  if (f.tile_rows < 0 || f.tile_rows > 256 || f.stages < 0 || f.stages == 1 ||
      f.stages > nvfp4::kTmaMaxStages)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "tile_rows must be 1..256, stages 2..%d",
                nvfp4::kTmaMaxStages);
  const int64_t nseg = slice_segs(ceil_div(K, nvfp4::kStep), S);  // segments of a CTA's slice
  int64_t Wc = f.warps_per_cta ? f.warps_per_cta : 8, nsw = 1;
  if (rv) {
    // the unaligned form needs more registers (about 88-96 a thread): at most 8 consumer warps
    // keep two CTAs per SM
    Wc = rv_warps(nseg, f.warps_per_cta, &nsw, ua ? 8 : 16);
    if (!Wc)
      return fail(NVFP4_ERR_UNSUPPORTED_SHAPE,
                  "register-vector TMA kernel: no warp count fits %lld K segments",
                  (long long)nseg);
  }
  const int64_t slots = rv ? std::min(Wc, nseg) : Wc;
  const int64_t rg_step = (rv && nseg < Wc) ? Wc / nseg : 1;
  const TmaLayout one_row = tma_layout(rv, K, 1, 1, 1, slots, ua, S);
  const int64_t row_bytes = one_row.rs_a + one_row.rs_s;
  const int64_t unit = 4 * rg_step;  // rows one round of the consumer warps covers
  // Tile rows and ring depth for P CTAs per batch within `budget` bytes of shared memory; false
  // if the partial sums and a two-stage ring do not fit.
  int occ_try = 2;  // the occupancy being tried (set by the loop below)
  // a call of at least 8 rows per CTA slot and 85 KB per SM: stages of 20-24 KB keep two slots
  // (four measured slower on such calls: K = 3584 on 12 rows, K = 5120 on 8), smaller ones four
  // (K = 8192 on 4 rows, 18 KB: two measured 5-7% slower)
  const bool large_call =
      (M * L) / std::max<int64_t>(1, 2 * (int64_t)d.sms) >= 8 && !small_call(d, M, K, L);
  auto shape = [&](int64_t P, int64_t budget, int64_t* TR_out, int64_t* NS_out) -> bool {
    const int64_t rows_cap = ceil_div(M, P);
    int64_t TR = f.tile_rows;
    // one unsplit CTA per SM (by registers) on 19-22 segments with early weights: two stages of
    // about twice the bytes in place of four
    const bool one_cta = rv && S == 1 && occ_try == 1 && nseg <= 22 &&
                         (f.flags & NVFP4_FLAG_EARLY_WEIGHTS);
    if (TR == 0) {
      TR = std::min<int64_t>(
          256, std::max<int64_t>(1, (one_cta ? kTmaStageTargetOneCta : kTmaStageTarget) / row_bytes));
      if (TR >= unit) TR -= TR % unit;
      else if (TR >= 4) TR -= TR % 4;
      // a warp's item is 4 rows: a tile of fewer re-reads its last row for the rest, so rows of
      // more than a quarter of the stage target (K past 24 segments) still take 4-row tiles
      // (shrunk below if two stages do not fit).  Measured on GB300 (13 warps of two segments,
      // one CTA per SM, 152 CTAs; us per call, 3-row tiles x 4 stages against 4-row tiles x 3 or
      // 4, early weights / strict order): 3584 x 25600 12.91 -> 11.36 / 12.49 -> 10.83, 8192 x
      // 25600 24.33 -> 20.03 / 24.69 -> 20.57, 14336 x 26624 42.13 -> 33.18 / 42.68 -> 33.73.
      else TR = 4;
      TR = std::min<int64_t>(TR, std::max<int64_t>(4, align_up(rows_cap, 4)));
      // at least ~4 tiles per CTA, so the last tile's compute is a small part of the CTA's time
      TR = std::min<int64_t>(TR, std::max<int64_t>(unit, align_up(ceil_div(rows_cap, 4), unit)));
      // shrink by whole rounds until two stages fit this occupancy's budget
      while (TR > unit && tma_layout(rv, K, TR, 2, rows_cap, slots, ua, S).total > budget) TR -= unit;
      while (TR > 4 && tma_layout(rv, K, TR, 2, rows_cap, slots, ua, S).total > budget) TR -= 4;
      // rows so long that two stages of 4 do not fit (the shared-memory-vector kernel at large K)
      while (TR > 1 && tma_layout(rv, K, TR, 2, rows_cap, slots, ua, S).total > budget) --TR;
    }
    int64_t NS = f.stages;
    if (NS == 0) {
      const int64_t stage = tma_layout(rv, K, TR, 1, rows_cap, slots, ua, S).stage_bytes;
      // three CTAs per SM keep two stages (4-stage rings of small tiles measured 5-10% slower);
      // one CTA per SM (where the registers allow no more) takes four, the bytes in flight of two
      int64_t want =
          (stage < (large_call ? kTmaSmallStageLarge : kTmaSmallStage) && occ_try < 3) ||
                  (occ_try == 1 && !one_cta)
              ? 4
              : 2;
      // large stages (>= 32 KB) of at least 8 rows, of a CTA that holds at most four of them: a
      // third stage where it fits.  Measured on GB300 (K = 8192, 8-row tiles, 8 warps; us per
      // call, two stages against three, early weights / strict order): 8192 x 8192 9.33 -> 8.28
      // / 10.15 -> 8.22, 9216 x 8192 10.09 -> 8.88 / 11.08 -> 8.89, 3072 x 8192 x 3 10.10 -> 8.81
      // / 11.09 -> 8.90, 5120 x 8192 6.77 -> 6.85 / 8.86 -> 6.68.  Stages of 4 rows (K = 16384)
      // measured 6-10% slower with early weights, and 27.6 KB stages (c4, K = 4096 on 12 rows)
      // 1-5% slower.
      if (want == 2 && occ_try == 2 && stage >= kTmaLargeStage && TR >= 8 &&
          ceil_div(rows_cap, TR) <= 4)
        want = 3;
      for (int64_t ns = want; ns >= 2; --ns)
        if (tma_layout(rv, K, TR, ns, rows_cap, slots, ua, S).total <= budget) {
          NS = ns;
          break;
        }
      if (NS == 0) return false;
    }
    if (tma_layout(rv, K, TR, NS, rows_cap, slots, ua, S).total > d.max_smem_optin) return false;
    *TR_out = TR;
    *NS_out = NS;
    return true;
  };
  // Two CTAs per SM if the ring fits, else one.  With at most 7 consumer warps of one segment each,
  // three CTAs per SM first: more warps to hide the decode's latency and fewer rows per CTA.
  // Measured on GB300 (K = 7168, 7 warps, early weights; us per call, automatic two-CTA plan
  // against three CTAs with 8-row tiles, 4-row where a CTA has few rows): 7168 x 7168 x 1 7.97 ->
  // 6.50, 4096 x 7168 x 8 (c3) 21.21 -> 20.63, 7168 x 7168 x 4 19.09 -> 18.31, 2048 x 7168 x 8
  // 12.22 -> 11.64, 16384 x 7168 x 1 12.23 -> 11.73, 1536 x 7168 x 16 16.51 -> 16.01.  Plans
  // with 12 warps (c4, c5) did not gain from three CTAs of 8 warps.
  // In strict stream order the three-CTA plans lost as often as they won (4096 x 7168 x 8 21.5 ->
  // 22.5 us, 16384 x 7168 x 1 13.0 -> 12.7), so they are for calls with early weights only.
  const bool three = rv && !ua && S == 1 && nsw == 1 && Wc + 1 <= 8 &&
                     (f.flags & NVFP4_FLAG_EARLY_WEIGHTS) && d.rv1_regs <= kRv1RegsForThreeCtas;
  // and never more CTAs than the registers hold: 11 or more warps of two segments (K of 20 to 32
  // segments unsplit) take one CTA per SM; planned as two they ran as a second wave (8192 x 24576:
  // 22.97 us on 304 CTAs, 20.54 on 152)
  const int occ_max = (int)std::min<int64_t>(three ? 3 : 2,
                                             rv && !ua ? rv_ctas_by_regs(d, Wc, nsw) : 2);
  for (int occ = occ_max; occ >= 1; --occ) {
    occ_try = occ;
    const int64_t budget = std::min<int64_t>(d.max_smem_optin, d.max_smem_sm / occ - 1024);
    const int64_t slots_sm = (int64_t)d.sms * occ;
    const int64_t LS = L * S;  // CTAs per row range: one per batch and slice
    int64_t P = 0, TR = 0, NS = 0;
    if (f.ctas_per_batch) {
      P = std::min<int64_t>(f.ctas_per_batch, M);
      if (!shape(P, budget, &TR, &NS)) continue;
    } else {
      // CTAs per batch: start from one wave of CTA slots; where L does not divide the slots (or
      // the rows of one wave's CTAs overflow shared memory) take more CTAs when they fill their
      // last wave at least 1% better.  Measured on GB300: a grid of 0.84 waves ran at 77% of the
      // bandwidth of four exact waves, and an 80-batch call (5.29 GB) ran at 2.1x the stream
      // kernel's rate.
      // A wave is the CTA slots, or under split K the clusters the GPCs hold at once (fewer than
      // the slots past S = 2); P CTAs (clusters) per batch take P * L of it.
      const int64_t wave = S > 1 ? clusters_resident(d, occ, S) : slots_sm;
      const int64_t per_p = S > 1 ? L : LS;
      const int64_t P0 = std::min<int64_t>(M, std::max<int64_t>(1, wave / per_p));
      // the smallest P >= P0 whose partial sums and two-stage ring fit: more CTAs per batch means
      // fewer rows per CTA, so whether a P fits is monotone in P (doubling, then bisection)
      int64_t P_fit = P0, tr = 0, ns = 0;
      if (!shape(P0, budget, &tr, &ns)) {
        int64_t hi = P0;
        while (hi < M && !shape(hi, budget, &tr, &ns)) hi = std::min<int64_t>(M, 2 * hi);
        if (!shape(hi, budget, &tr, &ns)) continue;  // nothing fits at this occupancy
        int64_t lo = std::max<int64_t>(P0, hi / 2);    // does not fit
        while (hi - lo > 1) {
          const int64_t mid = lo + (hi - lo) / 2;
          if (shape(mid, budget, &tr, &ns)) hi = mid;
          else lo = mid;
        }
        P_fit = hi;
      }
      const int64_t P_hi = std::min<int64_t>(M, P_fit + 8 * P0 + 8);
      double best_fill = -1.0;
      for (int64_t p = P_fit; p <= P_hi; ++p) {
        const int64_t grid = p * per_p;
        const double fill = (double)grid / (double)(ceil_div(grid, wave) * wave);
        if (fill <= best_fill + 0.01) continue;
        if (!shape(p, budget, &tr, &ns)) continue;
        P = p;
        TR = tr;
        NS = ns;
        best_fill = fill;
        if (fill >= 0.999) break;
      }
      if (P == 0) continue;
    }
    if (P * LS > (int64_t(1) << 31) - 1)
      return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "grid too large");
    pl->kernel = rv ? NVFP4_KERNEL_TMA_RV : NVFP4_KERNEL_TMA;
    pl->rows_per_warp = 4;
    pl->k_split = (int32_t)nsw;
    pl->k_slices = (int32_t)S;
    pl->ctas_per_batch = (int32_t)P;
    pl->warps_per_cta = (int32_t)Wc;
    pl->tile_rows = (int32_t)TR;
    pl->stages = (int32_t)NS;
    return NVFP4_OK;
  }
  return fail(NVFP4_ERR_UNSUPPORTED_SHAPE,
              "TMA kernel: K=%lld with this plan does not fit shared memory", (long long)K);
}

// Fills every field of *pl for (M, K, L); `forced` fields (non-zero) are honoured or rejected.
// Tensor-core kernel: 128-row output tiles, K cut into S slices (a cluster of S CTAs) so that
// groups x tiles x S CTAs fill the GPU at two CTAs per SM; NS ring stages of 256 K elements.
constexpr int kTcDefaultStages = 5;

// Shared memory of a tensor-core CTA: alignment slack, header, NS stages, split-K partials when
// S > 1; at least 80 KB, so that no more than two CTAs (2 x 256 TMEM columns) share an SM (a
// third would wait in its TMEM allocation).
int64_t tc_smem_bytes(int64_t NS, int64_t S) {
  return std::max<int64_t>(80 * 1024, 1024 + nvfp4::kTcHeaderBytes +
                                          NS * (nvfp4::kTcStageBytes + nvfp4::kTcSbBytes) +
                                          (S > 1 ? nvfp4::kTcRedBytes : 0));
}

int plan_tc(const DeviceInfo& d, int64_t M, int64_t K, int64_t groups, const nvfp4_plan& f,
            nvfp4_plan* pl) {
  if (K % 256 != 0)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "tensor-core kernel needs K %% 256 == 0 (K=%lld)",
                (long long)K);
  if ((f.warps_per_cta && f.warps_per_cta != 4) || (f.tile_rows && f.tile_rows != 128))
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE,
                "tensor-core kernel: 4 epilogue warps and 128-row tiles are fixed");
  const int64_t tiles = ceil_div(M, (int64_t)nvfp4::kTcRows), chunks = K / 256;
  const int64_t total = groups * tiles, slots = 2 * (int64_t)d.sms;
  int64_t S = f.k_split;
  if (S == 0) {  // split K only while the tiles leave at least half of the CTA slots empty
    S = 2 * total >= slots ? 1
                           : std::min<int64_t>(std::min<int64_t>(8, chunks),
                                               std::max<int64_t>(1, slots / total));
    // and in one wave: no more clusters than the GPCs hold at once (two CTAs per SM)
    while (S > 1 && total > clusters_resident(d, 2, S)) --S;
  }
  if (S < 1 || S > 8 || S > chunks)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE,
                "tensor-core kernel: K slices must be 1..8 and at most K/256 (S=%lld)",
                (long long)S);
  const int64_t per = ceil_div(chunks, S);
  S = ceil_div(chunks, per);  // every slice gets at least one chunk
  // default ring depth: the deepest up to kTcDefaultStages that still lets two CTAs share an SM
  int64_t NS = f.stages;
  if (NS == 0) {
    NS = kTcDefaultStages;
    while (NS > 2 && 2 * (tc_smem_bytes(NS, S) + 1024) > d.max_smem_sm) --NS;
  }
  if (NS < 2 || NS > nvfp4::kTcMaxStages || tc_smem_bytes(NS, S) > d.max_smem_optin)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE,
                "tensor-core kernel: stages must be 2..%d within shared memory",
                nvfp4::kTcMaxStages);
  if (total * S > (int64_t(1) << 31) - 1 || tiles > (int64_t(1) << 24))
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "grid too large");
  // ctas_per_batch: with S == 1 the number of persistent CTAs for the whole launch (forced, or 0
  // for as many as fit); with S > 1 one CTA per (tile, slice)
  int64_t ctas = S > 1 ? total * S : f.ctas_per_batch;
  if (S == 1 && ctas > total) ctas = total;
  pl->kernel = NVFP4_KERNEL_TC;
  pl->rows_per_warp = 0;
  pl->k_split = (int32_t)S;
  pl->ctas_per_batch = (int32_t)ctas;
  pl->warps_per_cta = 4;
  pl->tile_rows = nvfp4::kTcRows;
  pl->stages = (int32_t)NS;
  return NVFP4_OK;
}

// aligned16: A, sfa, b and sfb all 16-byte aligned; mat16: A and sfa 16-byte aligned (the
// register-vector kernel's aligned form takes a vector at any alignment).
int make_plan(const DeviceInfo& d, int64_t M, int64_t K, int64_t L, const nvfp4_plan* forced,
              nvfp4_plan* pl, bool aligned16, bool mat16, int64_t tc_groups = -1) {
  if (tc_groups < 0) tc_groups = L;
  nvfp4_plan f;
  memset(&f, 0, sizeof f);
  if (forced) f = *forced;
  if (!aligned16 && f.kernel != NVFP4_KERNEL_AUTO && f.kernel != NVFP4_KERNEL_SIMPLE &&
      f.kernel != NVFP4_KERNEL_SHIFT && f.kernel != NVFP4_KERNEL_TMA_RV)
    return fail(NVFP4_ERR_MISALIGNED,
                "kernel %d needs 16-byte aligned A, sfa, b and sfb (TMA_RV, SHIFT and SIMPLE take "
                "any)", f.kernel);
  if (f.flags & ~(NVFP4_FLAG_EARLY_WEIGHTS | NVFP4_FLAG_NO_PDL | NVFP4_FLAG_QUANTIZE_IN_GEMV |
                  NVFP4_FLAG_TEST_STALL | NVFP4_FLAG_NO_L2_PREFETCH))
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "unknown plan flags 0x%x", (unsigned)f.flags);
  if (f.warps_per_cta < 0 || f.rows_per_warp < 0 || f.k_split < 0 || f.ctas_per_batch < 0 ||
      f.tile_rows < 0 || f.stages < 0 || f.k_slices < 0)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "negative plan field");
  if (f.k_slices > 1 && f.kernel != NVFP4_KERNEL_TMA_RV)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE,
                "k_slices > 1 (split K over a cluster) needs the register-vector TMA kernel");
  memset(pl, 0, sizeof *pl);
  int st = NVFP4_OK;
  switch (f.kernel) {
    case NVFP4_KERNEL_SIMPLE: st = plan_simple(d, M, L, f, pl); break;
    case NVFP4_KERNEL_STREAM: st = plan_stream(d, M, K, L, f, pl); break;
    case NVFP4_KERNEL_TMA: st = plan_tma(d, M, K, L, f, false, pl); break;
    case NVFP4_KERNEL_TMA_RV:
      st = plan_tma(d, M, K, L, f, true, pl, !mat16, f.k_slices > 1 ? f.k_slices : 1);
      break;
    case NVFP4_KERNEL_TC: st = plan_tc(d, M, K, tc_groups, f, pl); break;
    case NVFP4_KERNEL_SHIFT: st = plan_shift(d, M, K, L, f, pl); break;
    case NVFP4_KERNEL_AUTO: {
      // K % 256 == 0 and at least 8 rows per CTA: the TMA ring (vector in registers if the warp
      // mapping allows; the register-vector kernel alone for operands not 16-byte aligned); else
      // aligned operands with K % 32 == 0: the stream kernel; else the shift kernel, else the
      // simple kernel
      const int64_t rows_per_cta = (M * L) / std::max<int64_t>(1, (int64_t)d.sms * 2);
      st = -1;
      // small calls (few bytes, or few rows): the ring on a grid sized by the call's bytes
      if (K % 256 == 0 && mat16 && (rows_per_cta < 8 || small_call(d, M, K, L))) {
        int64_t S = 0, P = 0;
        small_call_plan(d, M, K, L, &S, &P);
        if (S >= 1) {
          nvfp4_plan f2 = f;
          if (!f2.ctas_per_batch) f2.ctas_per_batch = (int32_t)P;
          // CTAs of one row group (at most 4 rows) and at most 6 segments: one warp per segment
          // (four for one or two), not 12 of which most would hold no item
          const int64_t nseg = ceil_div(K, nvfp4::kStep);
          if (S == 1 && !f2.warps_per_cta && nseg <= 6 && ceil_div(M, f2.ctas_per_batch) <= 4)
            f2.warps_per_cta = nseg <= 2 ? 4 : (int32_t)nseg;
          char saved[sizeof g_last_error];
          memcpy(saved, g_last_error, sizeof saved);
          st = plan_tma(d, M, K, L, f2, true, pl, false, S);
          // With early weights a ring of two stages requests one tile before the launch wait; a
          // small call whose CTAs hold more tiles than that takes a third stage where it fits, on
          // grids of at most 3/4 of the CTA slots (on full grids of 4-row stages a third stage
          // measured 9-10% slower: 2000 x 16384 5.27 -> 5.73 us; on 152: 1024 x 16384 3.79 ->
          // 3.28)
          if (st == NVFP4_OK && (f.flags & NVFP4_FLAG_EARLY_WEIGHTS) && !f.stages &&
              pl->stages == 2 && ceil_div(ceil_div(M, pl->ctas_per_batch), pl->tile_rows) > 1 &&
              (int64_t)pl->ctas_per_batch * L * S <= (int64_t)d.sms * 3 / 2) {
            nvfp4_plan f3 = f2;
            f3.warps_per_cta = pl->warps_per_cta;
            f3.tile_rows = pl->tile_rows;
            f3.stages = 3;
            nvfp4_plan p3;
            if (plan_tma(d, M, K, L, f3, true, &p3, false, S) == NVFP4_OK) *pl = p3;
          }
          memcpy(g_last_error, saved, sizeof saved);
          if (st == NVFP4_OK) break;
          memset(pl, 0, sizeof *pl);
        }
        st = -1;
      }
      if (K % 256 == 0 && rows_per_cta >= 8) {
        char saved[sizeof g_last_error];
        memcpy(saved, g_last_error, sizeof saved);
        // Wide K whose unsplit warps hold only one CTA per SM: when half of K runs on two-segment
        // warps that fit two CTAs, split K over clusters of 2.  Measured on GB300 (early weights,
        // us per call, one CTA per SM with a four-stage ring against the split): 8192 x 28672 x 1
        // 25.87 -> 23.74, 4096 x 28672 x 4 47.28 -> 42.56, 8192 x 32768 x 1 27.01 -> 25.80,
        // 4096 x 32768 x 4 49.39 -> 46.05.  Where the halves take one-segment warps (K of 20 to 24
        // segments) the split lost (8192 x 24576 x 1: 19.41 unsplit, 21.21 split).
        // Beyond 32 segments no warp mapping holds the whole vector: split K over 2, 4 or 8 CTAs
        // (the first whose slices are at most 24 segments, 12 warps of two), else 3, 5, 6 or 7,
        // else the first whose slices fit (at most 32); slices are ceil(segments / S) each, the
        // last the rest.  Slices of 26-32 segments (13-16 warps of two, one CTA per SM) streamed
        // 5-15% slower than smaller ones, and clusters of 3, 5 and 6 CTAs were 5-20% slower than
        // 2 or 4 on the same K.  Sweep on GB300, 8192 rows, grids of the resident clusters (us
        // per call, early weights): K of 33-48 segments take 2 (33: 27.0, 30.5 on 3; 48: 35.3,
        // 95% of the copy peak), 52-96 take 4 (53: 43.0, 50.9 on 3; 64: 47.8, 52.0 on 2; 67:
        // 50.5, 55.4 on 3; 96: 68.7, 82.7 on 3), 128 takes 8 (99.7, 103.0 on 4); 60 and 112 lose
        // 4-5% against 2 and 7.  The shared-memory-vector kernel these shapes used to take ran
        // 8192 x 40960 x 1 in 60.8 us (32.7 now) and 8192 x 65536 x 1 in 169.8.
        if (mat16 && f.k_slices == 0 && st != NVFP4_OK) {
          const int64_t nseg = ceil_div(K, nvfp4::kStep);
          int64_t nsw1 = 1, nsw2 = 1;
          const int64_t W1 = rv_warps(nseg, f.warps_per_cta, &nsw1);
          int64_t S = 0;
          if (W1 && rv_ctas_by_regs(d, W1, nsw1) < 2) {
            const int64_t W2 = rv_warps(slice_segs(nseg, 2), f.warps_per_cta, &nsw2);
            if (W2 && nsw2 == 2 && rv_ctas_by_regs(d, W2, nsw2) >= 2) S = 2;
          } else if (!W1) {
            for (int64_t most : {24, 32})
              for (int64_t s2 : {2, 4, 8, 3, 5, 6, 7})
                if (!S && slices_valid(nseg, s2) && slice_segs(nseg, s2) <= most &&
                    rv_warps(slice_segs(nseg, s2), f.warps_per_cta, &nsw2))
                  S = s2;
          }
          if (S && plan_tma(d, M, K, L, f, true, pl, false, S) == NVFP4_OK)
            st = NVFP4_OK;
          else
            memset(pl, 0, sizeof *pl);
        }
        for (bool rv : {true, false}) {
          if (st == NVFP4_OK) break;
          if (!aligned16 && !rv) break;  // unaligned operands: the register-vector kernel only
          if (plan_tma(d, M, K, L, f, rv, pl, rv && !mat16) == NVFP4_OK) {
            st = NVFP4_OK;
            break;
          }
          memset(pl, 0, sizeof *pl);
        }
        memcpy(g_last_error, saved, sizeof saved);
      }
      if (st == NVFP4_OK) break;
      memset(pl, 0, sizeof *pl);
      if (aligned16 && stream_ok(d, K)) {
        st = plan_stream(d, M, K, L, f, pl);
        break;
      }
      // any alignment, any K % 16 == 0: aligned loads shifted into place when the vector fits
      char saved[sizeof g_last_error];
      memcpy(saved, g_last_error, sizeof saved);
      st = plan_shift(d, M, K, L, f, pl);
      memcpy(g_last_error, saved, sizeof saved);
      if (st != NVFP4_OK) {
        memset(pl, 0, sizeof *pl);
        st = plan_simple(d, M, L, f, pl);
      }
      break;
    }
    default: return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "unknown kernel %d", f.kernel);
  }
  pl->flags = f.flags;
  return st;
}

// The fused-quantization inputs of a TMA_RV launch (NULL: the vector arrives packed).
struct FusedVector {
  const uint16_t* x;
  float gs;
  int rounding;
  uint8_t* b_out;
  uint8_t* sfb_out;
};

// ---------------------------------------------------------------- tensor-core launch
int encode_map(const DeviceInfo& d, CUtensorMap* m, const void* base, uint64_t row_bytes,
               uint64_t rows, uint32_t box_bytes, uint32_t box_rows, bool swizzle128) {
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_bytes, box_rows};
  cuuint32_t elem[2] = {1, 1};
  const CUresult r = d.encode_tiled(
      m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, elem,
      CU_TENSOR_MAP_INTERLEAVE_NONE,
      swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
      CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(NVFP4_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return NVFP4_OK;
}

// groups: independent (A, vectors) problems in one launch, each with N vectors; A is [groups][M]
// rows when a_rows_per_batch == M (the batched GEMV), else one shared [M] matrix.
int launch_tc(const DeviceInfo& d, const nvfp4_plan& pl, const uint8_t* A, const uint8_t* sfa,
              float g_a, const uint8_t* b, const uint8_t* sfb, float g_b, uint16_t* c, int64_t M,
              int64_t K, int64_t groups, int64_t N, int64_t a_rows_per_batch,
              cudaStream_t stream) {
  if (!d.encode_tiled)
    return fail(NVFP4_ERR_CUDA, "the driver's tensor-map encoder is not available");
  if (N < 1 || N > nvfp4::kTcCols)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "tensor-core kernel: 1..16 vectors per launch");
  const int64_t rowsA = a_rows_per_batch ? groups * M : M;
  const int64_t kI32 = (int64_t(1) << 31) - 1;
  if (rowsA > kI32 || groups * N > kI32 || K / 2 > kI32)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "tensor-core kernel: coordinates exceed 2^31");
  CUtensorMap mA, mB, mSA, mSB;
  int st;
  if ((st = encode_map(d, &mA, A, K / 2, rowsA, 128, nvfp4::kTcRows, true)) ||
      (st = encode_map(d, &mSA, sfa, K / 16, rowsA, 16, nvfp4::kTcRows, false)) ||
      (st = encode_map(d, &mB, b, K / 2, groups * N, 128, (uint32_t)N, true)) ||
      (st = encode_map(d, &mSB, sfb, K / 16, groups * N, 16, (uint32_t)N, false)))
    return st;
  nvfp4::TcArgs a;
  a.c = c;
  a.g_a = g_a;
  a.g_b = g_b;
  a.M = M;
  a.K = (int32_t)K;
  a.L = (int32_t)groups;
  a.N = (int32_t)N;
  a.tiles = (int32_t)ceil_div(M, (int64_t)nvfp4::kTcRows);
  a.S = pl.k_split;
  a.chunks = (int32_t)(K / 256);
  a.stages = pl.stages;
  a.a_rows_per_batch = (int32_t)a_rows_per_batch;
  a.early_weights = (pl.flags & NVFP4_FLAG_EARLY_WEIGHTS) ? 1 : 0;
  a.test_stall = (pl.flags & NVFP4_FLAG_TEST_STALL) ? 1 : 0;
  a.total_tiles = (int32_t)(groups * a.tiles);
  a.red_off = nvfp4::kTcHeaderBytes +
              (uint32_t)pl.stages * (nvfp4::kTcStageBytes + nvfp4::kTcSbBytes);
  const int64_t smem = tc_smem_bytes(pl.stages, a.S);
  // S == 1: persistent CTAs, as many as fit at once (at most two per SM); S > 1: one per
  // (tile, slice)
  const int64_t occ =
      std::max<int64_t>(1, std::min<int64_t>(2, d.max_smem_sm / (smem + 1024)));
  const int64_t grid = a.S > 1 ? (int64_t)a.total_tiles * a.S
                      : pl.ctas_per_batch > 0 ? std::min<int64_t>(a.total_tiles, pl.ctas_per_batch)
                                              : std::min<int64_t>(a.total_tiles, occ * d.sms);
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(nvfp4::kTcThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int na = 0;
  if (!(pl.flags & NVFP4_FLAG_NO_PDL)) {
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
  }
  if (a.S > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)a.S;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, nvfp4::gemv_tc_kernel, mA, mB, mSA, mSB, a);
  if (e != cudaSuccess) return cuda_fail(e, "tensor-core kernel launch");
  return NVFP4_OK;
}

// The grouped-form inputs of a launch (E == 0: the batched form) and the output type.
struct GroupedOut {
  nvfp4::Groups G;
  int out_bf16;
};

int launch(const DeviceInfo& d, const nvfp4_plan& pl, const uint8_t* A, const uint8_t* sfa,
           float g_a, const uint8_t* b, const uint8_t* sfb, float g_b, uint16_t* c, int64_t M,
           int64_t K, int64_t L, cudaStream_t stream, const FusedVector* fx = nullptr,
           const GroupedOut* go = nullptr) {
  const int threads = pl.warps_per_cta * 32;
  nvfp4::Groups G;
  memset(&G, 0, sizeof G);
  int out_bf16 = 0;
  if (go) {
    G = go->G;
    out_bf16 = go->out_bf16;
  }
  if (pl.kernel == NVFP4_KERNEL_TC) {
    if (fx || G.E > 0 || G.shared_a || out_bf16)
      return fail(NVFP4_ERR_UNSUPPORTED_SHAPE,
                  "the tensor-core kernel takes packed vectors and fp16 output only");
    return launch_tc(d, pl, A, sfa, g_a, b, sfb, g_b, c, M, K, L, 1, M, stream);
  }
  if (pl.kernel == NVFP4_KERNEL_SHIFT) {
    if (fx) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "the shift kernel takes a packed vector");
    nvfp4::ShiftArgs a;
    a.A = A; a.sfa = sfa; a.b = b; a.sfb = sfb; a.c = c;
    a.g_a = g_a; a.g_b = g_b;
    a.M = M; a.K = K; a.L = L;
    const int64_t n_mats = G.E > 0 ? (int64_t)G.E : (G.shared_a ? 1 : L);  // matrices in A
    a.a_bytes = n_mats * M * (K / 2);
    a.P = pl.ctas_per_batch;
    a.rows_q = (int32_t)(M / pl.ctas_per_batch);
    a.rows_r = (int32_t)(M % pl.ctas_per_batch);
    a.G = G;
    a.out_bf16 = out_bf16;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)(pl.ctas_per_batch * L));
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = (size_t)nvfp4::shift_smem_bytes(K);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (pl.flags & NVFP4_FLAG_NO_PDL) ? 0 : 1;
    const cudaError_t le = cudaLaunchKernelEx(&cfg, nvfp4::gemv_shift_kernel, a);
    if (le != cudaSuccess) return cuda_fail(le, "kernel launch");
    return NVFP4_OK;
  }
  if (pl.kernel == NVFP4_KERNEL_SIMPLE) {
    const int64_t grid = std::min<int64_t>((int64_t)pl.ctas_per_batch * L, (int64_t(1) << 31) - 1);
    nvfp4::gemv_simple_kernel<<<(unsigned)grid, threads, 0, stream>>>(A, sfa, b, sfb, g_a, g_b, c,
                                                                      M, K, L, G, out_bf16);
  } else if (pl.kernel == NVFP4_KERNEL_STREAM) {
    nvfp4::StreamArgs a;
    a.A = A; a.sfa = sfa; a.b = b; a.sfb = sfb; a.c = c;
    a.g_a = g_a; a.g_b = g_b;
    a.M = M; a.K = K; a.L = L;
    a.G = G;
    a.out_bf16 = out_bf16;
    a.P = pl.ctas_per_batch;
    a.rows_q = (int32_t)(M / pl.ctas_per_batch);
    a.rows_r = (int32_t)(M % pl.ctas_per_batch);
    const int64_t steps = ceil_div(K, nvfp4::kStep);
    a.slice_steps = (int32_t)ceil_div(steps, pl.k_split);
    a.S = (int32_t)ceil_div(steps, a.slice_steps);
    a.rows_cap = (int32_t)ceil_div(M, pl.ctas_per_batch);
    const size_t smem = (size_t)stream_smem_bytes(K, a.S, a.rows_cap);
    const unsigned grid = (unsigned)(pl.ctas_per_batch * L);
    switch (pl.rows_per_warp) {
      case 1: nvfp4::gemv_stream_kernel<1><<<grid, threads, smem, stream>>>(a); break;
      case 2: nvfp4::gemv_stream_kernel<2><<<grid, threads, smem, stream>>>(a); break;
      default: nvfp4::gemv_stream_kernel<4><<<grid, threads, smem, stream>>>(a); break;
    }
  } else {
    const bool rv = pl.kernel == NVFP4_KERNEL_TMA_RV;
    nvfp4::TmaArgs a;
    a.A = A; a.sfa = sfa; a.b = b; a.sfb = sfb; a.c = c;
    a.g_a = g_a; a.g_b = g_b;
    a.M = M; a.K = K; a.L = L;
    a.G = G;
    a.out_bf16 = out_bf16;
    a.P = pl.ctas_per_batch;
    a.tile_rows = pl.tile_rows;
    a.stages = pl.stages;
    a.rows_cap = (int32_t)ceil_div(M, pl.ctas_per_batch);
    a.rows_q = (int32_t)(M / pl.ctas_per_batch);
    a.rows_r = (int32_t)(M % pl.ctas_per_batch);
    const int64_t nseg = ceil_div(K, nvfp4::kStep);
    a.slots = (int32_t)(rv ? std::min<int64_t>(pl.warps_per_cta, nseg) : pl.warps_per_cta);
    a.early_weights = (pl.flags & NVFP4_FLAG_EARLY_WEIGHTS) ? 1 : 0;
    a.test_stall = (pl.flags & NVFP4_FLAG_TEST_STALL) ? 1 : 0;
    // A or sfa not 16-byte aligned: the register-vector kernel's unaligned form, the aligned
    // interiors of A and sfa and the ends of b and sfb bounding every read.  Only b or sfb not
    // aligned: the aligned form, its vector loaded once per CTA with shifted loads inside [b,
    // b_end) and [sfb, sfb_end).
    const bool ua = !matrix_aligned16(A, sfa);
    const bool va = (((uintptr_t)b | (uintptr_t)sfb) & 15u) != 0;
    if ((ua || va) && (!rv || fx))
      return fail(NVFP4_ERR_MISALIGNED, "this TMA plan needs 16-byte aligned operands");
    a.A_lo = a.A_hi = a.S_lo = a.S_hi = a.b_end = a.sfb_end = nullptr;
    if (va) {
      a.b_end = b + L * (K / 2);
      a.sfb_end = sfb + L * (K / 16);
    }
    if (ua) {
      const int64_t n_mats = G.E > 0 ? (int64_t)G.E : (G.shared_a ? 1 : L);  // matrices in A
      auto up16 = [](const uint8_t* q) {
        return reinterpret_cast<const uint8_t*>(((uintptr_t)q + 15) & ~(uintptr_t)15);
      };
      auto down16 = [](const uint8_t* q) {
        return reinterpret_cast<const uint8_t*>((uintptr_t)q & ~(uintptr_t)15);
      };
      a.A_lo = up16(A);
      a.A_hi = down16(A + n_mats * M * (K / 2));
      a.S_lo = up16(sfa);
      a.S_hi = down16(sfa + n_mats * M * (K / 16));
      a.b_end = b + L * (K / 2);
      a.sfb_end = sfb + L * (K / 16);
    }
    const int64_t S = pl.k_slices > 1 ? pl.k_slices : 1;
    if (S > 1 && (!rv || ua))
      return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "split K needs the aligned register-vector kernel");
    if (S > 1) a.slots = (int32_t)std::min<int64_t>(pl.warps_per_cta, slice_segs(nseg, S));
    const TmaLayout t = tma_layout(rv, K, pl.tile_rows, pl.stages, a.rows_cap, a.slots, ua, S);
    a.k_slices = (int32_t)S;
    a.slice_segs = (int32_t)slice_segs(nseg, S);
    a.rs_a = (uint32_t)t.rs_a;
    a.rs_s = (uint32_t)t.rs_s;
    a.red_off = (uint32_t)t.red_off;
    a.red_rows = (int32_t)t.red_rows;
    // strict stream order: the first ring fill is prefetched into L2 before the launch wait
    // (batched rows, aligned and unsplit; the grouped form learns its expert only after it; for
    // the unaligned form the prefetch measured 18.6 -> 17.9 us on c2 but 12.1 -> 13.0 us on c4)
    // The depth, from sweeps on GB300 of 1 to 8 tiles: the whole first fill (two tiles) for c2
    // (13.36 -> 11.74 us) and c3 (23.58 -> 21.96), one tile for c4 (8.41 -> 7.44; 7.65 with two)
    // and c5 (31.94 -> 30.04; 31.16 with two); deeper was slower everywhere.  The rule that fits:
    // at most a third of a CTA's rows, and at most 7/8 of an SM's shared memory in prefetched bytes
    // per SM (c3: 2 x 2 x 48 KB = 194 KB per SM; c5 would be 221 KB).
    a.pf_row0 = 0;
    a.pf_rows = 0;
    if (!a.early_weights && G.E == 0 && !ua && S == 1 && !(pl.flags & NVFP4_FLAG_NO_L2_PREFETCH)) {
      const int64_t grid = (int64_t)pl.ctas_per_batch * L;
      const int64_t per_sm = std::max<int64_t>(1, ceil_div(grid, (int64_t)d.sms));
      int64_t tiles = pl.stages;
      while (tiles > 1 && (3 * tiles * pl.tile_rows > a.rows_cap ||
                           8 * tiles * t.stage_bytes * per_sm > 7 * (int64_t)d.max_smem_sm))
        --tiles;
      a.pf_rows = (int32_t)(tiles * pl.tile_rows);
    }
    a.stage_bytes = (uint32_t)t.stage_bytes;
    a.sfa_off = (uint32_t)t.sfa_off;
    a.b_off = (uint32_t)t.b_off;
    a.sb_off = (uint32_t)t.sb_off;
    a.part_off = (uint32_t)t.part_off;
    a.ring_off = (uint32_t)t.ring_off;
    void (*kern)(const nvfp4::TmaArgs) = nvfp4::gemv_tma_kernel;
    a.x = nullptr;
    a.x_gs = 1.f;
    a.rounding = 0;
    a.b_out = a.sfb_out = nullptr;
    if (fx) {
      a.x = fx->x;
      a.x_gs = fx->gs;
      a.rounding = fx->rounding;
      a.b_out = fx->b_out;
      a.sfb_out = fx->sfb_out;
    }
    if (rv && S > 1) {
      if (fx)
        kern = pl.k_split == 2 ? nvfp4::gemv_tma_rv_kernel<2, true, false, true>
                               : nvfp4::gemv_tma_rv_kernel<1, true, false, true>;
      else if (va)
        kern = pl.k_split == 2 ? nvfp4::gemv_tma_rv_kernel<2, false, false, true, true>
                               : nvfp4::gemv_tma_rv_kernel<1, false, false, true, true>;
      else
        kern = pl.k_split == 2 ? nvfp4::gemv_tma_rv_kernel<2, false, false, true>
                               : nvfp4::gemv_tma_rv_kernel<1, false, false, true>;
    } else if (rv) {
      if (fx)
        kern = pl.k_split == 2 ? nvfp4::gemv_tma_rv_kernel<2, true, false>
                               : nvfp4::gemv_tma_rv_kernel<1, true, false>;
      else if (ua)
        kern = pl.k_split == 2 ? nvfp4::gemv_tma_rv_kernel<2, false, true>
                               : nvfp4::gemv_tma_rv_kernel<1, false, true>;
      else if (va)
        kern = pl.k_split == 2 ? nvfp4::gemv_tma_rv_kernel<2, false, false, false, true>
                               : nvfp4::gemv_tma_rv_kernel<1, false, false, false, true>;
      else
        kern = pl.k_split == 2 ? nvfp4::gemv_tma_rv_kernel<2, false, false>
                               : nvfp4::gemv_tma_rv_kernel<1, false, false>;
    }
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.gridDim = dim3((unsigned)(pl.ctas_per_batch * L * S));
    cfg.blockDim = dim3((unsigned)(threads + 32));
    cfg.dynamicSmemBytes = (size_t)t.total;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (!(pl.flags & NVFP4_FLAG_NO_PDL)) {
      attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[na].val.programmaticStreamSerializationAllowed = 1;
      ++na;
    }
    if (S > 1) {  // the S CTAs of a row range form one cluster (consecutive CTA indices)
      attr[na].id = cudaLaunchAttributeClusterDimension;
      attr[na].val.clusterDim.x = (unsigned)S;
      attr[na].val.clusterDim.y = 1;
      attr[na].val.clusterDim.z = 1;
      ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    const cudaError_t le = cudaLaunchKernelEx(&cfg, kern, a);
    if (le != cudaSuccess) return cuda_fail(le, "kernel launch");
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return NVFP4_OK;
}

int gemv_impl(const uint8_t* A, const uint8_t* sfa, float g_a, const uint8_t* b,
              const uint8_t* sfb, float g_b, uint16_t* c, int64_t M, int64_t K, int64_t L,
              void* stream, const nvfp4_plan* forced) {
  g_last_error[0] = '\0';
  bool noop = false, aligned16 = true;
  int st = check_args(A, sfa, b, sfb, c, M, K, L, &noop, &aligned16);
  if (st != NVFP4_OK || noop) return st;
  const DeviceInfo* d = nullptr;
  if ((st = current_device(&d)) != NVFP4_OK) return st;
  if ((st = check_access(*d, A, "A")) || (st = check_access(*d, sfa, "sfa")) ||
      (st = check_access(*d, b, "b")) || (st = check_access(*d, sfb, "sfb")) ||
      (st = check_access(*d, c, "c")))
    return st;
  if (forced && (forced->flags & NVFP4_FLAG_QUANTIZE_IN_GEMV))
    return fail(NVFP4_ERR_INVALID_VALUE, "NVFP4_FLAG_QUANTIZE_IN_GEMV needs a bf16 vector");
  nvfp4_plan pl;
  if ((st = make_plan(*d, M, K, L, forced, &pl, aligned16, matrix_aligned16(A, sfa))) != NVFP4_OK)
    return st;
  return launch(*d, pl, A, sfa, g_a, b, sfb, g_b, c, M, K, L, (cudaStream_t)stream);
}

// ---------------------------------------------------------------- activation quantization
int check_quant_args(const uint16_t* x, float gs, const uint8_t* b, const uint8_t* sfb,
                     int64_t K, int64_t L, int rounding, bool* noop) {
  *noop = false;
  if (K <= 0 || L < 0 || K % 16)
    return fail(NVFP4_ERR_INVALID_VALUE, "need K > 0, K %% 16 == 0, L >= 0 (K=%lld L=%lld)",
                (long long)K, (long long)L);
  if (rounding != NVFP4_ROUND_HALF_STEP_TABLE && rounding != NVFP4_ROUND_NEAREST_EVEN)
    return fail(NVFP4_ERR_INVALID_VALUE, "unknown rounding %d", rounding);
  if (!(gs > 0.f) || !std::isfinite(gs))
    return fail(NVFP4_ERR_INVALID_VALUE, "the global scale must be finite and > 0 (%g)", (double)gs);
  const int64_t kMax = (int64_t(1) << 31) - 1;
  if (L > kMax || K > kMax) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "L and K must be below 2^31");
  if (L == 0) {
    *noop = true;
    return NVFP4_OK;
  }
  if (!x || !b || !sfb) return fail(NVFP4_ERR_INVALID_VALUE, "NULL pointer");
  if (((uintptr_t)x | (uintptr_t)b | (uintptr_t)sfb) & 15u)
    return fail(NVFP4_ERR_MISALIGNED, "x, b and sfb must be 16-byte aligned");
  const int64_t nx = 2 * L * K, nb = L * K / 2, ns = L * K / 16;
  if (overlaps(x, nx, b, nb) || overlaps(x, nx, sfb, ns) || overlaps(b, nb, sfb, ns))
    return fail(NVFP4_ERR_INVALID_VALUE, "x, b and sfb must not overlap");
  return NVFP4_OK;
}

int launch_quantize(const uint16_t* x, float gs, int rounding, uint8_t* b, uint8_t* sfb,
                    int64_t K, int64_t L, cudaStream_t stream, bool pdl) {
  const int64_t n_pairs = L * K / 2;
  const int64_t grid = ceil_div(n_pairs, 256);
  if (grid > (int64_t(1) << 31) - 1) return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "grid too large");
  cudaLaunchConfig_t cfg;
  memset(&cfg, 0, sizeof cfg);
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  const cudaError_t e =
      cudaLaunchKernelEx(&cfg, nvfp4::quantize_activation_kernel, x, gs, rounding, b, sfb, n_pairs);
  if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
  return NVFP4_OK;
}

int quantize_impl(const uint16_t* x, float gs, int rounding, uint8_t* b, uint8_t* sfb, int64_t K,
                  int64_t L, void* stream) {
  g_last_error[0] = '\0';
  bool noop = false;
  int st = check_quant_args(x, gs, b, sfb, K, L, rounding, &noop);
  if (st != NVFP4_OK || noop) return st;
  const DeviceInfo* d = nullptr;
  if ((st = current_device(&d)) != NVFP4_OK) return st;
  if ((st = check_access(*d, x, "x")) || (st = check_access(*d, b, "b")) ||
      (st = check_access(*d, sfb, "sfb")))
    return st;
  return launch_quantize(x, gs, rounding, b, sfb, K, L, (cudaStream_t)stream, true);
}

int gemv_bf16_impl(const uint8_t* A, const uint8_t* sfa, float g_a, const uint16_t* x, float x_gs,
                   int rounding, uint8_t* b_out, uint8_t* sfb_out, uint16_t* c, int64_t M,
                   int64_t K, int64_t L, void* stream, const nvfp4_plan* forced) {
  g_last_error[0] = '\0';
  bool noop = false, aligned16 = true;
  int st = check_args(A, sfa, b_out, sfb_out, c, M, K, L, &noop, &aligned16);
  if (st != NVFP4_OK || noop) return st;
  if ((st = check_quant_args(x, x_gs, b_out, sfb_out, K, L, rounding, &noop)) != NVFP4_OK)
    return st;
  const int64_t nx = 2 * L * K, nA = M * L * (K / 2), nSA = M * L * (K / 16), nC = 2 * M * L,
                nb = L * K / 2, ns = L * K / 16;
  if (overlaps(c, nC, x, nx) || overlaps(A, nA, b_out, nb) || overlaps(A, nA, sfb_out, ns) ||
      overlaps(sfa, nSA, b_out, nb) || overlaps(sfa, nSA, sfb_out, ns))
    return fail(NVFP4_ERR_INVALID_VALUE, "outputs overlap inputs");
  const DeviceInfo* d = nullptr;
  if ((st = current_device(&d)) != NVFP4_OK) return st;
  if ((st = check_access(*d, A, "A")) || (st = check_access(*d, sfa, "sfa")) ||
      (st = check_access(*d, x, "x")) || (st = check_access(*d, b_out, "b_out")) ||
      (st = check_access(*d, sfb_out, "sfb_out")) || (st = check_access(*d, c, "c")))
    return st;
  nvfp4_plan pl;
  if ((st = make_plan(*d, M, K, L, forced, &pl, aligned16, matrix_aligned16(A, sfa))) != NVFP4_OK)
    return st;
  if (pl.flags & NVFP4_FLAG_QUANTIZE_IN_GEMV) {  // quantize inside the GEMV's vector staging
    if (pl.kernel != NVFP4_KERNEL_TMA_RV)
      return fail(NVFP4_ERR_UNSUPPORTED_SHAPE,
                  "quantizing inside the GEMV needs the register-vector TMA kernel (plan kernel %d)",
                  pl.kernel);
    const FusedVector fx{x, x_gs, rounding, b_out, sfb_out};
    return launch(*d, pl, A, sfa, g_a, nullptr, nullptr, x_gs, c, M, K, L, (cudaStream_t)stream,
                  &fx);
  }
  // the quantizer first (it releases the GEMV at once: the GEMV can stream A meanwhile when the
  // weights are static), then the GEMV on the packed vector, in stream order
  if ((st = launch_quantize(x, x_gs, rounding, b_out, sfb_out, K, L, (cudaStream_t)stream,
                            !(pl.flags & NVFP4_FLAG_NO_PDL))))
    return st;
  return launch(*d, pl, A, sfa, g_a, b_out, sfb_out, x_gs, c, M, K, L, (cudaStream_t)stream);
}

// ---------------------------------------------------------------- grouped (mixture of experts)
constexpr int64_t kMaxExperts = 65536;

int grouped_impl(const uint8_t* A, const uint8_t* sfa, const float* g_a, const uint8_t* b,
                 const uint8_t* sfb, const float* g_b, const int32_t* offsets,
                 const int32_t* expert_of, uint16_t* c, int out_dtype, int64_t M, int64_t K,
                 int64_t E, int64_t T, void* stream, const nvfp4_plan* forced) {
  g_last_error[0] = '\0';
  if (E < 1 || E > kMaxExperts)
    return fail(E < 1 ? NVFP4_ERR_INVALID_VALUE : NVFP4_ERR_UNSUPPORTED_SHAPE,
                "need 1 <= E <= %lld experts (E=%lld)", (long long)kMaxExperts, (long long)E);
  if ((offsets == nullptr) == (expert_of == nullptr))
    return fail(NVFP4_ERR_INVALID_VALUE,
                "give exactly one of expert_offsets and expert_of_token");
  if (out_dtype != NVFP4_OUT_F16 && out_dtype != NVFP4_OUT_BF16)
    return fail(NVFP4_ERR_INVALID_VALUE, "unknown output type %d", out_dtype);
  if (forced && (forced->flags & (NVFP4_FLAG_EARLY_WEIGHTS | NVFP4_FLAG_QUANTIZE_IN_GEMV)))
    return fail(NVFP4_ERR_INVALID_VALUE,
                "the grouped form reads each token's expert after the launch wait: no early "
                "weights, no in-GEMV quantization");
  bool noop = false, aligned16 = true;
  int st = check_args(A, sfa, b, sfb, c, M, K, T, &noop, &aligned16, E);
  if (st != NVFP4_OK || noop) return st;
  if (!g_a || !g_b) return fail(NVFP4_ERR_INVALID_VALUE, "NULL global-scale array");
  const void* idx = offsets ? (const void*)offsets : (const void*)expert_of;
  if (((uintptr_t)g_a | (uintptr_t)g_b | (uintptr_t)idx) & 3u)
    return fail(NVFP4_ERR_MISALIGNED, "g_a, g_b and the expert indices must be 4-byte aligned");
  const int64_t nC = 2 * M * T, nIdx = 4 * (offsets ? E : T);
  if (overlaps(c, nC, g_a, 4 * E) || overlaps(c, nC, g_b, 4 * E) || overlaps(c, nC, idx, nIdx))
    return fail(NVFP4_ERR_INVALID_VALUE, "c overlaps an input");
  const DeviceInfo* d = nullptr;
  if ((st = current_device(&d)) != NVFP4_OK) return st;
  if ((st = check_access(*d, A, "A")) || (st = check_access(*d, sfa, "sfa")) ||
      (st = check_access(*d, b, "b")) || (st = check_access(*d, sfb, "sfb")) ||
      (st = check_access(*d, c, "c")) || (st = check_access(*d, g_a, "g_a")) ||
      (st = check_access(*d, g_b, "g_b")) || (st = check_access(*d, idx, "expert indices")))
    return st;
  nvfp4_plan pl;
  if ((st = make_plan(*d, M, K, T, forced, &pl, aligned16, matrix_aligned16(A, sfa))) != NVFP4_OK)
    return st;
  GroupedOut go;
  go.G.offsets = offsets;
  go.G.expert_of = expert_of;
  go.G.g_a = g_a;
  go.G.g_b = g_b;
  go.G.E = (int32_t)E;
  go.out_bf16 = out_dtype == NVFP4_OUT_BF16 ? 1 : 0;
  return launch(*d, pl, A, sfa, 1.f, b, sfb, 1.f, c, M, K, T, (cudaStream_t)stream, nullptr, &go);
}

// ---------------------------------------------------------------- small N (vectors share A)
int small_n_impl(const uint8_t* A, const uint8_t* sfa, float g_a, const uint8_t* b,
                 const uint8_t* sfb, float g_b, uint16_t* c, int64_t M, int64_t K, int64_t N,
                 void* stream, const nvfp4_plan* forced) {
  g_last_error[0] = '\0';
  bool noop = false, aligned16 = true;
  int st = check_args(A, sfa, b, sfb, c, M, K, N, &noop, &aligned16, 1);
  if (st != NVFP4_OK || noop) return st;
  if (forced && (forced->flags & NVFP4_FLAG_QUANTIZE_IN_GEMV))
    return fail(NVFP4_ERR_INVALID_VALUE, "NVFP4_FLAG_QUANTIZE_IN_GEMV needs a bf16 vector");
  const DeviceInfo* d = nullptr;
  if ((st = current_device(&d)) != NVFP4_OK) return st;
  if ((st = check_access(*d, A, "A")) || (st = check_access(*d, sfa, "sfa")) ||
      (st = check_access(*d, b, "b")) || (st = check_access(*d, sfb, "sfb")) ||
      (st = check_access(*d, c, "c")))
    return st;
  nvfp4_plan pl;
  memset(&pl, 0, sizeof pl);
  const bool automatic = !forced || forced->kernel == NVFP4_KERNEL_AUTO;
  bool tc = false;
  if (automatic && aligned16 && K % 256 == 0) {  // the tensor cores when they can take it
    nvfp4_plan f;
    memset(&f, 0, sizeof f);
    if (forced) f = *forced;
    f.kernel = NVFP4_KERNEL_TC;
    char saved[sizeof g_last_error];
    memcpy(saved, g_last_error, sizeof saved);
    tc = make_plan(*d, M, K, std::min<int64_t>(N, nvfp4::kTcCols), &f, &pl, true, true, 1) ==
         NVFP4_OK;
    memcpy(g_last_error, saved, sizeof saved);
  }
  if (!tc) {
    if ((st = make_plan(*d, M, K, N, forced, &pl, aligned16, matrix_aligned16(A, sfa), 1)) !=
        NVFP4_OK)
      return st;
    tc = pl.kernel == NVFP4_KERNEL_TC;
  }
  if (tc) {  // groups of up to 16 vectors, one launch each
    for (int64_t n0 = 0; n0 < N; n0 += nvfp4::kTcCols) {
      const int64_t n = std::min<int64_t>(nvfp4::kTcCols, N - n0);
      if ((st = launch_tc(*d, pl, A, sfa, g_a, b + n0 * (K / 2), sfb + n0 * (K / 16), g_b,
                          c + n0 * M, M, K, 1, n, 0, (cudaStream_t)stream)))
        return st;
    }
    return NVFP4_OK;
  }
  GroupedOut go;
  memset(&go, 0, sizeof go);
  go.G.shared_a = 1;
  return launch(*d, pl, A, sfa, g_a, b, sfb, g_b, c, M, K, N, (cudaStream_t)stream, nullptr, &go);
}

}  // namespace

extern "C" {

int nvfp4_gemm_small_n(const uint8_t* A, const uint8_t* sfa, float g_a, const uint8_t* b,
                       const uint8_t* sfb, float g_b, uint16_t* c, int64_t M, int64_t K, int64_t N,
                       void* stream, const nvfp4_plan* plan) {
  return small_n_impl(A, sfa, g_a, b, sfb, g_b, c, M, K, N, stream, plan);
}

int nvfp4_gemv_batched(const uint8_t* A, const uint8_t* sfa, float g_a, const uint8_t* b,
                       const uint8_t* sfb, float g_b, uint16_t* c, int64_t M, int64_t K, int64_t L,
                       void* stream) {
  return gemv_impl(A, sfa, g_a, b, sfb, g_b, c, M, K, L, stream, nullptr);
}

int nvfp4_gemv_grouped(const uint8_t* A, const uint8_t* sfa, const float* g_a, const uint8_t* b,
                       const uint8_t* sfb, const float* g_b, const int32_t* expert_offsets,
                       const int32_t* expert_of_token, uint16_t* c, int out_dtype, int64_t M,
                       int64_t K, int64_t E, int64_t T, void* stream, const nvfp4_plan* plan) {
  return grouped_impl(A, sfa, g_a, b, sfb, g_b, expert_offsets, expert_of_token, c, out_dtype, M,
                      K, E, T, stream, plan);
}

int nvfp4_gemv_batched_ex(const uint8_t* A, const uint8_t* sfa, float g_a, const uint8_t* b,
                          const uint8_t* sfb, float g_b, uint16_t* c, int64_t M, int64_t K,
                          int64_t L, void* stream, const nvfp4_plan* plan) {
  return gemv_impl(A, sfa, g_a, b, sfb, g_b, c, M, K, L, stream, plan);
}

int nvfp4_gemv_plan(int64_t M, int64_t K, int64_t L, nvfp4_plan* out) {
  g_last_error[0] = '\0';
  if (!out) return fail(NVFP4_ERR_INVALID_VALUE, "out is NULL");
  if (M <= 0 || L <= 0 || K <= 0 || K % 16)
    return fail(NVFP4_ERR_INVALID_VALUE, "need M, L > 0 and K a positive multiple of 16");
  const DeviceInfo* d = nullptr;
  int st = current_device(&d);
  if (st != NVFP4_OK) return st;
  return make_plan(*d, M, K, L, nullptr, out, true, true);
}

int nvfp4_plan_for_limits(const nvfp4_device_limits* lim, int64_t M, int64_t K, int64_t L,
                          const nvfp4_plan* forced, nvfp4_plan* out) {
  g_last_error[0] = '\0';
  if (!lim || !out) return fail(NVFP4_ERR_INVALID_VALUE, "lim and out must not be NULL");
  if (lim->sms < 1 || lim->max_smem_optin < 1024 || lim->max_smem_sm < lim->max_smem_optin)
    return fail(NVFP4_ERR_INVALID_VALUE, "implausible device limits (sms %d, smem %d / %d)",
                lim->sms, lim->max_smem_optin, lim->max_smem_sm);
  if (M <= 0 || L <= 0 || K <= 0 || K % 16)
    return fail(NVFP4_ERR_INVALID_VALUE, "need M, L > 0 and K a positive multiple of 16");
  const int64_t kI32 = (int64_t(1) << 31) - 1;
  if (M > kI32 || L > kI32 || K / 2 > kI32)
    return fail(NVFP4_ERR_UNSUPPORTED_SHAPE, "M, L and K/2 must be below 2^31");
  DeviceInfo d;
  d.sms = lim->sms;
  d.max_smem_optin = lim->max_smem_optin;
  d.max_smem_sm = lim->max_smem_sm;
  return make_plan(d, M, K, L, forced, out, true, true);
}

int64_t nvfp4_max_stream_k(void) {
  const DeviceInfo* d = nullptr;
  if (current_device(&d) != NVFP4_OK) return 0;
  return max_stream_k(*d);
}

const char* nvfp4_status_string(int status) {
  switch (status) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID_VALUE: return "invalid value";
    case NVFP4_ERR_MISALIGNED: return "misaligned pointer";
    case NVFP4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape or plan";
    case NVFP4_ERR_ARCH: return "unsupported device architecture";
    case NVFP4_ERR_CUDA: return "CUDA error";
    default: return "unknown status";
  }
}

const char* nvfp4_last_error(void) { return g_last_error; }

int nvfp4_quantize_activation(const uint16_t* x, float global_scale, int rounding, uint8_t* b,
                              uint8_t* sfb, int64_t K, int64_t L, void* stream) {
  return quantize_impl(x, global_scale, rounding, b, sfb, K, L, stream);
}

int nvfp4_gemv_batched_bf16(const uint8_t* A, const uint8_t* sfa, float g_a, const uint16_t* x,
                            float x_global_scale, int rounding, uint8_t* b_out, uint8_t* sfb_out,
                            uint16_t* c, int64_t M, int64_t K, int64_t L, void* stream,
                            const nvfp4_plan* plan) {
  return gemv_bf16_impl(A, sfa, g_a, x, x_global_scale, rounding, b_out, sfb_out, c, M, K, L,
                        stream, plan);
}

int nvfp4_abi_version(void) { return NVFP4_ABI_VERSION; }

}  // extern "C"

/*
 * nvfp4_ref.c -- the NVFP4 block-scaled batched GEMV and its neighbours, written out as plain C
 * from their definitions, in fp64 (fp32 where the definition itself works in fp32).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU legs of the benchmark
 * load this library (through oracle/cref.py).  It shares no code, header, table or constant with
 * the CUDA library; the two meet only in the seeded input generator, which draws bytes.
 *
 * Sources (web pages, by title):
 *   [Blog]   "nvFP4 Batch GEMV算子系列(下)": section "NVFP4 Batched GEMV 概念阐述" (16-element blocks
 *            share one FP8 scale, one fp32 global scale per operand multiplies the result, floor(k/16)
 *            is the block id of element k; the formula image is lost, its written form is used),
 *            section "准备数据" (block scales are float8_e4m3fn; fp16 output).
 *   [Bridge] cutedsl/bridge.py (nvfp4-megamoe-kernel): section "Constants" (E2M1_MAGNITUDES
 *            0, 0.5, 1, 1.5, 2, 3, 4, 6), section "Quantization" (packed = (odd << 4) | even;
 *            quantize_activation_nvfp4), "compute_expert_offsets" and "Kernel Launch" (grouped).
 *
 * Built with plain gcc (-O2 -ffp-contract=off, no fast-math, OpenMP when available).  Every sum
 * runs in the order the definition states; OpenMP only distributes whole output rows, so the
 * result does not depend on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ element decoders */

/* E2M1: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.  e == 0 is the subnormal range
 * 0.5 * m; otherwise 2^(e-1) * (1 + m/2).  ([Bridge] "Constants" prints the magnitudes in code
 * order; the tests check this closed form against that list.) */
double nv_e2m1(unsigned code) {
  const unsigned e = (code >> 1) & 3u, m = code & 1u;
  const double mag = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, (int)e - 1);
  return (code & 8u) ? -mag : mag;
}

/* E4M3FN (torch.float8_e4m3fn, [Blog] "准备数据"): sign bit 7, exponent bits 6..3 (bias 7),
 * mantissa bits 2..0.  E == 0: m * 2^-9; otherwise 2^(E-7) * (1 + m/8).  S.1111.111 is NaN and
 * there is no infinity. */
double nv_e4m3(unsigned byte) {
  const unsigned E = (byte >> 3) & 15u, m = byte & 7u;
  if (E == 15u && m == 7u) return NAN;
  const double mag = E == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, (int)E - 7);
  return (byte & 0x80u) ? -mag : mag;
}

static double E2M1_VAL[16];
static double E4M3_VAL[256];
static int tables_ready = 0;

static void init_tables(void) {
  if (tables_ready) return;
  for (unsigned c = 0; c < 16; ++c) E2M1_VAL[c] = nv_e2m1(c);
  for (unsigned v = 0; v < 256; ++v) E4M3_VAL[v] = nv_e4m3(v);
  tables_ready = 1;
}

/* Code of element k of a packed row: the even k in the low nibble ([Bridge] "Quantization"). */
static unsigned nibble(const uint8_t* row, int64_t k) {
  const uint8_t byte = row[k >> 1];
  return (k & 1) ? (unsigned)(byte >> 4) : (unsigned)(byte & 15u);
}

/* ------------------------------------------------------------------------ the GEMV */

/* One output of batch l, row m:
 *   S = sum_{k<K} e2m1(A[l][m][k]) e2m1(b[l][k]) e4m3(sfa[l][m][k/16]) e4m3(sfb[l][k/16]),
 * a running fp64 sum in increasing k (each term is exact in fp64), and sum_k |term|.
 * Layouts: A [L][M][K/2], sfa [L][M][K/16], b [L][K/2], sfb [L][K/16]. */
static void one_row(const uint8_t* A, const uint8_t* sfa, const uint8_t* b, const uint8_t* sfb,
                    int64_t M, int64_t K, int64_t l, int64_t m, double* S_out, double* T_out) {
  const uint8_t* a_row = A + (l * M + m) * (K / 2);
  const uint8_t* sa_row = sfa + (l * M + m) * (K / 16);
  const uint8_t* b_row = b + l * (K / 2);
  const uint8_t* sb_row = sfb + l * (K / 16);
  double S = 0.0, T = 0.0;
  for (int64_t k = 0; k < K; ++k) {
    const double term = E2M1_VAL[nibble(a_row, k)] * E4M3_VAL[sa_row[k / 16]] *
                        E2M1_VAL[nibble(b_row, k)] * E4M3_VAL[sb_row[k / 16]];
    S += term;
    T += fabs(term);
  }
  *S_out = S;
  *T_out = T;
}

/* c_ref[i] = (S * g_a) * g_b and T[i] = sum_k |term_k| * |g_a * g_b| at the outputs
 * (ls[i], ms[i]), i < n (the global scales are fp32 values widened exactly).  threads <= 0: all
 * the OpenMP threads.  Returns 0, or -1 for an index outside [0, L) x [0, M). */
int nv_gemv_rows(const uint8_t* A, const uint8_t* sfa, float g_a, const uint8_t* b,
                 const uint8_t* sfb, float g_b, int64_t M, int64_t K, int64_t L,
                 const int64_t* ls, const int64_t* ms, int64_t n, double* c_ref, double* T,
                 int threads) {
  init_tables();
  for (int64_t i = 0; i < n; ++i)
    if (ls[i] < 0 || ls[i] >= L || ms[i] < 0 || ms[i] >= M) return -1;
  const double ga = (double)g_a, gb = (double)g_b, gg = fabs(ga * gb);
#ifdef _OPENMP
  const int nt = threads > 0 ? threads : omp_get_max_threads();
#pragma omp parallel for num_threads(nt) schedule(dynamic, 4)
#endif
  for (int64_t i = 0; i < n; ++i) {
    double S, T0;
    one_row(A, sfa, b, sfb, M, K, ls[i], ms[i], &S, &T0);
    c_ref[i] = (S * ga) * gb;
    T[i] = T0 * gg;
  }
  (void)threads;
  return 0;
}

/* Every output, c_ref and T as [L][M]. */
int nv_gemv(const uint8_t* A, const uint8_t* sfa, float g_a, const uint8_t* b, const uint8_t* sfb,
            float g_b, int64_t M, int64_t K, int64_t L, double* c_ref, double* T, int threads) {
  init_tables();
  const double ga = (double)g_a, gb = (double)g_b, gg = fabs(ga * gb);
#ifdef _OPENMP
  const int nt = threads > 0 ? threads : omp_get_max_threads();
#pragma omp parallel for num_threads(nt) schedule(dynamic, 4)
#endif
  for (int64_t i = 0; i < L * M; ++i) {
    double S, T0;
    one_row(A, sfa, b, sfb, M, K, i / M, i % M, &S, &T0);
    c_ref[i] = (S * ga) * gb;
    T[i] = T0 * gg;
  }
  (void)threads;
  return 0;
}

/* ------------------------------------------------------------------------ exact integer sums */

/* A second formulation in integers only.  E2M1 in half units: 2 * value = m for e == 0, else
 * (2 + m) << (e - 1).  E4M3 in units of 2^-9: m for E == 0, else (8 + m) << (E - 1).  A term in
 * units of 2^-20 is (2a)(2b)(2^9 sa)(2^9 sb), exact in int64; so is the sum while K < 2^20. */
static int64_t half_units(unsigned code) {
  const unsigned e = (code >> 1) & 3u, m = code & 1u;
  const int64_t mag = e == 0 ? (int64_t)m : (int64_t)(2u + m) << (e - 1u);
  return (code & 8u) ? -mag : mag;
}

static int scale_units(unsigned byte, int64_t* out) {
  const unsigned E = (byte >> 3) & 15u, m = byte & 7u;
  if (E == 15u && m == 7u) return 0; /* NaN: no integer */
  const int64_t mag = E == 0 ? (int64_t)m : (int64_t)(8u + m) << (E - 1u);
  *out = (byte & 0x80u) ? -mag : mag;
  return 1;
}

/* units[i]: the exact sum S at (ls[i], ms[i]) in units of 2^-20; nan[i] = 1 (units 0) when the
 * row or the vector uses a NaN scale byte.  Returns -1 for a bad index or K >= 2^20. */
int nv_gemv_exact_units(const uint8_t* A, const uint8_t* sfa, const uint8_t* b, const uint8_t* sfb,
                        int64_t M, int64_t K, int64_t L, const int64_t* ls, const int64_t* ms,
                        int64_t n, int64_t* units, uint8_t* nan_out, int threads) {
  if (K >= ((int64_t)1 << 20)) return -1;
  for (int64_t i = 0; i < n; ++i)
    if (ls[i] < 0 || ls[i] >= L || ms[i] < 0 || ms[i] >= M) return -1;
#ifdef _OPENMP
  const int nt = threads > 0 ? threads : omp_get_max_threads();
#pragma omp parallel for num_threads(nt) schedule(dynamic, 4)
#endif
  for (int64_t i = 0; i < n; ++i) {
    const int64_t l = ls[i], m = ms[i];
    const uint8_t* a_row = A + (l * M + m) * (K / 2);
    const uint8_t* sa_row = sfa + (l * M + m) * (K / 16);
    const uint8_t* b_row = b + l * (K / 2);
    const uint8_t* sb_row = sfb + l * (K / 16);
    int64_t sum = 0;
    int is_nan = 0;
    for (int64_t j = 0; j < K / 16; ++j) {
      int64_t sa = 0, sb = 0;
      if (!scale_units(sa_row[j], &sa) || !scale_units(sb_row[j], &sb)) {
        is_nan = 1; /* a NaN scale of the row or of the vector: the output has no integer sum */
        break;
      }
      for (int64_t k = 16 * j; k < 16 * j + 16; ++k)
        sum += half_units(nibble(a_row, k)) * half_units(nibble(b_row, k)) * sa * sb;
    }
    units[i] = is_nan ? 0 : sum;
    nan_out[i] = (uint8_t)is_nan;
  }
  (void)threads;
  return 0;
}

/* ------------------------------------------------------------------------ grouped (MoE) form */

/* Owner of each token 0..T-1 under the bridge's inclusive cumulative offsets ("compute_expert_offsets":
 * tokens sorted by expert, offsets[e] = tokens of experts 0..e), so expert e owns
 * offsets[e-1] <= t < offsets[e] (offsets[-1] read as 0); the first expert to claim a token owns
 * it; -1 for a token that no range covers. */
void nv_experts_from_offsets(const int32_t* offsets, int64_t E, int64_t T, int64_t* owner) {
  for (int64_t t = 0; t < T; ++t) owner[t] = -1;
  for (int64_t e = 0; e < E; ++e) {
    int64_t start = e > 0 ? offsets[e - 1] : 0, end = offsets[e];
    if (start < 0) start = 0;
    if (end > T) end = T;
    for (int64_t t = start; t < end; ++t)
      if (owner[t] < 0) owner[t] = e;
  }
}

/* c_ref[t][m] and T[t][m] ([T][M]) for tokens t with owner e = owner[t] >= 0: the GEMV of expert
 * e's matrix (A [E][M][K/2], sfa [E][M][K/16]) with the token's vector (b [T][K/2],
 * sfb [T][K/16]) and the expert's global scales g_a[e], g_b[e] ([Bridge] "Kernel Launch");
 * zeros for a token without an owner (the bridge's output starts as zeros). */
int nv_gemv_grouped(const uint8_t* A, const uint8_t* sfa, const float* g_a, const uint8_t* b,
                    const uint8_t* sfb, const float* g_b, const int64_t* owner, int64_t M,
                    int64_t K, int64_t E, int64_t T, double* c_ref, double* Tb, int threads) {
  init_tables();
  for (int64_t t = 0; t < T; ++t)
    if (owner[t] >= E) return -1;
#ifdef _OPENMP
  const int nt = threads > 0 ? threads : omp_get_max_threads();
#pragma omp parallel for num_threads(nt) schedule(dynamic, 4)
#endif
  for (int64_t i = 0; i < T * M; ++i) {
    const int64_t t = i / M, m = i % M, e = owner[t];
    if (e < 0) {
      c_ref[i] = 0.0;
      Tb[i] = 0.0;
      continue;
    }
    /* expert e's matrix as batch 0 of a one-batch problem, the token's vector as its vector */
    double S, T0;
    one_row(A + e * M * (K / 2), sfa + e * M * (K / 16), b + t * (K / 2), sfb + t * (K / 16), M,
            K, 0, m, &S, &T0);
    const double ga = (double)g_a[e], gb = (double)g_b[e];
    c_ref[i] = (S * ga) * gb;
    Tb[i] = T0 * fabs(ga * gb);
  }
  (void)threads;
  return 0;
}

/* ------------------------------------------------------------------------ activation quantizer */

/* The E4M3FN byte nearest to a non-negative fp32 value v, ties to the even byte, as torch's
 * float -> float8_e4m3fn cast gives: a value that rounds past the largest finite magnitude (448,
 * i.e. v > 464) has no finite encoding and becomes NaN (0x7F). */
static uint8_t e4m3_nearest(float v) {
  if (!(v == v)) return 0x7Fu;
  if (v > 464.0f) return 0x7Fu;
  uint8_t best = 0;
  double best_d = INFINITY;
  for (unsigned byte = 0; byte < 0x7Fu; ++byte) {
    const double d = fabs(E4M3_VAL[byte] - (double)v);
    if (d < best_d || (d == best_d && (byte & 1u) == 0)) {
      best = (uint8_t)byte;
      best_d = d;
    }
  }
  return best;
}

/* E2M1 magnitude code for a magnitude in [0, 6]:
 *   rounding 0: the page's half-step table, table[rint(2 * mag)] with
 *               table = 0,1,2,3,4,4,5,5,6,6,6,7,7 ([Bridge] "Quantization");
 *   rounding 1: the nearest E2M1 magnitude, ties to the even code. */
static unsigned e2m1_magnitude_code(float mag, int rounding) {
  if (rounding == 0) {
    static const unsigned table[13] = {0, 1, 2, 3, 4, 4, 5, 5, 6, 6, 6, 7, 7};
    float h = rintf(2.0f * mag);
    if (h < 0.0f) h = 0.0f;
    if (h > 12.0f) h = 12.0f;
    return table[(int)h];
  }
  unsigned best = 0;
  float best_d = INFINITY;
  for (unsigned c = 0; c < 8; ++c) {
    const float d = fabsf(mag - (float)E2M1_VAL[c]);
    if (d < best_d || (d == best_d && (c & 1u) == 0)) {
      best = c;
      best_d = d;
    }
  }
  return best;
}

/* quantize_activation_nvfp4 with a fixed global scale gs ([Bridge] "Quantization"): each
 * 16-element block of x ([L][K] fp32 holding bf16 values) is quantized on its own:
 *   the block scale is the E4M3 rounding of max(max_k |x_k / gs|, 1e-8) / 6;
 *   each element's code is the E2M1 rounding of min(|(x_k / gs) / max(scale, 1e-8)|, 6) with the
 *   sign of that quotient,
 * every operation in fp32 with IEEE division (the page's torch ops).  Reading for the case the
 * page leaves open: a block whose scale is NaN (its amax rounds past 448) gets the codes 0, since
 * the page's table lookup has no index for a NaN.  Output: packed [L][K/2] ((odd << 4) | even),
 * scales [L][K/16].  Returns -1 if K % 16 != 0. */
int nv_quantize_activation(const float* x, float gs, int rounding, int64_t K, int64_t L,
                           uint8_t* packed, uint8_t* scales) {
  init_tables();
  if (K % 16 != 0 || (rounding != 0 && rounding != 1)) return -1;
  for (int64_t blk = 0; blk < L * (K / 16); ++blk) {
    const float* xb = x + 16 * blk;
    float xn[16], amax = 0.0f;
    for (int i = 0; i < 16; ++i) {
      xn[i] = xb[i] / gs;
      if (fabsf(xn[i]) > amax) amax = fabsf(xn[i]);
    }
    if (amax < 1e-8f) amax = 1e-8f;
    const uint8_t sbyte = e4m3_nearest(amax / 6.0f);
    scales[blk] = sbyte;
    uint8_t* out = packed + 8 * blk;
    if (sbyte == 0x7Fu) {
      memset(out, 0, 8);
      continue;
    }
    float d = (float)E4M3_VAL[sbyte];
    if (d < 1e-8f) d = 1e-8f;
    for (int i = 0; i < 16; i += 2) {
      unsigned nib[2];
      for (int h = 0; h < 2; ++h) {
        const float xs = xn[i + h] / d;
        float mag = fabsf(xs);
        if (mag > 6.0f) mag = 6.0f;
        nib[h] = e2m1_magnitude_code(mag, rounding) | (xs < 0.0f ? 8u : 0u);
      }
      out[i / 2] = (uint8_t)(nib[0] | (nib[1] << 4));
    }
  }
  return 0;
}

/* ------------------------------------------------------------------------ fp16 rounding */

/* IEEE binary16 bits of x rounded to nearest, ties to even, straight from fp64; overflow to
 * +-inf, gradual underflow; NaN -> 0x7E00. */
uint16_t nv_fp16_bits(double x) {
  if (x != x) return 0x7E00u;
  const uint16_t sign = signbit(x) ? 0x8000u : 0u;
  const double a = fabs(x);
  if (a >= 65520.0) return sign | 0x7C00u; /* at or past the midpoint 65504 .. 65536 */
  if (a < ldexp(1.0, -14)) {                /* subnormal: multiples of 2^-24 */
    const double q = rint(ldexp(a, 24));    /* exact scaling, then round half to even */
    return sign | (uint16_t)q;              /* q == 1024 is the smallest normal, bits 0x0400 */
  }
  int E;
  frexp(a, &E);                             /* a = f 2^E, f in [0.5, 1) */
  int e = E - 1;                            /* a = (1 + frac) 2^e */
  double q = rint((ldexp(a, -e) - 1.0) * 1024.0);
  if (q == 1024.0) {
    q = 0.0;
    ++e;
  }
  if (e + 15 >= 31) return sign | 0x7C00u;
  return sign | (uint16_t)(((e + 15) << 10) | (int)q);
}

void nv_fp16_bits_array(const double* x, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = nv_fp16_bits(x[i]);
}

/* ------------------------------------------------------------------------ build facts */

/* Threads an OpenMP region would use by default (1 without OpenMP). */
int nv_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

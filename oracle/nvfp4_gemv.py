"""The NVFP4 block-scaled batched GEMV, written out as its definition, in fp64.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Definition ("nvFP4 Batch GEMV算子系列(下)", section "NVFP4 Batched GEMV 概念阐述": each block of
16 consecutive K elements shares one FP8 scale, a single fp32 global scale multiplies the result,
and floor(k/16) is the block id of element k; the formula image on that page is lost, so its
written form is taken as)

    c[l][m] = g_a * g_b * sum_{k<K} e2m1(A[l][m][k]) * e2m1(b[l][k])
                                    * e4m3(sfa[l][m][k//16]) * e4m3(sfb[l][k//16])

Layouts (all C-contiguous, K fastest; the page's "准备数据" section builds the same tensors as
(l, m, k//2) uint8 for A, (l, n, k//2) for b with n = 1, and (l, mn, k//16) for the scales):

    A   uint8 [L][M][K/2]   two E2M1 codes per byte, even k in the low nibble
    sfa uint8 [L][M][K/16]  E4M3FN bytes
    b   uint8 [L][K/2]
    sfb uint8 [L][K/16]
    c   [L][M]              fp16 on the GPU; here unrounded fp64 plus its binary16 rounding

``gemv`` accumulates in fp64 in increasing k (``np.cumsum`` is a sequential running sum).
``gemv_exact_units`` is a second, independent formulation in integers: every term is an integer
multiple of 2**-20, so the sum is computed exactly in int64 units of 2**-20.  Wherever the fp64
sum is itself exact (every input the tests and the bench use), the two agree bit for bit.
"""
from __future__ import annotations

import numpy as np

from .codecs import E2M1_TABLE, E4M3FN_TABLE, fp16_round, unpack_e2m1_codes

BLOCK = 16  # K elements per scale block (sf_vec_size in the blog's data preparation)

# Rows are processed in chunks so that one fp64 temporary stays near 32 MiB.
_CHUNK_ELEMS = 1 << 22


def _as_layout(A, sfa, b, sfb, M, K, L):
    if K % BLOCK:
        raise ValueError("K must be a multiple of 16")
    A = np.asarray(A, dtype=np.uint8).reshape(L, M, K // 2)
    sfa = np.asarray(sfa, dtype=np.uint8).reshape(L, M, K // BLOCK)
    b = np.asarray(b, dtype=np.uint8).reshape(L, K // 2)
    sfb = np.asarray(sfb, dtype=np.uint8).reshape(L, K // BLOCK)
    return A, sfa, b, sfb


def _vector_terms(b_l: np.ndarray, sfb_l: np.ndarray) -> np.ndarray:
    """e2m1(b[k]) * e4m3(sfb[k//16]) for one batch, fp64 [K] (exact: <= 6 significant bits)."""
    b_val = E2M1_TABLE[unpack_e2m1_codes(b_l)]
    sb = np.repeat(E4M3FN_TABLE[sfb_l], BLOCK)
    return b_val * sb


def _row_terms(A_rows: np.ndarray, sfa_rows: np.ndarray, bterm: np.ndarray) -> np.ndarray:
    """Every product term of a set of rows, fp64 [rows][K] (each term is exact in fp64)."""
    a_val = E2M1_TABLE[unpack_e2m1_codes(A_rows)]
    sa = np.repeat(E4M3FN_TABLE[sfa_rows], BLOCK, axis=-1)
    return a_val * sa * bterm


def _sum_rows(A_rows, sfa_rows, bterm):
    """(S, T0): the running fp64 sum over increasing k, and sum_k |term|."""
    with np.errstate(invalid="ignore"):
        terms = _row_terms(A_rows, sfa_rows, bterm)
        S = np.cumsum(terms, axis=-1)[..., -1]
        T0 = np.cumsum(np.abs(terms), axis=-1)[..., -1]
    return S, T0


def gemv(A, sfa, g_a, b, sfb, g_b, M: int, K: int, L: int):
    """Full batched GEMV.

    Returns ``(c_ref, T)``, both fp64 ``[L][M]``:
      c_ref = (S * g_a) * g_b with S the fp64 sum above (not rounded to fp16);
      T     = sum_k |term_k| * |g_a * g_b|, the scale the parity tolerance is stated against.
    ``g_a`` and ``g_b`` are taken as fp32 values (one global scale per operand) and widened exactly.
    """
    A, sfa, b, sfb = _as_layout(A, sfa, b, sfb, M, K, L)
    ga = float(np.float32(g_a))
    gb = float(np.float32(g_b))
    c_ref = np.empty((L, M), dtype=np.float64)
    T = np.empty((L, M), dtype=np.float64)
    rows_per_chunk = max(1, _CHUNK_ELEMS // max(K, 1))
    for l in range(L):
        bterm = _vector_terms(b[l], sfb[l])
        for m0 in range(0, M, rows_per_chunk):
            m1 = min(M, m0 + rows_per_chunk)
            S, T0 = _sum_rows(A[l, m0:m1], sfa[l, m0:m1], bterm)
            c_ref[l, m0:m1] = (S * ga) * gb
            T[l, m0:m1] = T0 * abs(ga * gb)
    return c_ref, T


def gemv_rows(A, sfa, g_a, b, sfb, g_b, M: int, K: int, L: int, ls, ms):
    """The same definition, evaluated only at the outputs (ls[i], ms[i]).

    Used to check full-size launches on a sample of outputs.  Returns ``(c_ref, T)`` as fp64
    vectors aligned with ``ls``/``ms``.
    """
    A, sfa, b, sfb = _as_layout(A, sfa, b, sfb, M, K, L)
    ls = np.asarray(ls, dtype=np.int64)
    ms = np.asarray(ms, dtype=np.int64)
    ga = float(np.float32(g_a))
    gb = float(np.float32(g_b))
    c_ref = np.empty(ls.shape, dtype=np.float64)
    T = np.empty(ls.shape, dtype=np.float64)
    for l in np.unique(ls):
        sel = np.nonzero(ls == l)[0]
        bterm = _vector_terms(b[l], sfb[l])
        S, T0 = _sum_rows(A[l, ms[sel]], sfa[l, ms[sel]], bterm)
        c_ref[sel] = (S * ga) * gb
        T[sel] = T0 * abs(ga * gb)
    return c_ref, T


def gemv_fp16(A, sfa, g_a, b, sfb, g_b, M, K, L) -> np.ndarray:
    """``gemv`` followed by round-to-nearest-even to binary16 (for reporting and fixtures)."""
    c_ref, _ = gemv(A, sfa, g_a, b, sfb, g_b, M, K, L)
    return fp16_round(c_ref)


# ---------------------------------------------------------------------------------------------
# Independent exact formulation (integers only).
#
# E2M1 in half units: 2 * value for codes 0..7 is 0, 1, 2, 3, 4, 6, 8, 12 (exponent bits e, mantissa
# bit m: e == 0 -> m, else (2 + m) << (e - 1)); bit 3 negates.
# E4M3FN in units of 2**-9: E == 0 -> m; else (8 + m) << (E - 1); 0x7F/0xFF are NaN (no integer).
# term_units = (2a)(2b)(2**9 sa)(2**9 sb) = term * 2**20.
# ---------------------------------------------------------------------------------------------

def _e2m1_half_units(code: int) -> int:
    e = (code >> 1) & 0x3
    m = code & 0x1
    mag = m if e == 0 else (2 + m) << (e - 1)
    return -mag if code & 0x8 else mag


def _e4m3_units(byte: int):
    E = (byte >> 3) & 0xF
    m = byte & 0x7
    if E == 0xF and m == 0x7:
        return None
    mag = m if E == 0 else (8 + m) << (E - 1)
    return -mag if byte & 0x80 else mag


_E2M1_HALF_UNITS = np.array([_e2m1_half_units(c) for c in range(16)], dtype=np.int64)
_E4M3_UNITS = np.array([_e4m3_units(v) or 0 for v in range(256)], dtype=np.int64)
_E4M3_IS_NAN = np.array([_e4m3_units(v) is None for v in range(256)], dtype=bool)

TERM_UNIT_EXP = -20  # one integer unit of a term is 2**-20


def gemv_exact_units(A, sfa, b, sfb, M: int, K: int, L: int, ls=None, ms=None):
    """Exact sum S in int64 units of 2**-20 (no global scales), plus a NaN mask.

    Evaluated for all outputs, or for the sample (ls, ms).  Rows that use a NaN scale byte have
    no integer sum: their mask entry is True and their units entry 0.  Valid while
    K * 12 * 12 * 229376**2 < 2**63, i.e. K < 2**20.
    """
    A, sfa, b, sfb = _as_layout(A, sfa, b, sfb, M, K, L)
    if K >= (1 << 20):
        raise ValueError("exact checker supports K < 2**20")
    if ls is None:
        ls, ms = np.divmod(np.arange(L * M, dtype=np.int64), M)
    ls = np.asarray(ls, dtype=np.int64)
    ms = np.asarray(ms, dtype=np.int64)
    units = np.zeros(ls.shape, dtype=np.int64)
    nan = np.zeros(ls.shape, dtype=bool)
    codes_per_row = max(1, _CHUNK_ELEMS // max(K, 1))
    for l in np.unique(ls):
        bu = _E2M1_HALF_UNITS[unpack_e2m1_codes(b[l])]
        sbu = _E4M3_UNITS[sfb[l]]
        b_nan = bool(_E4M3_IS_NAN[sfb[l]].any())
        sel_all = np.nonzero(ls == l)[0]
        for i0 in range(0, len(sel_all), codes_per_row):
            sel = sel_all[i0:i0 + codes_per_row]
            rows = ms[sel]
            au = _E2M1_HALF_UNITS[unpack_e2m1_codes(A[l, rows])]
            sau = _E4M3_UNITS[sfa[l, rows]]
            # per block: scale product (exact int), per element: code product (exact int)
            scale = np.repeat(sau * sbu[None, :], BLOCK, axis=-1)
            units[sel] = (au * bu[None, :] * scale).sum(axis=-1)
            nan[sel] = _E4M3_IS_NAN[sfa[l, rows]].any(axis=-1) | b_nan
    units[nan] = 0
    return units, nan

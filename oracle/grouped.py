"""Grouped (mixture-of-experts) NVFP4 decode GEMV, by its definition.  TEST INFRASTRUCTURE ONLY.

cutedsl/bridge.py (nvfp4-megamoe-kernel):
* "compute_expert_offsets": with the tokens sorted by expert, offsets[e] is the number of tokens
  of experts 0..e, so expert e owns the tokens t with offsets[e-1] <= t < offsets[e] (offsets[-1]
  read as 0);
* "Kernel Launch", run_nvfp4_grouped_gemm: the tokens (rows of the 2-D operand) times the 3-D
  expert operand, with one fp32 global scale per expert on each side.
flashinfer, group_deepgemm_fp8_nt_groupwise: ``m_indices`` names the group of each row directly.

Per token t owned by expert e, c[t] is the batched GEMV definition (``oracle.gemv``) applied to
expert e's matrix A[e], sfa[e] with global scale g_a[e] and to the token's vector b[t], sfb[t]
with global scale g_b[e].  A token that no expert owns gets zeros: the bridge allocates its output
filled with zeros and writes only the experts' token ranges.

Pinned by tests/test_oracle_grouped.py.
"""
from __future__ import annotations

import numpy as np

from .nvfp4_gemv import gemv, gemv_rows


def experts_from_offsets(offsets, T: int) -> np.ndarray:
    """Owner of each token 0..T-1 under inclusive cumulative offsets, or -1."""
    offsets = [int(v) for v in np.asarray(offsets).ravel()]
    owner = np.full(T, -1, dtype=np.int64)
    for e, end in enumerate(offsets):
        start = offsets[e - 1] if e > 0 else 0
        for t in range(max(start, 0), min(end, T)):
            if owner[t] < 0:
                owner[t] = e
    return owner


def experts_from_map(expert_of, E: int) -> np.ndarray:
    """Owner of each token from a per-token expert index; indices outside [0, E) own nothing."""
    e = np.asarray(expert_of, dtype=np.int64).ravel()
    return np.where((e >= 0) & (e < E), e, -1)


def gemv_grouped(A, sfa, g_a, b, sfb, g_b, experts, M: int, K: int):
    """A [E][M][K/2], sfa [E][M][K/16], g_a/g_b [E] (fp32 values), b [T][K/2], sfb [T][K/16],
    experts [T] (owner or -1).  Returns (c_ref, T_bound), fp64 [T][M], unrounded."""
    experts = np.asarray(experts, dtype=np.int64).ravel()
    T = len(experts)
    E = len(np.asarray(g_a).ravel())
    A = np.asarray(A).reshape(E, M, K // 2)
    sfa = np.asarray(sfa).reshape(E, M, K // 16)
    b = np.asarray(b).reshape(T, K // 2)
    sfb = np.asarray(sfb).reshape(T, K // 16)
    ga = np.asarray(g_a, dtype=np.float32).ravel()
    gb = np.asarray(g_b, dtype=np.float32).ravel()
    c_ref = np.zeros((T, M), dtype=np.float64)
    bound = np.zeros((T, M), dtype=np.float64)
    for t in range(T):
        e = int(experts[t])
        if e < 0:
            continue
        c, tb = gemv(A[e][None], sfa[e][None], ga[e], b[t][None], sfb[t][None], gb[e], M, K, 1)
        c_ref[t] = c[0]
        bound[t] = tb[0]
    return c_ref, bound


def gemv_grouped_rows(A, sfa, g_a, b, sfb, g_b, experts, M: int, K: int, ts, ms):
    """The same definition at the outputs (ts[i], ms[i]) only (full-size sampled checks)."""
    experts = np.asarray(experts, dtype=np.int64).ravel()
    T = len(experts)
    E = len(np.asarray(g_a).ravel())
    A = np.asarray(A).reshape(E, M, K // 2)
    sfa = np.asarray(sfa).reshape(E, M, K // 16)
    b = np.asarray(b).reshape(T, K // 2)
    sfb = np.asarray(sfb).reshape(T, K // 16)
    ga = np.asarray(g_a, dtype=np.float32).ravel()
    gb = np.asarray(g_b, dtype=np.float32).ravel()
    ts = np.asarray(ts, dtype=np.int64)
    ms = np.asarray(ms, dtype=np.int64)
    c_ref = np.zeros(len(ts), dtype=np.float64)
    bound = np.zeros(len(ts), dtype=np.float64)
    for i, (t, m) in enumerate(zip(ts, ms)):
        e = int(experts[t])
        if e < 0:
            continue
        c, tb = gemv_rows(A[e][None], sfa[e][None], ga[e], b[t][None], sfb[t][None], gb[e], M, K,
                          1, [0], [int(m)])
        c_ref[i] = c[0]
        bound[i] = tb[0]
    return c_ref, bound

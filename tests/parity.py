"""The parity criterion between the GPU's fp16 outputs and the oracle's unrounded fp64 values.

Tolerance (the decode configurations state it): |c_gpu - c_ref| <= 1e-3 * |c_ref| + 1e-4 * T,
T = sum_k |term_k| * |g_a * g_b|.  Why it is met by a correct kernel: every 16-element block
partial is exact (quarter-integer sums of at most 576 in magnitude, times a scale product with at
most 8 significant bits), so the only roundings are the fp32 cross-block additions (each at most
2**-24 of a running sum bounded by T, at most K/16 + 31 of them) and the final fp16 rounding
(half an ulp, at most 2**-11 of |c|).  For K = 16384 that is below 7e-5 * T + 4.9e-4 * |c|.

Readings for the edge cases:
* NaN: where the oracle is NaN the GPU must be NaN, and nowhere else.
* fp16 overflow: where |c_ref| is within the tolerance of the overflow threshold 65520, either the
  largest finite value 65504 or the infinity of the same sign is accepted; beyond it, only inf.
* fp16 subnormal outputs: half a subnormal ulp (2**-25) of absolute error is accepted as well.
* zeros of either sign are equal.
"""
from __future__ import annotations

import numpy as np

RTOL = 1e-3
TTOL = 1e-4
FP16_MAX = 65504.0
FP16_OVERFLOW = 65520.0
SUBNORMAL_SLACK = 2.0 ** -25


def parity_report(c_gpu, c_ref, T, rtol=RTOL, ttol=TTOL):
    """Returns (ok_mask, err, bound) over all outputs."""
    g = np.asarray(c_gpu).astype(np.float64).ravel()
    r = np.asarray(c_ref, dtype=np.float64).ravel()
    t = np.asarray(T, dtype=np.float64).ravel()
    if g.shape != r.shape:
        raise ValueError(f"shape mismatch {g.shape} vs {r.shape}")
    bound = rtol * np.abs(r) + ttol * t
    bound = bound + np.where(np.abs(r) < 2.0 ** -14, SUBNORMAL_SLACK, 0.0)
    nan_r = np.isnan(r)
    nan_g = np.isnan(g)
    with np.errstate(invalid="ignore", over="ignore"):
        err = np.abs(g - r)
        ok = err <= bound
        near = np.abs(np.abs(r) - FP16_OVERFLOW) <= bound
        big = np.abs(r) >= FP16_OVERFLOW
        same_inf = np.isinf(g) & (np.sign(g) == np.sign(r))
        max_finite = (np.abs(g) == FP16_MAX) & (np.sign(g) == np.sign(r))
    ok = np.where(big & ~near, same_inf, ok)
    ok = np.where(near, same_inf | max_finite | ok, ok)
    ok = np.where(nan_r | nan_g, nan_r & nan_g, ok)
    return ok, err, bound


def assert_parity(c_gpu, c_ref, T, what="", rtol=RTOL, ttol=TTOL):
    ok, err, bound = parity_report(c_gpu, c_ref, T, rtol, ttol)
    if not ok.all():
        bad = np.nonzero(~ok)[0]
        g = np.asarray(c_gpu).astype(np.float64).ravel()
        r = np.asarray(c_ref, dtype=np.float64).ravel()
        lines = [f"{what}: {len(bad)} of {ok.size} outputs out of tolerance"]
        for i in bad[:8]:
            lines.append(f"  [{i}] gpu={g[i]!r} ref={r[i]!r} err={err[i]:.3e} bound={bound[i]:.3e}")
        raise AssertionError("\n".join(lines))
    finite = np.isfinite(err)
    worst = float(np.max(err[finite] / bound[finite])) if finite.any() else 0.0
    return worst

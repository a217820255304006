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

bfloat16 outputs (the grouped form's NVFP4_OUT_BF16): the same reading with bf16's rounding,
|c_gpu - c_ref| <= 4e-3 * |c_ref| + 1e-4 * T (half a bf16 ulp is at most 2**-8 = 3.9e-3 of |c|;
the fp32 accumulation term is unchanged), overflow at (2 - 2**-8) * 2**127 and a subnormal slack
of 2**-134.
"""
from __future__ import annotations

import numpy as np

RTOL = 1e-3
TTOL = 1e-4
FP16_MAX = 65504.0
FP16_OVERFLOW = 65520.0
SUBNORMAL_SLACK = 2.0 ** -25


BF16_RTOL = 4e-3
FORMATS = {  # max finite, overflow threshold, smallest normal, subnormal slack
    "f16": (FP16_MAX, FP16_OVERFLOW, 2.0 ** -14, SUBNORMAL_SLACK),
    "bf16": ((2 - 2.0 ** -7) * 2.0 ** 127, (2 - 2.0 ** -8) * 2.0 ** 127, 2.0 ** -126, 2.0 ** -134),
}


def bf16_bits_to_f64(bits) -> np.ndarray:
    u = np.asarray(bits).astype(np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def parity_report(c_gpu, c_ref, T, rtol=RTOL, ttol=TTOL, fmt="f16"):
    """Returns (ok_mask, err, bound) over all outputs."""
    fmax, fover, fnormal, fslack = FORMATS[fmt]
    g = np.asarray(c_gpu).astype(np.float64).ravel()
    r = np.asarray(c_ref, dtype=np.float64).ravel()
    t = np.asarray(T, dtype=np.float64).ravel()
    if g.shape != r.shape:
        raise ValueError(f"shape mismatch {g.shape} vs {r.shape}")
    bound = rtol * np.abs(r) + ttol * t
    bound = bound + np.where(np.abs(r) < fnormal, fslack, 0.0)
    nan_r = np.isnan(r)
    nan_g = np.isnan(g)
    with np.errstate(invalid="ignore", over="ignore"):
        err = np.abs(g - r)
        ok = err <= bound
        near = np.abs(np.abs(r) - fover) <= bound
        big = np.abs(r) >= fover
        same_inf = np.isinf(g) & (np.sign(g) == np.sign(r))
        max_finite = (np.abs(g) == fmax) & (np.sign(g) == np.sign(r))
    ok = np.where(big & ~near, same_inf, ok)
    ok = np.where(near, same_inf | max_finite | ok, ok)
    ok = np.where(nan_r | nan_g, nan_r & nan_g, ok)
    return ok, err, bound


def assert_parity(c_gpu, c_ref, T, what="", rtol=None, ttol=TTOL, fmt="f16"):
    if rtol is None:
        rtol = BF16_RTOL if fmt == "bf16" else RTOL
    ok, err, bound = parity_report(c_gpu, c_ref, T, rtol, ttol, fmt)
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

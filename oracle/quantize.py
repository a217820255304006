"""NVFP4 activation quantizer with a fixed global scale, step by step.  TEST INFRASTRUCTURE ONLY.

Follows cutedsl/bridge.py (nvfp4-megamoe-kernel), section "Quantization", function
``quantize_activation_nvfp4``: the global scale is given (not measured, so the step needs no
reduction over the whole tensor), and every step is fp32:

  1. x_norm = x / global_scale
  2. per block of 16 consecutive elements: block_amax = max(|x_norm|), at least 1e-8
  3. block scale = block_amax / 6, cast to float8_e4m3fn (round to nearest even)
  4. x_scaled = x_norm / max(decoded block scale, 1e-8)
  5. sign = x_scaled < 0; magnitude = min(|x_scaled|, 6)
  6. E2M1 magnitude code, by one of two roundings:
       "lut" (the page's): half_steps = round(2 * magnitude) (ties to even), clamped to 0..12,
             then the table [0, 1, 2, 3, 4, 4, 5, 5, 6, 6, 6, 7, 7] printed on the page;
       "rne": the nearest E2M1 grid point, ties to the even code (the reading used for the
             quantized-normal workload).
  7. nibble = code | 8 if negative; packed = (odd << 4) | even.

Reading (the page is silent): a block scale that rounds above the largest finite E4M3 value (448)
saturates to 448 (byte 0x7E) instead of becoming NaN, as the GPU's saturating conversion does.
The global scale multiplies back: x ~= global_scale * e4m3(scale) * e2m1(code).

Pinned by tests/test_oracle_quantize.py.
"""
from __future__ import annotations

import numpy as np

from .codecs import E2M1_TABLE, E4M3FN_TABLE

BLOCK = 16
# finite non-negative E4M3 values in byte order 0x00 .. 0x7E (strictly increasing)
_E4M3_POS = E4M3FN_TABLE[:0x7F].astype(np.float64)
_HALF_STEP_CODE = np.array([0, 1, 2, 3, 4, 4, 5, 5, 6, 6, 6, 7, 7], dtype=np.uint8)
_E2M1_MAG = E2M1_TABLE[:8].astype(np.float32)               # 0, .5, 1, 1.5, 2, 3, 4, 6


def e4m3_encode_rne(v) -> np.ndarray:
    """Non-negative fp32 values -> E4M3FN bytes, round to nearest (ties to even byte), saturating
    at 448.  Works on the exact values: the nearest of the 127 finite non-negative E4M3 values."""
    v = np.asarray(v, dtype=np.float64)
    if np.any(v < 0) or np.any(np.isnan(v)):
        raise ValueError("block scales are non-negative")
    idx = np.searchsorted(_E4M3_POS, v, side="left")        # first value >= v
    idx = np.clip(idx, 1, len(_E4M3_POS) - 1)
    lo = _E4M3_POS[idx - 1]
    hi = _E4M3_POS[idx]
    pick_hi = (v - lo > hi - v) | ((v - lo == hi - v) & (idx % 2 == 0))
    out = np.where(pick_hi, idx, idx - 1)
    out = np.where(v >= _E4M3_POS[-1], len(_E4M3_POS) - 1, out)   # saturate at 448
    out = np.where(v <= 0, 0, out)
    return out.astype(np.uint8)


def e2m1_code_lut(mag: np.ndarray) -> np.ndarray:
    hs = np.clip(np.rint(2.0 * mag.astype(np.float32)), 0, 12).astype(np.int64)
    return _HALF_STEP_CODE[hs]


def e2m1_code_rne(mag: np.ndarray) -> np.ndarray:
    mag = mag.astype(np.float32)
    d = np.abs(mag[..., None] - _E2M1_MAG)                    # distance to each grid point
    best = d.min(axis=-1, keepdims=True)
    cand = d == best
    # ties: prefer the even code (two candidates at most, adjacent codes)
    even = cand & (np.arange(8) % 2 == 0)
    pick = np.where(even.any(axis=-1, keepdims=True), even, cand)
    return np.argmax(pick, axis=-1).astype(np.uint8)


def quantize_activation(x, global_scale: float, rounding: str = "lut"):
    """x: float32 [..., K] (bf16 values), K % 16 == 0.  Returns (packed uint8 [..., K/2],
    scale bytes uint8 [..., K/16])."""
    x = np.asarray(x, dtype=np.float32)
    K = x.shape[-1]
    if K % BLOCK:
        raise ValueError("K must be a multiple of 16")
    gs = np.float32(global_scale)
    xn = (x / gs).astype(np.float32)
    blocks = xn.reshape(*xn.shape[:-1], K // BLOCK, BLOCK)
    bamax = np.maximum(np.abs(blocks).max(axis=-1), np.float32(1e-8)).astype(np.float32)
    sf_byte = e4m3_encode_rne((bamax / np.float32(6.0)).astype(np.float32))
    sf_val = E4M3FN_TABLE[sf_byte].astype(np.float32)
    xs = (blocks / np.maximum(sf_val, np.float32(1e-8))[..., None]).astype(np.float32)
    neg = xs < 0
    mag = np.minimum(np.abs(xs), np.float32(6.0))
    if rounding == "lut":
        code = e2m1_code_lut(mag)
    elif rounding == "rne":
        code = e2m1_code_rne(mag)
    else:
        raise ValueError(rounding)
    nib = (code | np.where(neg, 8, 0)).astype(np.uint8).reshape(*x.shape[:-1], K)
    packed = (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)
    return packed, sf_byte.reshape(*x.shape[:-1], K // BLOCK)

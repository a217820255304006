"""NVFP4 activation quantizer with a fixed global scale, by its definition.  TEST INFRASTRUCTURE ONLY.

What it computes (cutedsl/bridge.py, nvfp4-megamoe-kernel, section "Quantization",
``quantize_activation_nvfp4``, which fixes the semantics: fp32 torch arithmetic, a caller-given
global scale gs, blocks of 16 consecutive elements, block scales of type float8_e4m3fn, E2M1 codes
packed two per byte with the even element in the low nibble).  For one block of values x_k:

    n_k   = x_k / gs                                   (fp32 division)
    scale = e4m3( max(max_k |n_k|, 1e-8) / 6 )         (nearest E4M3, ties to even; no finite
                                                        encoding past 448: NaN, as torch's cast)
    q_k   = n_k / max(scale, 1e-8)                     (fp32 division)
    code  = E2M1 rounding of min(|q_k|, 6), sign bit set when q_k < 0

so that x_k ~= gs * scale * e2m1(code_k).  Two roundings of the magnitude are offered:

    "lut": the page's rule, a table indexed by the number of half steps rint(2 * m) (ties to even),
           table = [0, 1, 2, 3, 4, 4, 5, 5, 6, 6, 6, 7, 7] as printed on the page;
    "rne": the E2M1 value nearest to m, ties to the even code (the reading used for the
           quantized-normal workload).

Readings where the page is silent: a block whose scale is NaN (its largest |n_k| / 6 lies past
464, so the cast gives NaN) gets the codes 0, since the page's table lookup has no index for a NaN
quotient; inputs are finite.

Pinned by tests/test_oracle_quantize.py; the plain C formulation in nvfp4_ref.c must agree with
this one byte for byte.
"""
from __future__ import annotations

import numpy as np

from .codecs import E2M1_TABLE, E4M3FN_TABLE

BLOCK = 16
E4M3_NAN = 0x7F
# finite non-negative E4M3 values in byte order 0x00 .. 0x7E (strictly increasing)
_E4M3_POS = E4M3FN_TABLE[:0x7F].astype(np.float64)
_HALF_STEP_CODE = np.array([0, 1, 2, 3, 4, 4, 5, 5, 6, 6, 6, 7, 7], dtype=np.uint8)
_E2M1_MAG = E2M1_TABLE[:8].astype(np.float32)               # 0, .5, 1, 1.5, 2, 3, 4, 6


def e4m3_encode_rne(v) -> np.ndarray:
    """Non-negative fp32 values -> the nearest E4M3FN byte (ties to the even byte), computed on
    the exact values.  Past the midpoint between 448 and the next step (464), and for NaN, there
    is no finite encoding: the byte is 0x7F (NaN)."""
    v = np.asarray(v, dtype=np.float64)
    if np.any(v < 0):
        raise ValueError("block scales are non-negative")
    idx = np.searchsorted(_E4M3_POS, np.nan_to_num(v), side="left")   # first value >= v
    idx = np.clip(idx, 1, len(_E4M3_POS) - 1)
    lo = _E4M3_POS[idx - 1]
    hi = _E4M3_POS[idx]
    pick_hi = (v - lo > hi - v) | ((v - lo == hi - v) & (idx % 2 == 0))
    out = np.where(pick_hi, idx, idx - 1)
    out = np.where(v >= _E4M3_POS[-1], len(_E4M3_POS) - 1, out)  # 448 .. 464 round to 448
    out = np.where(v <= 0, 0, out)
    out = np.where((v > 464.0) | np.isnan(v), E4M3_NAN, out)
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


_MAGNITUDE_CODE = {"lut": e2m1_code_lut, "rne": e2m1_code_rne}


def block_scale_bytes(n_blocks: np.ndarray) -> np.ndarray:
    """Scale byte of each block of normalised values n ([..., 16] fp32)."""
    amax = np.maximum(np.abs(n_blocks).max(axis=-1), np.float32(1e-8)).astype(np.float32)
    return e4m3_encode_rne((amax / np.float32(6.0)).astype(np.float32))


def quantize_activation(x, global_scale: float, rounding: str = "lut"):
    """x: float32 [..., K] (bf16 values), K % 16 == 0.  Returns (packed uint8 [..., K/2],
    scale bytes uint8 [..., K/16])."""
    if rounding not in _MAGNITUDE_CODE:
        raise ValueError(rounding)
    x = np.asarray(x, dtype=np.float32)
    K = x.shape[-1]
    if K % BLOCK:
        raise ValueError("K must be a multiple of 16")
    n = (x / np.float32(global_scale)).astype(np.float32)
    n = n.reshape(*n.shape[:-1], K // BLOCK, BLOCK)
    scale_byte = block_scale_bytes(n)
    finite = scale_byte != E4M3_NAN
    scale = np.where(finite, E4M3FN_TABLE[scale_byte], 1.0).astype(np.float32)
    q = (n / np.maximum(scale, np.float32(1e-8))[..., None]).astype(np.float32)
    code = _MAGNITUDE_CODE[rounding](np.minimum(np.abs(q), np.float32(6.0)))
    nib = np.where(q < 0, code | 8, code).astype(np.uint8)
    nib = np.where(finite[..., None], nib, 0).astype(np.uint8)   # reading: NaN scale, codes 0
    nib = nib.reshape(*x.shape[:-1], K)
    packed = (nib[..., 0::2] | (nib[..., 1::2] << 4)).astype(np.uint8)
    return packed, scale_byte.reshape(*x.shape[:-1], K // BLOCK)

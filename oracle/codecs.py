"""Scalar codecs of the NVFP4 format, written from their bit-level definitions.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

* E2M1 (FP4): 1 sign bit (bit 3), 2 exponent bits (bits 2..1, bias 1), 1 mantissa bit (bit 0).
  The magnitudes this gives, in code order 0..7, are the list ``E2M1_MAGNITUDES`` printed in
  cutedsl/bridge.py (nvfp4-megamoe-kernel), section "Constants".
* E4M3FN (FP8 block scale, ``torch.float8_e4m3fn``): 1 sign bit, 4 exponent bits (bias 7),
  3 mantissa bits; no infinities; S.1111.111 is NaN; largest finite 448.  The block-scale type is
  fixed in "nvFP4 Batch GEMV算子系列(下)", section "准备数据" (scales created as
  float8_e4m3fn) and in bridge.py, "Quantization" (block scales cast to float8_e4m3fn).
* Packing: two FP4 codes per byte, the element with even k in the low nibble and the odd one in
  the high nibble (bridge.py, "Quantization": ``packed = (odd << 4) | even``).

Every function here is pinned by ``tests/test_oracle_codecs.py``.
"""
from __future__ import annotations

import math

import numpy as np


def e2m1_value(code: int) -> float:
    """Value of one 4-bit E2M1 code.

    e = bits 2..1, m = bit 0.  e == 0 is the subnormal range (value 0.5*m); otherwise the value is
    2**(e-1) * (1 + m/2).  Bit 3 is the sign, so code 8 is -0.0.
    """
    if not 0 <= code <= 15:
        raise ValueError(f"E2M1 code out of range: {code}")
    sign = -1.0 if code & 0x8 else 1.0
    e = (code >> 1) & 0x3
    m = code & 0x1
    magnitude = 0.5 * m if e == 0 else 2.0 ** (e - 1) * (1.0 + 0.5 * m)
    return sign * magnitude


def e4m3fn_value(byte: int) -> float:
    """Value of one E4M3FN byte (float8_e4m3fn), exactly, as a Python float.

    E = bits 6..3, m = bits 2..0, bias 7.  E == 0: subnormal m * 2**-9.  Otherwise
    2**(E-7) * (1 + m/8).  0x7F and 0xFF are NaN; the format has no infinity.
    """
    if not 0 <= byte <= 255:
        raise ValueError(f"E4M3 byte out of range: {byte}")
    sign = -1.0 if byte & 0x80 else 1.0
    E = (byte >> 3) & 0xF
    m = byte & 0x7
    if E == 0xF and m == 0x7:
        return math.nan
    if E == 0:
        return sign * m * 2.0 ** -9
    return sign * 2.0 ** (E - 7) * (1.0 + m / 8.0)


#: fp64 value of every E2M1 code (index = code).
E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)

#: fp64 value of every E4M3FN byte (index = byte).
E4M3FN_TABLE = np.array([e4m3fn_value(b) for b in range(256)], dtype=np.float64)


def unpack_e2m1_codes(packed: np.ndarray) -> np.ndarray:
    """Split packed FP4 bytes ``[..., K/2]`` into codes ``[..., K]``.

    Element 2j is the low nibble of byte j and element 2j+1 its high nibble.
    """
    packed = np.asarray(packed, dtype=np.uint8)
    codes = np.empty(packed.shape[:-1] + (2 * packed.shape[-1],), dtype=np.uint8)
    codes[..., 0::2] = packed & 0x0F
    codes[..., 1::2] = packed >> 4
    return codes


def fp16_round(x) -> np.ndarray:
    """Round fp64 values to IEEE binary16, round-half-to-even, overflow to +-inf.

    numpy's float64 -> float16 conversion is used as the library primitive; the tests pin it
    (exhaustively over all binary16 values and their midpoints) against exact rational rounding.
    """
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float16)

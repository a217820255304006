"""Pins of the oracle's codecs against values fixed outside the oracle.

* E2M1: the magnitude list printed in cutedsl/bridge.py, section "Constants" (E2M1_MAGNITUDES),
  retyped here as the page prints it; bit 3 is the sign.
* E4M3FN: torch's float8_e4m3fn -> float32 cast (an independent library routine) on all 256 bytes,
  plus hand anchors.
* fp16 rounding: exhaustively, every binary16 value and every midpoint, against exact arithmetic.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import codecs

PRINTED_E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_equals_printed_magnitudes():
    for code in range(8):
        assert oracle.e2m1_value(code) == PRINTED_E2M1_MAGNITUDES[code]
        assert oracle.E2M1_TABLE[code] == PRINTED_E2M1_MAGNITUDES[code]


def test_e2m1_sign_symmetry():
    for code in range(8):
        assert oracle.e2m1_value(code | 8) == -oracle.e2m1_value(code)
    assert math.copysign(1.0, oracle.e2m1_value(8)) == -1.0      # code 8 is -0


def test_e2m1_rejects_out_of_range():
    with pytest.raises(ValueError):
        oracle.e2m1_value(16)


def test_e4m3_equals_torch_cast_all_bytes():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    ref = ref.to(torch.float32).to(torch.float64).numpy()
    mine = oracle.E4M3FN_TABLE
    assert np.array_equal(np.isnan(ref), np.isnan(mine))
    fin = ~np.isnan(ref)
    assert np.array_equal(ref[fin], mine[fin])
    assert np.array_equal(np.signbit(ref[fin]), np.signbit(mine[fin]))


@pytest.mark.parametrize("byte,value", [
    (0x38, 1.0), (0x40, 2.0), (0x30, 0.5), (0x48, 4.0), (0x7E, 448.0), (0x08, 2.0 ** -6),
    (0x01, 2.0 ** -9), (0x07, 7 * 2.0 ** -9), (0x00, 0.0), (0xB8, -1.0), (0xFE, -448.0),
])
def test_e4m3_anchors(byte, value):
    assert oracle.e4m3fn_value(byte) == value


def test_e4m3_nan_and_monotone():
    assert math.isnan(oracle.e4m3fn_value(0x7F))
    assert math.isnan(oracle.e4m3fn_value(0xFF))
    pos = oracle.E4M3FN_TABLE[:0x7F]
    assert np.all(np.diff(pos) > 0)                              # bytes 0..0x7E strictly increase
    assert np.nanmax(oracle.E4M3FN_TABLE) == 448.0


def test_code_products_brute_force():
    """All 16 x 16 products: integer quarter-units, and exactly the products of the printed list."""
    mags = set()
    for a in range(16):
        for b in range(16):
            p = oracle.E2M1_TABLE[a] * oracle.E2M1_TABLE[b]
            expect = PRINTED_E2M1_MAGNITUDES[a & 7] * PRINTED_E2M1_MAGNITUDES[b & 7]
            sign = -1.0 if ((a ^ b) & 8) else 1.0
            assert p == sign * expect
            assert (4 * p) == int(4 * p)
            mags.add(abs(p))
    assert sorted(mags) == [0.0, 0.25, 0.5, 0.75, 1.0, 1.5, 2.0, 2.25, 3.0, 4.0, 4.5, 6.0, 8.0,
                            9.0, 12.0, 16.0, 18.0, 24.0, 36.0]


def test_unpack_low_nibble_is_even_k():
    codes = oracle.unpack_e2m1_codes(np.array([[0x21, 0xA9]], dtype=np.uint8))
    assert codes.tolist() == [[1, 2, 9, 10]]


def _all_fp16_values():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    return bits, bits.view(np.float16).astype(np.float64)


def test_fp16_round_trips_every_value():
    bits, vals = _all_fp16_values()
    fin = np.isfinite(vals)
    out = codecs.fp16_round(vals[fin]).view(np.uint16)
    # -0 and +0 both round-trip with their sign
    assert np.array_equal(out, bits[fin])


def test_fp16_midpoints_tie_to_even_and_neighbours_round_to_nearest():
    bits = np.arange(0, 0x7C00, dtype=np.uint16)            # +0 .. 65504, ascending
    v = bits.view(np.float16).astype(np.float64)
    lo, hi = v[:-1], v[1:]
    mid = (lo + hi) / 2                                       # exact in fp64 (<= 12 bits)
    got = codecs.fp16_round(mid).view(np.uint16)
    even_lo = (bits[:-1] % 2) == 0
    expect = np.where(even_lo, bits[:-1], bits[1:])
    assert np.array_equal(got, expect)
    below = np.nextafter(mid, -np.inf)
    above = np.nextafter(mid, np.inf)
    assert np.array_equal(codecs.fp16_round(below).view(np.uint16), bits[:-1])
    assert np.array_equal(codecs.fp16_round(above).view(np.uint16), bits[1:])
    # mirrored for negative values
    assert np.array_equal(codecs.fp16_round(-mid).view(np.uint16), expect | 0x8000)


def test_fp16_overflow_threshold():
    assert codecs.fp16_round(65519.99).view(np.uint16) == 0x7BFF            # 65504
    assert codecs.fp16_round(65520.0).view(np.uint16) == 0x7C00             # +inf (tie to even)
    assert codecs.fp16_round(-1e9).view(np.uint16) == 0xFC00
    assert codecs.fp16_round(2.0 ** -25).view(np.uint16) == 0x0000          # tie -> even (zero)
    assert codecs.fp16_round(3 * 2.0 ** -26).view(np.uint16) == 0x0001

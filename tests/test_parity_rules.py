"""The parity criterion itself (tests/parity.py), on hand-made cases: the bound, NaN positions,
fp16 overflow near 65520, signed zeros, and the bfloat16 variant."""
import numpy as np
import pytest

from parity import assert_parity, bf16_bits_to_f64, parity_report


def test_bound_is_relative_plus_term_scale():
    ok, _, bound = parity_report([1.001, 1.0], [1.0, 1.0], [0.0, 10.0])
    assert bound.tolist() == pytest.approx([1e-3, 1e-3 + 1e-3])
    assert ok.tolist() == [True, True]
    ok, _, _ = parity_report([1.0011], [1.0], [0.0])
    assert not ok[0]


def test_nan_must_match_in_position():
    assert parity_report([np.nan, 1.0], [np.nan, 1.0], [1, 1])[0].all()
    assert not parity_report([np.nan], [1.0], [1])[0][0]
    assert not parity_report([1.0], [np.nan], [1])[0][0]


def test_fp16_overflow_rules():
    # just above the threshold: inf (or, within tolerance of it, 65504) accepted
    assert parity_report([np.inf], [65530.0], [0.0])[0][0]
    assert parity_report([65504.0], [65521.0], [0.0])[0][0]
    assert not parity_report([65504.0], [70000.0], [0.0])[0][0]
    assert not parity_report([-np.inf], [70000.0], [0.0])[0][0]


def test_signed_zeros_equal():
    assert parity_report([-0.0], [0.0], [0.0])[0][0]


def test_bf16_variant():
    # 1 + 2^-8 is a bf16 tie: either neighbour is within 4e-3
    lo = bf16_bits_to_f64([0x3F80])[0]
    hi = bf16_bits_to_f64([0x3F81])[0]
    assert (lo, hi) == (1.0, 1.0 + 2.0 ** -7)
    assert_parity([lo], [1.0 + 2.0 ** -8], [0.0], fmt="bf16")
    assert_parity([hi], [1.0 + 2.0 ** -8], [0.0], fmt="bf16")
    with pytest.raises(AssertionError):
        assert_parity([1.0 + 2.0 ** -6], [1.0], [0.0], fmt="bf16")
    # 70000 is an ordinary bf16-range value: no fp16 overflow rule applies
    assert_parity([bf16_bits_to_f64([0x4789])[0]], [70144.0], [0.0], fmt="bf16")
    assert bf16_bits_to_f64([0x4789])[0] == 70144.0

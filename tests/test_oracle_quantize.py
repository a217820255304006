"""Pins of the activation quantizer oracle (oracle/quantize.py) against things other than itself:
the half-step table printed in cutedsl/bridge.py, torch's float8_e4m3fn cast, exact grid
round-trips, brute-force nearest rounding, error bounds, sign symmetry, and the independently
written quantizer of the seeded workload generator."""
import numpy as np
import pytest
import torch

import workloads
from oracle import E2M1_TABLE, E4M3FN_TABLE
from oracle import quantize as Q

# bridge.py, imports section: _get_step_to_idx_lut's table, as the page prints it
PRINTED_HALF_STEP_TABLE = [0, 1, 2, 3, 4, 4, 5, 5, 6, 6, 6, 7, 7]
GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_half_step_table_is_the_printed_one():
    assert Q._HALF_STEP_CODE.tolist() == PRINTED_HALF_STEP_TABLE


def _torch_e4m3(v):
    t = torch.from_numpy(np.asarray(v, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def _encoder_inputs():
    """Every finite E4M3 value, every midpoint between neighbours and the fp32 values next to
    them, the edge past 448 (the midpoint 464 and the NaN range above it), and random values over
    the whole fp32 range the block scale can take."""
    pos = E4M3FN_TABLE[:0x7F]
    mids = np.concatenate([(pos[:-1] + pos[1:]) / 2, [464.0]])
    rng = np.random.default_rng(0)
    return np.concatenate([pos, mids, np.nextafter(mids.astype(np.float32), 0),
                           np.nextafter(mids.astype(np.float32), np.inf),
                           rng.uniform(0, 500, 20000), rng.uniform(440, 490, 5000),
                           np.exp2(rng.uniform(-40, 40, 5000)), [479.99, 480.0, 1e30, 3e38],
                           [np.inf, np.nan]]).astype(np.float32)


def test_e4m3_encoder_matches_torch_over_the_whole_range():
    """[Bridge] casts block_amax / 6 with torch's float8_e4m3fn conversion; the encoder must give
    the same byte for every non-negative fp32 input, NaN (0x7F) past 464 included."""
    vals = _encoder_inputs()
    assert np.array_equal(Q.e4m3_encode_rne(vals), _torch_e4m3(vals))


def test_e4m3_encoder_nan_past_464():
    got = Q.e4m3_encode_rne(np.float32([448.0, 463.9, 464.0, 464.01, 470.0, 1e6, np.nan]))
    assert got.tolist() == [0x7E, 0x7E, 0x7E, 0x7F, 0x7F, 0x7F, 0x7F]


@pytest.mark.parametrize("rounding", ["lut", "rne"])
def test_overflowing_block_scale_is_nan_with_zero_codes(rounding):
    """A block whose largest normalised magnitude / 6 lies past 464 has no finite scale: the
    cast gives NaN (byte 0x7F); its codes are 0 (reading), other blocks are unaffected."""
    gs = np.float32(0.25)
    x = np.random.default_rng(5).standard_normal((2, 64)).astype(np.float32)
    x[0, 16:32] = np.linspace(-3000, 3000, 16, dtype=np.float32)   # 3000 / 0.25 / 6 = 2000
    x[1, 48] = np.float32(464.5 * 6 * 0.25)
    packed, sfb = Q.quantize_activation(x, gs, rounding)
    assert sfb[0, 1] == 0x7F and sfb[1, 3] == 0x7F
    assert (packed[0, 8:16] == 0).all() and (packed[1, 24:32] == 0).all()
    keep = np.ones_like(sfb, dtype=bool)
    keep[0, 1] = keep[1, 3] = False
    assert (sfb[keep] != 0x7F).all()
    x2 = x.copy()
    x2[0, 16:32] = 0.0
    x2[1, 48:64] = 0.0
    p2, s2 = Q.quantize_activation(x2, gs, rounding)
    assert np.array_equal(s2[keep], sfb[keep])
    for r, blk in ((0, 1), (1, 3)):
        p2[r, 8 * blk:8 * blk + 8] = packed[r, 8 * blk:8 * blk + 8]
    assert np.array_equal(p2, packed)


@pytest.mark.parametrize("rounding", ["lut", "rne"])
def test_grid_values_round_trip(rounding):
    gs = np.float32(0.013)
    for sf_byte in (0x30, 0x38, 0x41, 0x7E, 0x08):
        sf = np.float32(E4M3FN_TABLE[sf_byte])
        # a block whose largest magnitude is 6 (so the block scale is exactly sf), then all codes
        mags = np.array(GRID * 2, dtype=np.float32)
        signs = np.array([1, -1] * 8, dtype=np.float32)
        x = (mags * signs * sf * gs).astype(np.float32)
        x[0] = np.float32(6.0) * sf * gs
        packed, sfb = Q.quantize_activation(x[None, :], gs, rounding)
        codes = np.empty(16, dtype=np.uint8)
        codes[0::2] = packed[0] & 15
        codes[1::2] = packed[0] >> 4
        deq = E2M1_TABLE[codes] * E4M3FN_TABLE[sfb[0, 0]] * gs
        assert np.allclose(deq, x, rtol=1e-6, atol=0), (rounding, sf_byte)


def test_lut_and_rne_disagree_at_the_half_steps():
    mags = np.float32([0.2, 0.25, 0.75, 1.25, 1.3, 2.5, 2.6, 3.6, 5.1, 5.6])
    lut = [GRID[c] for c in Q.e2m1_code_lut(mags)]
    rne = [GRID[c] for c in Q.e2m1_code_rne(mags)]
    assert lut == [0.0, 0.0, 1.0, 1.0, 1.5, 2.0, 2.0, 3.0, 4.0, 6.0]
    assert rne == [0.0, 0.0, 1.0, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0, 6.0]


def test_rne_is_nearest_brute_force():
    mags = np.random.default_rng(1).uniform(0, 6, 50000).astype(np.float32)
    codes = Q.e2m1_code_rne(mags)
    got = np.abs(mags - np.float32(GRID)[codes])
    best = np.abs(mags[:, None] - np.float32(GRID)[None, :]).min(axis=1)
    assert np.array_equal(got, best)


@pytest.mark.parametrize("rounding,bound", [("rne", 1.0), ("lut", 1.25)])
def test_dequantization_error_bound(rounding, bound):
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((8, 256)) * 3).astype(np.float32)
    gs = np.float32(np.abs(x).max() / 2688.0)
    packed, sfb = Q.quantize_activation(x, gs, rounding)
    codes = np.empty(x.shape, dtype=np.uint8)
    codes[:, 0::2] = packed & 15
    codes[:, 1::2] = packed >> 4
    sf = np.repeat(E4M3FN_TABLE[sfb], 16, axis=1)
    err = np.abs(E2M1_TABLE[codes] * sf * gs - x)
    assert np.all(err <= bound * sf * gs * (1 + 1e-6))


def test_sign_symmetry():
    x = np.random.default_rng(3).standard_normal((4, 64)).astype(np.float32)
    p1, s1 = Q.quantize_activation(x, 0.01)
    p2, s2 = Q.quantize_activation(-x, 0.01)
    assert np.array_equal(s1, s2)
    nz = (p1 != 0)
    # every nonzero magnitude code flips its sign bit
    c1 = np.stack([p1 & 15, p1 >> 4], -1)
    c2 = np.stack([p2 & 15, p2 >> 4], -1)
    mask = (c1 & 7) != 0
    assert np.array_equal((c1 ^ c2)[mask], np.full(mask.sum(), 8, dtype=np.uint8))
    assert nz.any()


def test_agrees_with_the_workload_generator():
    """workloads.quantize_bf16_to_nvfp4 is a separate implementation (torch's fp8 cast, its own
    E2M1 rounding); with its global scale and RNE rounding the two must give the same bytes."""
    x = workloads.normal_bf16(9, "A", 64 * 512).reshape(64, 512)
    packed_w, sf_w, gs = workloads.quantize_bf16_to_nvfp4(x)
    packed_o, sf_o = Q.quantize_activation(x, gs, "rne")
    assert np.array_equal(sf_o, sf_w)
    assert np.array_equal(packed_o, packed_w)


def test_rejects_ragged_k():
    with pytest.raises(ValueError):
        Q.quantize_activation(np.zeros((1, 24), np.float32), 1.0)

"""Pins of the oracle's GEMV against things other than itself.

* hand-worked examples (tests/golden/worked_examples.json; each derivation cites the pages);
* the independent exact-integer formulation, bit for bit, on all five workloads;
* algebraic invariants of the definition;
* planted mistakes: each plausible slip in the oracle (nibble order, sign, a dropped scale, a
  shifted block index, a transposed layout, a wrong exponent bias, a dropped global scale) must
  make at least one pin fail.
"""
import json
import os
import sys

import numpy as np
import pytest

import oracle
import workloads

NV = sys.modules["oracle.nvfp4_gemv"]
HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = json.load(open(os.path.join(HERE, "golden", "worked_examples.json")))["examples"]


def _tensors(ex):
    def h(key):
        return np.frombuffer(bytes.fromhex(ex[key]), dtype=np.uint8).copy()
    return h("A"), h("sfa"), h("b"), h("sfb")


def golden_failures(gemv_fn):
    """Ids of the worked examples that ``gemv_fn`` gets wrong."""
    bad = []
    for ex in GOLDEN:
        A, sfa, b, sfb = _tensors(ex)
        try:
            c, _ = gemv_fn(A, sfa, ex["g_a"], b, sfb, ex["g_b"], ex["M"], ex["K"], ex["L"])
        except Exception:
            bad.append(ex["id"])
            continue
        c = np.asarray(c, dtype=np.float64).ravel()
        want = [np.nan if v is None else v for v in ex["c"]]
        rel = ex.get("rel_tol", 0.0)
        for got, w in zip(c, want):
            if np.isnan(w):
                if not np.isnan(got):
                    bad.append(ex["id"])
                    break
            elif not (abs(got - w) <= rel * abs(w)):
                bad.append(ex["id"])
                break
    return bad


def test_worked_examples():
    assert golden_failures(oracle.gemv) == []


def test_worked_examples_fp16():
    for ex in GOLDEN:
        A, sfa, b, sfb = _tensors(ex)
        c16 = oracle.gemv_fp16(A, sfa, ex["g_a"], b, sfb, ex["g_b"], ex["M"], ex["K"], ex["L"])
        for got, want in zip(c16.ravel().view(np.uint16), ex["c_fp16_hex"]):
            if want == "nan":
                assert np.isnan(np.uint16(got).view(np.float16)), ex["id"]
            elif int(want, 16) & 0x7FFF == 0:
                assert int(got) & 0x7FFF == 0, ex["id"]           # either signed zero
            else:
                assert int(got) == int(want, 16), ex["id"]


def test_gemv_rows_matches_full():
    w = workloads.random_workload(7, 96, 3, seed=11)
    c, T = oracle.gemv(w.A, w.sfa, 1.5, w.b, w.sfb, 0.75, w.M, w.K, w.L)
    ls = np.array([0, 2, 1, 2, 0])
    ms = np.array([6, 0, 3, 3, 0])
    c2, T2 = oracle.gemv_rows(w.A, w.sfa, 1.5, w.b, w.sfb, 0.75, w.M, w.K, w.L, ls, ms)
    assert np.array_equal(c2, c[ls, ms]) and np.array_equal(T2, T[ls, ms])


def _assert_exact(w, ls=None, ms=None):
    if ls is None:
        c, _ = oracle.gemv(w.A, w.sfa, 1.0, w.b, w.sfb, 1.0, w.M, w.K, w.L)
        c = c.ravel()
    else:
        c, _ = oracle.gemv_rows(w.A, w.sfa, 1.0, w.b, w.sfb, 1.0, w.M, w.K, w.L, ls, ms)
    units, nan = oracle.gemv_exact_units(w.A, w.sfa, w.b, w.sfb, w.M, w.K, w.L, ls, ms)
    assert not nan.any()
    assert np.all(np.abs(units) < 2 ** 53)
    assert np.array_equal(c * 2.0 ** 20, units.astype(np.float64))


def test_exact_integer_agreement_c1(workload):
    _assert_exact(workload("c1"))


@pytest.mark.slow
@pytest.mark.parametrize("name", ["c2", "c3", "c4", "c5"])
def test_exact_integer_agreement_full_configs(workload, name):
    w = workload(name)
    rng = np.random.default_rng(100)
    n = 96
    ls = rng.integers(0, w.L, n)
    ms = rng.integers(0, w.M, n)
    ls[:2] = [0, w.L - 1]
    ms[:2] = [0, w.M - 1]
    _assert_exact(w, ls, ms)


def test_exact_integer_agreement_extreme_scales():
    # full E4M3 range including subnormals, largest values and every code
    finite = [v for v in range(256) if v not in (0x7F, 0xFF)]
    w = workloads.random_workload(9, 512, 2, seed=21, scale_bytes=finite)
    _assert_exact(w)


def test_exact_checker_flags_nan_rows():
    w = workloads.random_workload(4, 64, 2, seed=5)
    w.sfa[1, 2, 3] = 0x7F
    c, _ = oracle.gemv(w.A, w.sfa, 1.0, w.b, w.sfb, 1.0, w.M, w.K, w.L)
    _, nan = oracle.gemv_exact_units(w.A, w.sfa, w.b, w.sfb, w.M, w.K, w.L)
    assert np.array_equal(np.isnan(c).ravel(), nan)
    assert nan.sum() == 1


# ------------------------------------------------------------------ invariants of the definition

def _small(seed, M=5, K=64, L=3, scale_bytes=workloads.pow2_scale_bytes(-3, 3)):
    return workloads.random_workload(M, K, L, seed, scale_bytes=scale_bytes)


def _c(w, g_a=1.0, g_b=1.0, A=None, sfa=None, b=None, sfb=None):
    c, _ = oracle.gemv(w.A if A is None else A, w.sfa if sfa is None else sfa, g_a,
                       w.b if b is None else b, w.sfb if sfb is None else sfb, g_b, w.M, w.K, w.L)
    return c


def _block_contribution(w, l, m, j):
    """The j-th 16-element block of output (l, m), as its own K = 16 GEMV."""
    A = w.A[l, m, 8 * j:8 * j + 8]
    b = w.b[l, 8 * j:8 * j + 8]
    c, _ = oracle.gemv(A, w.sfa[l, m, j:j + 1], 1.0, b, w.sfb[l, j:j + 1], 1.0, 1, 16, 1)
    return c[0, 0]


def test_zero_scale_removes_block():
    w = _small(1)
    base = _c(w)
    sfa = w.sfa.copy()
    sfa[1, 2, 3] = 0x00
    assert _c(w, sfa=sfa)[1, 2] == base[1, 2] - _block_contribution(w, 1, 2, 3)
    sfb = w.sfb.copy()
    sfb[0, 1] = 0x80                                        # -0 also zeroes the block
    changed = _c(w, sfb=sfb)
    for m in range(w.M):
        assert changed[0, m] == base[0, m] - _block_contribution(w, 0, m, 1)


def test_doubling_a_scale_byte_adds_the_block_once_more():
    w = _small(2)
    base = _c(w)
    sfa = w.sfa.copy()
    assert 0x08 <= sfa[2, 4, 1] <= 0x6F
    sfa[2, 4, 1] += 0x08                                    # exponent + 1: the scale doubles
    assert _c(w, sfa=sfa)[2, 4] == base[2, 4] + _block_contribution(w, 2, 4, 1)


def _swap_nibbles(x):
    return ((x << 4) | (x >> 4)).astype(np.uint8)


def test_nibble_swap_permutes_k():
    w = _small(3)
    base = _c(w)
    assert np.array_equal(_c(w, A=_swap_nibbles(w.A), b=_swap_nibbles(w.b)), base)
    assert np.array_equal(_c(w, A=_swap_nibbles(w.A)), _c(w, b=_swap_nibbles(w.b)))


def test_sign_flip_of_b_negates():
    w = _small(4)
    assert np.array_equal(_c(w, b=w.b ^ 0x88), -_c(w))


def test_global_scales_multiply():
    w = _small(5)
    assert np.array_equal(_c(w, g_a=2.0), 2.0 * _c(w))
    assert np.array_equal(_c(w, g_a=0.5, g_b=4.0), 2.0 * _c(w))


def test_block_permutation_invariance():
    w = _small(6, K=128)
    perm = np.random.default_rng(0).permutation(w.K // 16)
    A = w.A.reshape(w.L, w.M, -1, 8)[:, :, perm].reshape(w.A.shape)
    b = w.b.reshape(w.L, -1, 8)[:, perm].reshape(w.b.shape)
    assert np.array_equal(_c(w, A=A, sfa=w.sfa[:, :, perm], b=b, sfb=w.sfb[:, perm]), _c(w))


def test_k_additivity():
    w = _small(7, K=96)
    h = w.K // 2
    full = _c(w)
    first, _ = oracle.gemv(w.A[..., :h // 2], w.sfa[..., :h // 16], 1.0, w.b[..., :h // 2],
                           w.sfb[..., :h // 16], 1.0, w.M, h, w.L)
    second, _ = oracle.gemv(w.A[..., h // 2:], w.sfa[..., h // 16:], 1.0, w.b[..., h // 2:],
                            w.sfb[..., h // 16:], 1.0, w.M, h, w.L)
    assert np.array_equal(full, first + second)


def test_batch_independence():
    w = _small(8)
    base = _c(w)
    A = w.A.copy()
    A[1] ^= 0x5A
    b = w.b.copy()
    b[1] ^= 0x33
    out = _c(w, A=A, b=b)
    assert np.array_equal(out[0], base[0]) and np.array_equal(out[2], base[2])
    assert not np.array_equal(out[1], base[1])


def test_T_bounds_c():
    w = _small(9)
    c, T = oracle.gemv(w.A, w.sfa, 0.3, w.b, w.sfb, -2.0, w.M, w.K, w.L)
    assert np.all(np.abs(c) <= T * (1 + 1e-15))


# ------------------------------------------------------------------ planted mistakes

def _mutant(monkeypatch, **attrs):
    for name, value in attrs.items():
        monkeypatch.setattr(NV, name, value)
    return NV.gemv


def _unpack_high_first(packed):
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (2 * packed.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = packed >> 4
    out[..., 1::2] = packed & 0x0F
    return out


def _row_terms_a_high_first(A_rows, sfa_rows, bterm):
    a_val = NV.E2M1_TABLE[_unpack_high_first(A_rows)]
    sa = np.repeat(NV.E4M3FN_TABLE[sfa_rows], 16, axis=-1)
    return a_val * sa * bterm


def _vector_terms_without_sfb(b_l, sfb_l):
    return NV.E2M1_TABLE[NV.unpack_e2m1_codes(b_l)]


def _row_terms_shifted_blocks(A_rows, sfa_rows, bterm):
    a_val = NV.E2M1_TABLE[NV.unpack_e2m1_codes(A_rows)]
    sa = np.repeat(NV.E4M3FN_TABLE[np.roll(sfa_rows, 1, axis=-1)], 16, axis=-1)
    return a_val * sa * bterm


def _layout_m_major(A, sfa, b, sfb, M, K, L):
    A = np.asarray(A, np.uint8).reshape(M, L, K // 2).transpose(1, 0, 2)
    sfa = np.asarray(sfa, np.uint8).reshape(M, L, K // 16).transpose(1, 0, 2)
    return A, sfa, np.asarray(b, np.uint8).reshape(L, K // 2), \
        np.asarray(sfb, np.uint8).reshape(L, K // 16)


MUTANTS = {
    # (reading the high nibble first for BOTH operands only permutes k within each pair, which
    # leaves every output unchanged; test_unpack_low_nibble_is_even_k pins the codec itself)
    "A read high nibble first": dict(_row_terms=_row_terms_a_high_first),
    "sign bit ignored": dict(E2M1_TABLE=np.abs(oracle.E2M1_TABLE)),
    "sfb dropped": dict(_vector_terms=_vector_terms_without_sfb),
    "block index off by one": dict(_row_terms=_row_terms_shifted_blocks),
    "rows and batches transposed": dict(_as_layout=_layout_m_major),
    "E4M3 bias off by one": dict(E4M3FN_TABLE=oracle.E4M3FN_TABLE * 2.0),
}


@pytest.mark.parametrize("mistake", sorted(MUTANTS))
def test_planted_mistake_is_caught(monkeypatch, mistake):
    gemv = _mutant(monkeypatch, **MUTANTS[mistake])
    assert golden_failures(gemv), f"no pin catches: {mistake}"


def test_planted_dropped_global_scale_is_caught():
    def drop_gb(A, sfa, g_a, b, sfb, g_b, M, K, L):
        return oracle.gemv(A, sfa, g_a, b, sfb, 1.0, M, K, L)
    assert "W7" in golden_failures(drop_gb)


def test_c1_fixture_matches_oracle(workload):
    """tests/golden/c1_oracle.json (written by make_c1_golden.py) freezes the oracle's c1 output."""
    fx = json.load(open(os.path.join(HERE, "golden", "c1_oracle.json")))
    w = workload("c1")
    c, T = oracle.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, w.M, w.K, w.L)
    assert np.array_equal(c.ravel(), np.array([float(v) for v in fx["c_ref"]]))
    assert np.array_equal(T.ravel(), np.array([float(v) for v in fx["T"]]))

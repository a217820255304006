"""Pins of the plain C oracle (oracle/nvfp4_ref.c, through oracle/cref.py) against things other
than itself:

* its decoders against the E2M1 magnitudes printed in cutedsl/bridge.py ("Constants") and torch's
  float8_e4m3fn -> float32 cast on all 256 bytes;
* the hand-worked examples under tests/golden/ (the GEMV tests run them through ``oracle.gemv``,
  which is the C function; here once more through the row-sampled entry point);
* the numpy formulation (oracle/nvfp4_gemv.py, oracle/grouped.py, oracle/quantize.py), written
  independently: bit for bit on all five workloads (whole c1, sampled rows at full size), on
  extreme and NaN scales, on the grouped workloads and on the quantizer;
* the exact-integer formulation, and independence from the OpenMP thread count;
* torch's float8_e4m3fn cast for the quantizer's block-scale bytes over the whole range;
* fp16 rounding: every binary16 value and every midpoint;
* planted mistakes: mutated copies of the C source, compiled on the side, each fail a pin.
"""
import ctypes
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import cref
from oracle import grouped as G
from oracle import nvfp4_gemv as NV
from oracle import quantize as Q

PRINTED_E2M1_MAGNITUDES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_c_e2m1_equals_printed_magnitudes():
    v = cref.e2m1_values()
    assert v[:8].tolist() == PRINTED_E2M1_MAGNITUDES
    assert np.array_equal(v[8:], -v[:8]) and np.signbit(v[8])


def test_c_e4m3_equals_torch_cast_all_bytes():
    ref = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    ref = ref.to(torch.float32).to(torch.float64).numpy()
    mine = cref.e4m3_values()
    assert np.array_equal(np.isnan(ref), np.isnan(mine))
    fin = ~np.isnan(ref)
    assert np.array_equal(ref[fin], mine[fin])
    assert np.array_equal(np.signbit(ref[fin]), np.signbit(mine[fin]))


def _same_bits(x, y):
    return np.array_equal(np.asarray(x, np.float64).view(np.uint64),
                          np.asarray(y, np.float64).view(np.uint64))


def test_c_equals_numpy_c1_whole(workload):
    w = workload("c1")
    c, T = cref.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, w.M, w.K, w.L)
    cn, Tn = NV.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, w.M, w.K, w.L)
    assert _same_bits(c, cn) and _same_bits(T, Tn)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["c2", "c3", "c4", "c5"])
def test_c_equals_numpy_full_size_samples(workload, name):
    w = workload(name)
    rng = np.random.default_rng(7)
    n = 64
    ls = rng.integers(0, w.L, n)
    ms = rng.integers(0, w.M, n)
    ls[:2] = [0, w.L - 1]
    ms[:2] = [0, w.M - 1]
    c, T = cref.gemv_rows(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, w.M, w.K, w.L, ls, ms)
    cn, Tn = NV.gemv_rows(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, w.M, w.K, w.L, ls, ms)
    assert _same_bits(c, cn) and _same_bits(T, Tn)
    u, nan = cref.gemv_exact_units(w.A, w.sfa, w.b, w.sfb, w.M, w.K, w.L, ls, ms)
    un, nann = NV.gemv_exact_units(w.A, w.sfa, w.b, w.sfb, w.M, w.K, w.L, ls, ms)
    assert np.array_equal(u, un) and np.array_equal(nan, nann) and not nan.any()


def test_c_equals_numpy_every_scale_byte_and_nan():
    every = list(range(256))                          # NaN bytes 0x7F / 0xFF included
    w = workloads.random_workload(11, 384, 3, seed=31, scale_bytes=every)
    c, T = cref.gemv(w.A, w.sfa, 0.375, w.b, w.sfb, -3.0, w.M, w.K, w.L)
    cn, Tn = NV.gemv(w.A, w.sfa, 0.375, w.b, w.sfb, -3.0, w.M, w.K, w.L)
    assert np.isnan(c).any()
    assert np.array_equal(np.isnan(c), np.isnan(cn))
    fin = ~np.isnan(cn)
    assert _same_bits(c[fin], cn[fin]) and _same_bits(T[fin], Tn[fin])
    u, nan = cref.gemv_exact_units(w.A, w.sfa, w.b, w.sfb, w.M, w.K, w.L)
    un, nann = NV.gemv_exact_units(w.A, w.sfa, w.b, w.sfb, w.M, w.K, w.L)
    assert np.array_equal(u, un) and np.array_equal(nan, nann)
    assert np.array_equal(nan, np.isnan(c).ravel())


def test_c_fp64_sum_equals_exact_integers():
    finite = [v for v in range(256) if v not in (0x7F, 0xFF)]
    w = workloads.random_workload(9, 1024, 2, seed=21, scale_bytes=finite)
    c, _ = cref.gemv(w.A, w.sfa, 1.0, w.b, w.sfb, 1.0, w.M, w.K, w.L)
    u, nan = cref.gemv_exact_units(w.A, w.sfa, w.b, w.sfb, w.M, w.K, w.L)
    assert not nan.any() and np.all(np.abs(u) < 2 ** 53)
    assert np.array_equal(c.ravel() * 2.0 ** 20, u.astype(np.float64))


def test_thread_count_does_not_change_a_bit(workload):
    w = workload("c1")
    outs = [cref.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, w.M, w.K, w.L, threads=t)
            for t in (1, 2, max(2, cref.max_threads()))]
    for c, T in outs[1:]:
        assert _same_bits(c, outs[0][0]) and _same_bits(T, outs[0][1])


def test_rows_entry_matches_whole_and_rejects_bad_indices():
    w = workloads.random_workload(7, 96, 3, seed=11)
    c, T = cref.gemv(w.A, w.sfa, 1.5, w.b, w.sfb, 0.75, w.M, w.K, w.L)
    ls, ms = np.array([0, 2, 1, 2, 0]), np.array([6, 0, 3, 3, 0])
    c2, T2 = cref.gemv_rows(w.A, w.sfa, 1.5, w.b, w.sfb, 0.75, w.M, w.K, w.L, ls, ms)
    assert _same_bits(c2, c[ls, ms]) and _same_bits(T2, T[ls, ms])
    with pytest.raises(IndexError):
        cref.gemv_rows(w.A, w.sfa, 1.0, w.b, w.sfb, 1.0, w.M, w.K, w.L, [3], [0])
    with pytest.raises(ValueError):
        cref.gemv(w.A, w.sfa, 1.0, w.b, w.sfb, 1.0, w.M, w.K + 16, w.L)


# ------------------------------------------------------------------ grouped form

def test_c_offsets_ownership_equals_numpy():
    rng = np.random.default_rng(3)
    assert cref.experts_from_offsets([2, 2, 5, 6], 8).tolist() == [0, 0, 2, 2, 2, 3, -1, -1]
    for _ in range(200):
        E = int(rng.integers(1, 10))
        offs = rng.integers(-2, 12, E)                 # decreasing and negative ones too
        T = int(rng.integers(0, 14))
        assert np.array_equal(cref.experts_from_offsets(offs, T), G.experts_from_offsets(offs, T))


@pytest.mark.parametrize("name", ["g0"])
def test_c_grouped_equals_numpy(name):
    g = workloads.make_grouped(name)
    owner = np.asarray(g.expert_of).copy()
    owner[::5] = -1                                    # tokens without an expert
    c, T = cref.gemv_grouped(g.A, g.sfa, g.g_a, g.b, g.sfb, g.g_b, owner, g.M, g.K)
    cn, Tn = G.gemv_grouped(g.A, g.sfa, g.g_a, g.b, g.sfb, g.g_b, owner, g.M, g.K)
    assert _same_bits(c, cn) and _same_bits(T, Tn)
    assert (c[::5] == 0).all()


# ------------------------------------------------------------------ quantizer

def _torch_e4m3(v):
    return torch.from_numpy(np.asarray(v, dtype=np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


@pytest.mark.parametrize("rounding", ["lut", "rne"])
def test_c_quantizer_equals_numpy(rounding):
    rng = np.random.default_rng(11)
    K, L = 1024, 6
    x = rng.standard_normal((L, K)).astype(np.float32)
    x *= np.exp2(rng.integers(-30, 14, (L, K // 16, 1))).repeat(16, axis=2).reshape(L, K)
    x[0, :16] = 0.0
    x[1, 16:32] = np.float32(-0.0)
    x[2, 32:48] = np.linspace(-5e4, 5e4, 16)           # block scale NaN: codes 0
    x[3, 48:64] = np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 2)
    for gs in (1.0, 0.0123, 2.0 ** -7, 37.5):
        p, s = cref.quantize_activation(x, gs, rounding)
        pn, sn = Q.quantize_activation(x, gs, rounding)
        assert np.array_equal(s, sn), gs
        assert np.array_equal(p, pn), gs
    p, s = cref.quantize_activation(x, 1.0, rounding)
    assert s[2, 2] == 0x7F and (p[2, 16:24] == 0).all()


def test_c_quantizer_scale_bytes_equal_torch_cast_over_the_range():
    """One block per value v: its largest element is 6 v (gs = 1), so the scale byte is the
    E4M3 cast of fp32(6 v / 6) = v; it must equal torch's cast of the same fp32 value."""
    pos = oracle.E4M3FN_TABLE[:0x7F]
    mids = np.concatenate([(pos[:-1] + pos[1:]) / 2, [464.0]])
    rng = np.random.default_rng(2)
    v = np.concatenate([pos, mids, np.nextafter(mids.astype(np.float32), 0),
                        np.nextafter(mids.astype(np.float32), np.inf), rng.uniform(0, 520, 4000),
                        np.exp2(rng.uniform(-30, 20, 2000))]).astype(np.float32)
    six_v = (v * np.float32(6.0)).astype(np.float32)
    v = (six_v / np.float32(6.0)).astype(np.float32)          # the value the quantizer casts
    x = np.zeros((v.size, 16), np.float32)
    x[:, 0] = six_v
    _, s = cref.quantize_activation(x, 1.0, "lut")
    want = _torch_e4m3(np.maximum(v, np.float32(1e-8)))
    assert np.array_equal(s[:, 0], want)


# ------------------------------------------------------------------ fp16

def test_c_fp16_every_value_and_midpoint():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    fin = np.isfinite(vals)
    assert np.array_equal(cref.fp16_bits(vals[fin]), bits[fin])
    pos = np.arange(0, 0x7C00, dtype=np.uint16)
    v = pos.view(np.float16).astype(np.float64)
    mid = (v[:-1] + v[1:]) / 2
    expect = np.where(pos[:-1] % 2 == 0, pos[:-1], pos[1:])
    assert np.array_equal(cref.fp16_bits(mid), expect)
    assert np.array_equal(cref.fp16_bits(np.nextafter(mid, -np.inf)), pos[:-1])
    assert np.array_equal(cref.fp16_bits(np.nextafter(mid, np.inf)), pos[1:])
    assert np.array_equal(cref.fp16_bits(-mid), expect | 0x8000)
    assert cref.fp16_bits(np.array([65519.99, 65520.0, -1e9, 2.0 ** -25, 3 * 2.0 ** -26,
                                    np.inf, np.nan])).tolist() == \
        [0x7BFF, 0x7C00, 0xFC00, 0x0000, 0x0001, 0x7C00, 0x7E00]


# ------------------------------------------------------------------ planted mistakes

# (source text, its replacement): each a plausible slip in the C oracle
C_MUTANTS = {
    "E2M1 sign ignored": ("return (code & 8u) ? -mag : mag;", "return mag;"),
    "E4M3 bias off by one": ("ldexp(1.0 + m / 8.0, (int)E - 7)", "ldexp(1.0 + m / 8.0, (int)E - 6)"),
    "high nibble read as even k": ("return (k & 1) ? (unsigned)(byte >> 4) : (unsigned)(byte & 15u);",
                                   "return (k & 1) ? (unsigned)(byte & 15u) : (unsigned)(byte >> 4);"),
    "sfb dropped": ("E2M1_VAL[nibble(b_row, k)] * E4M3_VAL[sb_row[k / 16]]",
                    "E2M1_VAL[nibble(b_row, k)]"),
    "block index shifted": ("E4M3_VAL[sa_row[k / 16]]", "E4M3_VAL[sa_row[(k / 16 + 1) % (K / 16)]]"),
    "g_b dropped": ("c_ref[i] = (S * ga) * gb;", "c_ref[i] = S * ga;"),
    "rows and batches transposed": ("const uint8_t* a_row = A + (l * M + m) * (K / 2);\n"
                                    "  const uint8_t* sa_row = sfa + (l * M + m) * (K / 16);",
                                    "const uint8_t* a_row = A + (m * L_ + l) * (K / 2);\n"
                                    "  const uint8_t* sa_row = sfa + (m * L_ + l) * (K / 16);"),
}

# mistakes in the quantizer, caught by the torch cast and the numpy formulation
Q_MUTANTS = {
    "scale saturates instead of NaN": ("if (v > 464.0f) return 0x7Fu;", "if (v > 464.0f) return 0x7Eu;"),
    "scale ties to the odd byte": ("(d == best_d && (byte & 1u) == 0)", "(d == best_d && (byte & 1u) == 1)"),
    "half-step table misprinted": ("{0, 1, 2, 3, 4, 4, 5, 5, 6, 6, 6, 7, 7}",
                                   "{0, 1, 2, 3, 4, 5, 5, 5, 6, 6, 6, 7, 7}"),
    "global scale multiplies": ("xn[i] = xb[i] / gs;", "xn[i] = xb[i] * gs;"),
}


def _build_mutant(tmp_path, old, new, name):
    src = open(cref.SOURCE).read()
    assert src.count(old) >= 1, f"mutation target of {name!r} not in the source"
    if name == "rows and batches transposed":
        # one_row has no L: thread it through as a file-scope variable for this mutant only
        src = src.replace("static void one_row(", "static int64_t L_ = 1;\nstatic void one_row(")
        src = src.replace("  init_tables();\n  for (int64_t i = 0; i < n; ++i)\n    if (ls[i]",
                          "  init_tables();\n  L_ = L;\n  for (int64_t i = 0; i < n; ++i)\n    if (ls[i]")
        src = src.replace("  init_tables();\n  const double ga = (double)g_a, gb = (double)g_b, gg",
                          "  init_tables();\n  L_ = L;\n  const double ga = (double)g_a, gb = (double)g_b, gg")
    src = src.replace(old, new)
    path = tmp_path / "mutant.c"
    path.write_text(src)
    so = tmp_path / f"mutant_{abs(hash(name))}.so"
    cc = os.environ.get("CC", "gcc")
    r = subprocess.run([cc, *cref.CFLAGS, str(path), "-o", str(so), "-lm"], capture_output=True,
                       text=True)
    assert r.returncode == 0, r.stderr
    return str(so)


@pytest.fixture
def use_library(monkeypatch):
    def use(path):
        monkeypatch.setattr(cref, "_lib", None)
        monkeypatch.setattr(cref, "LIB_PATH", path)
        monkeypatch.setattr(cref, "build", lambda verbose=False: path)
        return cref.lib()
    return use


@pytest.mark.skipif(shutil.which(os.environ.get("CC", "gcc")) is None, reason="no C compiler")
@pytest.mark.parametrize("mistake", sorted(C_MUTANTS))
def test_c_planted_gemv_mistake_is_caught(tmp_path, use_library, mistake):
    from test_oracle_gemv import golden_failures

    use_library(_build_mutant(tmp_path, *C_MUTANTS[mistake], mistake))
    caught = bool(golden_failures(cref.gemv))
    if mistake == "high nibble read as even k":
        # both operands read the same way: a permutation of k inside each pair, which leaves
        # every output unchanged; the quantizer's packing (same source) catches it instead
        assert not caught
        x = np.float32([[6.0, 0.5] + [0.0] * 14])
        p, _ = cref.quantize_activation(x, 1.0, "lut")
        assert p[0, 0] == (1 << 4) | 7                 # quantizer writes (odd << 4) | even
        return
    assert caught, f"no pin catches: {mistake}"


@pytest.mark.skipif(shutil.which(os.environ.get("CC", "gcc")) is None, reason="no C compiler")
@pytest.mark.parametrize("mistake", sorted(Q_MUTANTS))
def test_c_planted_quantizer_mistake_is_caught(tmp_path, use_library, mistake):
    use_library(_build_mutant(tmp_path, *Q_MUTANTS[mistake], mistake))
    caught = False
    try:
        test_c_quantizer_scale_bytes_equal_torch_cast_over_the_range()
        for r in ("lut", "rne"):
            test_c_quantizer_equals_numpy(r)
    except AssertionError:
        caught = True
    assert caught, f"no pin catches: {mistake}"

"""GPU parity of the activation quantizer and of the GEMV with a bf16 vector, through the C ABI.

The quantized bytes (packed E2M1 codes and E4M3 block scales) are compared bit for bit with
oracle/quantize.py: both sides take every decision in fp32 with correctly rounded divisions, so
the bytes are unique.  The GEMV output is compared with the oracle GEMV of the oracle's quantized
vector (global scale g_b = the activation's global scale) under the parity tolerance, and the fused
path (quantization inside the register-vector TMA kernel) must equal, bit for bit, the same plan
run on the packed vector.  Inputs: seeded normal bf16 values at block magnitudes across the whole
E4M3 range, plus planted blocks of zeros, signed zeros, grid points, exact rounding midpoints and
their bf16 neighbours, saturating magnitudes, tiny and subnormal values.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import quantize as Q
from parity import assert_parity

pytestmark = pytest.mark.gpu

ROUNDINGS = [(0, "lut"), (1, "rne")]
GRID = np.float32([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
MIDS = np.float32([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


@pytest.fixture(scope="module")
def pkg():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    from decode_nvfp4_gemv_gb300 import build

    build.build()
    import decode_nvfp4_gemv_gb300 as p

    p.load_library()
    return p


def bf16_round(x):
    """fp32 -> nearest bf16 (ties to even), returned as fp32 (finite inputs)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def bf16_bits(x32):
    return (np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def dev_bf16(x32):
    return torch.from_numpy(bf16_bits(x32).view(np.int16)).cuda()


def special_blocks(gs):
    """16-element blocks of edge values for global scale gs (bf16-rounded), all with a finite
    block scale (overflow_blocks has the ones whose scale is NaN)."""
    up, down = np.float32(1 + 2.0 ** -7), np.float32(1 - 2.0 ** -8)   # bf16 neighbours of 1
    mids = np.concatenate([MIDS, -MIDS, [0.3]]).astype(np.float32)      # 15 values
    rows = [
        np.zeros(16, np.float32),
        np.array([0.0, -0.0] * 8, np.float32),
        np.concatenate([GRID, -GRID]) * gs,                      # grid points, scale 1
        np.concatenate([[6.0], mids]) * gs,                      # exact midpoints, scale 1
        np.concatenate([[6.0], mids * up]) * gs,                 # just above the midpoints
        np.concatenate([[6.0], mids * down]) * gs,               # just below
        np.concatenate([[-6.0], mids]) * gs * 448,               # the largest scale, exactly
        np.concatenate([[6.0 * 460], mids * 460]) * gs,          # 448 < amax / 6 < 464: 448
        np.full(16, 1e-12, np.float32),                          # scale 0 (floor 1e-8)
        np.array([1e-40, -1e-39, 3e-38, 0.0] * 4, np.float32),   # subnormal and tiny
        np.concatenate([[6.0, 0.0], GRID[1:], -GRID[1:]]) * gs * 2.0 ** -9,   # smallest scale
        np.concatenate([[6.0], mids]) * gs * 2.0 ** -7,
        np.linspace(0.01, 7.0, 16, dtype=np.float32) * gs,
    ]
    return bf16_round(np.stack(rows).astype(np.float32))


def overflow_blocks(gs):
    """Blocks whose largest |x / gs| / 6 lies past 464: no finite E4M3 scale, so the page's cast
    gives NaN (0x7F) and the block's codes are 0."""
    rows = [np.full(16, 3000.0 * 6, np.float32) * gs,
            np.linspace(-1e5, 1e5, 16, dtype=np.float32) * gs,
            np.concatenate([[6.0 * 466.0, 0.0], GRID[1:], -GRID[1:]]).astype(np.float32) * gs]
    return bf16_round(np.stack(rows).astype(np.float32))


def activation(K, L, seed, gs, plant=True, overflow=False):
    """Seeded normal bf16 values, each 16-block multiplied by 2^e (e spread so that block scales
    cover the E4M3 range for this gs), with the special blocks planted at seeded positions (and
    the overflowing ones too, if asked: their scales are NaN)."""
    x = workloads.normal_bf16(seed, "x", K * L).reshape(L, K // 16, 16)
    e = (np.arange(L * (K // 16)) * 7 % 31 - 22).reshape(L, K // 16, 1).astype(np.float32)
    x = bf16_round(x * np.float32(gs) * np.exp2(e))
    if plant:
        sp = special_blocks(np.float32(gs))
        if overflow:
            sp = np.concatenate([sp, overflow_blocks(np.float32(gs))])
        flat = x.reshape(-1, 16)
        idx = (np.arange(len(sp)) * 2654435761 + seed) % len(flat)
        flat[idx] = sp[: len(idx)]
    return x.reshape(L, K)


def run_quantize(pkg, x, gs, rounding):
    L, K = x.shape
    guard = 64
    b = torch.full((L * K // 2 + guard,), 0xA5, dtype=torch.uint8, device="cuda")
    s = torch.full((L * K // 16 + guard,), 0x5A, dtype=torch.uint8, device="cuda")
    pkg.nvfp4_quantize_activation(dev_bf16(x), gs, b, s, K, L, rounding=rounding)
    torch.cuda.synchronize()
    b, s = b.cpu().numpy(), s.cpu().numpy()
    assert (b[L * K // 2:] == 0xA5).all() and (s[L * K // 16:] == 0x5A).all(), "wrote past the end"
    return b[: L * K // 2].reshape(L, K // 2), s[: L * K // 16].reshape(L, K // 16)


def assert_bytes_equal(got, ref, what):
    if not np.array_equal(got, ref):
        bad = np.argwhere(got != ref)
        raise AssertionError(f"{what}: {len(bad)} bytes differ, first at {bad[0].tolist()}: "
                             f"gpu={got[tuple(bad[0])]:#04x} oracle={ref[tuple(bad[0])]:#04x}")


# ------------------------------------------------------------------ the quantizer on its own

QSHAPES = [(16, 1), (48, 3), (256, 2), (1040, 1), (4096, 5), (16384, 1), (7168, 8)]


@pytest.mark.parametrize("rounding,name", ROUNDINGS, ids=[r[1] for r in ROUNDINGS])
@pytest.mark.parametrize("gs", [1.0, 2.0 ** -7, 0.0123, 37.5])
def test_quantizer_bytes_bit_exact(pkg, rounding, name, gs):
    for K, L in QSHAPES:
        x = activation(K, L, seed=K + 31 * L, gs=gs, overflow=True)
        b, s = run_quantize(pkg, x, gs, rounding)
        pr, sr = Q.quantize_activation(x, gs, name)
        assert_bytes_equal(s, sr, f"sfb K={K} L={L} gs={gs} {name}")
        assert_bytes_equal(b, pr, f"b K={K} L={L} gs={gs} {name}")


def test_special_blocks_alone(pkg):
    """Each edge block in a K=16 vector of its own (one thread, one block)."""
    for gs in (1.0, 0.0123):
        sp = special_blocks(np.float32(gs))
        for rounding, name in ROUNDINGS:
            b, s = run_quantize(pkg, sp, gs, rounding)
            pr, sr = Q.quantize_activation(sp, gs, name)
            assert_bytes_equal(s, sr, f"special sfb gs={gs} {name}")
            assert_bytes_equal(b, pr, f"special b gs={gs} {name}")
            if gs == 1.0:
                assert s[6, 0] == 0x7E                     # the largest finite block scale
                assert s[7, 0] == 0x7E                     # rounds down to 448
                assert s[8, 0] == 0x00                     # below the smallest subnormal
            ob = overflow_blocks(np.float32(gs))
            b, s = run_quantize(pkg, ob, gs, rounding)
            pr, sr = Q.quantize_activation(ob, gs, name)
            assert_bytes_equal(s, sr, f"overflow sfb gs={gs} {name}")
            assert_bytes_equal(b, pr, f"overflow b gs={gs} {name}")
            assert (s == 0x7F).all() and (b == 0).all()    # NaN scales, codes 0
    # the edge itself (global scale 1, exact): amax / 6 == 464 ties to 448; the next bf16 above
    # 2784 (= 6 * 464) gives NaN
    edge = np.zeros((2, 16), np.float32)
    edge[0, 0], edge[1, 0] = 2784.0, 2800.0
    for rounding, name in ROUNDINGS:
        b, s = run_quantize(pkg, edge, 1.0, rounding)
        assert s[:, 0].tolist() == [0x7E, 0x7F] and (b[1] == 0).all()
        pr, sr = Q.quantize_activation(edge, 1.0, name)
        assert_bytes_equal(s, sr, f"edge sfb {name}")
        assert_bytes_equal(b, pr, f"edge b {name}")


@pytest.mark.parametrize("flags", [1, 1 | 4], ids=["quantizer-then-gemv", "in-gemv"])
def test_overflowing_block_gives_nan_on_both_sides(pkg, flags):
    """A planted block whose scale has no finite E4M3 encoding: its scale byte is NaN on the GPU
    as in the oracle, so every output of that batch is NaN on both sides; the other batch is
    unaffected and within tolerance."""
    M, K, L = 256, 2048, 2
    gs = 0.0173
    w = workloads.random_workload(M, K, L, seed=77, scale_bytes=workloads.pow2_scale_bytes(-3, 2))
    x = activation(K, L, seed=78, gs=gs, plant=False)
    x[1, 512:528] = overflow_blocks(np.float32(gs))[0]
    pr, sr = Q.quantize_activation(x, gs, "lut")
    assert sr[1, 32] == 0x7F and (sr[0] != 0x7F).all()
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, pr, sr, gs, M, K, L)
    assert np.isnan(ref[1]).all() and not np.isnan(ref[0]).any()
    A, sfa = torch.from_numpy(w.A).cuda(), torch.from_numpy(w.sfa).cuda()
    c, b, s = gemv_bf16(pkg, A, sfa, w.g_a, x, gs, 0, M, {"kernel": 4, "flags": flags})
    assert_bytes_equal(s, sr, "sfb_out with an overflowing block")
    assert_bytes_equal(b, pr, "b_out with an overflowing block")
    assert np.isnan(c[1]).all()
    assert_parity(c, ref, T, "overflowing block")


def test_the_two_roundings_differ_where_expected(pkg):
    """Midpoints 2.5, 3.5 and 5 round down under the half-step table but 3.5 rounds up to 4 under
    nearest-even (and 2.5, 5 stay): the GPU shows the same split as the oracle."""
    x = bf16_round(np.float32([[6.0, 2.5, 3.5, 5.0] + [0.0] * 12]))
    b_lut, _ = run_quantize(pkg, x, 1.0, 0)
    b_rne, _ = run_quantize(pkg, x, 1.0, 1)
    codes = lambda b: [int(b[0, j // 2] >> (4 * (j % 2)) & 15) for j in range(4)]
    assert codes(b_lut) == [7, 4, 5, 6]
    assert codes(b_rne) == [7, 4, 6, 6]


def test_quantizer_statuses(pkg):
    x = dev_bf16(np.zeros((1, 256), np.float32))
    b = torch.empty(128, dtype=torch.uint8, device="cuda")
    s = torch.empty(16, dtype=torch.uint8, device="cuda")
    for kw in (dict(rounding=7), dict(gs=0.0)):
        with pytest.raises(pkg.NVFP4Error) as e:
            pkg.nvfp4_quantize_activation(x, kw.get("gs", 1.0), b, s, 256, 1,
                                          rounding=kw.get("rounding", 0))
        assert e.value.status == 1
    with pytest.raises(pkg.NVFP4Error) as e:
        pkg.nvfp4_quantize_activation(x, 1.0, b[1:], s, 240, 1)
    assert e.value.status == 2


# ------------------------------------------------------------------ the GEMV with a bf16 vector

def tma_plan(TR=0, NS=0, P=0, W=0, rv=False, flags=0):
    return dict(kernel=4 if rv else 3, tile_rows=TR, stages=NS, ctas_per_batch=P,
                warps_per_cta=W, flags=flags)


IN_GEMV = 4        # NVFP4_FLAG_QUANTIZE_IN_GEMV
FUSED_PLANS = [tma_plan(rv=True, flags=IN_GEMV), tma_plan(rv=True, flags=IN_GEMV | 1),
               tma_plan(rv=True, flags=IN_GEMV | 2), tma_plan(rv=True, TR=3, NS=5, P=2, flags=IN_GEMV),
               tma_plan(rv=True, TR=16, NS=2, P=1, flags=IN_GEMV | 1)]
UNFUSED_PLANS = [None, dict(kernel=1), dict(kernel=2), dict(kernel=2, rows_per_warp=4, k_split=2),
                 tma_plan(), tma_plan(TR=5, NS=3, P=2, W=3, flags=1), tma_plan(rv=True),
                 tma_plan(rv=True, flags=1), tma_plan(rv=True, flags=2)]
GSHAPES = [(129, 256, 3), (7, 1024, 2), (64, 2048, 1), (33, 3072, 2), (300, 5120, 1),
           (40, 16384, 2)]


def gemv_bf16(pkg, A, sfa, g_a, x, gs, rounding, M, plan):
    L, K = x.shape
    b = torch.full((L * K // 2 + 64,), 0xA5, dtype=torch.uint8, device="cuda")
    s = torch.full((L * K // 16 + 64,), 0x5A, dtype=torch.uint8, device="cuda")
    c = torch.full((L, M), float("nan"), dtype=torch.float16, device="cuda")
    pkg.nvfp4_gemv_batched_bf16(A, sfa, g_a, dev_bf16(x), gs, b, s, c, M, K, L,
                                rounding=rounding, plan=plan)
    torch.cuda.synchronize()
    b, s = b.cpu().numpy(), s.cpu().numpy()
    assert (b[L * K // 2:] == 0xA5).all() and (s[L * K // 16:] == 0x5A).all(), "wrote past the end"
    return c.cpu().numpy(), b[: L * K // 2].reshape(L, K // 2), s[: L * K // 16].reshape(L, K // 16)


def packed_gemv(pkg, A, sfa, g_a, b, s, g_b, M, K, L, plan):
    c = torch.full((L, M), float("nan"), dtype=torch.float16, device="cuda")
    pkg.nvfp4_gemv_batched_ex(A, sfa, g_a, torch.from_numpy(b).cuda(), torch.from_numpy(s).cuda(),
                              g_b, c, M, K, L, plan=plan)
    torch.cuda.synchronize()
    return c.cpu().numpy()


@pytest.mark.parametrize("rounding,name", ROUNDINGS, ids=[r[1] for r in ROUNDINGS])
@pytest.mark.parametrize("shape", GSHAPES, ids=[f"{m}x{k}x{l}" for m, k, l in GSHAPES])
def test_gemv_bf16_all_plans(pkg, shape, rounding, name):
    M, K, L = shape
    gs = 0.0173
    w = workloads.random_workload(M, K, L, seed=M + K + 7 * L,
                                  scale_bytes=workloads.pow2_scale_bytes(-4, 3), g_a=0.75, g_b=1.0)
    x = activation(K, L, seed=M * 3 + K, gs=gs, plant=K >= 1024)
    pr, sr = Q.quantize_activation(x, gs, name)
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, pr, sr, gs, M, K, L)
    A, sfa = torch.from_numpy(w.A).cuda(), torch.from_numpy(w.sfa).cuda()
    for plan in FUSED_PLANS + UNFUSED_PLANS:
        if plan is not None and plan.get("k_split", 0) > -(-K // 1024):
            continue                      # more K splits than 1024-element steps
        if plan is not None and plan.get("ctas_per_batch", 0) > M:
            plan = dict(plan, ctas_per_batch=M)
        try:
            c, b, s = gemv_bf16(pkg, A, sfa, w.g_a, x, gs, rounding, M, plan)
        except pkg.NVFP4Error as e:       # a forced ring too large for shared memory
            assert e.status == 3 and ("shared memory" in e.message or "warp count" in e.message), e
            continue
        what = f"{shape} {name} {plan}"
        assert_bytes_equal(s, sr, what + " sfb_out")
        assert_bytes_equal(b, pr, what + " b_out")
        assert not np.isnan(c).any(), what
        assert_parity(c, ref, T, what)
        packed_plan = None if plan is None else dict(plan, flags=plan.get("flags", 0) & ~IN_GEMV)
        c_packed = packed_gemv(pkg, A, sfa, w.g_a, pr, sr, gs, M, K, L, packed_plan)
        assert np.array_equal(c.view(np.uint16), c_packed.view(np.uint16)), what + " vs packed"


@pytest.mark.parametrize("flags", [1, 1 | IN_GEMV], ids=["quantizer-then-gemv", "in-gemv"])
def test_gemv_bf16_full_decode_shape(pkg, workload, flags):
    """The decode projection's shape (M=7168, K=16384, L=1) with the automatic plan and the flags
    the bench times: b_out / sfb_out bit exact, c within tolerance, deterministic."""
    w = workload("c2")
    M, K, L = w.M, w.K, w.L
    assert pkg.nvfp4_gemv_plan(M, K, L).kernel == 4
    x = workloads.normal_bf16(12, "x", K * L).reshape(L, K)
    gs = float(np.abs(x).max() / (448.0 * 6.0))
    pr, sr = Q.quantize_activation(x, gs, "lut")
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, pr, sr, gs, M, K, L)
    A, sfa = torch.from_numpy(w.A).cuda(), torch.from_numpy(w.sfa).cuda()
    c, b, s = gemv_bf16(pkg, A, sfa, w.g_a, x, gs, 0, M, {"flags": flags})
    assert_bytes_equal(s, sr, "c2 sfb_out")
    assert_bytes_equal(b, pr, "c2 b_out")
    assert_parity(c, ref, T, "c2 bf16 vector")
    c2, _, _ = gemv_bf16(pkg, A, sfa, w.g_a, x, gs, 0, M, {"flags": flags})
    assert np.array_equal(c.view(np.uint16), c2.view(np.uint16))


def test_back_to_back_calls_reuse_the_vector_buffers(pkg):
    """Decode reuses b_out / sfb_out every step: a chain of calls on one stream with new
    activations each time (no host sync between them) must give each step's own result."""
    M, K, L = 4096, 4096, 1
    assert pkg.nvfp4_gemv_plan(M, K, L).kernel == 4
    w = workloads.random_workload(M, K, L, seed=5, g_a=0.5, g_b=1.0)
    A, sfa = torch.from_numpy(w.A).cuda(), torch.from_numpy(w.sfa).cuda()
    gs = 0.01
    xs = [activation(K, L, seed=100 + i, gs=gs, plant=False) for i in range(6)]
    xd = [dev_bf16(x) for x in xs]
    b = torch.empty(L * K // 2, dtype=torch.uint8, device="cuda")
    s = torch.empty(L * K // 16, dtype=torch.uint8, device="cuda")
    for flags in (1, 1 | IN_GEMV):
        cs = [torch.empty((L, M), dtype=torch.float16, device="cuda") for _ in xs]
        for x, c in zip(xd, cs):
            pkg.nvfp4_gemv_batched_bf16(A, sfa, w.g_a, x, gs, b, s, c, M, K, L,
                                        plan={"flags": flags})
        torch.cuda.synchronize()
        for i, (x, c) in enumerate(zip(xs, cs)):
            pr, sr = Q.quantize_activation(x, gs, "lut")
            ref, T = oracle.gemv(w.A, w.sfa, w.g_a, pr, sr, gs, M, K, L)
            assert_parity(c.cpu().numpy(), ref, T, f"step {i} flags {flags}")


def test_in_gemv_flag_rules(pkg):
    M, K, L = 64, 1024, 1
    w = workloads.random_workload(M, K, L, seed=6)
    A, sfa = torch.from_numpy(w.A).cuda(), torch.from_numpy(w.sfa).cuda()
    x = activation(K, L, seed=1, gs=1.0, plant=False)
    with pytest.raises(pkg.NVFP4Error) as e:          # needs the register-vector kernel
        gemv_bf16(pkg, A, sfa, 1.0, x, 1.0, 0, M, dict(kernel=2, flags=IN_GEMV))
    assert e.value.status == 3
    with pytest.raises(pkg.NVFP4Error) as e:          # meaningless for a packed vector
        packed_gemv(pkg, A, sfa, 1.0, w.b, w.sfb, 1.0, M, K, L, {"flags": IN_GEMV})
    assert e.value.status == 1
    # a matrix off a 16-byte boundary: the in-GEMV form refuses it; the two-launch form (the
    # default) quantizes first and runs the GEMV's unaligned form
    raw = torch.empty(A.numel() + 16, dtype=torch.uint8, device="cuda")
    A1 = raw[3:3 + A.numel()]
    A1.copy_(A.reshape(-1))
    with pytest.raises(pkg.NVFP4Error) as e:          # the automatic plan here: not the ring
        gemv_bf16(pkg, A1, sfa, 1.0, x, 1.0, 0, M, {"flags": IN_GEMV})
    assert e.value.status == 3
    with pytest.raises(pkg.NVFP4Error) as e:          # the ring forced: its unaligned form
        gemv_bf16(pkg, A1, sfa, 1.0, x, 1.0, 0, M, {"kernel": 4, "flags": IN_GEMV})
    assert e.value.status == 2
    c1, b1, s1 = gemv_bf16(pkg, A1, sfa, 1.0, x, 1.0, 0, M, None)
    pr, sr = Q.quantize_activation(x, 1.0, "lut")
    assert_bytes_equal(b1, pr, "b_out, misaligned A")
    assert_bytes_equal(s1, sr, "sfb_out, misaligned A")
    ref, T = oracle.gemv(w.A, w.sfa, 1.0, pr, sr, 1.0, M, K, L)
    assert_parity(c1, ref, T, "bf16 vector, misaligned A")


def test_gemv_bf16_empty_and_statuses(pkg):
    A = torch.zeros(4 * 128, dtype=torch.uint8, device="cuda")
    sfa = torch.zeros(4 * 16, dtype=torch.uint8, device="cuda")
    x = dev_bf16(np.ones((1, 256), np.float32))
    b = torch.full((128,), 7, dtype=torch.uint8, device="cuda")
    s = torch.full((16,), 7, dtype=torch.uint8, device="cuda")
    c = torch.zeros((1, 4), dtype=torch.float16, device="cuda")
    pkg.nvfp4_gemv_batched_bf16(A, sfa, 1.0, x, 1.0, b, s, c, 0, 256, 1)
    torch.cuda.synchronize()
    assert (b.cpu().numpy() == 7).all() and (s.cpu().numpy() == 7).all()
    with pytest.raises(pkg.NVFP4Error) as e:
        pkg.nvfp4_gemv_batched_bf16(A, sfa, 1.0, x, -2.0, b, s, c, 4, 256, 1)
    assert e.value.status == 1


@pytest.mark.parametrize("case", list(range(100)))
def test_random_bf16_vector_cases(pkg, case):
    """Seeded random bf16-vector GEMVs: K (any multiple of 16), L, M, global scale, rounding, the
    matrix's alignment and the plan drawn at random.  The packed vector the call writes must equal
    the oracle's quantization byte for byte; the output is checked under the tolerance."""
    rng = np.random.default_rng(21_000 + case)
    K = 16 * int(rng.choice([1, 3, 16, 17, 64, 65, 128, 256, 513]))
    L = int(rng.integers(1, 5))
    M = int(rng.integers(1, 300))
    gs = float(np.float32(rng.choice([1.0, 2.0 ** -5, 0.0173, 3.7])))
    rounding, name = ROUNDINGS[int(rng.integers(0, 2))]
    w = workloads.random_workload(M, K, L, seed=22_000 + case,
                                  scale_bytes=workloads.pow2_scale_bytes(-4, 3), g_a=0.75)
    x = activation(K, L, seed=23_000 + case, gs=gs, plant=K >= 256)
    pr, sr = Q.quantize_activation(x, gs, name)
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, pr, sr, gs, M, K, L)
    A = torch.from_numpy(w.A).cuda()
    if rng.random() < 0.4:                            # the matrix off a 16-byte boundary
        off = int(rng.integers(1, 16))
        raw = torch.empty(A.numel() + 32, dtype=torch.uint8, device="cuda")
        A = raw[off:off + w.A.size]
        A.copy_(torch.from_numpy(w.A.ravel()).cuda())
    sfa = torch.from_numpy(w.sfa).cuda()
    plan = [None, {"flags": 1}, {"flags": 1 | IN_GEMV}, {"kernel": 6}][int(rng.integers(0, 4))]
    try:
        c, b, s = gemv_bf16(pkg, A, sfa, w.g_a, x, gs, rounding, M, plan)
    except pkg.NVFP4Error as e:   # the in-GEMV form needs the aligned register-vector kernel
        assert plan is not None and plan["flags"] & IN_GEMV and e.status in (2, 3), (plan, e)
        return
    what = f"case {case}: M={M} K={K} L={L} gs={gs} {name} plan={plan}"
    assert_bytes_equal(b, pr, what + " b_out")
    assert_bytes_equal(s, sr, what + " sfb_out")
    assert not np.isnan(c).any(), what
    assert_parity(c, ref, T, what)

"""Seeded random sweeps on the GPU: shapes, operand alignments and forced plans drawn at random,
every output checked against the oracle under the parity tolerance, for the batched GEMV (below),
the small-N entry point and the grouped form (their own tests at the end).

Each batched case draws M in [1, 300], K in 16..4096 (multiples of 16, with K % 32, K % 256 and
K % 1024 each varied), L in [1, 4]; each of A, sfa, b, sfb lands 0 to 15 bytes past a 16-byte
boundary (aligned half of the time); the plan is automatic or forces a kernel with random fields.
A forced plan the planner refuses for that shape (UNSUPPORTED_SHAPE or MISALIGNED) is skipped: the
refusal itself is the host-side rule under test, and the automatic plan still runs on the same
inputs.  Block scales are positive powers of two, 2^-4 to 2^3 (the tensor cores read them as
unsigned E4M3).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import assert_parity

pytestmark = pytest.mark.gpu

N_CASES = 400


@pytest.fixture(scope="module")
def pkg():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    from decode_nvfp4_gemv_gb300 import build

    build.build()
    import decode_nvfp4_gemv_gb300 as p

    p.load_library()
    return p


def placed(x, offset):
    raw = torch.full((x.size + offset + 64,), 0xEE, dtype=torch.uint8, device="cuda")
    view = raw[offset:offset + x.size]
    view.copy_(torch.from_numpy(np.ascontiguousarray(x).ravel()))
    return view, raw


def random_plan(rng):
    kind = rng.integers(0, 8)
    if kind <= 1:
        return None                                   # automatic, twice as likely
    kernel = int(rng.choice([1, 2, 3, 4, 5, 6]))
    plan = {"kernel": kernel}
    if rng.random() < 0.5:
        plan["warps_per_cta"] = int(rng.integers(1, 9))
    if rng.random() < 0.5:
        plan["ctas_per_batch"] = int(rng.integers(1, 20))
    if kernel in (3, 4) and rng.random() < 0.5:
        plan["tile_rows"] = int(rng.integers(1, 33))
        plan["stages"] = int(rng.integers(2, 5))
    if kernel == 5:
        plan.pop("warps_per_cta", None)
        plan.pop("ctas_per_batch", None)
        if rng.random() < 0.5:
            plan["k_split"] = int(rng.integers(1, 4))
    if kernel == 2 and rng.random() < 0.5:
        plan["rows_per_warp"] = int(rng.choice([1, 2, 4]))
    plan["flags"] = int(rng.choice([0, 1, 2]))
    return plan


CASES = list(range(N_CASES))


@pytest.mark.parametrize("case", CASES)
def test_random_case(pkg, case):
    rng = np.random.default_rng(1000 + case)
    M = int(rng.integers(1, 301))
    K = 16 * int(rng.choice([1, 2, 3, 16, 17, 32, 64, 65, 128, 129, 256]))
    L = int(rng.integers(1, 5))
    aligned = rng.random() < 0.5
    offsets = (0, 0, 0, 0) if aligned else tuple(int(x) for x in rng.integers(0, 16, 4))
    w = workloads.random_workload(M, K, L, seed=50_000 + case,
                                  scale_bytes=workloads.pow2_scale_bytes(-4, 3),
                                  g_a=float(rng.choice([0.5, 1.0, 1.25])),
                                  g_b=float(rng.choice([0.75, 1.0, 2.0])))
    keep, args = [], []
    for name, off in zip(("A", "sfa", "b", "sfb"), offsets):
        v, raw = placed(getattr(w, name), off)
        keep.append(raw)
        args.append(v)
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, M, K, L)
    plan = random_plan(rng)
    for p in (plan, None) if plan is not None else (None,):
        c = torch.full((L, M), float("nan"), dtype=torch.float16, device="cuda")
        try:
            pkg.nvfp4_gemv_batched_ex(args[0], args[1], w.g_a, args[2], args[3], w.g_b, c, M, K,
                                      L, plan=p)
        except pkg.NVFP4Error as e:
            assert p is not None and e.status in (2, 3), (p, e)   # a refusal of a forced plan
            continue
        torch.cuda.synchronize()
        out = c.cpu().numpy()
        what = f"case {case}: M={M} K={K} L={L} offsets={offsets} plan={p}"
        assert not np.isnan(out).any(), what
        assert_parity(out, ref, T, what)


@pytest.mark.parametrize("case", list(range(40)))
def test_random_wide_k(pkg, case):
    """Wide K on the register-vector ring: 17 to 96 segments (odd and prime counts, a partial last
    segment a quarter of the time), M up to 3000, L up to 2, the vector aligned or not (A aligned,
    as split K needs); the automatic plan, and forced K slices 2 to 8 (equal slices and a shorter
    last one; a split that leaves a slice empty or a slice past 32 segments is refused)."""
    rng = np.random.default_rng(9000 + case)
    nseg = int(rng.integers(17, 97))
    K = nseg * 1024 - (256 * int(rng.integers(1, 4)) if rng.random() < 0.25 else 0)
    M = int(rng.integers(1, 3001))
    L = int(rng.integers(1, 3))
    offsets = (0, 0, 0, 0) if rng.random() < 0.5 else \
        (0, 0, int(rng.integers(0, 16)), int(rng.integers(0, 16)))
    w = workloads.random_workload(M, K, L, seed=60_000 + case,
                                  scale_bytes=workloads.pow2_scale_bytes(-4, 3), g_a=0.75,
                                  g_b=1.25)
    keep, args = [], []
    for name, off in zip(("A", "sfa", "b", "sfb"), offsets):
        v, raw = placed(getattr(w, name), off)
        keep.append(raw)
        args.append(v)
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, M, K, L)
    plans = [None]
    if rng.random() < 0.5:
        plans.append({"kernel": 4, "k_slices": int(rng.integers(2, 9)),
                      "flags": int(rng.choice([0, 1]))})
    for p in plans:
        c = torch.full((L, M), float("nan"), dtype=torch.float16, device="cuda")
        try:
            pkg.nvfp4_gemv_batched_ex(args[0], args[1], w.g_a, args[2], args[3], w.g_b, c, M, K,
                                      L, plan=p)
        except pkg.NVFP4Error as e:
            # refused: a slice left empty, or slices too long for one CTA's warps
            assert p is not None and e.status == 3, (p, e)
            nsl, S = -(-K // 1024), p["k_slices"]
            assert (S - 1) * -(-nsl // S) >= nsl or -(-nsl // S) > 32, (p, e)
            continue
        torch.cuda.synchronize()
        out = c.cpu().numpy()
        what = f"wide case {case}: M={M} K={K} L={L} offsets={offsets} plan={p}"
        assert not np.isnan(out).any(), what
        assert_parity(out, ref, T, what)


@pytest.mark.parametrize("case", list(range(150)))
def test_random_small_n(pkg, case):
    """nvfp4_gemm_small_n: N vectors (1 to 40: above 16 the tensor-core path takes several
    launches) sharing one matrix, any alignment, automatic or forced plans."""
    rng = np.random.default_rng(7000 + case)
    M = int(rng.integers(1, 401))
    K = 16 * int(rng.choice([1, 17, 16, 32, 64, 128, 129, 256]))
    N = int(rng.choice([1, 2, 3, 5, 8, 13, 16, 17, 31, 40]))
    aligned = rng.random() < 0.6
    offsets = (0, 0, 0, 0) if aligned else tuple(int(x) for x in rng.integers(0, 16, 4))
    wa = workloads.random_workload(M, K, 1, seed=80_000 + case,
                                   scale_bytes=workloads.pow2_scale_bytes(-3, 2), g_a=0.5)
    wv = workloads.random_workload(1, K, N, seed=90_000 + case,
                                   scale_bytes=workloads.pow2_scale_bytes(-3, 2), g_b=1.5)
    keep, args = [], []
    for x, off in zip((wa.A[0], wa.sfa[0], wv.b, wv.sfb), offsets):
        v, raw = placed(x, off)
        keep.append(raw)
        args.append(v)
    ref, T = oracle.gemv(np.repeat(wa.A, N, 0), np.repeat(wa.sfa, N, 0), wa.g_a, wv.b, wv.sfb,
                         wv.g_b, M, K, N)
    plans = [None]
    r = rng.random()
    if r < 0.4:
        plans.append({"kernel": 5, "k_split": int(rng.integers(1, 5)),
                      "stages": int(rng.integers(2, 7)), "flags": int(rng.choice([0, 1, 2]))})
    elif r < 0.7:
        plans.append({"kernel": int(rng.choice([1, 2, 4, 6])), "flags": int(rng.choice([0, 1]))})
    for p in plans:
        c = torch.full((N, M), float("nan"), dtype=torch.float16, device="cuda")
        try:
            pkg.nvfp4_gemm_small_n(args[0], args[1], wa.g_a, args[2], args[3], wv.g_b, c, M, K,
                                   N, plan=p)
        except pkg.NVFP4Error as e:
            assert p is not None and e.status in (2, 3), (p, e)
            continue
        torch.cuda.synchronize()
        out = c.cpu().numpy()
        what = f"small-N case {case}: M={M} K={K} N={N} offsets={offsets} plan={p}"
        assert not np.isnan(out).any(), what
        assert_parity(out, ref, T, what)


@pytest.mark.parametrize("case", list(range(150)))
def test_random_grouped(pkg, case):
    """nvfp4_gemv_grouped: random experts, token routing (either form, tokens without an expert),
    output type, alignment and plan."""
    from oracle import grouped as G
    from parity import bf16_bits_to_f64

    rng = np.random.default_rng(11_000 + case)
    E = int(rng.integers(1, 9))
    T_tok = int(rng.integers(1, 13))
    M = int(rng.integers(1, 257))
    K = 16 * int(rng.choice([1, 16, 17, 32, 64, 65, 128]))
    use_offsets = rng.random() < 0.5
    if use_offsets:   # cumulative token counts per expert; tokens past the last count get zeros
        counts = rng.multinomial(T_tok, np.ones(E) / E)
        if rng.random() < 0.3 and counts.sum() > 0:
            counts[-1] = max(0, counts[-1] - 1)
        offsets = np.cumsum(counts).astype(np.int32)
        expert_of = G.experts_from_offsets(offsets, T_tok)
    else:
        expert_of = rng.integers(-1, E, T_tok).astype(np.int32)
    out_bf16 = rng.random() < 0.3
    aligned = rng.random() < 0.6
    offs = (0, 0, 0, 0) if aligned else tuple(int(x) for x in rng.integers(0, 16, 4))
    wa = workloads.random_workload(M, K, E, seed=12_000 + case,
                                   scale_bytes=workloads.pow2_scale_bytes(-3, 2))
    wv = workloads.random_workload(1, K, T_tok, seed=13_000 + case,
                                   scale_bytes=workloads.pow2_scale_bytes(-3, 2))
    g_a = (0.5 + rng.random(E)).astype(np.float32)
    g_b = (0.5 + rng.random(E)).astype(np.float32)
    keep, args = [], []
    for x, off in zip((wa.A, wa.sfa, wv.b, wv.sfb), offs):
        v, raw = placed(x, off)
        keep.append(raw)
        args.append(v)
    ref, Tb = G.gemv_grouped(wa.A, wa.sfa, g_a, wv.b, wv.sfb, g_b, expert_of, M, K)
    plans = [None]
    if rng.random() < 0.5:
        plans.append({"kernel": int(rng.choice([1, 2, 4, 6])), "flags": int(rng.choice([0, 2]))})
    dga, dgb = torch.from_numpy(g_a).cuda(), torch.from_numpy(g_b).cuda()
    route = torch.from_numpy(offsets if use_offsets else expert_of).cuda()
    for p in plans:
        c = torch.full((T_tok, M), -1, dtype=torch.int16, device="cuda")   # 0xFFFF: NaN
        kw = {"expert_offsets": route} if use_offsets else {"expert_of_token": route}
        try:
            pkg.nvfp4_gemv_grouped(args[0], args[1], dga, args[2], args[3], dgb, c, M, K, E,
                                   T_tok, out_dtype=1 if out_bf16 else 0, plan=p, **kw)
        except pkg.NVFP4Error as e:
            assert p is not None and e.status in (2, 3), (p, e)
            continue
        torch.cuda.synchronize()
        bits = c.cpu().numpy().view(np.uint16)
        out = bf16_bits_to_f64(bits) if out_bf16 else bits.view(np.float16).astype(np.float64)
        what = (f"grouped case {case}: E={E} T={T_tok} M={M} K={K} offsets_form={use_offsets} "
                f"bf16={out_bf16} align={offs} plan={p}")
        assert not np.isnan(out).any(), what
        assert_parity(out, ref, Tb, what, fmt="bf16" if out_bf16 else "f16")

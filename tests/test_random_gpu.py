"""Seeded random sweep on the GPU: shapes, operand alignments and forced plans drawn at random,
every output checked against the oracle under the parity tolerance.

Each case draws M in [1, 300], K in 16..4096 (multiples of 16, with K % 32, K % 256 and
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

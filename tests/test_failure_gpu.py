"""Failure detection on the GPU, without a fault.

Every wait in the TMA and tensor-core kernels gives up after one second of wall time; the CTA then
sets its abort flag, lets any copy it issued land, writes NaN to its outputs and exits, so the host
sees the failure in c and the context stays usable.  NVFP4_FLAG_TEST_STALL makes the producer
issue no copies at all, so those waits run out for real.  The tests check that the launch ends
(no hang), that every output is NaN, that CUDA reports no error, and that the next, normal call
on the same stream gives the oracle's values.  Nothing here traps, faults or spins without a
limit.
"""
import time

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import assert_parity

pytestmark = pytest.mark.gpu

STALL = 8


@pytest.fixture(scope="module")
def pkg():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    from decode_nvfp4_gemv_gb300 import build

    build.build()
    import decode_nvfp4_gemv_gb300 as p

    p.load_library()
    return p


PLANS = [dict(kernel=4), dict(kernel=4, flags=1), dict(kernel=4, k_slices=2),
         dict(kernel=4, k_slices=2, flags=1), dict(kernel=3), dict(kernel=5),
         dict(kernel=5, k_split=2), dict(kernel=5, flags=1)]


@pytest.mark.parametrize("plan", PLANS, ids=lambda p: ",".join(f"{k}={v}" for k, v in p.items()))
def test_stalled_producer_gives_nan_and_the_context_recovers(pkg, plan):
    M, K, L = 300, 2048, 2
    w = workloads.random_workload(M, K, L, seed=5, scale_bytes=workloads.pow2_scale_bytes(-3, 2))
    t = {k: torch.from_numpy(getattr(w, k)).cuda() for k in ("A", "sfa", "b", "sfb")}
    s = torch.cuda.Stream()
    c = torch.zeros((L, M), dtype=torch.float16, device="cuda")   # zeros: NaN is the kernel's
    stalled = dict(plan, flags=plan.get("flags", 0) | STALL)
    torch.cuda.synchronize()
    t0 = time.time()
    pkg.nvfp4_gemv_batched_ex(t["A"], t["sfa"], w.g_a, t["b"], t["sfb"], w.g_b, c, M, K, L,
                              stream=s, plan=stalled)
    s.synchronize()                     # raises if the launch faulted
    elapsed = time.time() - t0
    assert elapsed < 60, elapsed        # bounded: each wait gives up after one second
    out = c.cpu().numpy()
    assert np.isnan(out).all(), f"{plan}: {np.count_nonzero(~np.isnan(out))} outputs not NaN"
    # the same stream and context, a normal call: the oracle's values
    c2 = torch.full((L, M), float("nan"), dtype=torch.float16, device="cuda")
    pkg.nvfp4_gemv_batched_ex(t["A"], t["sfa"], w.g_a, t["b"], t["sfb"], w.g_b, c2, M, K, L,
                              stream=s, plan=plan)
    s.synchronize()
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, M, K, L)
    assert_parity(c2.cpu().numpy(), ref, T, f"after a stalled launch, {plan}")


def test_the_flag_is_ignored_by_kernels_without_a_producer(pkg):
    """The stream, shift and simple kernels have no producer to stall: their results stand."""
    M, K, L = 64, 1024, 1
    w = workloads.random_workload(M, K, L, seed=6)
    t = {k: torch.from_numpy(getattr(w, k)).cuda() for k in ("A", "sfa", "b", "sfb")}
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, M, K, L)
    for kernel in (1, 2, 6):
        c = torch.full((L, M), float("nan"), dtype=torch.float16, device="cuda")
        pkg.nvfp4_gemv_batched_ex(t["A"], t["sfa"], w.g_a, t["b"], t["sfb"], w.g_b, c, M, K, L,
                                  plan=dict(kernel=kernel, flags=STALL))
        torch.cuda.synchronize()
        assert_parity(c.cpu().numpy(), ref, T, f"kernel {kernel} with the stall flag")

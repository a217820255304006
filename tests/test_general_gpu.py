"""GPU parity of the general path: any byte alignment of A, sfa, b and sfb, and any K % 16 == 0
(K not a multiple of 32 included), through the C ABI against the oracle.  The planner sends such
calls to the simple kernel (byte loads); the vector-load and TMA kernels refuse them."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import assert_parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def pkg():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    from decode_nvfp4_gemv_gb300 import build

    build.build()
    import decode_nvfp4_gemv_gb300 as p

    p.load_library()
    return p


def placed(x, offset):
    """A device copy of the bytes of x starting `offset` bytes past a 256-byte boundary."""
    raw = torch.full((x.size + offset + 64,), 0xEE, dtype=torch.uint8, device="cuda")
    view = raw[offset:offset + x.size]
    view.copy_(torch.from_numpy(np.ascontiguousarray(x).ravel()))
    return view, raw


@pytest.mark.parametrize("offsets", [(1, 0, 0, 0), (0, 3, 0, 0), (0, 0, 7, 0), (0, 0, 0, 15),
                                     (5, 9, 2, 13), (8, 8, 8, 8)])
def test_unaligned_inputs(pkg, offsets):
    w = workloads.random_workload(70, 1056, 3, seed=31, scale_bytes=workloads.pow2_scale_bytes(-3, 3),
                                  g_a=0.5, g_b=1.5)
    keep = []
    args = []
    for name, off in zip(("A", "sfa", "b", "sfb"), offsets):
        v, raw = placed(getattr(w, name), off)
        keep.append(raw)
        args.append(v)
    c = torch.full((w.L, w.M), float("nan"), dtype=torch.float16, device="cuda")
    pkg.nvfp4_gemv_batched(args[0], args[1], w.g_a, args[2], args[3], w.g_b, c, w.M, w.K, w.L)
    torch.cuda.synchronize()
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, w.M, w.K, w.L)
    assert_parity(c.cpu().numpy(), ref, T, f"offsets {offsets}")
    for plan in (dict(kernel=2), dict(kernel=3), dict(kernel=4)):
        with pytest.raises(pkg.NVFP4Error) as e:
            pkg.nvfp4_gemv_batched_ex(args[0], args[1], w.g_a, args[2], args[3], w.g_b, c, w.M,
                                      w.K, w.L, plan=plan)
        assert e.value.status == 2


@pytest.mark.parametrize("K", [16, 272, 2064, 16368])
def test_k_multiple_of_16_only(pkg, K):
    M, L = 257, 2
    w = workloads.random_workload(M, K, L, seed=K, scale_bytes=workloads.pow2_scale_bytes(-4, 3),
                                  g_a=0.25, g_b=4.0)
    c = torch.full((L, M), float("nan"), dtype=torch.float16, device="cuda")
    t = {k: torch.from_numpy(getattr(w, k)).cuda() for k in ("A", "sfa", "b", "sfb")}
    pkg.nvfp4_gemv_batched(t["A"], t["sfa"], w.g_a, t["b"], t["sfb"], w.g_b, c, M, K, L)
    torch.cuda.synchronize()
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, M, K, L)
    assert_parity(c.cpu().numpy(), ref, T, f"K={K}")


def test_unaligned_grouped(pkg):
    w = workloads.make_grouped("g0")
    A, rA = placed(w.A, 3)
    sfa, rS = placed(w.sfa, 1)
    b, rB = placed(w.b, 6)
    sfb = torch.from_numpy(w.sfb).cuda()
    g_a = torch.from_numpy(np.ascontiguousarray(w.g_a)).cuda()
    g_b = torch.from_numpy(np.ascontiguousarray(w.g_b)).cuda()
    emap = torch.from_numpy(w.expert_of).cuda()
    c = torch.full((w.T, w.M), float("nan"), dtype=torch.float16, device="cuda")
    pkg.nvfp4_gemv_grouped(A, sfa, g_a, b, sfb, g_b, c, w.M, w.K, w.E, w.T, expert_of_token=emap)
    torch.cuda.synchronize()
    from oracle import grouped as G
    ref, T = G.gemv_grouped(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, w.expert_of, w.M, w.K)
    assert_parity(c.cpu().numpy(), ref, T, "unaligned grouped")

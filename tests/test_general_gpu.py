"""GPU parity of the general path: any byte alignment of A, sfa, b and sfb, and any K % 16 == 0
(K not a multiple of 32 included), through the C ABI against the oracle.  The planner sends such
calls to the register-vector TMA kernel when K % 256 == 0 (bulk copies of each tile's aligned
interior, edge bytes stored one by one, shifted out of shared memory) and otherwise to the shift
kernel (aligned 16-byte loads funnel-shifted into place); the simple kernel (byte loads) takes them
when forced; the vector-load, shared-memory-vector TMA and tensor-core kernels refuse them.  The buffers sit
inside larger allocations filled with other bytes, so a read before the first or past the last
byte of an operand would change the result."""
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
    auto = c.cpu().numpy()
    for plan in (dict(kernel=6), dict(kernel=6, warps_per_cta=3, ctas_per_batch=5),
                 dict(kernel=6, flags=2), dict(kernel=1)):
        c2 = torch.full((w.L, w.M), float("nan"), dtype=torch.float16, device="cuda")
        pkg.nvfp4_gemv_batched_ex(args[0], args[1], w.g_a, args[2], args[3], w.g_b, c2, w.M, w.K,
                                  w.L, plan=plan)
        torch.cuda.synchronize()
        assert_parity(c2.cpu().numpy(), ref, T, f"offsets {offsets} {plan}")
        if plan.get("kernel") == 6:   # the automatic plan is the shift kernel: same bits
            assert np.array_equal(c2.cpu().numpy().view(np.uint16), auto.view(np.uint16))
    # the vector-load and shared-memory-vector TMA kernels refuse unaligned operands; the
    # register-vector TMA kernel takes them but needs K % 256 == 0 (here K = 1056)
    for plan, status in ((dict(kernel=2), 2), (dict(kernel=3), 2), (dict(kernel=4), 3),
                         (dict(kernel=5), 2)):
        with pytest.raises(pkg.NVFP4Error) as e:
            pkg.nvfp4_gemv_batched_ex(args[0], args[1], w.g_a, args[2], args[3], w.g_b, c, w.M,
                                      w.K, w.L, plan=plan)
        assert e.value.status == status, plan


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


SHIFT_SHAPES = [(1, 16, 1), (5, 1040, 3), (257, 2064, 2), (130, 4096, 1), (33, 16400, 2),
                (1000, 7184, 1)]


@pytest.mark.parametrize("shape", SHIFT_SHAPES, ids=[f"{m}x{k}x{l}" for m, k, l in SHIFT_SHAPES])
@pytest.mark.parametrize("offset", [0, 1, 7, 8, 15])
def test_shift_kernel_shapes_and_offsets(pkg, shape, offset):
    """Ragged M, K % 32 == 16 and K % 1024 != 0, every row-start residue mod 16 (K % 32 == 16
    alternates it), A placed so that its first chunk begins before it and its last ends past it."""
    M, K, L = shape
    w = workloads.random_workload(M, K, L, seed=M * 7 + K + offset,
                                  scale_bytes=workloads.pow2_scale_bytes(-4, 3), g_a=0.75, g_b=1.25)
    keep, args = [], []
    for name, off in zip(("A", "sfa", "b", "sfb"), (offset, (offset * 3) % 16, offset, 0)):
        v, raw = placed(getattr(w, name), off)
        keep.append(raw)
        args.append(v)
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, M, K, L)
    for plan in (None, dict(kernel=6), dict(kernel=6, warps_per_cta=1, ctas_per_batch=1),
                 dict(kernel=6, warps_per_cta=8, ctas_per_batch=M)):
        c = torch.full((L, M), float("nan"), dtype=torch.float16, device="cuda")
        pkg.nvfp4_gemv_batched_ex(args[0], args[1], w.g_a, args[2], args[3], w.g_b, c, M, K, L,
                                  plan=plan)
        torch.cuda.synchronize()
        out = c.cpu().numpy()
        assert not np.isnan(out).any(), plan
        assert_parity(out, ref, T, f"{shape} offset {offset} {plan}")


def test_shift_kernel_small_n_shares_a(pkg):
    """Unaligned operands of the small-N entry point: the shift kernel reads the one matrix for
    every vector."""
    M, K, N = 300, 2064, 5
    wa = workloads.random_workload(M, K, 1, seed=77, scale_bytes=workloads.pow2_scale_bytes(-3, 2))
    wv = workloads.random_workload(1, K, N, seed=78, scale_bytes=workloads.pow2_scale_bytes(-3, 2))
    A, rA = placed(wa.A[0], 5)
    sfa, rS = placed(wa.sfa[0], 3)
    b, rB = placed(wv.b, 9)
    sfb, rSB = placed(wv.sfb, 1)
    c = torch.full((N, M), float("nan"), dtype=torch.float16, device="cuda")
    pkg.nvfp4_gemm_small_n(A, sfa, wa.g_a, b, sfb, wv.g_b, c, M, K, N)
    torch.cuda.synchronize()
    ref, T = oracle.gemv(np.repeat(wa.A, N, 0), np.repeat(wa.sfa, N, 0), wa.g_a, wv.b, wv.sfb,
                         wv.g_b, M, K, N)
    assert_parity(c.cpu().numpy(), ref, T, "small N, unaligned")


def test_shift_kernel_grouped_forms(pkg):
    """The grouped form (per-token routing) through the shift kernel, with a token that no expert
    owns."""
    w = workloads.make_grouped("g0")
    A, rA = placed(w.A, 11)
    sfa, rS = placed(w.sfa, 2)
    b, rB = placed(w.b, 4)
    sfb, rSB = placed(w.sfb, 7)
    g_a = torch.from_numpy(np.ascontiguousarray(w.g_a)).cuda()
    g_b = torch.from_numpy(np.ascontiguousarray(w.g_b)).cuda()
    emap = np.array(w.expert_of, dtype=np.int32).copy()
    emap[-1] = -1                                          # this token has no expert
    from oracle import grouped as G
    ref, T = G.gemv_grouped(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, emap, w.M, w.K)
    for plan in (None, dict(kernel=6), dict(kernel=1)):
        c = torch.full((w.T, w.M), float("nan"), dtype=torch.float16, device="cuda")
        pkg.nvfp4_gemv_grouped(A, sfa, g_a, b, sfb, g_b, c, w.M, w.K, w.E, w.T,
                               expert_of_token=torch.from_numpy(emap).cuda(), plan=plan)
        torch.cuda.synchronize()
        out = c.cpu().numpy()
        assert np.all(out[-1] == 0), plan
        assert_parity(out, ref, T, f"grouped unaligned {plan}")


RING_SHAPES = [(2432, 2048, 1), (300, 4096, 9), (97, 1024, 3), (1000, 16384, 1),
               (600, 4352, 2),                                # a partial last segment
               (400, 11264, 2)]                               # 11 segments: 6 warps, one idle


@pytest.mark.parametrize("shape", RING_SHAPES, ids=[f"{m}x{k}x{l}" for m, k, l in RING_SHAPES])
@pytest.mark.parametrize("offsets", [(1, 0, 0, 0), (0, 5, 0, 0), (0, 0, 3, 9), (15, 13, 11, 7),
                                     (8, 8, 0, 0)])
def test_unaligned_operands_on_the_tma_ring(pkg, shape, offsets):
    """K % 256 == 0 with operands off 16-byte boundaries: the register-vector TMA kernel copies each
    tile's aligned interior in bulk and the buffer's first and last partial chunks byte by byte.
    Every plan gives the oracle's values; the ring plans agree bit for bit with each other."""
    M, K, L = shape
    w = workloads.random_workload(M, K, L, seed=M + K + sum(offsets),
                                  scale_bytes=workloads.pow2_scale_bytes(-4, 3), g_a=0.5, g_b=1.5)
    keep, args = [], []
    for name, off in zip(("A", "sfa", "b", "sfb"), offsets):
        v, raw = placed(getattr(w, name), off)
        keep.append(raw)
        args.append(v)
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, M, K, L)
    ring = None
    for plan in (None, dict(kernel=4), dict(kernel=4, flags=1), dict(kernel=4, flags=2),
                 dict(kernel=4, tile_rows=3, stages=3, ctas_per_batch=2),
                 dict(kernel=4, tile_rows=5, stages=2), dict(kernel=6), dict(kernel=1)):
        c = torch.full((L, M), float("nan"), dtype=torch.float16, device="cuda")
        pkg.nvfp4_gemv_batched_ex(args[0], args[1], w.g_a, args[2], args[3], w.g_b, c, M, K, L,
                                  plan=plan)
        torch.cuda.synchronize()
        out = c.cpu().numpy()
        assert not np.isnan(out).any(), plan
        assert_parity(out, ref, T, f"{shape} {offsets} {plan}")
        if plan == dict(kernel=4):
            ring = out
        elif plan is not None and plan.get("kernel") == 4 and "tile_rows" not in plan:
            assert np.array_equal(out.view(np.uint16), ring.view(np.uint16)), plan


VEC_SHAPES = [(2432, 2048, 1), (300, 4096, 9), (64, 65536, 1), (40, 16384, 3),
              (700, 2304, 2), (1500, 1280, 1),                # partial last segments
              (2560, 17408, 1),                               # 17 segments: 9 warps, one idle
              (700, 37888, 1)]                                # 37: slices of 13, 13 and 11


@pytest.mark.parametrize("shape", VEC_SHAPES, ids=[f"{m}x{k}x{l}" for m, k, l in VEC_SHAPES])
@pytest.mark.parametrize("offsets", [(0, 0, 1, 0), (0, 0, 0, 3), (0, 0, 9, 5), (0, 0, 15, 15)])
def test_unaligned_vector_keeps_the_aligned_ring(pkg, shape, offsets):
    """Only b or sfb off a 16-byte boundary: the aligned ring form with its usual plan (split K
    and small-call grids included), the vector loaded with shifted loads.  The outputs are the
    oracle's and bit-identical to the same call on aligned copies, for the automatic plan and with
    early weights."""
    M, K, L = shape
    w = workloads.random_workload(M, K, L, seed=M + K + L + sum(offsets),
                                  scale_bytes=workloads.pow2_scale_bytes(-4, 3), g_a=0.5, g_b=1.5)
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, M, K, L)
    keep = []

    def run(offs, plan):
        args = []
        for name, off in zip(("A", "sfa", "b", "sfb"), offs):
            v, raw = placed(getattr(w, name), off)
            keep.append(raw)
            args.append(v)
        c = torch.full((L, M), float("nan"), dtype=torch.float16, device="cuda")
        pkg.nvfp4_gemv_batched_ex(args[0], args[1], w.g_a, args[2], args[3], w.g_b, c, M, K, L,
                                  plan=plan)
        torch.cuda.synchronize()
        return c.cpu().numpy()

    for plan in (None, dict(flags=1)):
        aligned = run((0, 0, 0, 0), plan)
        out = run(offsets, plan)
        assert not np.isnan(out).any(), plan
        assert_parity(out, ref, T, f"{shape} {offsets} {plan}")
        assert np.array_equal(out.view(np.uint16), aligned.view(np.uint16)), plan


def test_unaligned_vector_grouped_keeps_the_aligned_ring(pkg):
    """The grouped form with aligned experts and token vectors off 16-byte boundaries: the aligned
    ring form, bit-identical to the same call on aligned vectors."""
    w = workloads.make_grouped("g0")
    A = torch.from_numpy(w.A).cuda()
    sfa = torch.from_numpy(w.sfa).cuda()
    g_a = torch.from_numpy(np.ascontiguousarray(w.g_a)).cuda()
    g_b = torch.from_numpy(np.ascontiguousarray(w.g_b)).cuda()
    emap = torch.from_numpy(np.ascontiguousarray(w.expert_of, dtype=np.int32)).cuda()
    from oracle import grouped as G
    ref, T = G.gemv_grouped(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, w.expert_of, w.M, w.K)
    outs = []
    for ob, osb in ((0, 0), (3, 0), (0, 5), (11, 7)):
        b, rb = placed(w.b, ob)
        sfb, rsb = placed(w.sfb, osb)
        c = torch.full((w.T, w.M), float("nan"), dtype=torch.float16, device="cuda")
        pkg.nvfp4_gemv_grouped(A, sfa, g_a, b, sfb, g_b, c, w.M, w.K, w.E, w.T,
                               expert_of_token=emap, plan=dict(kernel=4))
        torch.cuda.synchronize()
        out = c.cpu().numpy()
        assert_parity(out, ref, T, f"grouped vector +{ob}/+{osb}")
        outs.append(out)
    for out in outs[1:]:
        assert np.array_equal(out.view(np.uint16), outs[0].view(np.uint16))


def test_unaligned_grouped_on_the_tma_ring(pkg):
    """The grouped form with unaligned experts on the register-vector TMA kernel."""
    w = workloads.make_grouped("g0")
    A, rA = placed(w.A, 9)
    sfa, rS = placed(w.sfa, 14)
    b, rB = placed(w.b, 1)
    sfb, rSB = placed(w.sfb, 6)
    g_a = torch.from_numpy(np.ascontiguousarray(w.g_a)).cuda()
    g_b = torch.from_numpy(np.ascontiguousarray(w.g_b)).cuda()
    from oracle import grouped as G
    ref, T = G.gemv_grouped(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, w.expert_of, w.M, w.K)
    for plan in (dict(kernel=4), dict(kernel=4, tile_rows=7, stages=4)):
        c = torch.full((w.T, w.M), float("nan"), dtype=torch.float16, device="cuda")
        pkg.nvfp4_gemv_grouped(A, sfa, g_a, b, sfb, g_b, c, w.M, w.K, w.E, w.T,
                               expert_of_token=torch.from_numpy(w.expert_of).cuda(), plan=plan)
        torch.cuda.synchronize()
        assert_parity(c.cpu().numpy(), ref, T, f"grouped unaligned ring {plan}")

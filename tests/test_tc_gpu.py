"""GPU parity of the tensor-core kernel (tcgen05 block-scaled MMA) through the C ABI.

Two uses: the small-N GEMM (N vectors sharing one matrix, nvfp4_gemm_small_n) and the batched
GEMV with a forced tensor-core plan (N = 1 per batch).  Every output is compared with the oracle
(the batched definition, with A repeated for every vector) under the parity tolerance, across
ragged M (partial 128-row tiles), N from 1 to 19 (19: two launches of at most 16 vectors), K
splits over clusters of 1 to 8 CTAs (including splits that do not divide the K chunks), ring
depths, the launch flags, the CUDA-core plans on the same inputs, and determinism.  The MMA reads
block scales as unsigned E4M3; the kernel negates the blocks whose scales are negative, and the
signed-scale tests check every finite E4M3FN byte, negative ones included, and NaN bytes.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import assert_parity

pytestmark = pytest.mark.gpu
TC = 5


@pytest.fixture(scope="module")
def pkg():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    from decode_nvfp4_gemv_gb300 import build

    build.build()
    import decode_nvfp4_gemv_gb300 as p

    p.load_library()
    return p


def make(M, K, N, seed):
    """One matrix A [M][K/2] and N vectors, non-negative power-of-two scales."""
    w = workloads.random_workload(M, K, 1, seed=seed, scale_bytes=workloads.pow2_scale_bytes(-4, 3),
                                  g_a=0.5, g_b=1.5)
    v = workloads.random_workload(1, K, N, seed=seed + 7,
                                  scale_bytes=workloads.pow2_scale_bytes(-3, 2))
    return w.A[0], w.sfa[0], v.b, v.sfb, w.g_a, w.g_b


def small_n(pkg, A, sfa, b, sfb, g_a, g_b, M, K, N, plan=None):
    t = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (A, sfa, b, sfb)]
    c = torch.full((N, M), float("nan"), dtype=torch.float16, device="cuda")
    pkg.nvfp4_gemm_small_n(t[0], t[1], g_a, t[2], t[3], g_b, c, M, K, N, plan=plan)
    torch.cuda.synchronize()
    return c.cpu().numpy()


def ref_small_n(A, sfa, b, sfb, g_a, g_b, M, K, N):
    return oracle.gemv(np.repeat(A[None], N, 0), np.repeat(sfa[None], N, 0), g_a, b, sfb, g_b,
                       M, K, N)


SHAPES = [(128, 256, 1), (128, 256, 16), (1, 256, 3), (300, 512, 5), (257, 2304, 7),
          (1000, 4096, 8), (64, 1024, 19), (520, 7168, 16)]


@pytest.mark.parametrize("shape", SHAPES, ids=[f"{m}x{k}x{n}" for m, k, n in SHAPES])
def test_small_n_tensor_cores(pkg, shape):
    M, K, N = shape
    A, sfa, b, sfb, g_a, g_b = make(M, K, N, seed=M + K + N)
    ref, T = ref_small_n(A, sfa, b, sfb, g_a, g_b, M, K, N)
    chunks = K // 256
    plans = [None, dict(kernel=TC), dict(kernel=TC, stages=2), dict(kernel=TC, stages=6),
             dict(kernel=TC, flags=1), dict(kernel=TC, flags=2)]
    plans += [dict(kernel=TC, k_split=s) for s in (1, 2, 3, 8) if s <= chunks]
    first = None
    for plan in plans:
        c = small_n(pkg, A, sfa, b, sfb, g_a, g_b, M, K, N, plan)
        assert not np.isnan(c).any(), plan
        assert_parity(c, ref, T, f"{shape} {plan}")
        if plan is None:
            first = c
    again = small_n(pkg, A, sfa, b, sfb, g_a, g_b, M, K, N)
    assert np.array_equal(first.view(np.uint16), again.view(np.uint16))   # deterministic


@pytest.mark.parametrize("plan", [dict(kernel=1), dict(kernel=2), dict(kernel=4),
                                  dict(kernel=4, flags=1)], ids=["simple", "stream", "rv", "rv-ew"])
def test_small_n_cuda_core_plans(pkg, plan):
    M, K, N = 300, 2048, 6
    A, sfa, b, sfb, g_a, g_b = make(M, K, N, seed=5)
    ref, T = ref_small_n(A, sfa, b, sfb, g_a, g_b, M, K, N)
    try:
        c = small_n(pkg, A, sfa, b, sfb, g_a, g_b, M, K, N, plan)
    except pkg.NVFP4Error as e:        # a forced ring that does not fit this shape
        assert e.status == 3, e
        return
    assert_parity(c, ref, T, f"cuda-core {plan}")


def test_small_n_general_k_falls_back(pkg):
    """K % 256 != 0: the automatic plan leaves the tensor cores; a forced TC plan is refused."""
    M, K, N = 200, 1056, 4
    A, sfa, b, sfb, g_a, g_b = make(M, K, N, seed=9)
    ref, T = ref_small_n(A, sfa, b, sfb, g_a, g_b, M, K, N)
    assert_parity(small_n(pkg, A, sfa, b, sfb, g_a, g_b, M, K, N), ref, T, "K=1056")
    with pytest.raises(pkg.NVFP4Error) as e:
        small_n(pkg, A, sfa, b, sfb, g_a, g_b, M, K, N, dict(kernel=TC))
    assert e.value.status == 3


def test_small_n_decode_shape(pkg):
    """The decode projection shape with 16 tokens: M=7168, K=16384, N=16, sampled rows checked
    by the oracle one by one."""
    M, K, N = 7168, 16384, 16
    A, sfa, b, sfb, g_a, g_b = make(M, K, N, seed=2)
    c = small_n(pkg, A, sfa, b, sfb, g_a, g_b, M, K, N)
    rng = np.random.default_rng(0)
    ls = rng.integers(0, N, 400)
    ms = rng.integers(0, M, 400)
    ref, T = oracle.gemv_rows(np.repeat(A[None], N, 0), np.repeat(sfa[None], N, 0), g_a, b, sfb,
                              g_b, M, K, N, ls, ms)
    assert_parity(c[ls, ms], ref, T, "decode shape, 16 tokens")


BATCHED = [(129, 256, 3), (7, 1024, 2), (130, 4096, 1), (64, 7168, 3), (300, 2304, 2)]


@pytest.mark.parametrize("shape", BATCHED, ids=[f"{m}x{k}x{l}" for m, k, l in BATCHED])
def test_batched_gemv_on_tensor_cores(pkg, shape):
    M, K, L = shape
    w = workloads.random_workload(M, K, L, seed=M * 3 + K + L,
                                  scale_bytes=workloads.pow2_scale_bytes(-4, 3), g_a=0.75, g_b=1.25)
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, M, K, L)
    t = {k: torch.from_numpy(getattr(w, k)).cuda() for k in ("A", "sfa", "b", "sfb")}
    for plan in (dict(kernel=TC), dict(kernel=TC, k_split=1), dict(kernel=TC, k_split=2, stages=3),
                 dict(kernel=TC, flags=1)):
        if plan.get("k_split", 0) > K // 256:
            continue
        c = torch.full((L, M), float("nan"), dtype=torch.float16, device="cuda")
        pkg.nvfp4_gemv_batched_ex(t["A"], t["sfa"], w.g_a, t["b"], t["sfb"], w.g_b, c, M, K, L,
                                  plan=plan)
        torch.cuda.synchronize()
        assert_parity(c.cpu().numpy(), ref, T, f"{shape} {plan}")


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5"])
def test_workloads_on_tensor_cores(pkg, workload, name):
    w = workload(name)
    t = {k: torch.from_numpy(getattr(w, k)).cuda() for k in ("A", "sfa", "b", "sfb")}
    c = torch.full((w.L, w.M), float("nan"), dtype=torch.float16, device="cuda")
    pkg.nvfp4_gemv_batched_ex(t["A"], t["sfa"], w.g_a, t["b"], t["sfb"], w.g_b, c, w.M, w.K, w.L,
                              plan=dict(kernel=TC, flags=1))
    torch.cuda.synchronize()
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, w.M, w.K, w.L)
    assert_parity(c.cpu().numpy(), ref, T, f"{name} on tensor cores")


def test_tensor_core_plan_rules(pkg):
    """Forced TC plans outside the kernel's range are refused on the host (UNSUPPORTED_SHAPE),
    and the TC kernel takes neither the grouped form nor bf16 output."""
    M, K, N = 128, 512, 2
    A, sfa, b, sfb, g_a, g_b = make(M, K, N, seed=4)
    for plan in (dict(kernel=TC, k_split=3), dict(kernel=TC, k_split=9), dict(kernel=TC, stages=1),
                 dict(kernel=TC, stages=7), dict(kernel=TC, warps_per_cta=8),
                 dict(kernel=TC, tile_rows=64)):
        with pytest.raises(pkg.NVFP4Error) as e:
            small_n(pkg, A, sfa, b, sfb, g_a, g_b, M, K, N, plan)
        assert e.value.status == 3, plan
    g = workloads.make_grouped("g0")
    d = {k: torch.from_numpy(np.ascontiguousarray(getattr(g, k))).cuda()
         for k in ("A", "sfa", "g_a", "g_b", "b", "sfb", "expert_of")}
    c = torch.empty((g.T, g.M), dtype=torch.float16, device="cuda")
    with pytest.raises(pkg.NVFP4Error) as e:
        pkg.nvfp4_gemv_grouped(d["A"], d["sfa"], d["g_a"], d["b"], d["sfb"], d["g_b"], c, g.M,
                               g.K, g.E, g.T, expert_of_token=d["expert_of"],
                               plan=dict(kernel=TC))
    assert e.value.status == 3


def test_tensor_cores_after_other_work_in_the_stream(pkg):
    """A TC call whose vectors are written by the kernel just before it (programmatic dependent
    launch must still see them), on a non-default stream, then captured in a graph."""
    M, K, N = 384, 1024, 3
    A, sfa, b, sfb, g_a, g_b = make(M, K, N, seed=6)
    ref, T = ref_small_n(A, sfa, b, sfb, g_a, g_b, M, K, N)
    tA, tS = torch.from_numpy(A).cuda(), torch.from_numpy(sfa).cuda()
    src_b, src_s = torch.from_numpy(b).cuda(), torch.from_numpy(sfb).cuda()
    tb, ts = torch.zeros_like(src_b), torch.zeros_like(src_s)
    c = torch.full((N, M), float("nan"), dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        tb.copy_(src_b)
        ts.copy_(src_s)
        pkg.nvfp4_gemm_small_n(tA, tS, g_a, tb, ts, g_b, c, M, K, N, stream=s,
                               plan={"flags": 1})
    s.synchronize()
    assert_parity(c.cpu().numpy(), ref, T, "after a copy kernel")
    g = torch.cuda.CUDAGraph()
    c2 = torch.full((N, M), float("nan"), dtype=torch.float16, device="cuda")
    with torch.cuda.graph(g, stream=s):
        pkg.nvfp4_gemm_small_n(tA, tS, g_a, tb, ts, g_b, c2, M, K, N, stream=s)
    with torch.cuda.stream(s):
        g.replay()
    s.synchronize()
    assert np.array_equal(c.cpu().numpy().view(np.uint16), c2.cpu().numpy().view(np.uint16))


# ------------------------------------------------------------------ signed and NaN block scales

FINITE = [v for v in range(256) if v not in (0x7F, 0xFF)]
SIGNED_SHAPES = [(128, 256, 1), (300, 1024, 5), (257, 2304, 16), (1000, 4096, 3)]


@pytest.mark.parametrize("shape", SIGNED_SHAPES, ids=[f"{m}x{k}x{n}" for m, k, n in SIGNED_SHAPES])
def test_signed_scales_on_the_automatic_small_n_path(pkg, shape):
    """Block scales drawn from every finite E4M3FN byte (half of them negative) on both operands:
    the automatic small-N plan takes the tensor cores and must give the oracle's result under
    every split and ring depth."""
    M, K, N = shape
    w = workloads.random_workload(M, K, 1, seed=M + 3 * K, scale_bytes=FINITE, g_a=0.5, g_b=2.0)
    v = workloads.random_workload(1, K, N, seed=M + 5 * K, scale_bytes=FINITE)
    A, sfa = w.A[0], w.sfa[0]
    assert (sfa & 0x80).any() and (v.sfb & 0x80).any()
    ref, T = ref_small_n(A, sfa, v.b, v.sfb, w.g_a, w.g_b, M, K, N)
    chunks = K // 256
    plans = [None, dict(kernel=TC, stages=2), dict(kernel=TC, flags=1)]
    plans += [dict(kernel=TC, k_split=s) for s in (2, 3) if s <= chunks]
    for plan in plans:
        c = small_n(pkg, A, sfa, v.b, v.sfb, w.g_a, w.g_b, M, K, N, plan)
        assert not np.isnan(c).any(), plan
        assert_parity(c, ref, T, f"signed scales {shape} {plan}")


def test_one_negative_scale_negates_its_block(pkg):
    """A single negative scale byte: flipping its sign bit changes the output by exactly minus two
    times that block's contribution, as the oracle says."""
    M, K, N = 128, 512, 2
    A, sfa, b, sfb, g_a, g_b = make(M, K, N, seed=91)
    sfa2 = sfa.copy()
    sfa2[7, 5] |= 0x80
    sfb2 = sfb.copy()
    sfb2[1, 30] |= 0x80
    for sa, sb in ((sfa2, sfb), (sfa, sfb2), (sfa2, sfb2)):
        c = small_n(pkg, A, sa, b, sb, g_a, g_b, M, K, N)
        ref, T = ref_small_n(A, sa, b, sb, g_a, g_b, M, K, N)
        assert_parity(c, ref, T, "one negative scale")


def test_nan_scale_bytes_give_nan_on_tensor_cores(pkg):
    """E4M3 NaN bytes (0x7F, 0xFF) in a matrix row's scales make that row's outputs NaN for every
    vector; in a vector's scales, that vector's outputs NaN: on the tensor cores as in the
    oracle."""
    M, K, N = 256, 1024, 4
    A, sfa, b, sfb, g_a, g_b = make(M, K, N, seed=93)
    sfa = sfa.copy()
    sfb = sfb.copy()
    sfa[17, 3] = 0x7F
    sfa[200, 60] = 0xFF
    sfb[2, 11] = 0x7F
    c = small_n(pkg, A, sfa, b, sfb, g_a, g_b, M, K, N)
    ref, T = ref_small_n(A, sfa, b, sfb, g_a, g_b, M, K, N)
    assert np.isnan(ref[:, 17]).all() and np.isnan(ref[2]).all()
    assert_parity(c, ref, T, "NaN scales on tensor cores")


def test_batched_gemv_forced_onto_tensor_cores_with_signed_scales(pkg):
    w = workloads.random_workload(200, 2048, 3, seed=95, scale_bytes=FINITE, g_a=0.25, g_b=4.0)
    t = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (w.A, w.sfa, w.b, w.sfb)]
    c = torch.full((w.L, w.M), float("nan"), dtype=torch.float16, device="cuda")
    pkg.nvfp4_gemv_batched_ex(t[0], t[1], w.g_a, t[2], t[3], w.g_b, c, w.M, w.K, w.L,
                              plan=dict(kernel=TC))
    torch.cuda.synchronize()
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, w.M, w.K, w.L)
    assert_parity(c.cpu().numpy(), ref, T, "batched GEMV on tensor cores, signed scales")

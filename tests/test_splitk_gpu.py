"""GPU parity of split K over a thread-block cluster (the register-vector TMA kernel with
k_slices > 1), through the C ABI, against the oracle.

Few output rows (M * L far below 8 rows per CTA slot) with long K: each cluster of S CTAs shares a
row range, CTA z streams K slice z and the partial sums meet in the owner CTA's shared memory.
Covered: the automatic plan on M * L in {16, 64, 128, 512} at K = 16384 and 65536, the automatic
plan on wide K (24576 to 131072) with many rows, forced slice
counts (2, 3, 4, 7, 8; a last slice shorter than the others), batches, one row range per batch,
tile and ring shapes, the launch flags (bit-identical with and without early weights),
determinism, NaN pre-fill and guard bands, the grouped, small-N and bf16-vector entry points on
the split kernel, and forced plans the split cannot take (refused on the host).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from oracle import grouped as G
from oracle import quantize as Q
from parity import assert_parity

pytestmark = pytest.mark.gpu
TMA_RV = 4


@pytest.fixture(scope="module")
def pkg():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    from decode_nvfp4_gemv_gb300 import build

    build.build()
    import decode_nvfp4_gemv_gb300 as p

    p.load_library()
    return p


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def run(pkg, w, plan=None, guard=0):
    t = {k: dev(getattr(w, k)) for k in ("A", "sfa", "b", "sfb")}
    n = w.L * w.M
    raw = torch.full((n + 2 * guard,), float("nan"), dtype=torch.float16, device="cuda")
    if guard:
        raw[:guard] = 1.5
        raw[guard + n:] = -2.5
    c = raw[guard:guard + n]
    pkg.nvfp4_gemv_batched_ex(t["A"], t["sfa"], w.g_a, t["b"], t["sfb"], w.g_b, c, w.M, w.K, w.L,
                              plan=plan)
    torch.cuda.synchronize()
    out = raw.cpu().numpy()
    if guard:
        assert (out[:guard] == 1.5).all() and (out[guard + n:] == -2.5).all(), "guard band"
    return out[guard:guard + n].reshape(w.L, w.M)


def check(w, c, what):
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, w.M, w.K, w.L)
    assert not np.isnan(c).any(), what + ": an output was not written"
    return assert_parity(c, ref, T, what)


def small(M, K, L=1, seed=0):
    return workloads.random_workload(M, K, L, seed=1000 + seed + M + K // 256,
                                     scale_bytes=workloads.pow2_scale_bytes(-4, 3), g_a=0.75,
                                     g_b=1.25)


FEW_ROWS = [(m, k) for k in (16384, 65536) for m in (16, 64, 128, 512)]


@pytest.mark.parametrize("shape", FEW_ROWS, ids=[f"{m}x{k}" for m, k in FEW_ROWS])
def test_automatic_plan_for_few_rows(pkg, shape):
    """Few rows take the register-vector ring on a smaller grid; K is split over a cluster when
    it holds more than 16 segments (K = 65536 here)."""
    M, K = shape
    w = small(M, K)
    p = pkg.nvfp4_gemv_plan(M, K, 1)
    assert p.kernel == TMA_RV and (p.k_slices > 1) == (K > 16384), p
    c = run(pkg, w, guard=64)
    check(w, c, f"{shape} auto {p}")
    c_ew = run(pkg, w, {"flags": 1})
    assert np.array_equal(c.view(np.uint16), c_ew.view(np.uint16)), "early weights changed bits"
    assert np.array_equal(run(pkg, w).view(np.uint16), c.view(np.uint16)), "not deterministic"


# (M, K, L) -> K slices of the automatic plan: wide K on enough rows for the full grid
WIDE_K = {(2432, 24576, 1): 1, (2560, 28672, 1): 2, (2560, 33792, 1): 2, (2560, 36864, 1): 2,
          (2560, 53248, 1): 4, (1280, 65536, 2): 4, (2560, 98304, 1): 4, (2560, 114688, 1): 8,
          (2560, 131072, 1): 8,
          # odd and prime segment counts: warps of two with one idle, slices with a shorter last
          (2560, 17408, 1): 1, (2560, 25600, 1): 1, (2560, 31744, 1): 2, (2560, 37888, 1): 2,
          (2560, 61440 + 1024, 1): 4}


@pytest.mark.parametrize("shape", list(WIDE_K), ids=lambda s: "x".join(map(str, s)))
def test_automatic_plan_for_wide_k(pkg, shape):
    """Wide K on many rows: one CTA per SM where the registers hold no more (24576), split over
    clusters of two for 28 segments, past 32 segments over the fewest CTAs whose slices are at most
    24 segments; grids of the clusters the GPU holds at once."""
    M, K, L = shape
    w = small(M, K, L, seed=11)
    p = pkg.nvfp4_gemv_plan(M, K, L)
    assert p.kernel == TMA_RV and max(1, p.k_slices) == WIDE_K[shape], p
    c = run(pkg, w, guard=64)
    check(w, c, f"{shape} auto {p}")
    c_ew = run(pkg, w, {"flags": 1})
    assert np.array_equal(c.view(np.uint16), c_ew.view(np.uint16)), "early weights changed bits"


FORCED = [
    # (M, K, L, plan)
    (40, 16384, 1, dict(k_slices=2)),
    (40, 16384, 1, dict(k_slices=4)),
    (40, 16384, 1, dict(k_slices=8)),
    (33, 7168, 2, dict(k_slices=7)),                          # 7 slices of one segment
    (50, 2304, 3, dict(k_slices=3)),                          # last slice 256 elements
    (50, 4352, 2, dict(k_slices=5)),                          # 5 segments, the last 256
    (97, 8192, 1, dict(k_slices=2, ctas_per_batch=1)),        # one row range: many tiles
    (97, 8192, 2, dict(k_slices=4, ctas_per_batch=3, tile_rows=5, stages=3)),
    (97, 8192, 1, dict(k_slices=8, tile_rows=1, stages=8)),
    (64, 16384, 1, dict(k_slices=2, warps_per_cta=4)),        # two segments per warp
    (64, 16384, 1, dict(k_slices=4, warps_per_cta=16)),       # four warps per segment
    (300, 4096, 2, dict(k_slices=2, flags=1)),
    (300, 4096, 2, dict(k_slices=2, flags=2)),
    (5, 32768, 1, dict(k_slices=8, flags=1)),                 # more CTAs than rows in a cluster
    (1, 16384, 3, dict(k_slices=8)),
    (100, 16384, 1, dict(k_slices=3)),                        # slices of 6, 6 and 4 segments
    (97, 37888, 1, dict(k_slices=2)),                         # 19 + 18: 10 warps, one idle
    (64, 10240, 2, dict(k_slices=4)),                         # 3, 3, 3 and 1
    (50, 9472, 1, dict(k_slices=3, flags=1)),                 # 4, 4 and a partial 2
]


@pytest.mark.parametrize("case", FORCED, ids=lambda c: f"{c[0]}x{c[1]}x{c[2]}-" +
                         ",".join(f"{k}={v}" for k, v in c[3].items()))
def test_forced_split_plans(pkg, case):
    M, K, L, plan = case
    w = small(M, K, L, seed=7)
    c = run(pkg, w, dict(plan, kernel=TMA_RV), guard=32)
    check(w, c, f"{case}")


def test_slices_agree_within_tolerance_and_differ_only_in_summation_order(pkg):
    w = small(128, 16384, 2, seed=3)
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, w.M, w.K, w.L)
    outs = [run(pkg, w, dict(kernel=TMA_RV, k_slices=s)) for s in (1, 2, 4, 8)]
    for c in outs:
        assert_parity(c, ref, T, "slices")


def test_nan_scale_poisons_only_its_row_under_split(pkg):
    w = small(24, 16384, 1, seed=4)
    w.sfa[0, 5, 700] = 0x7F                                   # slice 5 of 8
    c = run(pkg, w, dict(kernel=TMA_RV, k_slices=8))
    assert np.isnan(c[0, 5]) and np.count_nonzero(np.isnan(c)) == 1
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, w.M, w.K, w.L)
    assert_parity(c, ref, T, "NaN scale under split K")


@pytest.mark.parametrize("plan", [dict(kernel=TMA_RV, k_slices=7), dict(kernel=TMA_RV, k_slices=9),
                                  dict(kernel=2, k_slices=2), dict(kernel=3, k_slices=2),
                                  dict(kernel=TMA_RV, k_slices=-1)],
                         ids=["7-leaves-a-slice-empty", "9-too-many", "stream", "smem-vector",
                              "negative"])
def test_plans_the_split_cannot_take_are_refused(pkg, plan):
    w = small(64, 16384)
    with pytest.raises(pkg.NVFP4Error) as e:
        run(pkg, w, plan)
    assert e.value.status == 3


def test_split_needs_aligned_operands(pkg):
    w = small(64, 16384)
    raw = torch.empty(w.A.size + 16, dtype=torch.uint8, device="cuda")
    A1 = raw[5:5 + w.A.size]
    A1.copy_(dev(w.A.ravel()))
    c = torch.zeros((1, 64), dtype=torch.float16, device="cuda")
    with pytest.raises(pkg.NVFP4Error) as e:
        pkg.nvfp4_gemv_batched_ex(A1, dev(w.sfa), w.g_a, dev(w.b), dev(w.sfb), w.g_b, c, 64,
                                  16384, 1, plan=dict(kernel=TMA_RV, k_slices=4))
    assert e.value.status == 2
    # the automatic plan for misaligned few-row operands does not split and is still right
    pkg.nvfp4_gemv_batched_ex(A1, dev(w.sfa), w.g_a, dev(w.b), dev(w.sfb), w.g_b, c, 64, 16384, 1)
    torch.cuda.synchronize()
    check(w, c.cpu().numpy(), "misaligned A, automatic plan")


def test_grouped_tokens_on_the_split_kernel(pkg):
    """A handful of tokens routed to experts on the split kernel: each cluster finds its token's
    expert, and tokens without one get zeros."""
    E, M, K, T = 4, 256, 8192, 5
    a = workloads.random_workload(M, K, E, seed=51, scale_bytes=workloads.pow2_scale_bytes(-3, 2))
    v = workloads.random_workload(1, K, T, seed=52, scale_bytes=workloads.pow2_scale_bytes(-3, 2))
    g_a = np.float32([0.5, 1.0, 2.0, 0.25])
    g_b = np.float32([1.0, 0.5, 1.0, 2.0])
    expert_of = np.int32([2, 0, -1, 3, 0])
    c = torch.full((T, M), float("nan"), dtype=torch.float16, device="cuda")
    pkg.nvfp4_gemv_grouped(dev(a.A), dev(a.sfa), dev(g_a), dev(v.b), dev(v.sfb), dev(g_b), c, M,
                           K, E, T, expert_of_token=dev(expert_of),
                           plan=dict(kernel=TMA_RV, k_slices=4))
    torch.cuda.synchronize()
    ref, Tb = G.gemv_grouped(a.A, a.sfa, g_a, v.b, v.sfb, g_b, G.experts_from_map(expert_of, E),
                             M, K)
    out = c.cpu().numpy()
    assert (out[2] == 0).all()
    assert_parity(out, ref, Tb, "grouped on the split kernel")


def test_small_n_on_cuda_cores_with_split(pkg):
    """N vectors sharing one matrix through the CUDA-core path forced to split K: every batch
    reads the same A."""
    M, K, N = 96, 16384, 3
    a = small(M, K, 1, seed=61)
    v = small(1, K, N, seed=62)
    c = torch.full((N, M), float("nan"), dtype=torch.float16, device="cuda")
    pkg.nvfp4_gemm_small_n(dev(a.A[0]), dev(a.sfa[0]), a.g_a, dev(v.b), dev(v.sfb), v.g_b, c, M,
                           K, N, plan=dict(kernel=TMA_RV, k_slices=4))
    torch.cuda.synchronize()
    ref, T = oracle.gemv(np.repeat(a.A, N, 0), np.repeat(a.sfa, N, 0), a.g_a, v.b, v.sfb, v.g_b,
                         M, K, N)
    assert_parity(c.cpu().numpy(), ref, T, "small N, CUDA cores, split K")


@pytest.mark.parametrize("flags", [1, 1 | 4], ids=["quantizer-then-gemv", "in-gemv"])
def test_bf16_vector_on_the_split_kernel(pkg, flags):
    """The GEMV with a bf16 vector on few rows: with the in-GEMV flag every cluster CTA quantizes
    its own slice of the vector, and the first row range's CTAs write the packed vector."""
    M, K, L = 64, 16384, 2
    w = small(M, K, L, seed=71)
    x = workloads.normal_bf16(72, "x", K * L).reshape(L, K)
    gs = float(np.abs(x).max() / 2688.0)
    pr, sr = Q.quantize_activation(x, gs, "lut")
    bits = (x.view(np.uint32) >> 16).astype(np.uint16).view(np.int16)
    b = torch.full((L * K // 2,), 0xA5, dtype=torch.uint8, device="cuda")
    s = torch.full((L * K // 16,), 0x5A, dtype=torch.uint8, device="cuda")
    c = torch.full((L, M), float("nan"), dtype=torch.float16, device="cuda")
    pkg.nvfp4_gemv_batched_bf16(dev(w.A), dev(w.sfa), w.g_a, dev(bits), gs, b, s, c, M, K, L,
                                plan={"kernel": TMA_RV, "k_slices": 4, "flags": flags})
    torch.cuda.synchronize()
    assert np.array_equal(b.cpu().numpy(), pr.ravel()), "b_out"
    assert np.array_equal(s.cpu().numpy(), sr.ravel()), "sfb_out"
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, pr, sr, gs, M, K, L)
    assert_parity(c.cpu().numpy(), ref, T, f"bf16 vector, split K, flags {flags}")


@pytest.mark.parametrize("flags", [1, 1 | 4], ids=["quantizer-then-gemv", "in-gemv"])
def test_bf16_vector_with_an_idle_segment(pkg, flags):
    """17 segments on 9 warps of two, the last warp's second segment idle: the in-GEMV form still
    writes every segment of the packed vector once."""
    M, K, L = 2560, 17408, 1
    w = small(M, K, L, seed=73)
    x = workloads.normal_bf16(74, "x", K * L).reshape(L, K)
    gs = float(np.abs(x).max() / 2688.0)
    pr, sr = Q.quantize_activation(x, gs, "lut")
    bits = (x.view(np.uint32) >> 16).astype(np.uint16).view(np.int16)
    b = torch.full((L * K // 2,), 0xA5, dtype=torch.uint8, device="cuda")
    s = torch.full((L * K // 16,), 0x5A, dtype=torch.uint8, device="cuda")
    c = torch.full((L, M), float("nan"), dtype=torch.float16, device="cuda")
    p = pkg.nvfp4_gemv_plan(M, K, L)
    assert (p.kernel, p.warps_per_cta, p.k_split, max(1, p.k_slices)) == (TMA_RV, 9, 2, 1), p
    pkg.nvfp4_gemv_batched_bf16(dev(w.A), dev(w.sfa), w.g_a, dev(bits), gs, b, s, c, M, K, L,
                                plan={"flags": flags})
    torch.cuda.synchronize()
    assert np.array_equal(b.cpu().numpy(), pr.ravel()), "b_out"
    assert np.array_equal(s.cpu().numpy(), sr.ravel()), "sfb_out"
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, pr, sr, gs, M, K, L)
    assert_parity(c.cpu().numpy(), ref, T, f"bf16 vector, 17 segments, flags {flags}")


def test_graph_replays_of_split_calls(pkg):
    """Split calls captured in a CUDA graph and replayed: each replay recomputes the outputs."""
    w = small(128, 16384, 1, seed=81)
    t = {k: dev(getattr(w, k)) for k in ("A", "sfa", "b", "sfb")}
    c = torch.full((1, 128), float("nan"), dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    pkg.nvfp4_gemv_batched_ex(t["A"], t["sfa"], w.g_a, t["b"], t["sfb"], w.g_b, c, 128, 16384, 1,
                              stream=s, plan={"flags": 1})
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            pkg.nvfp4_gemv_batched_ex(t["A"], t["sfa"], w.g_a, t["b"], t["sfb"], w.g_b, c, 128,
                                      16384, 1, stream=s, plan={"flags": 1})
    for _ in range(2):
        c.fill_(float("nan"))
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        check(w, c.cpu().numpy(), "graph replay, split K")

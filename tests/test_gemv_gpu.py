"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle.

Every output is compared with the oracle's unrounded fp64 value under the stated tolerance
(tests/parity.py): the hand-worked examples, ragged small shapes under many forced plans, and all
five seeded workloads at full size with the plan the bench uses.  Also: invariants that must hold
bit for bit, determinism, untouched guard bands, poisoned tails, error statuses, non-default
streams and CUDA-graph capture.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import assert_parity

pytestmark = pytest.mark.gpu
HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = json.load(open(os.path.join(HERE, "golden", "worked_examples.json")))["examples"]


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


def run(pkg, w, plan=None, stream=None, g_a=None, g_b=None, A=None, sfa=None, b=None, sfb=None):
    t = {k: dev(getattr(w, k) if v is None else v)
         for k, v in (("A", A), ("sfa", sfa), ("b", b), ("sfb", sfb))}
    c = torch.full((w.L, w.M), float("nan"), dtype=torch.float16, device="cuda")
    pkg.nvfp4_gemv_batched_ex(t["A"], t["sfa"], w.g_a if g_a is None else g_a, t["b"], t["sfb"],
                              w.g_b if g_b is None else g_b, c, w.M, w.K, w.L, stream=stream,
                              plan=plan)
    torch.cuda.synchronize()
    return c.cpu().numpy()


def check(w, c, what=""):
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, w.M, w.K, w.L)
    return assert_parity(c, ref, T, what or w.name)


SIMPLE = dict(kernel=1)


def stream_plan(R=0, S=0, P=0, W=0):
    return dict(kernel=2, rows_per_warp=R, k_split=S, ctas_per_batch=P, warps_per_cta=W)


def tma_plan(TR=0, NS=0, P=0, W=0, rv=False, flags=0):
    return dict(kernel=4 if rv else 3, tile_rows=TR, stages=NS, ctas_per_batch=P,
                warps_per_cta=W, flags=flags)


# ------------------------------------------------------------------ worked examples (exact)

def _golden_workload(ex):
    def h(key):
        return np.frombuffer(bytes.fromhex(ex[key]), dtype=np.uint8).copy()
    M, K, L = ex["M"], ex["K"], ex["L"]
    return workloads.Workload(ex["id"], M, K, L, h("A").reshape(L, M, K // 2),
                              h("sfa").reshape(L, M, K // 16), h("b").reshape(L, K // 2),
                              h("sfb").reshape(L, K // 16), ex["g_a"], ex["g_b"], 0)


@pytest.mark.parametrize("ex", GOLDEN, ids=[e["id"] for e in GOLDEN])
@pytest.mark.parametrize("plan", [None, SIMPLE], ids=["auto", "simple"])
def test_worked_examples_exact(pkg, ex, plan):
    w = _golden_workload(ex)
    c = run(pkg, w, plan).ravel()
    for got, want in zip(c.view(np.uint16), ex["c_fp16_hex"]):
        if want == "nan":
            assert np.isnan(np.uint16(got).view(np.float16))
        elif int(want, 16) & 0x7FFF == 0:
            assert int(got) & 0x7FFF == 0
        else:
            assert int(got) == int(want, 16), (ex["id"], hex(got), want)


def test_worked_examples_through_stream_kernel(pkg):
    """Examples with K = 32 through every stream-kernel row grouping."""
    for ex in GOLDEN:
        if ex["K"] % 32:
            continue
        w = _golden_workload(ex)
        for R in (1, 2, 4):
            c = run(pkg, w, stream_plan(R=R)).ravel()
            assert c.view(np.uint16).tolist() == [int(h, 16) for h in ex["c_fp16_hex"]]


# ------------------------------------------------------------------ ragged shapes x plans

SHAPES = [(1, 32, 1), (3, 64, 2), (7, 1024, 1), (129, 256, 3), (5, 1056, 2), (17, 2080, 1),
          (33, 3104, 2), (130, 4096, 1), (2, 16384, 1), (64, 7168, 3)]
PLANS = [None, SIMPLE, stream_plan(R=1), stream_plan(R=2), stream_plan(R=4),
         stream_plan(R=4, S=2), stream_plan(R=2, S=3, P=2), stream_plan(R=4, P=1, W=1),
         stream_plan(R=1, P=1, W=16), stream_plan(R=4, S=5, P=3, W=3)]
TMA_PLANS = [tma_plan(), tma_plan(TR=1, NS=2), tma_plan(TR=4, NS=3, P=1), tma_plan(TR=8, W=1),
             tma_plan(TR=12, NS=2, W=16), tma_plan(TR=5, NS=8, P=2, W=3),
             tma_plan(rv=True), tma_plan(rv=True, TR=4, NS=2), tma_plan(rv=True, TR=3, NS=5, P=2),
             tma_plan(rv=True, flags=1), tma_plan(flags=1), tma_plan(rv=True, flags=2),
             tma_plan(rv=True, TR=16, NS=2, P=1)]


# Early weights: the last tile requested before the launch wait keeps the tail of its A bytes
# (one row of a tile of more than 4 rows, else 16 bytes) until after the wait.  (M, K, L, TR, NS,
# P): that tile with 1, 4 and 5 rows, at ring position 0, 1 and 2, partial last tiles, and CTAs
# with fewer tiles than the stages requested early (no tail held back, no producer wait).
EARLY_TAIL_CASES = [(1, 256, 1, 1, 2, 1), (5, 1024, 2, 5, 2, 1), (4, 2048, 1, 4, 2, 1),
                    (13, 512, 1, 4, 3, 1), (40, 1024, 2, 6, 3, 2), (30, 768, 1, 8, 4, 2),
                    (77, 256, 3, 9, 4, 3), (300, 2048, 1, 24, 2, 5)]


@pytest.mark.parametrize("case", EARLY_TAIL_CASES, ids=lambda c: "x".join(map(str, c)))
@pytest.mark.parametrize("rv", [False, True], ids=["smem_vector", "register_vector"])
def test_early_weights_tail_after_the_wait(pkg, case, rv):
    M, K, L, TR, NS, P = case
    w = workloads.random_workload(M, K, L, seed=M * 7 + K + TR,
                                  scale_bytes=workloads.pow2_scale_bytes(-3, 2))
    plain = run(pkg, w, tma_plan(TR=TR, NS=NS, P=P, rv=rv))
    early = run(pkg, w, tma_plan(TR=TR, NS=NS, P=P, rv=rv, flags=1))
    check(w, early, f"{case} rv={rv} early weights")
    # the copies' split changes nothing in the arithmetic: bit-identical to strict order
    assert np.array_equal(early.view(np.uint16), plain.view(np.uint16)), case


@pytest.mark.parametrize("shape", SHAPES, ids=[f"{m}x{k}x{l}" for m, k, l in SHAPES])
def test_ragged_shapes_all_plans(pkg, shape):
    M, K, L = shape
    w = workloads.random_workload(M, K, L, seed=M * 1000 + K + L,
                                  scale_bytes=workloads.pow2_scale_bytes(-4, 3), g_a=0.75,
                                  g_b=-1.25)
    steps = -(-K // 1024)
    for plan in PLANS:
        if plan is not None and plan.get("k_split", 0) > steps:
            with pytest.raises(pkg.NVFP4Error) as e:
                run(pkg, w, plan)
            assert e.value.status == 3
            continue
        if plan is not None and plan.get("ctas_per_batch", 0) > M:
            plan = dict(plan, ctas_per_batch=M)
        check(w, run(pkg, w, plan), f"{shape} {plan}")
    for plan in TMA_PLANS:
        if K % 256:
            with pytest.raises(pkg.NVFP4Error) as e:
                run(pkg, w, plan)
            assert e.value.status == 3
            continue
        if plan.get("ctas_per_batch", 0) > M:
            plan = dict(plan, ctas_per_batch=M)
        try:
            c = run(pkg, w, plan)
        except pkg.NVFP4Error as e:       # a forced ring too large for shared memory
            assert e.status == 3 and ("shared memory" in e.message or "warp count" in e.message), e
            continue
        check(w, c, f"{shape} {plan}")


@pytest.mark.parametrize("K", [16, 48, 80, 1040, 2064])
def test_k_not_multiple_of_32_uses_simple_kernel(pkg, K):
    w = workloads.random_workload(9, K, 2, seed=K)
    check(w, run(pkg, w), f"K={K}")
    with pytest.raises(pkg.NVFP4Error) as e:
        run(pkg, w, stream_plan())
    assert e.value.status == 3


def test_auto_plans_are_complete(pkg):
    for M, K, L in [(7168, 16384, 1), (4096, 7168, 8), (7168, 2048, 4), (3584, 6144, 16),
                    (128, 256, 1), (1, 16, 1)]:
        p = pkg.nvfp4_gemv_plan(M, K, L)
        assert p.kernel in (1, 2, 3, 4, 6) and p.warps_per_cta >= 1 and p.ctas_per_batch >= 1
        if K % 32 != 0:
            assert p.kernel == 6                            # the general-alignment kernel
        if K % 32 == 0:
            assert p.kernel in (2, 3, 4) and p.rows_per_warp in (1, 2, 4) and p.k_split >= 1
        if K % 256 == 0 and M * L >= 8 * 304:
            assert p.kernel in (3, 4) and p.stages >= 2 and p.tile_rows >= 1


def test_device_free_planner_matches_the_device(pkg):
    """nvfp4_plan_for_limits with this device's own limits gives the plans its launches use."""
    props = torch.cuda.get_device_properties(0)
    lim = {}
    for key, attr in (("sms", "multi_processor_count"),
                      ("max_smem_optin", "shared_memory_per_block_optin"),
                      ("max_smem_sm", "shared_memory_per_multiprocessor")):
        if not hasattr(props, attr):
            pytest.skip(f"torch does not report {attr}")
        lim[key] = int(getattr(props, attr))
    for M, K, L in [(7168, 16384, 1), (4096, 7168, 8), (7168, 2048, 4), (3584, 6144, 16),
                    (7168, 16384, 80), (4096, 7168, 64), (270000, 16384, 5), (128, 256, 1),
                    (1000, 1040, 3), (64, 7168, 3), (7168, 32768, 1)]:
        assert (pkg.nvfp4_plan_for_limits(M, K, L, **lim).as_dict()
                == pkg.nvfp4_gemv_plan(M, K, L).as_dict()), (M, K, L)


def test_auto_plans_fill_their_waves(pkg):
    """Batch counts that do not divide the CTA slots, or whose one-wave CTAs would hold too many
    rows, still get the register-vector kernel with a well-filled last wave."""
    slots = 2 * torch.cuda.get_device_properties(0).multi_processor_count
    for M, K, L in [(7168, 16384, 80), (4096, 7168, 64), (7168, 16384, 5), (270000, 16384, 5),
                    (3584, 6144, 16), (7168, 2048, 4), (4096, 7168, 8)]:
        p = pkg.nvfp4_gemv_plan(M, K, L)
        assert p.kernel == 4, (M, K, L, p.kernel)
        grid = p.ctas_per_batch * L
        fill = grid / (-(-grid // slots) * slots)
        assert fill >= 0.95, (M, K, L, p.ctas_per_batch, fill)


def test_largest_stream_k_and_beyond(pkg):
    kmax = pkg.nvfp4_max_stream_k()
    assert kmax >= 65536
    w = workloads.random_workload(6, kmax, 1, seed=3)
    assert pkg.nvfp4_gemv_plan(6, kmax, 1).kernel in (2, 3, 4)
    check(w, run(pkg, w), f"K={kmax}")
    w2 = workloads.random_workload(3, kmax + 32, 1, seed=4)
    assert pkg.nvfp4_gemv_plan(3, kmax + 32, 1).kernel == 6   # the shift kernel's bound is wider
    check(w2, run(pkg, w2), f"K={kmax + 32}")
    # past the shift kernel's shared memory (2.25 bytes per element of K): the byte-load kernel
    smem = torch.cuda.get_device_properties(0).shared_memory_per_block_optin \
        if hasattr(torch.cuda.get_device_properties(0), "shared_memory_per_block_optin") else 232448
    k3 = (int(smem / 2.25) // 32 + 1) * 32
    assert pkg.nvfp4_gemv_plan(3, k3, 1).kernel == 1
    w3 = workloads.random_workload(3, k3, 1, seed=5)
    check(w3, run(pkg, w3), f"K={k3}")


# ------------------------------------------------------------------ the five workloads, full size

@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5"])
def test_workloads_full_parity(pkg, workload, name):
    w = workload(name)
    c = run(pkg, w)
    assert not np.isnan(c).any()                         # every output written
    worst = check(w, c, name)
    assert worst <= 1.0
    c_again = run(pkg, w)
    assert np.array_equal(c.view(np.uint16), c_again.view(np.uint16))   # deterministic


def test_c1_matches_committed_oracle_fixture(pkg, workload):
    fx = json.load(open(os.path.join(HERE, "golden", "c1_oracle.json")))
    w = workload("c1")
    c = run(pkg, w)
    assert_parity(c, np.array([float(v) for v in fx["c_ref"]]),
                  np.array([float(v) for v in fx["T"]]), "c1 fixture")


@pytest.mark.parametrize("plan", [SIMPLE, stream_plan(), tma_plan(), tma_plan(rv=True, flags=1)],
                         ids=["simple", "stream", "tma", "tma-rv-early"])
def test_other_kernels_agree_at_full_size(pkg, workload, plan):
    w = workload("c2")
    check(w, run(pkg, w, plan), f"c2 {plan}")


# ------------------------------------------------------------------ invariants (bit for bit)

@pytest.mark.parametrize("shape", [(7168, 16384, 1), (300, 4096, 3), (2432, 2048, 2)],
                         ids=lambda s: "x".join(map(str, s)))
def test_l2_prefetch_in_strict_order_changes_no_bit(pkg, shape):
    """Strict stream order prefetches the first ring fill into L2 before the launch wait; the
    flag that turns the prefetch off must give the same bits, on both ring kernels."""
    M, K, L = shape
    w = workloads.random_workload(M, K, L, seed=M + K + L, scale_bytes=workloads.pow2_scale_bytes(-3, 2),
                                  g_a=0.25, g_b=0.5)
    for kernel in (3, 4):
        on = run(pkg, w, dict(kernel=kernel))
        off = run(pkg, w, dict(kernel=kernel, flags=16))
        assert np.array_equal(on.view(np.uint16), off.view(np.uint16)), kernel
    check(w, on, f"{shape} strict order, prefetch")


@pytest.fixture(scope="module")
def mid():
    return workloads.random_workload(300, 5120, 3, seed=77,
                                     scale_bytes=workloads.pow2_scale_bytes(-3, 3))


def test_negating_b_negates_exactly(pkg, mid):
    base = run(pkg, mid)
    neg = run(pkg, mid, b=mid.b ^ 0x88)
    # as values: an exact cancellation rounds to +0 whichever operand is negated
    assert np.array_equal(neg.astype(np.float64), -base.astype(np.float64))


def test_doubling_g_a_doubles_exactly(pkg, mid):
    base = run(pkg, mid).astype(np.float64)
    dbl = run(pkg, mid, g_a=2.0 * mid.g_a).astype(np.float64)
    assert np.array_equal(dbl, 2.0 * base)


def test_nibble_swap_of_both_operands_is_bit_identical(pkg, mid):
    sw = lambda x: ((x << 4) | (x >> 4)).astype(np.uint8)  # noqa: E731
    base = run(pkg, mid)
    assert np.array_equal(run(pkg, mid, A=sw(mid.A), b=sw(mid.b)).view(np.uint16),
                          base.view(np.uint16))


def test_batches_are_independent(pkg, mid):
    base = run(pkg, mid)
    A = mid.A.copy()
    A[1] ^= 0x5A
    sfb = mid.sfb.copy()
    sfb[1] = 0x40
    out = run(pkg, mid, A=A, sfb=sfb)
    assert np.array_equal(out[0].view(np.uint16), base[0].view(np.uint16))
    assert np.array_equal(out[2].view(np.uint16), base[2].view(np.uint16))


def test_plans_agree_within_tolerance(pkg, mid):
    for plan in PLANS + TMA_PLANS:
        check(mid, run(pkg, mid, plan), f"mid {plan}")
    assert pkg.nvfp4_gemv_plan(mid.M, mid.K, mid.L).kernel in (2, 3, 4)


def test_zero_scale_block(pkg, mid):
    sfa = mid.sfa.copy()
    sfa[2, 10, :] = 0
    c = run(pkg, mid, sfa=sfa)
    assert c[2, 10] == 0
    w = workloads.Workload("z", mid.M, mid.K, mid.L, mid.A, sfa, mid.b, mid.sfb, mid.g_a,
                           mid.g_b, 0)
    check(w, c, "zeroed row")


# ------------------------------------------------------------------ special values

def test_nan_scale_poisons_only_its_row(pkg):
    w = workloads.random_workload(40, 2048, 2, seed=9)
    w.sfa[1, 7, 33] = 0x7F
    c = run(pkg, w)
    nan = np.isnan(c)
    assert nan[1, 7] and nan.sum() == 1
    w.sfb[0, 5] = 0xFF
    c = run(pkg, w)
    assert np.isnan(c[0]).all() and np.isnan(c).sum() == w.M + 1


def test_overflow_gives_inf(pkg):
    w = workloads.random_workload(8, 1024, 1, seed=1, scale_bytes=(0x7E,), a_bytes=(0x77,),
                                  b_bytes=(0x77,))
    c = run(pkg, w)
    check(w, c, "overflow")
    assert np.isinf(c).all()


def test_empty_problem_leaves_c_untouched(pkg):
    c = torch.full((4,), 7.0, dtype=torch.float16, device="cuda")
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    pkg.nvfp4_gemv_batched(z, z, 1.0, z, z, 1.0, c, 0, 256, 1)
    pkg.nvfp4_gemv_batched(z, z, 1.0, z, z, 1.0, c, 4, 256, 0)
    torch.cuda.synchronize()
    assert (c == 7.0).all()


# ------------------------------------------------------------------ memory safety

@pytest.mark.parametrize("plan", [None, SIMPLE, stream_plan(R=4, S=3), tma_plan(TR=4, NS=2),
                                  tma_plan(TR=3, NS=5, P=2), tma_plan(rv=True, TR=3, NS=3),
                                  tma_plan(rv=True, flags=1)])
def test_guard_bands_and_poisoned_tails(pkg, plan):
    M, K, L = 77, 3328, 3
    w = workloads.random_workload(M, K, L, seed=5)
    G = 2048

    def padded(x, fill):
        flat = np.ascontiguousarray(x).ravel()
        buf = torch.full((flat.size + 256,), fill, dtype=torch.uint8, device="cuda")
        buf[:flat.size] = torch.from_numpy(flat).cuda()
        return buf, buf[:flat.size]

    A_buf, A = padded(w.A, 0xFF)
    sfa_buf, sfa = padded(w.sfa, 0x7F)       # E4M3 NaN: any over-read would show up as NaN
    b_buf, b = padded(w.b, 0xFF)
    sfb_buf, sfb = padded(w.sfb, 0x7F)
    out = torch.full((M * L + 2 * G,), -1, dtype=torch.int16, device="cuda")
    out[G:G + M * L] = torch.tensor(0x7E00, dtype=torch.int16)  # fp16 NaN pre-fill
    c = out[G:G + M * L]
    pkg.nvfp4_gemv_batched_ex(A, sfa, w.g_a, b, sfb, w.g_b, c, M, K, L, plan=plan)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert (o[:G] == -1).all() and (o[G + M * L:] == -1).all()
    got = o[G:G + M * L].view(np.float16).reshape(L, M)
    assert not np.isnan(got).any()
    check(w, got, f"guarded {plan}")


def test_error_statuses_with_real_buffers(pkg):
    w = workloads.random_workload(8, 256, 1, seed=2)
    t = {k: dev(getattr(w, k)) for k in ("A", "sfa", "b", "sfb")}
    c = torch.empty((1, 8), dtype=torch.float16, device="cuda")
    raw = torch.zeros(4096, dtype=torch.uint8, device="cuda")

    def status(**kw):
        args = dict(A=t["A"], sfa=t["sfa"], b=t["b"], sfb=t["sfb"], c=c, M=8, K=256, L=1)
        args.update(kw)
        try:
            pkg.nvfp4_gemv_batched(args["A"], args["sfa"], 1.0, args["b"], args["sfb"], 1.0,
                                   args["c"], args["M"], args["K"], args["L"])
            torch.cuda.synchronize()
            return 0
        except pkg.NVFP4Error as e:
            return e.status

    assert status() == 0
    assert status(A=raw[1:]) == 0                           # any alignment: the simple kernel
    with pytest.raises(pkg.NVFP4Error) as e:                # ... but no vector-load kernel
        pkg.nvfp4_gemv_batched_ex(raw[1:], t["sfa"], 1.0, t["b"], t["sfb"], 1.0, c, 8, 256, 1,
                                  plan=dict(kernel=2))
    assert e.value.status == 2
    assert status(c=c.data_ptr() + 1) == 2                  # misaligned c (raw address)
    assert status(c=raw[2:].view(torch.int16)[:8]) == 0     # 2-byte aligned c is fine
    assert status(K=24) == 1
    assert status(c=t["A"][:16].view(torch.float16)) == 1   # c overlaps A
    with pytest.raises(pkg.NVFP4Error) as e:
        pkg.nvfp4_gemv_batched_ex(t["A"], t["sfa"], 1.0, t["b"], t["sfb"], 1.0, c, 8, 256, 1,
                                  plan=pkg.Plan(kernel=2, flags=64))
    assert e.value.status == 3
    with pytest.raises(pkg.NVFP4Error) as e:
        pkg.nvfp4_gemv_batched_ex(t["A"], t["sfa"], 1.0, t["b"], t["sfb"], 1.0, c, 8, 256, 1,
                                  plan=dict(kernel=7))
    assert e.value.status == 3
    host = torch.zeros(4096, dtype=torch.uint8)
    with pytest.raises(ValueError):                        # the binding refuses CPU tensors
        pkg.nvfp4_gemv_batched(host, t["sfa"], 1.0, t["b"], t["sfb"], 1.0, c, 8, 256, 1)


# ------------------------------------------------------------------ streams and graphs

def test_non_default_stream_and_graph_capture(pkg):
    w = workloads.random_workload(1000, 4096, 2, seed=12)
    t = {k: dev(getattr(w, k)) for k in ("A", "sfa", "b", "sfb")}
    ref = run(pkg, w)
    s = torch.cuda.Stream()
    c = torch.full((w.L, w.M), float("nan"), dtype=torch.float16, device="cuda")
    with torch.cuda.stream(s):
        pkg.nvfp4_gemv_batched(t["A"], t["sfa"], w.g_a, t["b"], t["sfb"], w.g_b, c, w.M, w.K,
                               w.L)
    s.synchronize()
    assert np.array_equal(c.cpu().numpy().view(np.uint16), ref.view(np.uint16))

    c.fill_(float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(3):
            pkg.nvfp4_gemv_batched(t["A"], t["sfa"], w.g_a, t["b"], t["sfb"], w.g_b, c, w.M,
                                   w.K, w.L)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(c.cpu().numpy().view(np.uint16), ref.view(np.uint16))

"""GPU parity of the grouped (mixture-of-experts) decode GEMV through the C ABI against the oracle.

Every token's output row is compared with oracle/grouped.py under the parity tolerance (fp16, or
the bfloat16 variant), for both ways of naming experts (the bridge's cumulative offsets and a
per-token index), every kernel, tokens that no expert owns, identity routing against the batched
entry point (bit for bit), offsets that decrease (each row must be zeros or one expert's GEMV),
routing written on the device by preceding work, and CUDA-graph replays with new routing.
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import grouped as G
from parity import assert_parity, bf16_bits_to_f64

pytestmark = pytest.mark.gpu

OUT_F16, OUT_BF16 = 0, 1


@pytest.fixture(scope="module")
def pkg():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    from decode_nvfp4_gemv_gb300 import build

    build.build()
    import decode_nvfp4_gemv_gb300 as p

    p.load_library()
    return p


def offsets_of(expert_of, E):
    """Inclusive cumulative token counts per expert (the bridge's compute_expert_offsets)."""
    return np.cumsum(np.bincount(np.asarray(expert_of), minlength=E)).astype(np.int32)


class Dev:
    def __init__(self, w):
        self.w = w
        self.A = torch.from_numpy(w.A).cuda()
        self.sfa = torch.from_numpy(w.sfa).cuda()
        self.g_a = torch.from_numpy(np.ascontiguousarray(w.g_a, dtype=np.float32)).cuda()
        self.g_b = torch.from_numpy(np.ascontiguousarray(w.g_b, dtype=np.float32)).cuda()
        self.b = torch.from_numpy(w.b).cuda()
        self.sfb = torch.from_numpy(w.sfb).cuda()


def run(pkg, d, M, K, E, T, offsets=None, expert_of=None, out=OUT_F16, plan=None, stream=None,
        c=None):
    if c is None:
        c = torch.full((T, M), -1, dtype=torch.int16, device="cuda")   # poison: 0xFFFF is NaN
    po = None if offsets is None else torch.from_numpy(np.asarray(offsets, np.int32)).cuda()
    pm = None if expert_of is None else torch.from_numpy(np.asarray(expert_of, np.int32)).cuda()
    pkg.nvfp4_gemv_grouped(d.A, d.sfa, d.g_a, d.b, d.sfb, d.g_b, c, M, K, E, T,
                           expert_offsets=po, expert_of_token=pm, out_dtype=out, stream=stream,
                           plan=plan)
    torch.cuda.synchronize()
    return decode_out(c, out)


def decode_out(c, out):
    bits = c.cpu().numpy().view(np.uint16)
    return bf16_bits_to_f64(bits) if out == OUT_BF16 else bits.view(np.float16).astype(np.float64)


def oracle_of(w, experts):
    return G.gemv_grouped(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, experts, w.M, w.K)


def tma_plan(TR=0, NS=0, P=0, W=0, rv=False, flags=0):
    return dict(kernel=4 if rv else 3, tile_rows=TR, stages=NS, ctas_per_batch=P,
                warps_per_cta=W, flags=flags)


PLANS = [None, dict(kernel=1), dict(kernel=2), dict(kernel=2, rows_per_warp=4, ctas_per_batch=1),
         dict(kernel=2, rows_per_warp=1, ctas_per_batch=3, warps_per_cta=5), tma_plan(),
         tma_plan(TR=5, NS=3, P=2, W=3), tma_plan(rv=True), tma_plan(rv=True, TR=3, NS=4, P=2),
         tma_plan(rv=True, flags=2)]


@pytest.fixture(scope="module")
def g0():
    return workloads.make_grouped("g0")


@pytest.mark.parametrize("out", [OUT_F16, OUT_BF16], ids=["f16", "bf16"])
@pytest.mark.parametrize("form", ["offsets", "map"])
def test_small_all_plans(pkg, g0, form, out):
    w = g0
    d = Dev(w)
    experts = w.expert_of
    ref, T = oracle_of(w, experts)
    fmt = "bf16" if out == OUT_BF16 else "f16"
    for plan in PLANS:
        kw = dict(offsets=offsets_of(experts, w.E)) if form == "offsets" else dict(expert_of=experts)
        try:
            c = run(pkg, d, w.M, w.K, w.E, w.T, out=out, plan=plan, **kw)
        except pkg.NVFP4Error as e:
            assert e.status == 3 and ("shared memory" in e.message or "warp count" in e.message), e
            continue
        assert_parity(c, ref, T, f"g0 {form} {plan}", fmt=fmt)


def test_tokens_without_an_expert_get_zeros(pkg, g0):
    w = g0
    d = Dev(w)
    # offsets that stop two tokens short: the last two rows belong to no expert
    offs = offsets_of(w.expert_of, w.E)
    offs = np.minimum(offs, w.T - 2).astype(np.int32)
    experts = G.experts_from_offsets(offs, w.T)
    assert (experts[-2:] == -1).all()
    ref, T = oracle_of(w, experts)
    for plan in (None, dict(kernel=1), dict(kernel=2), tma_plan(), tma_plan(rv=True)):
        c = run(pkg, d, w.M, w.K, w.E, w.T, offsets=offs, plan=plan)
        assert (c[-2:] == 0).all()
        assert_parity(c, ref, T, f"short offsets {plan}")
    # an index map with -1 and E (both out of range)
    emap = w.expert_of.copy()
    emap[0] = -1
    emap[3] = w.E
    experts = G.experts_from_map(emap, w.E)
    ref, T = oracle_of(w, experts)
    for plan in (None, dict(kernel=1), tma_plan(rv=True)):
        c = run(pkg, d, w.M, w.K, w.E, w.T, expert_of=emap, plan=plan)
        assert (c[0] == 0).all() and (c[3] == 0).all()
        assert_parity(c, ref, T, f"map with holes {plan}")


@pytest.mark.parametrize("shape", [(300, 1024, 4), (2600, 17408, 2), (96, 37888, 3)],
                         ids=["300x1024x4", "17-segments-one-idle", "37-segments-split"])
def test_identity_routing_equals_the_batched_call(pkg, shape):
    """E experts, one token each, equal global scales: the same kernel and plan as the batched
    entry point with L = E, so the same bits (also with an idle segment, and with K split over a
    cluster into slices of 13, 13 and 11 segments)."""
    M, K, L = shape
    w = workloads.random_workload(M, K, L, seed=21, scale_bytes=workloads.pow2_scale_bytes(-3, 3),
                                  g_a=0.5, g_b=2.0)
    gw = workloads.GroupedWorkload("id", M, K, L, L, w.A, w.sfa, np.full(L, 0.5, np.float32),
                                   np.full(L, 2.0, np.float32), w.b, w.sfb,
                                   np.arange(L, dtype=np.int32), 21)
    d = Dev(gw)
    plans = [None, dict(kernel=1), dict(kernel=2), tma_plan()]
    if K <= 32768:   # past 32 segments the register-vector kernel needs K split over a cluster
        plans.append(tma_plan(rv=True))
    for plan in plans:
        cg = run(pkg, d, M, K, L, L, offsets=np.arange(1, L + 1), plan=plan)
        cb = torch.full((L, M), float("nan"), dtype=torch.float16, device="cuda")
        pkg.nvfp4_gemv_batched_ex(d.A, d.sfa, 0.5, d.b, d.sfb, 2.0, cb, M, K, L, plan=plan)
        torch.cuda.synchronize()
        assert np.array_equal(cg, cb.cpu().numpy().astype(np.float64)), plan


def test_decreasing_offsets_stay_in_bounds(pkg, g0):
    """Offsets that decrease name no valid grouping; each row must still be zeros or the GEMV of
    one of the experts (all in bounds, nothing else written)."""
    w = g0
    d = Dev(w)
    offs = np.array([5, 2, 7, 1, 6, 3], np.int32)[: w.E]
    c = run(pkg, d, w.M, w.K, w.E, w.T, offsets=offs)
    cands = [oracle_of(w, np.full(w.T, e))[0] for e in range(w.E)]
    for t in range(w.T):
        if (c[t] == 0).all():
            continue
        assert any(np.allclose(c[t], cand[t], rtol=2e-3, atol=1e-3) for cand in cands), t


def test_routing_written_by_preceding_work(pkg, g0):
    """The offsets are produced on the stream right before each call (as a router would): each
    call must see its own routing."""
    w = g0
    d = Dev(w)
    M, K, E, T = w.M, w.K, w.E, w.T
    routes = [offsets_of(w.expert_of, E), np.full(E, T, np.int32), np.arange(1, E + 1) % (T + 1)]
    routes[2] = np.maximum.accumulate(routes[2]).astype(np.int32)
    offs_dev = torch.zeros(E, dtype=torch.int32, device="cuda")
    srcs = [torch.from_numpy(np.asarray(r, np.int32)).cuda() for r in routes]
    outs = [torch.full((T, M), -1, dtype=torch.int16, device="cuda") for _ in routes]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for src, c in zip(srcs, outs):
            offs_dev.copy_(src)
            pkg.nvfp4_gemv_grouped(d.A, d.sfa, d.g_a, d.b, d.sfb, d.g_b, c, M, K, E, T,
                                   expert_offsets=offs_dev, stream=s)
    s.synchronize()
    for r, c in zip(routes, outs):
        experts = G.experts_from_offsets(r, T)
        ref, tb = oracle_of(w, experts)
        assert_parity(decode_out(c, OUT_F16), ref, tb, f"route {r.tolist()}")


def test_graph_replay_with_new_routing(pkg, g0):
    w = g0
    d = Dev(w)
    M, K, E, T = w.M, w.K, w.E, w.T
    emap = torch.from_numpy(w.expert_of.copy()).cuda()
    c = torch.zeros((T, M), dtype=torch.int16, device="cuda")
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):   # warm-up (device info cached outside the capture)
        pkg.nvfp4_gemv_grouped(d.A, d.sfa, d.g_a, d.b, d.sfb, d.g_b, c, M, K, E, T,
                               expert_of_token=emap, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pkg.nvfp4_gemv_grouped(d.A, d.sfa, d.g_a, d.b, d.sfb, d.g_b, c, M, K, E, T,
                               expert_of_token=emap, stream=s)
    rng = np.random.default_rng(3)
    for _ in range(3):
        new = np.sort(rng.integers(0, E, T)).astype(np.int32)
        with torch.cuda.stream(s):
            emap.copy_(torch.from_numpy(new).cuda())
            g.replay()
        s.synchronize()
        ref, tb = oracle_of(w, new)
        assert_parity(decode_out(c, OUT_F16), ref, tb, f"replay {new.tolist()}")


@pytest.mark.parametrize("form", ["offsets", "map"])
def test_full_size_decode_moe(pkg, form):
    """g1: 32 experts of 3584 x 6144, 2 tokens x top-8 (16 rows), the automatic plan, fp16 and
    bf16 outputs, two routings over the same weights."""
    w0 = workloads.make_grouped("g1")
    for route in (0, 1):
        w = w0 if route == 0 else workloads.make_grouped("g1", route=1, with_weights=w0)
        d = Dev(w)
        ref, T = oracle_of(w, w.expert_of)
        kw = (dict(offsets=offsets_of(w.expert_of, w.E)) if form == "offsets"
              else dict(expert_of=w.expert_of))
        for out, fmt in ((OUT_F16, "f16"), (OUT_BF16, "bf16")):
            c = run(pkg, d, w.M, w.K, w.E, w.T, out=out, **kw)
            assert not np.isnan(c).any()
            assert_parity(c, ref, T, f"g1 route {route} {form} {fmt}", fmt=fmt)

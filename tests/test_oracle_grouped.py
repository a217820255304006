"""Pins of the grouped (mixture-of-experts) oracle (oracle/grouped.py) against things other than
itself: a worked example of the bridge's cumulative offsets, a second formulation of token
ownership, the batched definition (identity routing, one shared expert), relabelling and scale
invariants, and a brute-force loop over tiny inputs.  Planted mistakes each fail a pin."""
import numpy as np
import pytest

import oracle
import workloads
from oracle import E2M1_TABLE, E4M3FN_TABLE
from oracle import grouped as G


def test_offsets_worked_example():
    # tokens per expert [2, 0, 3, 1]: offsets are the running totals [2, 2, 5, 6]
    # (compute_expert_offsets); tokens 0-1 -> expert 0, none -> 1, 2-4 -> 2, 5 -> 3, 6-7 -> none
    owner = G.experts_from_offsets([2, 2, 5, 6], 8)
    assert owner.tolist() == [0, 0, 2, 2, 2, 3, -1, -1]


def test_offsets_match_first_greater_formulation():
    rng = np.random.default_rng(0)
    for _ in range(50):
        E = int(rng.integers(1, 12))
        counts = rng.integers(0, 4, E)
        offsets = np.cumsum(counts)
        T = int(offsets[-1] + rng.integers(0, 3))
        # second formulation: the first e with t < offsets[e]
        want = [next((e for e in range(E) if t < offsets[e]), -1) for t in range(T)]
        assert G.experts_from_offsets(offsets, T).tolist() == want


def test_map_range():
    assert G.experts_from_map([0, 3, -1, 4, 2], 4).tolist() == [0, 3, -1, -1, 2]


def _tiny(E, M, K, T, seed):
    w = workloads.random_workload(M, K, E, seed=seed, scale_bytes=workloads.pow2_scale_bytes(-2, 2))
    v = workloads.random_workload(1, K, T, seed=seed + 1)
    rng = np.random.default_rng(seed)
    g_a = np.float32([0.25, 0.5, 1.0, 2.0])[rng.integers(0, 4, E)]
    g_b = np.float32([0.5, 1.0, 2.0])[rng.integers(0, 3, E)]
    return w.A, w.sfa, g_a, v.b, v.sfb, g_b


def brute(A, sfa, g_a, b, sfb, g_b, experts, M, K):
    """The formula as a plain loop over (token, row, k)."""
    T = len(experts)
    out = np.zeros((T, M))
    for t in range(T):
        e = int(experts[t])
        if e < 0:
            continue
        for m in range(M):
            s = 0.0
            for k in range(K):
                ca = (int(A[e, m, k // 2]) >> (4 * (k % 2))) & 15
                cb = (int(b[t, k // 2]) >> (4 * (k % 2))) & 15
                s += (E2M1_TABLE[ca] * E2M1_TABLE[cb] * E4M3FN_TABLE[sfa[e, m, k // 16]]
                      * E4M3FN_TABLE[sfb[t, k // 16]])
            out[t, m] = s * float(g_a[e]) * float(g_b[e])
    return out


def test_brute_force_tiny():
    A, sfa, g_a, b, sfb, g_b = _tiny(E=3, M=2, K=32, T=6, seed=5)
    experts = np.array([2, 0, -1, 2, 1, 0])
    c, bound = G.gemv_grouped(A, sfa, g_a, b, sfb, g_b, experts, 2, 32)
    assert np.array_equal(c, brute(A, sfa, g_a, b, sfb, g_b, experts, 2, 32))
    assert np.all(c[2] == 0) and np.all(bound[2] == 0)
    assert np.all(np.abs(c) <= bound)


def test_identity_routing_is_the_batched_gemv():
    w = workloads.random_workload(8, 256, 5, seed=3, scale_bytes=workloads.pow2_scale_bytes(-3, 3),
                                  g_a=0.5, g_b=2.0)
    E = w.L
    c, bound = G.gemv_grouped(w.A, w.sfa, np.full(E, w.g_a, np.float32), w.b, w.sfb,
                              np.full(E, w.g_b, np.float32),
                              G.experts_from_offsets(np.arange(1, E + 1), E), w.M, w.K)
    ref, tref = oracle.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, w.M, w.K, w.L)
    assert np.array_equal(c, ref) and np.array_equal(bound, tref)


def test_one_expert_is_the_batched_gemv_on_a_repeated_matrix():
    w = workloads.random_workload(6, 128, 1, seed=4)
    v = workloads.random_workload(1, 128, 4, seed=9)
    c, _ = G.gemv_grouped(w.A, w.sfa, np.float32([0.75]), v.b, v.sfb, np.float32([1.5]),
                          G.experts_from_offsets([4], 4), 6, 128)
    ref, _ = oracle.gemv(np.repeat(w.A, 4, axis=0), np.repeat(w.sfa, 4, axis=0), 0.75, v.b, v.sfb,
                         1.5, 6, 128, 4)
    assert np.array_equal(c, ref)


def test_relabelling_experts_changes_nothing():
    A, sfa, g_a, b, sfb, g_b = _tiny(E=4, M=3, K=64, T=7, seed=7)
    experts = np.array([1, 3, 3, 0, 2, 1, -1])
    perm = np.array([2, 0, 3, 1])          # old expert e becomes perm[e]
    inv = np.argsort(perm)
    c0, _ = G.gemv_grouped(A, sfa, g_a, b, sfb, g_b, experts, 3, 64)
    e1 = np.where(experts >= 0, perm[np.maximum(experts, 0)], -1)
    c1, _ = G.gemv_grouped(A[inv], sfa[inv], g_a[inv], b, sfb, g_b[inv], e1, 3, 64)
    assert np.array_equal(c0, c1)


def test_per_expert_scale_touches_only_its_tokens():
    A, sfa, g_a, b, sfb, g_b = _tiny(E=3, M=4, K=64, T=6, seed=8)
    experts = np.array([0, 1, 1, 2, 0, 1])
    c0, _ = G.gemv_grouped(A, sfa, g_a, b, sfb, g_b, experts, 4, 64)
    g2 = g_a.copy()
    g2[1] *= 2
    c1, _ = G.gemv_grouped(A, sfa, g2, b, sfb, g_b, experts, 4, 64)
    mine = experts == 1
    assert np.array_equal(c1[mine], 2 * c0[mine]) and np.array_equal(c1[~mine], c0[~mine])


# planted mistakes: each variant must fail one of the pins above
def _owner_off_by_one(offsets, T):
    offsets = [int(v) for v in offsets]
    return np.array([next((e for e in range(len(offsets)) if t <= offsets[e]), -1)
                     for t in range(T)])


def _grouped_scale_by_token(A, sfa, g_a, b, sfb, g_b, experts, M, K):
    c, bound = G.gemv_grouped(A, sfa, g_a, b, sfb, g_b, experts, M, K)
    for t, e in enumerate(experts):
        if e >= 0 and t < len(g_b) and g_b[t] != g_b[e]:
            c[t] *= float(g_b[t]) / float(g_b[e])
    return c, bound


def test_planted_mistakes_are_caught():
    assert _owner_off_by_one([2, 2, 5, 6], 8).tolist() != [0, 0, 2, 2, 2, 3, -1, -1]
    A, sfa, g_a, b, sfb, g_b = _tiny(E=3, M=2, K=32, T=6, seed=5)
    experts = np.array([2, 0, -1, 2, 1, 0])
    c, _ = _grouped_scale_by_token(A, sfa, g_a, b, sfb, g_b, experts, 2, 32)
    assert not np.array_equal(c, brute(A, sfa, g_a, b, sfb, g_b, experts, 2, 32))

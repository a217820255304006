"""GPU parity at operand sizes past 2^31 and 2^32 bytes, through the C ABI.

Offsets into A reach beyond 32-bit range only at sizes no other test touches:
- the batched GEMV with 80 batches of 7168 x 16384 (A is 4.7 GB);
- the grouped GEMV over 80 such experts;
- the small-N GEMM with one 270000 x 16384 matrix (A is 2.2 GB; M is not a multiple of 128).

The big matrices are built on the device from one seeded 7168 x 16384 block: copy q is the
block with every byte XORed with key(q).  The host knows each row's bytes without reading the
device.  Every kernel is checked against the oracle on sampled outputs: the first and last
batch, expert and row, plus random ones.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from parity import assert_parity

pytestmark = pytest.mark.gpu

M0, K = 7168, 16384
K2, K16 = K // 2, K // 16
L_BIG = 80


def key(q):
    return (37 * q + 11) & 0xFF


@pytest.fixture(scope="module")
def pkg():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    from decode_nvfp4_gemv_gb300 import build

    build.build()
    import decode_nvfp4_gemv_gb300 as p

    p.load_library()
    return p


@pytest.fixture(scope="module")
def block():
    """One seeded 7168 x 16384 matrix (power-of-two block scales) and 80 vectors."""
    w = workloads.random_workload(M0, K, 1, seed=31, scale_bytes=workloads.pow2_scale_bytes(-3, 2),
                                  g_a=0.75, g_b=1.25)
    v = workloads.random_workload(1, K, L_BIG, seed=32,
                                  scale_bytes=workloads.pow2_scale_bytes(-2, 1))
    return w.A[0], w.sfa[0], v.b, v.sfb, w.g_a, w.g_b


def tiled_rows(blk, blk_s, rows):
    """Device tensors [rows][K/2], [rows][K/16]: row m is block row m % M0 XOR key(m // M0)."""
    dA = torch.from_numpy(blk).cuda()
    dS = torch.from_numpy(blk_s).cuda()
    A = torch.empty((rows, K2), dtype=torch.uint8, device="cuda")
    S = torch.empty((rows, K16), dtype=torch.uint8, device="cuda")
    for q in range(0, (rows + M0 - 1) // M0):
        r0, r1 = q * M0, min(rows, (q + 1) * M0)
        torch.bitwise_xor(dA[: r1 - r0], key(q), out=A[r0:r1])
        S[r0:r1].copy_(dS[: r1 - r0])
    return A, S


def host_row(blk, blk_s, m):
    q, r = divmod(int(m), M0)
    return blk[r] ^ np.uint8(key(q)), blk_s[r]


def expected(blk, blk_s, rows, vec_idx, b, sfb, g_a, g_b):
    """Oracle values at the given global rows of the tiled matrix, each with its own vector."""
    A_s = np.stack([host_row(blk, blk_s, m)[0] for m in rows])[:, None]
    S_s = np.stack([host_row(blk, blk_s, m)[1] for m in rows])[:, None]
    c, T = oracle.gemv(A_s, S_s, g_a, b[vec_idx], sfb[vec_idx], g_b, 1, K, len(rows))
    return c[:, 0], T[:, 0]


def samples(n_outer, n_inner, seed, count=48):
    rng = np.random.default_rng(seed)
    outer = np.concatenate([[0, n_outer - 1, n_outer - 1, 0], rng.integers(0, n_outer, count)])
    inner = np.concatenate([[0, n_inner - 1, 0, n_inner - 1], rng.integers(0, n_inner, count)])
    return outer, inner


def test_batched_beyond_4gb(pkg, block):
    blk, blk_s, b, sfb, g_a, g_b = block
    A, S = tiled_rows(blk, blk_s, L_BIG * M0)
    assert A.numel() > 2 ** 32
    db, dsb = torch.from_numpy(b).cuda(), torch.from_numpy(sfb).cuda()
    ls, ms = samples(L_BIG, M0, seed=1)
    ref, T = expected(blk, blk_s, ls * M0 + ms, ls, b, sfb, g_a, g_b)
    for plan in (None, dict(kernel=1), dict(kernel=2), dict(kernel=5),
                 dict(kernel=4, ctas_per_batch=16, flags=1), dict(kernel=3, ctas_per_batch=38)):
        c = torch.full((L_BIG, M0), float("nan"), dtype=torch.float16, device="cuda")
        pkg.nvfp4_gemv_batched_ex(A, S, g_a, db, dsb, g_b, c, M0, K, L_BIG, plan=plan)
        torch.cuda.synchronize()
        out = c.cpu().numpy()
        assert not np.isnan(out).any(), plan
        assert_parity(out[ls, ms], ref, T, f"80 batches, A 4.7 GB, plan {plan}")
    del A, S
    torch.cuda.empty_cache()


def test_grouped_beyond_4gb(pkg, block):
    blk, blk_s, b, sfb, _, _ = block
    A, S = tiled_rows(blk, blk_s, L_BIG * M0)
    g_a = (0.5 + np.arange(L_BIG) / 64).astype(np.float32)
    g_b = (2.0 - np.arange(L_BIG) / 128).astype(np.float32)
    expert_of = np.array([79, 0, 41, 79, 63], dtype=np.int32)
    T_tok = len(expert_of)
    dga, dgb = torch.from_numpy(g_a).cuda(), torch.from_numpy(g_b).cuda()
    db = torch.from_numpy(np.ascontiguousarray(b[:T_tok])).cuda()
    dsb = torch.from_numpy(np.ascontiguousarray(sfb[:T_tok])).cuda()
    dmap = torch.from_numpy(expert_of).cuda()
    ts, ms = samples(T_tok, M0, seed=2, count=40)
    rows = expert_of[ts].astype(np.int64) * M0 + ms
    ref = np.empty(len(ts))
    bound = np.empty(len(ts))
    for i, (t, m) in enumerate(zip(ts, rows)):   # each token's own expert scales
        e = int(expert_of[t])
        c1, T1 = expected(blk, blk_s, [m], [t], b, sfb, g_a[e], g_b[e])
        ref[i], bound[i] = c1[0], T1[0]
    for plan in (None, dict(kernel=2), dict(kernel=4, ctas_per_batch=16)):
        c = torch.full((T_tok, M0), float("nan"), dtype=torch.float16, device="cuda")
        pkg.nvfp4_gemv_grouped(A, S, dga, db, dsb, dgb, c, M0, K, L_BIG, T_tok,
                               expert_of_token=dmap, plan=plan)
        torch.cuda.synchronize()
        out = c.cpu().numpy()
        assert not np.isnan(out).any(), plan
        assert_parity(out[ts, ms], ref, bound, f"80 experts, A 4.7 GB, plan {plan}")
    del A, S
    torch.cuda.empty_cache()


def test_small_n_beyond_2gb(pkg, block):
    blk, blk_s, b, sfb, g_a, g_b = block
    M, N = 270000, 5
    A, S = tiled_rows(blk, blk_s, M)
    assert A.numel() > 2 ** 31
    db = torch.from_numpy(np.ascontiguousarray(b[:N])).cuda()
    dsb = torch.from_numpy(np.ascontiguousarray(sfb[:N])).cuda()
    ns, ms = samples(N, M, seed=3)
    ref, T = expected(blk, blk_s, ms, ns, b, sfb, g_a, g_b)
    for plan in (None, dict(kernel=5, k_split=1), dict(kernel=4), dict(kernel=1)):
        c = torch.full((N, M), float("nan"), dtype=torch.float16, device="cuda")
        pkg.nvfp4_gemm_small_n(A, S, g_a, db, dsb, g_b, c, M, K, N, plan=plan)
        torch.cuda.synchronize()
        out = c.cpu().numpy()
        assert not np.isnan(out).any(), plan
        assert_parity(out[ns, ms], ref, T, f"M=270000, A 2.2 GB, plan {plan}")
    del A, S
    torch.cuda.empty_cache()

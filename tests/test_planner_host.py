"""The planner without a GPU, through nvfp4_plan_for_limits (the C ABI's device-free planning
entry point).

It checks:
- the plans the four large decode workloads get on GB300's limits (the ones the bench reports);
- that every automatic plan over a grid of shapes takes the register-vector TMA kernel with a
  well-filled last wave;
- that plans scale with the device's SM count;
- that a forced plan is honoured field by field, or refused with the status a launch would
  return;
- that implausible limits and shapes are rejected.
"""
import pytest

import decode_nvfp4_gemv_gb300 as pkg


KERNEL_STREAM, KERNEL_TMA, KERNEL_TMA_RV, KERNEL_TC = 2, 3, 4, 5
INVALID, UNSUPPORTED = 1, 3


@pytest.fixture(scope="module", autouse=True)
def lib():
    from decode_nvfp4_gemv_gb300 import build

    build.build()
    return pkg.load_library()


def plan(M, K, L, forced=None, **lim):
    return pkg.nvfp4_plan_for_limits(M, K, L, plan=forced, **lim).as_dict()


def status_of(M, K, L, forced=None, **lim):
    with pytest.raises(pkg.NVFP4Error) as e:
        pkg.nvfp4_plan_for_limits(M, K, L, plan=forced, **lim)
    return e.value.status


# (M, K, L): kernel, CTAs per batch, consumer warps, 1024-element segments per warp, tile rows,
# ring stages, CTAs per SM -- one wave of CTAs for each workload, with early weights
DECODE_PLANS = {
    (7168, 16384, 1): (KERNEL_TMA_RV, 304, 8, 2, 4, 2, 2),
    (4096, 7168, 8): (KERNEL_TMA_RV, 57, 7, 1, 8, 2, 3),    # 7 warps of one segment: 3 per SM
    (7168, 2048, 4): (KERNEL_TMA_RV, 76, 12, 1, 24, 2, 2),
    (3584, 6144, 16): (KERNEL_TMA_RV, 19, 12, 1, 16, 2, 2),
}


@pytest.mark.parametrize("shape", list(DECODE_PLANS), ids=lambda s: "x".join(map(str, s)))
def test_decode_workload_plans_on_gb300(shape):
    p = plan(*shape, forced={"flags": 1})
    got = (p["kernel"], p["ctas_per_batch"], p["warps_per_cta"], p["k_split"], p["tile_rows"],
           p["stages"])
    assert got == DECODE_PLANS[shape][:6]
    assert p["flags"] == 1 and p["rows_per_warp"] == 4
    assert p["ctas_per_batch"] * shape[2] == DECODE_PLANS[shape][6] * 152


def test_three_ctas_per_sm_only_with_early_weights():
    # in strict stream order the 7-warp plans keep two CTAs per SM
    p = plan(4096, 7168, 8, forced={"flags": 0})
    assert (p["ctas_per_batch"], p["warps_per_cta"], p["tile_rows"], p["stages"]) == (38, 7, 12, 2)
    # with early weights, three; a CTA with few rows keeps 4-row tiles and two stages
    q = plan(7168, 7168, 1, forced={"flags": 1})
    assert (q["ctas_per_batch"], q["tile_rows"], q["stages"]) == (456, 4, 2)
    # 8 or more consumer warps never take three CTAs per SM
    for shape in ((7168, 16384, 1), (7168, 8192, 1), (7168, 2048, 4)):
        r = plan(*shape, forced={"flags": 1})
        assert r["ctas_per_batch"] * shape[2] <= 2 * 152, shape


def _fill(grid, slots):
    return grid / (-(-grid // slots) * slots)


def test_automatic_plans_fill_their_waves():
    """Every shape with at least 8 rows per CTA slot, at least 85 KB per SM and K % 256 == 0
    (K <= 16384, two CTAs per SM) gets the register-vector kernel, a valid warp mapping and a last
    wave >= 95% full."""
    n = 0
    for K in (256, 512, 1024, 2048, 3072, 4096, 6144, 7168, 16384):
        nseg = -(-K // 1024)
        for M in (256, 1000, 3584, 4096, 7168, 20000, 100000):
            for L in (1, 2, 3, 5, 7, 8, 16, 24, 33, 50, 64, 80, 100, 150, 304, 500):
                if M * L < 8 * 304 or M * L * (K // 2 + K // 16) < 85 * 1024 * 152:
                    continue                              # small calls: sized by their bytes
                p = plan(M, K, L)
                n += 1
                assert p["kernel"] == KERNEL_TMA_RV, (M, K, L, p)
                W, P = p["warps_per_cta"], p["ctas_per_batch"]
                assert 1 <= P <= M and 1 <= W <= 16
                assert (nseg % W == 0 and p["k_split"] == nseg // W <= 2) or \
                       (W % nseg == 0 and p["k_split"] == 1), (M, K, L, p)
                assert 1 <= p["tile_rows"] <= 256 and 2 <= p["stages"] <= 8
                assert _fill(P * L, 304) >= 0.95, (M, K, L, p)
    assert n > 700


def test_plans_follow_the_sm_count():
    half = dict(sms=76, max_smem_optin=232448, max_smem_sm=233472)
    assert plan(7168, 16384, 1, **half)["ctas_per_batch"] == 152
    assert plan(7168, 2048, 4, **half)["ctas_per_batch"] == 38
    assert plan(4096, 7168, 8, **half)["ctas_per_batch"] == 19


def test_register_capped_rings_take_one_wave():
    """K of 20-24 segments unsplit: 10-12 consumer warps of two segments each hold ~90 registers a
    thread, so the register file takes one CTA per SM; the grid is one wave of 152 CTAs, with a
    four-stage ring to keep the SM's loads in flight (in strict order; with early weights two
    stages of twice the rows up to 22 segments)."""
    for M, K, L in ((8192, 20480, 1), (8192, 24576, 1), (4096, 24576, 4)):
        p = plan(M, K, L, forced={"flags": 0})
        assert p["kernel"] == KERNEL_TMA_RV and p["k_slices"] == 1, (M, K, L, p)
        assert p["ctas_per_batch"] * L == 152 and p["stages"] == 4, (M, K, L, p)
        assert p["k_split"] == 2 and p["warps_per_cta"] == K // 2048, (M, K, L, p)
        q = plan(M, K, L, forced={"flags": 1})
        assert q["ctas_per_batch"] * L == 152 and q["warps_per_cta"] == p["warps_per_cta"]
        assert (q["tile_rows"], q["stages"]) == ((8, 2) if K // 1024 <= 22 else (4, 4)), q


def test_odd_segment_counts_take_warps_of_two_with_one_idle():
    """An odd segment count past 16 has no warp count that divides it: ceil(segments / 2) warps of
    two segments, the last warp's second one idle (unsplit, or over clusters of two)."""
    for nseg in (17, 19, 21, 23, 25, 29):
        p = plan(8192, nseg * 1024, 1, forced={"flags": 1})
        assert p["kernel"] == KERNEL_TMA_RV and p["k_slices"] == 1, (nseg, p)
        assert p["warps_per_cta"] == (nseg + 1) // 2 and p["k_split"] == 2, (nseg, p)
    for nseg in (27, 31):
        p = plan(8192, nseg * 1024, 1, forced={"flags": 1})
        assert p["k_slices"] == 2 and p["warps_per_cta"] == (nseg + 3) // 4, (nseg, p)
    # a forced warp count must still divide the segments (or be a multiple of them)
    assert status_of(8192, 17 * 1024, 1, forced={"kernel": KERNEL_TMA_RV, "warps_per_cta": 9}) \
        == UNSUPPORTED


def test_one_cta_rings_with_early_weights_take_two_large_stages():
    """One unsplit CTA per SM on 19-22 segments with early weights: two stages of about twice the
    bytes (8-row tiles where the CTA's rows allow) in place of four; strict order keeps four."""
    for M, K, L in ((3584, 18944, 1), (14336, 22528, 1), (1792, 18944, 8)):
        ew = plan(M, K, L, forced={"flags": 1})
        st = plan(M, K, L, forced={"flags": 0})
        assert ew["ctas_per_batch"] * L == 152 and (ew["tile_rows"], ew["stages"]) == (8, 2), ew
        assert (st["tile_rows"], st["stages"]) == (4, 4), st
    # 24 segments keep four stages also with early weights
    assert plan(8192, 24576, 1, forced={"flags": 1})["stages"] == 4


def test_wide_k_splits_over_a_cluster_of_two():
    """K of 28-32 segments: split over a cluster of two CTAs, each slice on 7-8 warps of two
    segments, two clusters' CTAs per SM -- instead of one 14-16 warp CTA per SM."""
    for M, K in ((7168, 32768), (8192, 28672)):
        p = plan(M, K, 1, forced={"flags": 1})
        assert p["kernel"] == KERNEL_TMA_RV and p["k_slices"] == 2, (M, K, p)
        assert p["ctas_per_batch"] * 2 == 304 and p["k_split"] == 2, (M, K, p)
        assert p["warps_per_cta"] == K // 4096, (M, K, p)


# Thread-block clusters of S CTAs a GB300 holds at once, at one and at two CTAs per SM (the
# occupancy query's answers on a 152-SM GB300; a cluster's CTAs share one GPC)
CLUSTERS_RESIDENT = {1: {2: 76, 3: 46, 4: 36, 5: 28, 6: 23, 7: 15, 8: 15},
                     2: {2: 152, 3: 97, 4: 74, 5: 58, 6: 46, 7: 38, 8: 36}}


def _ctas_per_sm_by_regs(p):
    """CTAs per SM the register file holds: 96 (two segments a warp) or 72 (one) registers a
    thread, a quarter of the SM's 64 K registers per scheduler."""
    per_scheduler = 16384 // ((96 if p["k_split"] == 2 else 72) * 32)
    return max(1, 4 * per_scheduler // (p["warps_per_cta"] + 1))


def test_split_grids_fit_the_resident_clusters():
    """Every automatic split-K plan launches at most the clusters the GPU holds at once (small
    calls fewer, by their bytes), or, where the rows do not fit one wave's CTAs, waves at least 95%
    full."""
    n = 0
    for nseg in range(28, 129):
        for M, L in ((8192, 1), (2048, 4), (512, 1), (100000, 1)):
            p = plan(M, nseg * 1024, L, forced={"flags": 1})
            if p["k_slices"] < 2:
                continue
            n += 1
            occ = min(2, _ctas_per_sm_by_regs(p))
            cap = CLUSTERS_RESIDENT[occ][p["k_slices"]]
            grid = p["ctas_per_batch"] * L
            assert grid <= cap or _fill(grid, cap) >= 0.95, (M, nseg, L, p)
    assert n > 100


@pytest.mark.parametrize("K,S", [(36864, 2), (49152, 2), (53248, 4), (65536, 4), (98304, 4),
                                 (114688, 8), (131072, 8), (262144, 8), (33792, 2), (37888, 2),
                                 (52224, 4), (54272, 4), (99328, 8), (61440, 4)])
def test_huge_k_splits_into_slices_of_at_most_24_segments(K, S):
    """Past 32 segments no single CTA holds the vector slice: K splits over 2, 4 or 8 CTAs of a
    cluster, the first whose slices (ceil(segments / S) each, the last the rest) are at most 24
    segments (12 warps of two), else over 3, 5, 6 or 7, else the first whose slices are at most 32.
    The grid is the clusters the GPU holds at once."""
    p = plan(8192, K, 1, forced={"flags": 1})
    assert p["kernel"] == KERNEL_TMA_RV and p["k_slices"] == S, p
    nseg = -(-K // 1024)
    sl = lambda s: -(-nseg // s)
    order = [s for most in (24, 32) for s in (2, 4, 8, 3, 5, 6, 7)
             if (s - 1) * sl(s) < nseg and sl(s) <= most]
    assert S == order[0]
    occ = min(2, _ctas_per_sm_by_regs(p))
    assert p["ctas_per_batch"] == min(CLUSTERS_RESIDENT[occ][S], 8192)


def _small_call_grid(M, K, L, slots=304):
    """The grid the planner documents for small calls: 76, 152 or 304 CTAs by the call's bytes
    (below 10 KB and 85 KB per SM), at most 152 for more than 16 segments unsplit, at most 3/4 of
    the slots when K is split."""
    sms = slots // 2
    nbytes = M * L * (K // 2 + K // 16)
    G = slots // 4 if nbytes < 10 * 1024 * sms else slots // 2 if nbytes < 85 * 1024 * sms \
        else slots
    return G


def test_small_calls_take_the_ring_on_a_grid_sized_by_bytes():
    """Few rows (below 8 per CTA slot) or few bytes (below 85 KB per SM), K % 256 == 0: the
    register-vector kernel on 76 / 152 / 304 CTAs by the call's bytes; K split over a cluster
    into slices of at most 16 segments only past 32 segments."""
    n = 0
    for K in (256, 1024, 2048, 4096, 7168, 8192, 16384, 32768, 65536, 131072):
        nseg = -(-K // 1024)
        for M in (1, 5, 16, 64, 128, 300, 512, 1000, 2000, 2432, 7168):
            for L in (1, 2, 3):
                rows = M * L
                nbytes = rows * (K // 2 + K // 16)
                if rows >= 8 * 304 and nbytes >= 85 * 1024 * 152:
                    continue
                p = plan(M, K, L)
                S, P = p["k_slices"], p["ctas_per_batch"]
                if nseg > 32 and not any(nseg % s == 0 and nseg // s <= 16 for s in range(2, 9)):
                    assert p["kernel"] != KERNEL_TMA_RV or S <= 1, (M, K, L, p)
                    continue
                if nseg in (17, 19, 23, 29, 31):                 # no warp mapping: other kernels
                    continue
                n += 1
                assert p["kernel"] == KERNEL_TMA_RV, (M, K, L, p)
                G = _small_call_grid(M, K, L)
                if nseg <= 32:
                    assert S == 1, (M, K, L, p)
                    if nseg > 16:
                        G = min(G, 152)
                else:
                    assert S == min(s for s in range(2, 9) if nseg % s == 0 and nseg // s <= 16)
                    G = min(G, 228)
                assert P == min(M, max(1, G // (L * S))), (M, K, L, p, G)
    assert n > 250


def test_forced_k_slices():
    p = plan(64, 16384, 1, forced={"kernel": KERNEL_TMA_RV, "k_slices": 2})
    assert p["k_slices"] == 2 and p["kernel"] == KERNEL_TMA_RV
    assert plan(64, 16384, 1, forced={"kernel": KERNEL_TMA_RV})["k_slices"] == 1
    assert plan(7168, 16384, 1)["k_slices"] == 1
    for forced in ({"kernel": KERNEL_TMA_RV, "k_slices": 7}, {"kernel": KERNEL_TMA_RV, "k_slices": 9},
                   {"kernel": KERNEL_STREAM, "k_slices": 2}, {"kernel": KERNEL_TMA, "k_slices": 2},
                   {"kernel": KERNEL_TMA_RV, "k_slices": -1}):
        assert status_of(64, 16384, 1, forced=forced) == UNSUPPORTED, forced
    # slices need not divide the segments: 16 segments in three slices of 6, 6 and 4
    assert plan(64, 16384, 1, forced={"kernel": KERNEL_TMA_RV, "k_slices": 3})["k_slices"] == 3


def test_planning_is_deterministic_and_forced_plans_are_echoed():
    for shape in list(DECODE_PLANS) + [(20000, 4096, 33), (100000, 16384, 80), (64, 16384, 1),
                                       (512, 65536, 1), (100, 2304, 3)]:
        a = plan(*shape)
        assert plan(*shape) == a
        forced = {k: v for k, v in a.items()}
        assert plan(*shape, forced=forced) == a


@pytest.mark.parametrize("forced", [
    {"kernel": KERNEL_TC, "k_split": 9}, {"kernel": KERNEL_TC, "stages": 7},
    {"kernel": KERNEL_TC, "stages": 1}, {"kernel": KERNEL_TC, "warps_per_cta": 8},
    {"kernel": KERNEL_TC, "tile_rows": 64}, {"kernel": KERNEL_TMA, "tile_rows": 300},
    {"kernel": KERNEL_TMA_RV, "stages": 9}, {"kernel": KERNEL_TMA_RV, "stages": 1},
    {"kernel": KERNEL_TMA_RV, "warps_per_cta": 17}, {"kernel": KERNEL_TMA_RV, "rows_per_warp": 2},
    {"kernel": 9}, {"flags": 0x100}, {"ctas_per_batch": -1},
], ids=lambda f: ",".join(f"{k}={v}" for k, v in f.items()))
def test_forced_plans_out_of_range_are_refused(forced):
    assert status_of(7168, 2048, 4, forced=forced) == UNSUPPORTED


def test_kernels_that_need_k_multiples_refuse_other_k():
    for kernel in (KERNEL_TMA, KERNEL_TMA_RV, KERNEL_TC):
        assert status_of(512, 1056, 2, forced={"kernel": kernel}) == UNSUPPORTED
    assert status_of(512, 1040, 2, forced={"kernel": KERNEL_STREAM}) == UNSUPPORTED
    assert plan(512, 1040, 2)["kernel"] == 6            # K % 32 == 16: the shift kernel
    assert plan(512, 1056, 2)["kernel"] in (1, 2)       # K % 32 == 0: CUDA-core kernels


def test_shift_kernel_plans():
    """K % 32 == 16 takes the general-alignment kernel: 8 warps, 4 rows per warp, one wave of CTA
    slots (two per SM while the staged vector fits half an SM); a forced plan outside its range is
    refused, and a vector too long for shared memory falls back to the byte-load kernel."""
    p = plan(7168, 16400, 1)
    assert (p["kernel"], p["warps_per_cta"], p["rows_per_warp"], p["ctas_per_batch"]) == \
        (6, 8, 4, 304)
    assert plan(4096, 7184, 8)["ctas_per_batch"] == 38
    assert plan(7168, 2064, 1, forced={"kernel": 6})["kernel"] == 6
    assert status_of(7168, 2064, 1, forced={"kernel": 6, "warps_per_cta": 9}) == UNSUPPORTED
    assert status_of(7168, 2064, 1, forced={"kernel": 6, "rows_per_warp": 2}) == UNSUPPORTED
    assert plan(64, 160016, 2)["kernel"] == 1            # 2.25 B/element of K > 227 KB
    assert status_of(64, 160016, 2, forced={"kernel": 6}) == UNSUPPORTED


def test_tensor_core_plans():
    p = plan(7168, 16384, 1, forced={"kernel": KERNEL_TC})
    assert p["kernel"] == KERNEL_TC and p["tile_rows"] == 128 and p["warps_per_cta"] == 4
    assert 2 <= p["k_split"] <= 8 and 2 <= p["stages"] <= 6   # 56 tiles leave slots: split K
    q = plan(7168, 16384, 16, forced={"kernel": KERNEL_TC})
    assert q["k_split"] == 1                               # 896 tiles fill the GPU unsplit
    r = plan(7168, 512, 1, forced={"kernel": KERNEL_TC, "k_split": 2})
    assert r["k_split"] == 2
    assert status_of(7168, 512, 1, forced={"kernel": KERNEL_TC, "k_split": 3}) == UNSUPPORTED


def test_one_row_group_ctas_take_one_warp_per_segment():
    """Small calls whose CTAs hold at most 4 rows (one row group) and at most 6 segments: one
    consumer warp per segment (four for one or two segments) instead of 12 mostly idle ones."""
    n = 0
    for K in (256, 512, 1024, 2048, 3072, 4096, 5120, 6144, 7168, 16384):
        nseg = -(-K // 1024)
        for M, L in ((64, 1), (128, 1), (128, 2), (256, 1), (300, 1), (600, 2)):
            p = plan(M, K, L, forced={"flags": 1})
            rows = -(-M // p["ctas_per_batch"])
            if p["k_slices"] > 1 or rows > 4:
                continue
            n += 1
            if nseg <= 6:
                assert p["warps_per_cta"] == (4 if nseg <= 2 else nseg), (M, K, L, p)
            else:
                assert p["warps_per_cta"] >= 7, (M, K, L, p)
    assert n > 30
    # c1 (128 x 256 x 1): 76 CTAs of 2 rows, four warps
    assert plan(128, 256, 1)["warps_per_cta"] == 4


def test_small_calls_with_early_weights_request_two_tiles_early():
    """With early weights a two-stage ring requests one tile before the launch wait; small calls
    whose CTAs hold more than one tile take a third stage, so two go out early.  Strict-order plans
    and one-tile CTAs keep theirs."""
    for shape, strict_stages in (((2048, 7168, 1), 4), ((4096, 2048, 1), 2), ((768, 7168, 3), 4),
                                 ((2048, 3072, 2), 2)):
        ew = plan(*shape, forced={"flags": 1})
        st = plan(*shape, forced={"flags": 0})
        assert ew["stages"] == 3, (shape, ew)
        assert st["stages"] == strict_stages, (shape, st)
        assert -(-(-(-shape[0] // ew["ctas_per_batch"])) // ew["tile_rows"]) > 1
    assert plan(128, 7168, 1, forced={"flags": 1})["stages"] == 2      # one tile a CTA
    # full grids (more than 3/4 of the CTA slots) keep two: 2000 x 16384 on 304 CTAs
    assert plan(2000, 16384, 1, forced={"flags": 1})["stages"] == 2
    assert plan(1024, 16384, 1, forced={"flags": 1})["stages"] == 3    # on 152


def test_tiles_hold_whole_row_groups():
    """A warp's item is 4 rows: automatic tiles hold a multiple of 4 rows (or the CTA's rows),
    also where a row is more than a quarter of the stage target (K of 25-26 segments)."""
    for M, K, L in ((3584, 25600, 1), (8192, 25600, 1), (14336, 26624, 1), (2048, 26624, 1)):
        p = plan(M, K, L, forced={"flags": 1})
        assert p["tile_rows"] % 4 == 0 and p["k_slices"] == 1, (M, K, L, p)
    n = 0
    for K in range(256, 32768 + 1, 1024):
        for M in (2432, 4096, 8192, 20000):
            p = plan(M, K, 1)
            if p["kernel"] in (KERNEL_TMA, KERNEL_TMA_RV):
                n += 1
                rows = -(-M // p["ctas_per_batch"])
                assert p["tile_rows"] % 4 == 0 or p["tile_rows"] >= rows, (M, K, p)
    assert n > 100


def test_few_large_tiles_take_a_third_stage():
    """Stages of at least 32 KB and 8 rows, at most four a CTA, two CTAs per SM: three stages
    where they fit (K = 8192 on 8-row tiles); 4-row stages (K = 16384) and smaller stages keep
    two."""
    for shape in ((8192, 8192, 1), (7168, 8192, 1), (4096, 8192, 2), (3072, 8192, 3)):
        for flags in (0, 1):
            p = plan(*shape, forced={"flags": flags})
            assert (p["tile_rows"], p["stages"]) == (8, 3), (shape, flags, p)
    for shape in ((4096, 16384, 1), (7168, 16384, 1), (8192, 4096, 1)):
        assert plan(*shape, forced={"flags": 1})["stages"] == 2, shape
    # large calls (>= 8 rows per CTA slot, >= 85 KB per SM) keep two stages also when they are
    # small (below 24 KB: K = 3584 on 12 rows, K = 5120 on 8)
    for shape in ((5120, 5120, 1), (7168, 3584, 1), (14336, 3584, 1), (3584, 3584, 4)):
        for flags in (0, 1):
            p = plan(*shape, forced={"flags": flags})
            assert p["stages"] == 2 and p["k_slices"] == 1, (shape, flags, p)


def test_tensor_core_ring_keeps_two_ctas_per_sm():
    # five stages of 20,480 bytes plus the tokens' scales and the split-K partials: 114,944 bytes,
    # two CTAs in the 228 KB of an SM
    p = plan(7168, 16384, 1, forced={"kernel": KERNEL_TC})
    assert (p["k_split"], p["stages"]) == (5, 5)
    assert plan(7168, 16384, 16, forced={"kernel": KERNEL_TC})["stages"] == 5
    # with less shared memory per SM the ring gets shallower instead of leaving one CTA per SM
    r = plan(7168, 16384, 1, forced={"kernel": KERNEL_TC}, max_smem_sm=200 * 1024,
             max_smem_optin=199 * 1024)
    assert (r["k_split"], r["stages"]) == (5, 4)


def test_tensor_core_split_runs_in_one_wave_of_clusters():
    """The tensor-core kernel splits K over clusters of S CTAs, one cluster per 128-row tile: S is
    the largest (up to 8, and while the tiles leave half the CTA slots empty) whose clusters the
    GPU holds at once, so no tile waits for a second wave."""
    n = 0
    for M in range(128, 19 * 1024, 128):
        for L in (1, 2):
            p = plan(M, 16384, L, forced={"kernel": KERNEL_TC})
            tiles, S = -(-M // 128) * L, p["k_split"]
            if S > 1:
                n += 1
                assert tiles <= CLUSTERS_RESIDENT[2][S], (M, L, p)
                if S < 8 and 2 * tiles * (S + 1) <= 2 * 304:
                    assert tiles > CLUSTERS_RESIDENT[2][S + 1], (M, L, p)   # the largest that fits
    assert n > 100
    # 60 tiles: five slices would be 60 clusters of 5 where 58 fit; four it is
    assert plan(7680, 16384, 1, forced={"kernel": KERNEL_TC})["k_split"] == 4


@pytest.mark.parametrize("lim", [dict(sms=0), dict(max_smem_optin=512),
                                 dict(max_smem_sm=1000, max_smem_optin=2000)],
                         ids=["no SMs", "tiny smem", "sm smem below cta smem"])
def test_implausible_limits_are_rejected(lim):
    assert status_of(7168, 16384, 1, **lim) == INVALID


def test_shapes_are_checked_like_the_launching_entry_points():
    assert status_of(0, 256, 1) == INVALID
    assert status_of(16, 256, 0) == INVALID
    assert status_of(16, 40, 1) == INVALID                 # K % 16 != 0
    assert status_of(2 ** 31, 256, 1) == UNSUPPORTED

"""Seeded synthetic inputs for the NVFP4 batched GEMV.

This module is the only code shared by the CPU oracle's tests and the CUDA path's tests and bench.
It draws bytes; it holds none of the GEMV's arithmetic (no decoding, no products, no sums).

Random numbers: splitmix64 (S. Vigna's 64-bit mixing generator), written here from its published
definition: state_i = seed + i * 0x9E3779B97F4A7C15 (mod 2**64) and
z = state_i; z = (z ^ z>>30) * 0xBF58476D1CE4E5B9; z = (z ^ z>>27) * 0x94D049BB133111EB;
out = z ^ z>>31.  It is counter based, so every draw is a pure function of (seed, tensor, index).
Each tensor has its own sub-seed, splitmix64(seed * 16 + tensor id); ids: A=0, sfa=1, b=2, sfb=3.
Tensors are filled in memory order.  Uniform bytes take the 8 little-endian bytes of each draw;
a choice from a set of n values takes draw % n.

The five workloads (shapes and value distributions as the decode configurations specify them):

  c1  M=128,  K=256,   L=1   A, b uniform bytes (all 16 codes in each nibble); sfa, sfb the E4M3
                             values {0, 1, 2} (bytes 0x00, 0x38, 0x40); g_a = g_b = 1.  Seed 1.
  c2  M=7168, K=16384, L=1   A, b uniform bytes; scales uniform over powers of two 2**-3..2**2
                             (bytes 0x20..0x48 step 0x08); g_a = g_b = fp32(1/(6*448)).  Seed 2.
  c3  M=4096, K=7168,  L=8   as c1, independent per batch.  Seed 3.
  c4  M=7168, K=2048,  L=4   A [L][M][K] and b [L][K] drawn N(0, 1) (Box-Muller), rounded to bf16,
                             then quantized to NVFP4 (see ``quantize_bf16_to_nvfp4``).  Seed 4.
  c5  M=3584, K=6144,  L=16  A, b uniform bytes; scales powers of two 2**-4..2**3 (bytes
                             0x18..0x50 step 0x08); g_a = 0.5, g_b = 2.0.  Seed 5.

The c1/c3 recipe follows the blog's data preparation ("nvFP4 Batch GEMV算子系列(下)", section
"准备数据": integer scale values 0..2 converted numerically to float8_e4m3fn), widened to all byte
values for A and b and with sfa and sfb drawn independently.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_U64 = np.uint64

TENSOR_IDS = {"A": 0, "sfa": 1, "b": 2, "sfb": 3, "x": 4, "route": 5, "g": 6}
# x: a bf16 activation vector; route: expert choices of the grouped workloads; g: their scales


_CHUNK = 1 << 20  # draws per chunk: temporaries stay cache-resident


def _mix(z: np.ndarray) -> np.ndarray:
    """The splitmix64 output function, applied in place to a uint64 array of states."""
    t = np.empty_like(z)
    with np.errstate(over="ignore"):
        np.right_shift(z, _U64(30), out=t); z ^= t; z *= _U64(_M1)
        np.right_shift(z, _U64(27), out=t); z ^= t; z *= _U64(_M2)
        np.right_shift(z, _U64(31), out=t); z ^= t
    return z


def splitmix64(state: int, n: int, start: int = 0) -> np.ndarray:
    """Draws start+1 .. start+n of the splitmix64 sequence seeded with ``state`` (uint64 array)."""
    z = np.arange(start + 1, start + n + 1, dtype=_U64)
    with np.errstate(over="ignore"):
        z *= _U64(GOLDEN)
        z += _U64(state % (1 << 64))
    return _mix(z)


def _chunks(n: int):
    for i0 in range(0, n, _CHUNK):
        yield i0, min(n, i0 + _CHUNK)


def sub_seed(seed: int, tensor: str) -> int:
    """splitmix64(seed * 16 + tensor id): the first draw of the sequence seeded with that value."""
    return int(splitmix64((seed * 16 + TENSOR_IDS[tensor]) % (1 << 64), 1)[0])


def uniform_bytes(seed: int, tensor: str, n: int) -> np.ndarray:
    s = sub_seed(seed, tensor)
    out = np.empty(((n + 7) // 8) * 8, dtype=np.uint8)
    words = out.view("<u8")
    for i0, i1 in _chunks(len(words)):
        words[i0:i1] = splitmix64(s, i1 - i0, start=i0)
    return out[:n]


def choice_bytes(seed: int, tensor: str, n: int, values) -> np.ndarray:
    values = np.asarray(values, dtype=np.uint8)
    s = sub_seed(seed, tensor)
    out = np.empty(n, dtype=np.uint8)
    for i0, i1 in _chunks(n):
        draws = splitmix64(s, i1 - i0, start=i0)
        out[i0:i1] = values[(draws % _U64(len(values))).view(np.int64)]
    return out


def uniform01(seed: int, tensor: str, n: int, start: int = 0) -> np.ndarray:
    """n doubles in [0, 1) from the top 53 bits of each draw (draws start+1 .. start+n)."""
    draws = splitmix64(sub_seed(seed, tensor), n, start)
    return (draws >> _U64(11)).view(np.int64).astype(np.float64) * 2.0 ** -53


# E4M3FN byte encodings of the scale value sets used by the workloads (bit patterns, no decoding):
# 0 -> 0x00, 1 -> 0x38, 2 -> 0x40; 2**e -> (e + 7) << 3.
SCALES_0_1_2 = (0x00, 0x38, 0x40)


def pow2_scale_bytes(e_lo: int, e_hi: int):
    return tuple((e + 7) << 3 for e in range(e_lo, e_hi + 1))


@dataclass
class Workload:
    name: str
    M: int
    K: int
    L: int
    A: np.ndarray      # uint8 [L][M][K/2]
    sfa: np.ndarray    # uint8 [L][M][K/16]
    b: np.ndarray      # uint8 [L][K/2]
    sfb: np.ndarray    # uint8 [L][K/16]
    g_a: float         # fp32 value
    g_b: float         # fp32 value
    seed: int
    recipe: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def algorithmic_bytes(self) -> int:
        """Bytes the GEMV must move: A, sfa, b, sfb read once, c (fp16) written once."""
        M, K, L = self.M, self.K, self.L
        return M * K * L // 2 + M * K * L // 16 + K * L // 2 + K * L // 16 + 2 * M * L


def algorithmic_bytes(M: int, K: int, L: int) -> int:
    return M * K * L // 2 + M * K * L // 16 + K * L // 2 + K * L // 16 + 2 * M * L


def random_workload(M: int, K: int, L: int, seed: int, scale_bytes=SCALES_0_1_2,
                    g_a: float = 1.0, g_b: float = 1.0, name: str = "custom",
                    a_bytes=None, b_bytes=None) -> Workload:
    """Uniform packed bytes for A and b (or draws from ``a_bytes``/``b_bytes`` if given) and block
    scales drawn uniformly from ``scale_bytes``."""
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    if a_bytes is None:
        A = uniform_bytes(seed, "A", L * M * K // 2)
    else:
        A = choice_bytes(seed, "A", L * M * K // 2, a_bytes)
    if b_bytes is None:
        b = uniform_bytes(seed, "b", L * K // 2)
    else:
        b = choice_bytes(seed, "b", L * K // 2, b_bytes)
    sfa = choice_bytes(seed, "sfa", L * M * K // 16, scale_bytes)
    sfb = choice_bytes(seed, "sfb", L * K // 16, scale_bytes)
    return Workload(name, M, K, L, A.reshape(L, M, K // 2), sfa.reshape(L, M, K // 16),
                    b.reshape(L, K // 2), sfb.reshape(L, K // 16),
                    float(np.float32(g_a)), float(np.float32(g_b)), seed,
                    recipe=f"uniform bytes, scales from {len(scale_bytes)} values")


# ---------------------------------------------------------------------------------------------
# c4: N(0,1) bf16 data quantized to NVFP4.  This is input preparation, not the GEMV: it encodes
# samples into the input format.  It follows bridge.py's quantize_to_nvfp4 in its fp32 operation
# order (global scale amax/(6*448); x/gs; per-16 block amax/6 cast to float8_e4m3fn; divide by the
# quantized block scale with a 1e-8 guard; clamp to 6) but rounds to the E2M1 grid with
# round-to-nearest-even instead of that function's half-step lookup table.
# ---------------------------------------------------------------------------------------------

# E2M1 grid points in code order and the midpoints between neighbours.
_E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float32)
_E2M1_MID = (_E2M1_GRID[:-1] + _E2M1_GRID[1:]) / 2


def _e2m1_rne_code(mag: np.ndarray) -> np.ndarray:
    """Magnitude code (0..7) of the nearest E2M1 grid point, ties to the even code.

    code = number of midpoints strictly below mag, plus one when mag sits exactly on a midpoint
    whose lower neighbour has an odd code (so the tie goes to the even code above it).
    """
    code = np.zeros(mag.shape, dtype=np.uint8)
    for j, mid in enumerate(_E2M1_MID):
        code += mag > mid
        if j % 2 == 1:
            code += mag == mid
    return code


def _bf16_round(x32: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (round-to-nearest-even) -> fp32, for finite inputs."""
    bits = x32.astype(np.float32).view(np.uint32).astype(np.uint64)
    bits = (bits + 0x7FFF + ((bits >> 16) & 1)) & 0xFFFF0000
    return bits.astype(np.uint32).view(np.float32)


def normal_bf16(seed: int, tensor: str, n: int) -> np.ndarray:
    """n samples of N(0, 1) (Box-Muller on splitmix64 uniforms), rounded to bf16, as fp32.

    Draws 2i+1 and 2i+2 give samples 2i (cosine branch) and 2i+1 (sine branch).
    """
    out = np.empty(2 * ((n + 1) // 2), dtype=np.float32)
    pairs = len(out) // 2
    for p0 in range(0, pairs, _CHUNK // 2):
        p1 = min(pairs, p0 + _CHUNK // 2)
        u = uniform01(seed, tensor, 2 * (p1 - p0), start=2 * p0)
        r = np.sqrt(-2.0 * np.log(1.0 - u[0::2]))          # 1 - u in (0, 1]
        theta = (2.0 * np.pi) * u[1::2]
        z = np.empty(2 * (p1 - p0), dtype=np.float32)
        z[0::2] = r * np.cos(theta)
        z[1::2] = r * np.sin(theta)
        out[2 * p0:2 * p1] = _bf16_round(z)
    return out[:n]


def quantize_bf16_to_nvfp4(x: np.ndarray):
    """x: fp32 [..., K] (bf16 values).  Returns (packed [..., K/2], scale bytes [..., K/16], gs).

    One global scale over the whole tensor: gs = max(amax, 1e-8) / (6 * 448) in fp32.
    """
    import torch  # float8_e4m3fn round-to-nearest-even cast (library primitive)

    x = np.asarray(x, dtype=np.float32)
    K = x.shape[-1]
    lead = x.shape[:-1]
    rows = x.reshape(-1, K)
    amax = np.float32(max(float(np.abs(x).max()), 1e-8))
    gs = np.float32(amax / np.float32(6.0 * 448.0))
    packed = np.empty((rows.shape[0], K // 2), dtype=np.uint8)
    sf_bytes = np.empty((rows.shape[0], K // 16), dtype=np.uint8)
    step = max(1, _CHUNK // K)
    for r0 in range(0, rows.shape[0], step):
        r1 = min(rows.shape[0], r0 + step)
        xn = (rows[r0:r1] / gs).astype(np.float32)
        blocks = xn.reshape(r1 - r0, K // 16, 16)
        bamax = np.maximum(np.abs(blocks).max(axis=-1), np.float32(1e-8)).astype(np.float32)
        sf8 = torch.from_numpy(bamax / np.float32(6.0)).to(torch.float8_e4m3fn)
        sf_bytes[r0:r1] = sf8.view(torch.uint8).numpy()
        sf_val = sf8.to(torch.float32).numpy()
        xs = blocks / np.maximum(sf_val, np.float32(1e-8))[..., None]
        mag = np.minimum(np.abs(xs), np.float32(6.0))
        code = (_e2m1_rne_code(mag) | np.where(xs < 0, np.uint8(8), np.uint8(0))).astype(np.uint8)
        code = code.reshape(r1 - r0, K)
        packed[r0:r1] = code[:, 0::2] | (code[:, 1::2] << 4)
    return packed.reshape(*lead, K // 2), sf_bytes.reshape(*lead, K // 16), float(gs)


def quantized_normal_workload(M: int, K: int, L: int, seed: int, name: str = "custom") -> Workload:
    xa = normal_bf16(seed, "A", L * M * K).reshape(L, M, K)
    A, sfa, g_a = quantize_bf16_to_nvfp4(xa)
    del xa
    xb = normal_bf16(seed, "b", L * K).reshape(L, K)
    b, sfb, g_b = quantize_bf16_to_nvfp4(xb)
    return Workload(name, M, K, L, A, sfa, b, sfb, g_a, g_b, seed,
                    recipe="N(0,1) bf16 quantized to NVFP4 (RNE E2M1, amax/(6*448) global scale)")


CONFIGS = {
    "c1": dict(M=128, K=256, L=1, seed=1),
    "c2": dict(M=7168, K=16384, L=1, seed=2),
    "c3": dict(M=4096, K=7168, L=8, seed=3),
    "c4": dict(M=7168, K=2048, L=4, seed=4),
    "c5": dict(M=3584, K=6144, L=16, seed=5),
}


def make(name: str, seed: int | None = None) -> Workload:
    cfg = CONFIGS[name]
    M, K, L = cfg["M"], cfg["K"], cfg["L"]
    s = cfg["seed"] if seed is None else seed
    if name in ("c1", "c3"):
        w = random_workload(M, K, L, s, SCALES_0_1_2, 1.0, 1.0, name)
    elif name == "c2":
        g = float(np.float32(1.0) / np.float32(6.0 * 448.0))
        w = random_workload(M, K, L, s, pow2_scale_bytes(-3, 2), g, g, name)
    elif name == "c4":
        w = quantized_normal_workload(M, K, L, s, name)
    elif name == "c5":
        w = random_workload(M, K, L, s, pow2_scale_bytes(-4, 3), 0.5, 2.0, name)
    else:
        raise KeyError(name)
    return w


# ---------------------------------------------------------------------------------------------
# Grouped (mixture-of-experts) decode workloads.  E experts' weights [E][M][K/2] drawn like c5
# (M=3584, K=6144 is the expert shape of the bridge's grouped GEMM); each of `tokens` tokens picks
# `top_k` distinct experts uniformly at random; the (token, expert) rows are sorted by expert
# (stable) and each row gets its own packed vector.  Per-expert global scales are drawn from small
# sets of powers of two.  `route` selects an independent routing and vectors over the same
# weights.  Only draws here: the expert offsets are derived by the caller.
# ---------------------------------------------------------------------------------------------
@dataclass
class GroupedWorkload:
    name: str
    M: int
    K: int
    E: int
    T: int
    A: np.ndarray          # uint8 [E][M][K/2]
    sfa: np.ndarray        # uint8 [E][M][K/16]
    g_a: np.ndarray        # float32 [E]
    g_b: np.ndarray        # float32 [E]
    b: np.ndarray          # uint8 [T][K/2]
    sfb: np.ndarray        # uint8 [T][K/16]
    expert_of: np.ndarray  # int32 [T], non-decreasing
    seed: int
    recipe: str = ""

    @property
    def active_experts(self) -> int:
        return len(np.unique(self.expert_of[self.expert_of >= 0]))

    @property
    def algorithmic_bytes(self) -> int:
        """Bytes a call must move: the weights and scales of every expert that owns a token, once;
        the vectors, the outputs (16-bit) and the per-expert scales and offsets."""
        M, K, E, T = self.M, self.K, self.E, self.T
        return (self.active_experts * (M * K // 2 + M * K // 16) + T * (K // 2 + K // 16)
                + 2 * M * T + 12 * E)


GROUPED = {
    "g1": dict(M=3584, K=6144, E=32, tokens=2, top_k=8, seed=11),
    "g0": dict(M=96, K=512, E=6, tokens=3, top_k=2, seed=12),
}


def grouped_routing(seed: int, route: int, tokens: int, top_k: int, E: int) -> np.ndarray:
    keys = uniform01(seed * 1009 + route, "route", tokens * E).reshape(tokens, E)
    chosen = np.argsort(keys, axis=1, kind="stable")[:, :top_k]
    return np.sort(chosen.ravel(), kind="stable").astype(np.int32)


def make_grouped(name: str, route: int = 0, with_weights=None) -> GroupedWorkload:
    """with_weights: a GroupedWorkload of the same config whose weights are reused."""
    cfg = GROUPED[name]
    M, K, E, s = cfg["M"], cfg["K"], cfg["E"], cfg["seed"]
    expert_of = grouped_routing(s, route, cfg["tokens"], cfg["top_k"], E)
    T = len(expert_of)
    if with_weights is not None:
        A, sfa, g_a, g_b = with_weights.A, with_weights.sfa, with_weights.g_a, with_weights.g_b
    else:
        A = uniform_bytes(s, "A", E * M * K // 2).reshape(E, M, K // 2)
        sfa = choice_bytes(s, "sfa", E * M * K // 16, pow2_scale_bytes(-4, 3)).reshape(E, M, K // 16)
        gi = choice_bytes(s, "g", 2 * E, (0, 1, 2, 3))
        g_a = np.float32([0.25, 0.5, 1.0, 2.0])[gi[:E]]
        g_b = np.float32([0.5, 1.0, 2.0, 0.25])[gi[E:]]
    vs = s * 1009 + route
    b = uniform_bytes(vs, "b", T * K // 2).reshape(T, K // 2)
    sfb = choice_bytes(vs, "sfb", T * K // 16, pow2_scale_bytes(-4, 3)).reshape(T, K // 16)
    return GroupedWorkload(name, M, K, E, T, A, sfa, g_a, g_b, b, sfb, expert_of, s,
                           recipe=f"{E} experts, {cfg['tokens']} tokens x top-{cfg['top_k']}, "
                                  "uniform bytes, scales 2^-4..2^3, per-expert g in powers of two")


def describe(name: str) -> str:
    cfg = CONFIGS[name]
    return f"{name}: M={cfg['M']} K={cfg['K']} L={cfg['L']}"

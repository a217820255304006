"""ctypes shim of the plain C oracle (``oracle/nvfp4_ref.c``).  TEST INFRASTRUCTURE ONLY.

``build()`` compiles the C source with gcc into ``oracle/_build/libnvfp4_ref.so`` (OpenMP when the
compiler has it; fp contraction and fast math off, so every fp64 and fp32 operation is the one the
source writes).  The functions below take and return numpy arrays in the same layouts and with the
same meaning as the numpy formulation in ``oracle.nvfp4_gemv``, ``oracle.grouped`` and
``oracle.quantize``; the two formulations are written independently and must agree bit for bit.

``threads``: OpenMP threads for the sums (None = all of them; the results do not depend on it,
since each output row is one sequential sum).
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "nvfp4_ref.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libnvfp4_ref.so")
STAMP = os.path.join(BUILD_DIR, "stamp")
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]

_lib = None


def _digest(flags) -> str:
    with open(SOURCE, "rb") as f:
        return hashlib.sha256(f.read() + " ".join(flags).encode()).hexdigest()


def build(verbose: bool = False) -> str:
    """Compile the oracle library if the source changed; returns its path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = os.environ.get("CC", "gcc")
    for extra in (["-fopenmp"], []):               # without OpenMP if the compiler lacks it
        flags = CFLAGS + extra
        digest = _digest(flags)
        if os.path.exists(LIB_PATH) and os.path.exists(STAMP):
            with open(STAMP) as f:
                if f.read().strip() == digest:
                    return LIB_PATH
        tmp = LIB_PATH + f".{os.getpid()}.tmp"
        cmd = [cc, *flags, SOURCE, "-o", tmp, "-lm"]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode == 0:
            os.replace(tmp, LIB_PATH)
            with open(STAMP, "w") as f:
                f.write(digest + "\n")
            return LIB_PATH
        if verbose:
            print(r.stderr, flush=True)
    raise RuntimeError(f"could not compile {SOURCE}:\n{r.stderr}")


def lib():
    """The loaded oracle library (built on first use)."""
    global _lib
    if _lib is not None:
        return _lib
    build()
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, f32, c_int = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
    L.nv_e2m1.argtypes, L.nv_e2m1.restype = [ctypes.c_uint], ctypes.c_double
    L.nv_e4m3.argtypes, L.nv_e4m3.restype = [ctypes.c_uint], ctypes.c_double
    L.nv_gemv_rows.argtypes = [vp, vp, f32, vp, vp, f32, i64, i64, i64, vp, vp, i64, vp, vp, c_int]
    L.nv_gemv_rows.restype = c_int
    L.nv_gemv.argtypes = [vp, vp, f32, vp, vp, f32, i64, i64, i64, vp, vp, c_int]
    L.nv_gemv.restype = c_int
    L.nv_gemv_exact_units.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, vp, i64, vp, vp, c_int]
    L.nv_gemv_exact_units.restype = c_int
    L.nv_experts_from_offsets.argtypes = [vp, i64, i64, vp]
    L.nv_experts_from_offsets.restype = None
    L.nv_gemv_grouped.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, vp, vp, c_int]
    L.nv_gemv_grouped.restype = c_int
    L.nv_quantize_activation.argtypes = [vp, f32, c_int, i64, i64, vp, vp]
    L.nv_quantize_activation.restype = c_int
    L.nv_fp16_bits.argtypes, L.nv_fp16_bits.restype = [ctypes.c_double], ctypes.c_uint16
    L.nv_fp16_bits_array.argtypes = [vp, i64, vp]
    L.nv_fp16_bits_array.restype = None
    L.nv_max_threads.argtypes, L.nv_max_threads.restype = [], c_int
    _lib = L
    return L


def _u8(x, n, what):
    a = np.ascontiguousarray(np.asarray(x, dtype=np.uint8).ravel())
    if a.size != n:
        raise ValueError(f"{what} holds {a.size} bytes, the shape needs {n}")
    return a


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _threads(threads):
    return 0 if threads is None else int(threads)


def max_threads() -> int:
    """OpenMP threads the oracle uses by default (1 when built without OpenMP)."""
    return int(lib().nv_max_threads())


def e2m1_values() -> np.ndarray:
    """The C decoder's value of every E2M1 code 0..15."""
    return np.array([lib().nv_e2m1(c) for c in range(16)])


def e4m3_values() -> np.ndarray:
    """The C decoder's value of every E4M3FN byte 0..255."""
    return np.array([lib().nv_e4m3(v) for v in range(256)])


def _operands(A, sfa, b, sfb, M, K, L, n_mats=None):
    if K <= 0 or K % 16:
        raise ValueError("K must be a positive multiple of 16")
    n_mats = L if n_mats is None else n_mats
    return (_u8(A, n_mats * M * K // 2, "A"), _u8(sfa, n_mats * M * K // 16, "sfa"),
            _u8(b, L * K // 2, "b"), _u8(sfb, L * K // 16, "sfb"))


def gemv(A, sfa, g_a, b, sfb, g_b, M: int, K: int, L: int, threads=None):
    """(c_ref, T), fp64 [L][M]: c_ref = (S g_a) g_b with S the fp64 sum in increasing k, and
    T = sum_k |term_k| |g_a g_b|."""
    A, sfa, b, sfb = _operands(A, sfa, b, sfb, M, K, L)
    c = np.empty((L, M), np.float64)
    T = np.empty((L, M), np.float64)
    lib().nv_gemv(_p(A), _p(sfa), float(np.float32(g_a)), _p(b), _p(sfb), float(np.float32(g_b)),
                  M, K, L, _p(c), _p(T), _threads(threads))
    return c, T


def gemv_rows(A, sfa, g_a, b, sfb, g_b, M: int, K: int, L: int, ls, ms, threads=None):
    """(c_ref, T) at the outputs (ls[i], ms[i]) only."""
    A, sfa, b, sfb = _operands(A, sfa, b, sfb, M, K, L)
    ls = np.ascontiguousarray(np.asarray(ls, dtype=np.int64).ravel())
    ms = np.ascontiguousarray(np.asarray(ms, dtype=np.int64).ravel())
    if ls.shape != ms.shape:
        raise ValueError("ls and ms differ in length")
    c = np.empty(ls.shape, np.float64)
    T = np.empty(ls.shape, np.float64)
    st = lib().nv_gemv_rows(_p(A), _p(sfa), float(np.float32(g_a)), _p(b), _p(sfb),
                            float(np.float32(g_b)), M, K, L, _p(ls), _p(ms), ls.size, _p(c), _p(T),
                            _threads(threads))
    if st:
        raise IndexError("an output index is outside [0, L) x [0, M)")
    return c, T


def gemv_exact_units(A, sfa, b, sfb, M: int, K: int, L: int, ls=None, ms=None, threads=None):
    """(units, nan): the exact sum S in int64 units of 2**-20 at every output (or at (ls, ms)),
    and the mask of outputs that use a NaN scale (their units are 0)."""
    A, sfa, b, sfb = _operands(A, sfa, b, sfb, M, K, L)
    if ls is None:
        ls, ms = np.divmod(np.arange(L * M, dtype=np.int64), M)
    ls = np.ascontiguousarray(np.asarray(ls, dtype=np.int64).ravel())
    ms = np.ascontiguousarray(np.asarray(ms, dtype=np.int64).ravel())
    units = np.empty(ls.shape, np.int64)
    nan = np.empty(ls.shape, np.uint8)
    st = lib().nv_gemv_exact_units(_p(A), _p(sfa), _p(b), _p(sfb), M, K, L, _p(ls), _p(ms),
                                   ls.size, _p(units), _p(nan), _threads(threads))
    if st:
        raise ValueError("bad output index, or K >= 2**20")
    return units, nan.astype(bool)


def experts_from_offsets(offsets, T: int) -> np.ndarray:
    """Owner of each token 0..T-1 under inclusive cumulative offsets, or -1."""
    off = np.ascontiguousarray(np.asarray(offsets, dtype=np.int32).ravel())
    owner = np.empty(int(T), np.int64)
    lib().nv_experts_from_offsets(_p(off), off.size, int(T), _p(owner))
    return owner


def gemv_grouped(A, sfa, g_a, b, sfb, g_b, experts, M: int, K: int, threads=None):
    """Grouped decode GEMV: token t uses expert experts[t] (or has none: -1).  Returns (c_ref, T)
    fp64 [T][M]."""
    owner = np.ascontiguousarray(np.asarray(experts, dtype=np.int64).ravel())
    ga = np.ascontiguousarray(np.asarray(g_a, dtype=np.float32).ravel())
    gb = np.ascontiguousarray(np.asarray(g_b, dtype=np.float32).ravel())
    E, T = ga.size, owner.size
    A, sfa, b, sfb = _operands(A, sfa, b, sfb, M, K, T, n_mats=E)
    c = np.empty((T, M), np.float64)
    Tb = np.empty((T, M), np.float64)
    st = lib().nv_gemv_grouped(_p(A), _p(sfa), _p(ga), _p(b), _p(sfb), _p(gb), _p(owner), M, K, E,
                               T, _p(c), _p(Tb), _threads(threads))
    if st:
        raise ValueError("an owner index is >= E")
    return c, Tb


ROUNDINGS = {"lut": 0, "rne": 1}


def quantize_activation(x, global_scale: float, rounding: str = "lut"):
    """x: fp32 [..., K] (bf16 values), K % 16 == 0.  Returns (packed [..., K/2], scales
    [..., K/16]) as uint8."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    K = x.shape[-1]
    if K % 16:
        raise ValueError("K must be a multiple of 16")
    L = x.size // K if K else 0
    packed = np.empty(x.shape[:-1] + (K // 2,), np.uint8)
    scales = np.empty(x.shape[:-1] + (K // 16,), np.uint8)
    st = lib().nv_quantize_activation(_p(x), float(np.float32(global_scale)), ROUNDINGS[rounding],
                                      K, L, _p(packed), _p(scales))
    if st:
        raise ValueError("bad shape or rounding")
    return packed, scales


def fp16_bits(x) -> np.ndarray:
    """IEEE binary16 bits of fp64 values, round to nearest even (uint16 array of x's shape)."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    out = np.empty(x.shape, np.uint16)
    lib().nv_fp16_bits_array(_p(x), x.size, _p(out))
    return out

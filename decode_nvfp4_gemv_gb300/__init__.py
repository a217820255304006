"""GB300-native NVFP4 block-scaled batched GEMV.

Python binding of ``libnvfp4_gemv.so`` (C ABI in ``include/nvfp4_gemv.h``).  It only marshals
arguments: every step of the GEMV runs in the library's CUDA kernels.  PyTorch provides device
memory and streams.  The entry points have the C names:

    nvfp4_gemv_batched(A, sfa, g_a, b, sfb, g_b, c, M, K, L, stream=None)
    nvfp4_gemv_batched_ex(A, sfa, g_a, b, sfb, g_b, c, M, K, L, stream=None, plan=None)
    nvfp4_gemv_plan(M, K, L) -> Plan
    nvfp4_plan_for_limits(M, K, L, plan=None, sms=..., max_smem_optin=..., max_smem_sm=...) -> Plan
    nvfp4_max_stream_k(), nvfp4_status_string(status), nvfp4_last_error(), nvfp4_abi_version()

Tensor arguments are contiguous CUDA tensors (A, sfa, b, sfb: uint8; c: float16, or uint16/int16
holding fp16 bits) or raw integer device addresses.  The binding checks tensor sizes against
(M, K, L) before calling, so a shape mistake raises instead of reading out of bounds.  A non-zero
library status raises ``NVFP4Error``.  If the library is not built, calls raise ``RuntimeError``:
there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

__all__ = [
    "NVFP4Error", "Plan", "KERNEL_AUTO", "KERNEL_SIMPLE", "KERNEL_STREAM", "KERNEL_TMA",
    "KERNEL_TMA_RV", "KERNEL_TC", "KERNEL_SHIFT", "nvfp4_gemm_small_n", "FLAG_EARLY_WEIGHTS", "FLAG_NO_PDL", "FLAG_QUANTIZE_IN_GEMV",
    "FLAG_NO_L2_PREFETCH",
    "ROUND_HALF_STEP_TABLE",
    "ROUND_NEAREST_EVEN", "nvfp4_quantize_activation", "nvfp4_gemv_batched_bf16", "OUT_F16",
    "OUT_BF16", "nvfp4_gemv_grouped", "library_path",
    "load_library", "nvfp4_gemv_batched", "nvfp4_gemv_batched_ex", "nvfp4_gemv_plan",
    "nvfp4_max_stream_k", "nvfp4_status_string", "nvfp4_last_error", "nvfp4_abi_version", "gemv",
    "DeviceLimits", "GB300_LIMITS", "nvfp4_plan_for_limits",
]

KERNEL_AUTO, KERNEL_SIMPLE, KERNEL_STREAM, KERNEL_TMA, KERNEL_TMA_RV, KERNEL_TC, KERNEL_SHIFT = (
    0, 1, 2, 3, 4, 5, 6)
FLAG_EARLY_WEIGHTS, FLAG_NO_PDL, FLAG_QUANTIZE_IN_GEMV, FLAG_TEST_STALL = 1, 2, 4, 8
FLAG_NO_L2_PREFETCH = 16
ROUND_HALF_STEP_TABLE, ROUND_NEAREST_EVEN = 0, 1
OUT_F16, OUT_BF16 = 0, 1

OK, ERR_INVALID_VALUE, ERR_MISALIGNED, ERR_UNSUPPORTED_SHAPE, ERR_ARCH, ERR_CUDA = range(6)


class NVFP4Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"nvfp4 status {status} ({nvfp4_status_string(status)}): {message}")
        self.status = status
        self.message = message


class Plan(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("rows_per_warp", ctypes.c_int32),
                ("k_split", ctypes.c_int32), ("ctas_per_batch", ctypes.c_int32),
                ("warps_per_cta", ctypes.c_int32), ("tile_rows", ctypes.c_int32),
                ("stages", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("k_slices", ctypes.c_int32)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}

    def __repr__(self):
        return f"Plan({self.as_dict()})"


class DeviceLimits(ctypes.Structure):
    """The device limits the planner reads (nvfp4_device_limits)."""
    _fields_ = [("sms", ctypes.c_int32), ("max_smem_optin", ctypes.c_int32),
                ("max_smem_sm", ctypes.c_int32)]


# GB300: 152 SMs, 227 KiB of shared memory per CTA (opt-in), 228 KiB per SM
GB300_LIMITS = dict(sms=152, max_smem_optin=232448, max_smem_sm=233472)


_lib = None


def library_path() -> str:
    return LIB_PATH


def load_library():
    """Load libnvfp4_gemv.so once (raises RuntimeError if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m decode_nvfp4_gemv_gb300.build` (or __graft_entry__.build())")
    lib = ctypes.CDLL(LIB_PATH)
    u8p, u16p, vp = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
    i64, f32 = ctypes.c_int64, ctypes.c_float
    lib.nvfp4_gemv_batched.argtypes = [u8p, u8p, f32, u8p, u8p, f32, u16p, i64, i64, i64, vp]
    lib.nvfp4_gemv_batched.restype = ctypes.c_int
    lib.nvfp4_gemv_batched_ex.argtypes = [u8p, u8p, f32, u8p, u8p, f32, u16p, i64, i64, i64, vp,
                                          ctypes.POINTER(Plan)]
    lib.nvfp4_gemv_batched_ex.restype = ctypes.c_int
    lib.nvfp4_quantize_activation.argtypes = [vp, f32, ctypes.c_int, vp, vp, i64, i64, vp]
    lib.nvfp4_quantize_activation.restype = ctypes.c_int
    lib.nvfp4_gemv_batched_bf16.argtypes = [u8p, u8p, f32, vp, f32, ctypes.c_int, vp, vp, u16p,
                                            i64, i64, i64, vp, ctypes.POINTER(Plan)]
    lib.nvfp4_gemv_batched_bf16.restype = ctypes.c_int
    lib.nvfp4_gemv_grouped.argtypes = [u8p, u8p, vp, u8p, u8p, vp, vp, vp, u16p, ctypes.c_int,
                                       i64, i64, i64, i64, vp, ctypes.POINTER(Plan)]
    lib.nvfp4_gemv_grouped.restype = ctypes.c_int
    lib.nvfp4_gemm_small_n.argtypes = [u8p, u8p, f32, u8p, u8p, f32, u16p, i64, i64, i64, vp,
                                       ctypes.POINTER(Plan)]
    lib.nvfp4_gemm_small_n.restype = ctypes.c_int
    lib.nvfp4_gemv_plan.argtypes = [i64, i64, i64, ctypes.POINTER(Plan)]
    lib.nvfp4_gemv_plan.restype = ctypes.c_int
    lib.nvfp4_plan_for_limits.argtypes = [ctypes.POINTER(DeviceLimits), i64, i64, i64,
                                          ctypes.POINTER(Plan), ctypes.POINTER(Plan)]
    lib.nvfp4_plan_for_limits.restype = ctypes.c_int
    lib.nvfp4_max_stream_k.argtypes = []
    lib.nvfp4_max_stream_k.restype = ctypes.c_int64
    lib.nvfp4_status_string.argtypes = [ctypes.c_int]
    lib.nvfp4_status_string.restype = ctypes.c_char_p
    lib.nvfp4_last_error.argtypes = []
    lib.nvfp4_last_error.restype = ctypes.c_char_p
    lib.nvfp4_abi_version.argtypes = []
    lib.nvfp4_abi_version.restype = ctypes.c_int
    _lib = lib
    return lib


def nvfp4_status_string(status: int) -> str:
    return load_library().nvfp4_status_string(int(status)).decode()


def nvfp4_last_error() -> str:
    return load_library().nvfp4_last_error().decode()


def nvfp4_abi_version() -> int:
    return load_library().nvfp4_abi_version()


def nvfp4_plan_for_limits(M, K, L, plan=None, sms=GB300_LIMITS["sms"],
                          max_smem_optin=GB300_LIMITS["max_smem_optin"],
                          max_smem_sm=GB300_LIMITS["max_smem_sm"]) -> Plan:
    """The planner's choice (or its check of ``plan``) for a device with the given limits, without
    touching any device; raises NVFP4Error with the status a launch would return."""
    lim = DeviceLimits(int(sms), int(max_smem_optin), int(max_smem_sm))
    forced = None
    if plan is not None:
        forced = Plan(**plan) if isinstance(plan, dict) else plan
    out = Plan()
    _check(load_library().nvfp4_plan_for_limits(
        ctypes.byref(lim), int(M), int(K), int(L),
        ctypes.byref(forced) if forced is not None else None, ctypes.byref(out)))
    return out


def nvfp4_max_stream_k() -> int:
    return int(load_library().nvfp4_max_stream_k())


def _check(status: int):
    if status != OK:
        raise NVFP4Error(status, nvfp4_last_error())


# ------------------------------------------------------------------ argument marshalling

_ITEM = {"A": 1, "sfa": 1, "b": 1, "sfb": 1, "c": 2}


def _ptr(name, x, need_bytes):
    """Device address of a tensor (checking dtype, contiguity and size) or of a raw integer."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    import torch

    if not isinstance(x, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor or an integer address")
    if name == "c":
        if x.dtype not in (torch.float16, torch.uint16, torch.int16):
            raise TypeError("c must be float16 (or 16-bit integers holding fp16 bits)")
    elif x.dtype not in (torch.uint8, torch.int8):
        raise TypeError(f"{name} must be uint8 (packed FP4 / FP8 bytes)")
    if not x.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if not x.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (use the host path in bench/tests to copy)")
    have = x.numel() * x.element_size()
    if have < need_bytes:
        raise ValueError(f"{name} holds {have} bytes, (M, K, L) needs {need_bytes}")
    return x.data_ptr()


def _stream_handle(stream, tensors):
    if stream is None:
        import torch

        dev = next((t.device for t in tensors if hasattr(t, "device")), None)
        return torch.cuda.current_stream(dev).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _marshal(A, sfa, g_a, b, sfb, g_b, c, M, K, L, stream):
    M, K, L = int(M), int(K), int(L)
    if M <= 0 or K <= 0 or L <= 0 or K % 16:
        # empty problems touch no memory; invalid shapes get the library's status
        need = {k: 0 for k in _ITEM}
    else:
        need = {"A": M * L * K // 2, "sfa": M * L * K // 16, "b": L * K // 2, "sfb": L * K // 16,
                "c": 2 * M * L}
    ptrs = [_ptr(n, x, need[n]) for n, x in (("A", A), ("sfa", sfa), ("b", b), ("sfb", sfb),
                                                 ("c", c))]
    h = _stream_handle(stream, [A, sfa, b, sfb, c])
    return ptrs, ctypes.c_float(g_a), ctypes.c_float(g_b), M, K, L, h


class _on_device:
    """Makes the device of the first tensor argument current for the duration of a call (the
    library works on the calling thread's current device)."""

    def __init__(self, tensors):
        self.dev = next((t.device for t in tensors if hasattr(t, "device") and t.is_cuda), None)
        self.prev = None

    def __enter__(self):
        if self.dev is not None:
            import torch

            self.prev = torch.cuda.current_device()
            if self.prev != self.dev.index:
                torch.cuda.set_device(self.dev)
            else:
                self.prev = None

    def __exit__(self, *exc):
        if self.prev is not None:
            import torch

            torch.cuda.set_device(self.prev)


def nvfp4_gemv_batched(A, sfa, g_a, b, sfb, g_b, c, M, K, L, stream=None):
    """Enqueue c = fp16(g_a g_b A (x) b) per batch on ``stream`` (default: torch's current stream)."""
    with _on_device([A, sfa, b, sfb, c]):
        (pA, pSA, pB, pSB, pC), ga, gb, M, K, L, h = _marshal(A, sfa, g_a, b, sfb, g_b, c, M, K,
                                                              L, stream)
        _check(load_library().nvfp4_gemv_batched(pA, pSA, ga, pB, pSB, gb, pC, M, K, L, h))


def nvfp4_gemv_batched_ex(A, sfa, g_a, b, sfb, g_b, c, M, K, L, stream=None, plan=None):
    """As ``nvfp4_gemv_batched`` with a forced ``Plan`` (or a dict of its fields; None = auto)."""
    pl = None
    if plan is not None:
        pl = Plan(**plan) if isinstance(plan, dict) else plan
    with _on_device([A, sfa, b, sfb, c]):
        (pA, pSA, pB, pSB, pC), ga, gb, M, K, L, h = _marshal(A, sfa, g_a, b, sfb, g_b, c, M, K,
                                                              L, stream)
        _check(load_library().nvfp4_gemv_batched_ex(pA, pSA, ga, pB, pSB, gb, pC, M, K, L, h,
                                                    ctypes.byref(pl) if pl is not None else None))


def nvfp4_gemv_plan(M, K, L) -> Plan:
    out = Plan()
    _check(load_library().nvfp4_gemv_plan(int(M), int(K), int(L), ctypes.byref(out)))
    return out


def gemv(A, sfa, g_a, b, sfb, g_b, out=None, stream=None, plan=None):
    """Shape-inferring convenience wrapper: A [L][M][K/2], sfa [L][M][K/16], b [L][K/2],
    sfb [L][K/16] (uint8 CUDA tensors).  Returns c [L][M] float16 (allocated if ``out`` is None)."""
    import torch

    if A.dim() != 3:
        raise ValueError("A must be [L][M][K/2]")
    L, M, K2 = A.shape
    K = 2 * K2
    if out is None:
        out = torch.empty((L, M), dtype=torch.float16, device=A.device)
    nvfp4_gemv_batched_ex(A, sfa, g_a, b, sfb, g_b, out, M, K, L, stream, plan)
    return out


def _bf16_ptr(name, x, need_bytes):
    """Address of a bf16 tensor (or a 16-bit integer tensor holding bf16 bits)."""
    if x is None or isinstance(x, int):
        return x
    import torch

    if x.dtype not in (torch.bfloat16, torch.uint16, torch.int16):
        raise TypeError(f"{name} must be bfloat16 (or 16-bit integers holding bf16 bits)")
    if not x.is_contiguous() or not x.is_cuda:
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if x.numel() * 2 < need_bytes:
        raise ValueError(f"{name} holds {x.numel() * 2} bytes, (K, L) needs {need_bytes}")
    return x.data_ptr()


def nvfp4_quantize_activation(x, global_scale, b, sfb, K, L, rounding=ROUND_HALF_STEP_TABLE,
                              stream=None):
    """Quantize bf16 x [L][K] to packed E2M1 b [L][K/2] and E4M3 block scales sfb [L][K/16]."""
    K, L = int(K), int(L)
    ok = K > 0 and L > 0 and K % 16 == 0
    with _on_device([x, b, sfb]):
        px = _bf16_ptr("x", x, 2 * K * L if ok else 0)
        pb = _ptr("b", b, K * L // 2 if ok else 0)
        ps = _ptr("sfb", sfb, K * L // 16 if ok else 0)
        h = _stream_handle(stream, [x, b, sfb])
        _check(load_library().nvfp4_quantize_activation(px, ctypes.c_float(global_scale),
                                                        int(rounding), pb, ps, K, L, h))


def nvfp4_gemv_batched_bf16(A, sfa, g_a, x, x_global_scale, b_out, sfb_out, c, M, K, L,
                            rounding=ROUND_HALF_STEP_TABLE, stream=None, plan=None):
    """The GEMV with a bf16 vector x [L][K]: quantizes it (global scale x_global_scale, which is
    g_b) into b_out / sfb_out and computes c from A and that vector."""
    pl = None
    if plan is not None:
        pl = Plan(**plan) if isinstance(plan, dict) else plan
    M, K, L = int(M), int(K), int(L)
    ok = M > 0 and K > 0 and L > 0 and K % 16 == 0
    with _on_device([A, sfa, x, b_out, sfb_out, c]):
        (pA, pSA, pB, pSB, pC), ga, gb, M, K, L, h = _marshal(A, sfa, g_a, b_out, sfb_out,
                                                              x_global_scale, c, M, K, L, stream)
        px = _bf16_ptr("x", x, 2 * K * L if ok else 0)
        _check(load_library().nvfp4_gemv_batched_bf16(
            pA, pSA, ga, px, gb, int(rounding), pB, pSB, pC, M, K, L, h,
            ctypes.byref(pl) if pl is not None else None))


def _typed_ptr(name, x, dtypes, need_bytes):
    """Device address of a contiguous CUDA tensor of one of `dtypes` (names), or a raw integer."""
    if x is None or isinstance(x, int):
        return x
    import torch

    if not isinstance(x, torch.Tensor) or str(x.dtype).replace("torch.", "") not in dtypes:
        raise TypeError(f"{name} must be a tensor of {' or '.join(dtypes)}")
    if not x.is_contiguous() or not x.is_cuda:
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    if x.numel() * x.element_size() < need_bytes:
        raise ValueError(f"{name} holds {x.numel() * x.element_size()} bytes, needs {need_bytes}")
    return x.data_ptr()


def nvfp4_gemv_grouped(A, sfa, g_a, b, sfb, g_b, c, M, K, E, T, expert_offsets=None,
                       expert_of_token=None, out_dtype=OUT_F16, stream=None, plan=None):
    """Grouped (mixture-of-experts) decode GEMV: token t uses expert e(t)'s matrix A[e] and the
    global scales g_a[e], g_b[e] (fp32 device arrays); e(t) from inclusive cumulative
    ``expert_offsets`` [E] or from ``expert_of_token`` [T] (int32 device arrays, exactly one).
    c [T][M] is fp16 or bfloat16 (``out_dtype``); tokens without an expert get zeros."""
    pl = None
    if plan is not None:
        pl = Plan(**plan) if isinstance(plan, dict) else plan
    M, K, E, T = int(M), int(K), int(E), int(T)
    ok = M > 0 and K > 0 and T > 0 and E > 0 and K % 16 == 0
    tensors = [A, sfa, g_a, b, sfb, g_b, c, expert_offsets, expert_of_token]
    with _on_device([t for t in tensors if t is not None]):
        pA = _ptr("A", A, E * M * K // 2 if ok else 0)
        pSA = _ptr("sfa", sfa, E * M * K // 16 if ok else 0)
        pB = _ptr("b", b, T * K // 2 if ok else 0)
        pSB = _ptr("sfb", sfb, T * K // 16 if ok else 0)
        pga = _typed_ptr("g_a", g_a, ("float32",), 4 * E if ok else 0)
        pgb = _typed_ptr("g_b", g_b, ("float32",), 4 * E if ok else 0)
        po = _typed_ptr("expert_offsets", expert_offsets, ("int32",), 4 * E if ok else 0)
        pm = _typed_ptr("expert_of_token", expert_of_token, ("int32",), 4 * T if ok else 0)
        out_types = ("bfloat16", "int16", "uint16") if out_dtype == OUT_BF16 else \
            ("float16", "int16", "uint16")
        pC = _typed_ptr("c", c, out_types, 2 * M * T if ok else 0)
        h = _stream_handle(stream, [t for t in tensors if t is not None])
        _check(load_library().nvfp4_gemv_grouped(
            pA, pSA, pga, pB, pSB, pgb, po, pm, pC, int(out_dtype), M, K, E, T, h,
            ctypes.byref(pl) if pl is not None else None))


def nvfp4_gemm_small_n(A, sfa, g_a, b, sfb, g_b, c, M, K, N, stream=None, plan=None):
    """c[n][m] for N vectors b [N][K/2] sharing one matrix A [M][K/2] (tensor cores when they
    can take the shape)."""
    pl = None
    if plan is not None:
        pl = Plan(**plan) if isinstance(plan, dict) else plan
    M, K, N = int(M), int(K), int(N)
    ok = M > 0 and K > 0 and N > 0 and K % 16 == 0
    with _on_device([A, sfa, b, sfb, c]):
        pA = _ptr("A", A, M * K // 2 if ok else 0)
        pSA = _ptr("sfa", sfa, M * K // 16 if ok else 0)
        pB = _ptr("b", b, N * K // 2 if ok else 0)
        pSB = _ptr("sfb", sfb, N * K // 16 if ok else 0)
        pC = _ptr("c", c, 2 * M * N if ok else 0)
        h = _stream_handle(stream, [A, sfa, b, sfb, c])
        _check(load_library().nvfp4_gemm_small_n(pA, pSA, ctypes.c_float(g_a), pB, pSB,
                                                 ctypes.c_float(g_b), pC, M, K, N, h,
                                                 ctypes.byref(pl) if pl is not None else None))

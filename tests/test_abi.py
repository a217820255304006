"""The C ABI library without a GPU: it builds for sm_103a, loads, exports every function declared in
include/*.h, and returns the documented statuses for arguments rejected before any device work.
No call here reaches a kernel launch (every call is rejected on the host first)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from decode_nvfp4_gemv_gb300 import build

    build.build()
    import decode_nvfp4_gemv_gb300 as pkg

    return pkg.load_library()


def _declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text = open(os.path.join(inc, f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w\s\*]*?\b(nvfp4_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for n in ("nvfp4_gemv_batched", "nvfp4_gemv_batched_ex", "nvfp4_gemv_plan",
              "nvfp4_status_string", "nvfp4_last_error", "nvfp4_abi_version",
              "nvfp4_plan_for_limits"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/ but not exported"


def test_abi_version_and_status_strings(lib):
    import decode_nvfp4_gemv_gb300 as pkg

    assert pkg.nvfp4_abi_version() == 7
    assert pkg.nvfp4_status_string(0) == "ok"
    assert pkg.nvfp4_status_string(2) == "misaligned pointer"
    assert pkg.nvfp4_status_string(99) == "unknown status"


def _call(lib, A=0x1000, sfa=0x2000, b=0x3000, sfb=0x4000, c=0x5000, M=4, K=256, L=1):
    vp = ctypes.c_void_p
    return lib.nvfp4_gemv_batched(vp(A), vp(sfa), ctypes.c_float(1.0), vp(b), vp(sfb),
                                  ctypes.c_float(1.0), vp(c), M, K, L, None)


@pytest.mark.parametrize("kw,status", [
    (dict(M=-1), 1), (dict(L=-2), 1), (dict(K=0), 1), (dict(K=24), 1), (dict(K=-16), 1),
    (dict(A=0), 1), (dict(sfb=0), 1), (dict(c=0), 1),
    (dict(c=0x5001), 2),
    (dict(c=0x1000), 1),                        # c overlaps A
    (dict(M=1 << 31), 3), (dict(K=1 << 33), 3),
])
def test_rejected_before_device_work(lib, kw, status):
    """Every case is rejected by the host-side checks, which run before any CUDA call."""
    assert _call(lib, **kw) == status
    import decode_nvfp4_gemv_gb300 as pkg

    assert pkg.nvfp4_last_error() != ""


def test_empty_problem_is_a_noop(lib):
    assert _call(lib, M=0, A=0, sfa=0, b=0, sfb=0, c=0) == 0
    assert _call(lib, L=0, A=0, sfa=0, b=0, sfb=0, c=0) == 0


def test_binding_checks_sizes_before_calling(lib):
    torch = pytest.importorskip("torch")
    import decode_nvfp4_gemv_gb300 as pkg

    small = torch.zeros(10, dtype=torch.uint8)
    with pytest.raises((ValueError, TypeError)):
        pkg.nvfp4_gemv_batched(small, small, 1.0, small, small, 1.0,
                               torch.zeros(4, dtype=torch.float16), 4, 256, 1)


def test_plan_query_without_gpu(lib):
    import decode_nvfp4_gemv_gb300 as pkg
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present: covered by the GPU tests")
    with pytest.raises(pkg.NVFP4Error) as e:
        pkg.nvfp4_gemv_plan(128, 256, 1)
    assert e.value.status == 5          # CUDA error: no device


def _quant(lib, x=0x1000, gs=1.0, rounding=0, b=0x100000, sfb=0x200000, K=256, L=1):
    vp = ctypes.c_void_p
    return lib.nvfp4_quantize_activation(vp(x), ctypes.c_float(gs), rounding, vp(b), vp(sfb),
                                         K, L, None)


@pytest.mark.parametrize("kw,status", [
    (dict(K=24), 1), (dict(K=0), 1), (dict(L=-1), 1), (dict(rounding=2), 1),
    (dict(gs=0.0), 1), (dict(gs=-1.0), 1), (dict(gs=float("inf")), 1), (dict(gs=float("nan")), 1),
    (dict(x=0), 1), (dict(b=0), 1), (dict(sfb=0), 1),
    (dict(x=0x1002), 2), (dict(b=0x100008), 2), (dict(sfb=0x200001), 2),
    (dict(b=0x1100), 1),                        # b overlaps x (x holds 512 bytes)
    (dict(K=1 << 33), 3),
])
def test_quantize_rejected_before_device_work(lib, kw, status):
    assert _quant(lib, **kw) == status


def test_quantize_empty_batch_is_a_noop(lib):
    assert _quant(lib, L=0, x=0, b=0, sfb=0) == 0


def _gemv_bf16(lib, A=0x1000, sfa=0x2000, x=0x3000, b=0x100000, sfb=0x200000, c=0x5000, gs=1.0,
               M=4, K=256, L=1):
    vp = ctypes.c_void_p
    return lib.nvfp4_gemv_batched_bf16(vp(A), vp(sfa), ctypes.c_float(1.0), vp(x),
                                       ctypes.c_float(gs), 0, vp(b), vp(sfb), vp(c), M, K, L,
                                       None, None)


@pytest.mark.parametrize("kw,status", [
    (dict(K=24), 1), (dict(gs=0.0), 1), (dict(x=0), 1), (dict(b=0), 1), (dict(x=0x3002), 2),
    (dict(c=0x3000), 1),                        # c overlaps x
    (dict(b=0x1000 + 64), 1),                   # b_out overlaps A
])
def test_gemv_bf16_rejected_before_device_work(lib, kw, status):
    assert _gemv_bf16(lib, **kw) == status


def test_gemv_bf16_empty_is_a_noop(lib):
    assert _gemv_bf16(lib, M=0, A=0, sfa=0, c=0) == 0


def _grouped(lib, A=0x100000, sfa=0x200000, ga=0x300000, b=0x400000, sfb=0x500000, gb=0x600000,
             offs=0x700000, emap=0, c=0x800000, out=0, M=4, K=256, E=2, T=3, flags=None):
    vp = ctypes.c_void_p
    import decode_nvfp4_gemv_gb300 as pkg

    plan = ctypes.byref(pkg.Plan(flags=flags)) if flags is not None else None
    return lib.nvfp4_gemv_grouped(vp(A), vp(sfa), vp(ga), vp(b), vp(sfb), vp(gb),
                                  vp(offs) if offs else None, vp(emap) if emap else None, vp(c),
                                  out, M, K, E, T, None, plan)


@pytest.mark.parametrize("kw,status", [
    (dict(E=0), 1), (dict(E=70000), 3), (dict(offs=0), 1), (dict(emap=0x900000), 1),
    (dict(out=2), 1), (dict(flags=1), 1), (dict(flags=4), 1), (dict(K=24), 1),
    (dict(ga=0), 1), (dict(gb=0), 1), (dict(ga=0x300002), 2), (dict(offs=0x700001), 2),
    (dict(c=0x800001), 2), (dict(c=0x700000), 1),   # c overlaps the offsets
    (dict(c=0x300000), 1),                          # c overlaps g_a
])
def test_grouped_rejected_before_device_work(lib, kw, status):
    assert _grouped(lib, **kw) == status


def test_grouped_empty_is_a_noop(lib):
    assert _grouped(lib, T=0, A=0, sfa=0, b=0, sfb=0, c=0) == 0
    assert _grouped(lib, M=0, A=0, sfa=0, b=0, sfb=0, c=0) == 0


def _small_n(lib, A=0x100000, sfa=0x200000, b=0x300000, sfb=0x400000, c=0x500000, M=4, K=256,
             N=3, flags=None):
    vp = ctypes.c_void_p
    import decode_nvfp4_gemv_gb300 as pkg

    plan = ctypes.byref(pkg.Plan(flags=flags)) if flags is not None else None
    return lib.nvfp4_gemm_small_n(vp(A), vp(sfa), ctypes.c_float(1.0), vp(b), vp(sfb),
                                  ctypes.c_float(1.0), vp(c), M, K, N, None, plan)


@pytest.mark.parametrize("kw,status", [
    (dict(M=-1), 1), (dict(N=-1), 1), (dict(K=24), 1), (dict(K=0), 1), (dict(A=0), 1),
    (dict(c=0x500001), 2), (dict(c=0x100000), 1),   # c misaligned; c overlaps A
    (dict(flags=4), 1), (dict(M=1 << 31), 3),
])
def test_small_n_rejected_before_device_work(lib, kw, status):
    assert _small_n(lib, **kw) == status


def test_small_n_empty_is_a_noop(lib):
    assert _small_n(lib, N=0, A=0, sfa=0, b=0, sfb=0, c=0) == 0
    assert _small_n(lib, M=0, A=0, sfa=0, b=0, sfb=0, c=0) == 0

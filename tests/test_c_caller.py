"""The C ABI from a caller written in plain C (tests/c_caller/gemv_from_c.c): no Python binding,
no torch.  Without a GPU: the header compiles as strict C99 and the program links against the
library.  On a GPU (`-m gpu`): the program runs the batched GEMV on its own stream from operands
written to files here, and its output matches the oracle element by element; it also checks that
a misaligned pointer under a forced TMA plan is refused before any device work."""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
import workloads
from parity import assert_parity

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_caller", "gemv_from_c.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def build_caller(out_dir):
    """Compile and link the C caller (C11: the CUDA runtime's own headers use anonymous unions)."""
    from decode_nvfp4_gemv_gb300 import build

    so = build.build()
    libdir = os.path.dirname(so)
    exe = os.path.join(str(out_dir), "gemv_from_c")
    cmd = ["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"), SRC,
           "-L", libdir, "-lnvfp4_gemv", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{libdir}", "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_header_is_c99_and_the_caller_links(tmp_path):
    # the library's header alone is strict C99
    tu = tmp_path / "header_only.c"
    tu.write_text('#include "nvfp4_gemv.h"\nint main(void) { return nvfp4_abi_version() > 0 ? 0 : 1; }\n')
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), str(tu)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    exe = build_caller(tmp_path)
    assert os.access(exe, os.X_OK)


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(1000, 16384, 2), (128, 256, 1), (2600, 17408, 1),
                                   (300, 1040, 3)], ids=lambda s: "x".join(map(str, s)))
def test_c_caller_matches_the_oracle(tmp_path, shape):
    M, K, L = shape
    exe = build_caller(tmp_path)
    w = workloads.random_workload(M, K, L, seed=M + K + L,
                                  scale_bytes=workloads.pow2_scale_bytes(-4, 3), g_a=0.75,
                                  g_b=1.25)
    paths = []
    for name in ("A", "sfa", "b", "sfb"):
        p = tmp_path / f"{name}.bin"
        np.ascontiguousarray(getattr(w, name)).tofile(p)
        paths.append(str(p))
    out = tmp_path / "c.bin"
    r = subprocess.run([exe, str(M), str(K), str(L), repr(float(w.g_a)), repr(float(w.g_b)),
                        *paths, str(out)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    c = np.fromfile(out, dtype=np.float16).reshape(L, M)
    ref, T = oracle.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, M, K, L)
    assert_parity(c, ref, T, f"C caller {shape}")

"""Writes tests/golden/c1_oracle.json: the oracle's outputs for the seeded 128 x 256 x 1 workload.

It calls only the oracle and the seeded input generators.  The fixture freezes the oracle's results
so that any later change to its arithmetic shows up as a diff of this file.

    python tests/golden/make_c1_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle      # noqa: E402
import workloads   # noqa: E402


def main():
    w = workloads.make("c1")
    c_ref, T = oracle.gemv(w.A, w.sfa, w.g_a, w.b, w.sfb, w.g_b, w.M, w.K, w.L)
    c16 = oracle.fp16_round(c_ref)
    out = {
        "about": "Oracle outputs for the seeded workload M=128, K=256, L=1 (seed 1), written by "
                 "make_c1_golden.py from oracle.gemv; c_ref is unrounded fp64 (repr), T the "
                 "tolerance scale, c_fp16 the binary16 rounding as hex.",
        "M": w.M, "K": w.K, "L": w.L, "seed": w.seed,
        "c_ref": [repr(float(v)) for v in c_ref.ravel()],
        "T": [repr(float(v)) for v in T.ravel()],
        "c_fp16": ["%04x" % int(v) for v in c16.ravel().view("uint16")],
    }
    with open(os.path.join(HERE, "c1_oracle.json"), "w") as f:
        json.dump(out, f, indent=0)
        f.write("\n")


if __name__ == "__main__":
    main()

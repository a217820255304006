"""CPU oracle for the NVFP4 block-scaled batched GEMV.

THIS PACKAGE IS TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` may import it.  The product (``decode_nvfp4_gemv_gb300``:
the CUDA kernels, the C ABI and its Python binding) never imports, links or calls anything here,
and this package shares no code, table or helper with it.  The only module both sides use is the
seeded input generator ``workloads``, which holds none of the GEMV's arithmetic.

Contents, each written from the pages' definitions (citations in each module):

* ``nvfp4_ref.c`` (loaded by ``cref``) the plain C oracle: E2M1 / E4M3FN decoders from their
               closed forms, the GEMV definition in fp64 summed in increasing k (one output row per
               OpenMP work item, so the thread count does not change a bit), the exact-integer
               formulation, the grouped form, the activation quantizer (fp32, the page's
               operations) and fp16 rounding.  ``gemv``, ``gemv_rows``, ``gemv_exact_units`` and
               ``gemv_fp16`` below are these C functions.
* ``codecs``   E2M1 / E4M3FN decoders from their bit layouts, nibble unpacking, fp16 rounding.
* ``nvfp4_gemv`` the same GEMV definition written a second time, in numpy fp64 (its ``gemv``,
               ``gemv_rows``, ``gemv_exact_units``), kept as an independent cross-check of the C
               code: the two agree bit for bit.
* ``grouped``  the grouped (mixture-of-experts) decode GEMV: expert ownership from the bridge's
               cumulative offsets or from a per-token index, then the GEMV definition per token.
* ``quantize`` the NVFP4 activation quantizer with a fixed global scale (bridge.py,
               ``quantize_activation_nvfp4``) in numpy fp32: the page's half-step-table rounding
               and round-to-nearest-even; a block scale with no finite E4M3 encoding is NaN.

Pins (tests that tie the oracle to something other than itself):

* E2M1 table == the magnitude list printed in bridge.py "Constants", plus sign symmetry;
* E4M3FN: all 256 bytes == torch's float8_e4m3fn -> float32 cast, plus hand anchors;
* all 16 x 16 code products == exact integer quarter-units (brute force);
* fp16 rounding: every binary16 value round-trips, every midpoint ties to even, checked against
  exact rational arithmetic;
* hand-worked examples under ``tests/golden/`` (values derived from the pages' table and formula);
* algebraic invariants (zero scale, doubled scale, nibble swap, negation, block permutation,
  batch independence);
* ``gemv`` == ``gemv_exact_units`` bit for bit on all five workloads (sampled rows at full size);
* the C and numpy formulations bit for bit on all five workloads, the grouped workloads and the
  quantizer; C planted mistakes (mutated copies of the C source) each fail a pin;
* planted mistakes (swapped nibbles, dropped scale, off-by-one block index, ...) each fail a pin.
* quantizer: the printed half-step table; its E4M3 encoder against torch's cast; exact grid
  round-trips; brute-force nearest rounding; error bounds; sign symmetry; bit-for-bit agreement
  with the workload generator's independently written quantizer.

* grouped: ownership on a worked offsets example and against a second formulation; identity
  routing == the batched definition; one expert == the batched definition over a repeated
  matrix; expert relabelling; per-expert scales; a brute-force loop over tiny inputs; planted
  mistakes (off-by-one ownership, scales indexed by token) each fail a pin.

No function in this package is "parity unpinned".
"""
import numpy as _np

from . import cref
from .codecs import (E2M1_TABLE, E4M3FN_TABLE, e2m1_value, e4m3fn_value, fp16_round,
                     unpack_e2m1_codes)
from .cref import gemv, gemv_exact_units, gemv_rows
from .nvfp4_gemv import BLOCK, TERM_UNIT_EXP


def gemv_fp16(A, sfa, g_a, b, sfb, g_b, M, K, L):
    """``gemv`` rounded to binary16 (round to nearest even, from fp64), as float16 [L][M]."""
    c_ref, _ = gemv(A, sfa, g_a, b, sfb, g_b, M, K, L)
    return cref.fp16_bits(c_ref).view(_np.float16)


__all__ = [
    "cref", "E2M1_TABLE", "E4M3FN_TABLE", "e2m1_value", "e4m3fn_value", "fp16_round", "unpack_e2m1_codes",
    "BLOCK", "TERM_UNIT_EXP", "gemv", "gemv_exact_units", "gemv_fp16", "gemv_rows",
]

"""CPU oracle for the weight-only 4-bit / 16-bit decode GEMV path.

TEST INFRASTRUCTURE ONLY.  This package is the plain, slow, obviously correct
reference that the CUDA library is checked against.  It is imported by the
tests, by ``__graft_entry__.smoke()`` and by the CPU-baseline / reference leg
of ``bench.py`` -- never by the library itself, which has no CPU fallback.

It shares no code with the CUDA path: no kernels, headers, tables or
constant generators.  Everything here is numpy, with float64 accumulation for
every dot product and IEEE float32 arithmetic where the formats fix float32
decisions (scales, quotients, nearest-level searches), so that integer
outputs (quantised codes, block sums, argmax indices) are defined exactly.

Modules
-------
numerics  exact conversions (fp16/bf16 round-to-nearest-even), rounding,
          units in the last place.
formats   Q8_1 activation blocks, Q4_0 and Q8_0 weight blocks, NF4 blockwise codes and
          the NormalFloat codebook: quantise, pack, unpack, dequantise.
gemv      the dot products themselves (dense, Q4_0 x Q8_1, Q8_0 x Q8_1, NF4), greedy argmax
          and argmin,
          the streaming-read checksum, and the parity bound.

Every function with no independent pin would say "parity unpinned" here; at
present every function is pinned by the ``-m "not gpu"`` oracle tests
(worked examples, brute force, closed forms, invariants, library special
cases).
"""

from . import numerics, formats, gemv  # noqa: F401
from .numerics import (  # noqa: F401
    f16_rn, bf16_rn_bits, bf16_bits_to_f32, round_half_away, ulp,
)
from .formats import (  # noqa: F401
    quantize_q8_1, pack_q8_1, unpack_q8_1,
    quantize_q4_0, pack_q4_0, unpack_q4_0, dequantize_q4_0,
    quantize_q8_0, dequantize_q8_0,
    nf4_codebook, quantize_nf4, pack_nf4, unpack_nf4, dequantize_nf4, dequantize_nf4_bf16,
)
from .gemv import (  # noqa: F401
    gemv_dense, abs_dot_dense, q4_0_q8_1_blockdots, gemv_q4_0_q8_1,
    abs_dot_q4_0_q8_1, q8_0_q8_1_blockdots, gemv_q8_0_q8_1, abs_dot_q8_0_q8_1,
    gemv_nf4, abs_dot_nf4, argmax_rows, argmin_rows, xor_words,
    parity_bound,
)

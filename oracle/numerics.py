"""Exact scalar conversions used by the oracle.

TEST INFRASTRUCTURE ONLY (see the package docstring).

* ``f16_rn``: float32 -> IEEE binary16, round to nearest even, subnormals
  kept.  The pages stress that 16-bit subnormals must survive ("Capability
  Gain from ISA to Shared Execution on AMD MI300A and MI250X", section on
  rocHPL-MxP: the MI250X flushes them); weights drawn from N(0, 0.02^2)
  contain fp16 subnormals, so nothing here flushes.
* ``bf16_rn_bits`` / ``bf16_bits_to_f32``: bfloat16 is the upper half of a
  float32; rounding to it is round-to-nearest-even on the low 16 bits.
* ``round_half_away``: C ``roundf`` semantics (ties away from zero), applied
  to float32 quotients and evaluated exactly in float64.
* ``ulp``: spacing of a binary floating-point format at a magnitude.
"""

import numpy as np


def f16_rn(a):
    """Round float32 values to binary16 (RNE, subnormals kept)."""
    return np.asarray(a, dtype=np.float32).astype(np.float16)


def bf16_rn_bits(a):
    """Round float32 values to bfloat16; return the 16-bit patterns (uint16).

    Round to nearest, ties to even, on the 16 discarded bits.  Inputs must be
    finite (the oracle never rounds NaN or infinity).
    """
    f = np.asarray(a, dtype=np.float32)
    assert np.all(np.isfinite(f)), "bf16_rn_bits: non-finite input"
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits):
    """Exact widening of bfloat16 bit patterns (uint16) to float32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def round_half_away(q32):
    """Round float32 values to integers, ties away from zero (C ``roundf``).

    The float32 value is widened to float64 (exact), so ``|v| + 0.5`` is exact
    for every |v| < 2^29 and the floor gives the correctly rounded magnitude.
    Returns float64 integers.
    """
    v = np.asarray(q32, dtype=np.float32).astype(np.float64)
    assert np.all(np.abs(v) < 2.0 ** 29)
    return np.sign(v) * np.floor(np.abs(v) + 0.5)


_FORMATS = {
    # name: (mantissa bits stored, minimum normal exponent, exponent of the
    #        smallest subnormal spacing)
    "f16": (10, -14, -24),
    "bf16": (7, -126, -133),
    "f32": (23, -126, -149),
}


def ulp(v, fmt):
    """Spacing of ``fmt`` at magnitude |v| (float64 array).

    For |v| in [2^e, 2^(e+1)) with e at or above the format's minimum normal
    exponent this is 2^(e - mantissa_bits); below it (and at zero) it is the
    subnormal spacing.
    """
    mbits, emin, esub = _FORMATS[fmt]
    a = np.abs(np.asarray(v, dtype=np.float64))
    _, e = np.frexp(a)          # a = m * 2^e, m in [0.5, 1)
    e = e.astype(np.int64) - 1  # a in [2^e, 2^(e+1))
    e = np.maximum(e, emin)
    out = np.ldexp(1.0, e - mbits)
    return np.where(a == 0.0, np.ldexp(1.0, esub), out)

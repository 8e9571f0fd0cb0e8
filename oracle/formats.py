"""Quantised formats: Q8_1 activations, Q4_0 and Q8_0 weights, NF4 blockwise
weights.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The pages name the formats and what they are for; the exact recipes below
are the plainest reading of that naming, written out step by step.

Q8_1 (activations), named in "The kernel that waited for itself"
(sebastianhaas.dev m12-db-gemm case study), section "Seven variants, one
microbenchmark, many mistakes": a standalone harness with Q4_0/Q8_1
quantisation and a CPU reference.  Per block of 32 consecutive elements of
one activation column, in IEEE float32:

    amax = max_i |x_i|
    d    = amax / 127
    q_i  = round_half_away(x_i / d)        (q_i = 0 when d == 0)
    s    = d * sum_i q_i                   (float32 product)

and the block stores fp16(d), fp16(s) and the 32 int8 codes, 36 bytes:
``{half d; half s; int8 q[32]}``.

Q4_0 (weights), same page and section.  Per block of 32 consecutive
elements of one weight row, in IEEE float32:

    amax = the signed element of largest |w_i| (first one on ties)
    d    = amax / -8
    q_i  = clamp(round_half_away(w_i / d) + 8, 0, 15)   (q_i = 8 when d == 0)

and the block stores fp16(d) and 16 bytes of nibbles; byte j (j < 16) holds
element j in its low nibble and element j + 16 in its high nibble.
Dequantised value: fp16(d) * (q - 8).  In memory the library keeps two
planes per matrix: ``qs[N][K/2]`` (the nibble bytes, block after block) and
``d[N][K/32]`` (fp16 scales).

Q8_0 (weights), named in the same case study, section "What correctness
was measured against": the new matrix path is tested on Q4_0 and Q8_0
weights.  Per block of 32 consecutive elements of one weight row, in IEEE
float32 (the Q8_1 recipe without the sum field):

    amax = max_i |w_i|
    d    = amax / 127
    q_i  = round_half_away(w_i / d)        (q_i = 0 when d == 0)

and the block stores fp16(d) and the 32 int8 codes.  Planes: ``qs[N][K]``
(int8 codes, element order) and ``d[N][K/32]`` (fp16).  Dequantised value:
fp16(d) * q.

NF4 (weights), named in bitsandbytes issue #1842 "70B 4-bit LLM decode
bottlenecked by HIP kernel (kgemm_4bit_inference_naive) efficiency",
sections "Minimal Repro" (``F.quantize_4bit(w, quant_type='nf4')``) and
"Benchmark Data" (blocksize 64 is the kernel's).  Per block of 64
consecutive elements of one bf16 weight row, in IEEE float32:

    absmax = max_i |w_i|
    v_i    = w_i / absmax                  (v_i = 0 when absmax == 0)
    code_i = argmin_k |cb[k] - v_i|        (lowest k on ties)

with ``cb`` the 16-level NormalFloat codebook (``nf4_codebook``).  Two codes
per byte, the first (even) element in the HIGH nibble.  Planes:
``qs[N][K/2]`` and ``absmax[N][K/64]`` (float32).  Dequantised value:
absmax * cb[code].
"""

import math

import numpy as np

from .numerics import bf16_rn_bits, f16_rn, round_half_away

QK8_1 = 32
QK4_0 = 32
QK_NF4 = 64


# --------------------------------------------------------------------- Q8_1

def quantize_q8_1(x):
    """Quantise activations ``x`` (M, K) float32 to Q8_1.

    Returns ``(q, d16, s16)``: int8 codes (M, K), fp16 scales (M, K/32) and
    fp16 sum fields (M, K/32).
    """
    x = np.asarray(x, dtype=np.float32)
    assert x.ndim == 2 and x.shape[1] % QK8_1 == 0
    m, k = x.shape
    xb = x.reshape(m, k // QK8_1, QK8_1)
    amax = np.max(np.abs(xb), axis=2)                       # exact
    d = (amax / np.float32(127.0)).astype(np.float32)       # IEEE fp32 div
    zero = d == 0
    dsafe = np.where(zero, np.float32(1.0), d)
    quot = (xb / dsafe[..., None]).astype(np.float32)       # IEEE fp32 div
    q = round_half_away(quot)
    q = np.where(zero[..., None], 0.0, q)
    assert np.all(np.abs(q) <= 127)
    q = q.astype(np.int8)
    sumq = q.astype(np.int64).sum(axis=2)                   # exact
    s = (d * sumq.astype(np.float32)).astype(np.float32)    # fp32 product
    return q.reshape(m, k), f16_rn(d), f16_rn(s)


def pack_q8_1(q, d16, s16):
    """Pack Q8_1 fields into the 36-byte block layout; (M, K/32*36) uint8."""
    q = np.asarray(q, dtype=np.int8)
    m, k = q.shape
    nb = k // QK8_1
    out = np.zeros((m, nb, 36), dtype=np.uint8)
    out[:, :, 0:2] = np.asarray(d16, np.float16).reshape(m, nb, 1).view(np.uint8)
    out[:, :, 2:4] = np.asarray(s16, np.float16).reshape(m, nb, 1).view(np.uint8)
    out[:, :, 4:36] = q.reshape(m, nb, QK8_1).view(np.uint8)
    return out.reshape(m, nb * 36)


def unpack_q8_1(blocks, k):
    """Inverse of ``pack_q8_1``: returns ``(q, d16, s16)``."""
    b = np.ascontiguousarray(np.asarray(blocks, dtype=np.uint8))
    m = b.shape[0]
    nb = k // QK8_1
    b = b.reshape(m, nb, 36)
    d16 = np.ascontiguousarray(b[:, :, 0:2]).view(np.float16).reshape(m, nb)
    s16 = np.ascontiguousarray(b[:, :, 2:4]).view(np.float16).reshape(m, nb)
    q = np.ascontiguousarray(b[:, :, 4:36]).view(np.int8).reshape(m, k)
    return q, d16, s16


# --------------------------------------------------------------------- Q8_0

QK8_0 = 32


def quantize_q8_0(w):
    """Quantise weights ``w`` (N, K) float32 to Q8_0.

    Returns ``(q, d16)``: int8 codes (N, K), element order, and fp16 scales
    (N, K/32).  Both are the two planes the library stores.
    """
    w = np.asarray(w, dtype=np.float32)
    assert w.ndim == 2 and w.shape[1] % QK8_0 == 0
    n, k = w.shape
    nb = k // QK8_0
    q = np.zeros((n, k), dtype=np.int8)
    d16 = np.zeros((n, nb), dtype=np.float16)
    for b in range(nb):
        blk = w[:, QK8_0 * b:QK8_0 * (b + 1)]
        amax = np.max(np.abs(blk), axis=1)                      # exact
        d = (amax / np.float32(127.0)).astype(np.float32)       # IEEE fp32 div
        zero = d == 0
        quot = (blk / np.where(zero, np.float32(1.0), d)[:, None]).astype(np.float32)
        qb = np.where(zero[:, None], 0.0, round_half_away(quot))
        assert np.all(np.abs(qb) <= 127)
        q[:, QK8_0 * b:QK8_0 * (b + 1)] = qb.astype(np.int8)
        d16[:, b] = f16_rn(d)
    return q, d16


def dequantize_q8_0(q, d16):
    """fp16(d) * q as float64, (N, K)."""
    q = np.asarray(q, dtype=np.int8).astype(np.float64)
    d = np.repeat(np.asarray(d16, np.float16).astype(np.float64), QK8_0, axis=1)
    return q * d


# --------------------------------------------------------------------- Q4_0

def quantize_q4_0(w):
    """Quantise weights ``w`` (N, K) float32 to Q4_0.

    Returns ``(q, d16)``: codes 0..15 as uint8 (N, K), unpacked, and fp16
    scales (N, K/32).
    """
    w = np.asarray(w, dtype=np.float32)
    assert w.ndim == 2 and w.shape[1] % QK4_0 == 0
    n, k = w.shape
    wb = w.reshape(n, k // QK4_0, QK4_0)
    idx = np.argmax(np.abs(wb), axis=2)                     # first on ties
    amax = np.take_along_axis(wb, idx[..., None], axis=2)[..., 0]
    d = (amax / np.float32(-8.0)).astype(np.float32)        # IEEE fp32 div
    zero = d == 0
    dsafe = np.where(zero, np.float32(1.0), d)
    quot = (wb / dsafe[..., None]).astype(np.float32)       # IEEE fp32 div
    q = np.clip(round_half_away(quot) + 8.0, 0.0, 15.0)
    q = np.where(zero[..., None], 8.0, q).astype(np.uint8)
    return q.reshape(n, k), f16_rn(d)


def pack_q4_0(q):
    """Nibble-pack Q4_0 codes (N, K) into the ``qs`` plane (N, K/2) uint8.

    Byte j of a block: low nibble = element j, high nibble = element j + 16.
    """
    q = np.asarray(q, dtype=np.uint8)
    n, k = q.shape
    qb = q.reshape(n, k // QK4_0, QK4_0)
    lo = qb[:, :, :16]
    hi = qb[:, :, 16:]
    return (lo | (hi << 4)).astype(np.uint8).reshape(n, k // 2)


def unpack_q4_0(qs):
    """Inverse of ``pack_q4_0``: codes 0..15 (N, K) uint8."""
    qs = np.asarray(qs, dtype=np.uint8)
    n, kh = qs.shape
    qb = qs.reshape(n, kh // 16, 16)
    out = np.empty((n, kh // 16, 32), dtype=np.uint8)
    out[:, :, :16] = qb & 0x0F
    out[:, :, 16:] = qb >> 4
    return out.reshape(n, kh * 2)


def dequantize_q4_0(qs, d16):
    """Dequantised Q4_0 weights fp16(d) * (q - 8), float64 (N, K)."""
    q = unpack_q4_0(qs).astype(np.float64) - 8.0
    n, k = q.shape
    d = np.asarray(d16, np.float16).astype(np.float64).reshape(n, k // QK4_0, 1)
    return (q.reshape(n, k // QK4_0, QK4_0) * d).reshape(n, k)


# ---------------------------------------------------------------------- NF4

def _std_normal_quantile(p):
    """Inverse of the standard normal CDF by bisection (float64).

    Phi(z) = erfc(-z / sqrt(2)) / 2 is increasing; bisect on [-40, 40] until
    the bracket stops shrinking.
    """
    assert 0.0 < p < 1.0
    lo, hi = -40.0, 40.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if mid == lo or mid == hi:
            break
        if 0.5 * math.erfc(-mid / math.sqrt(2.0)) < p:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def nf4_codebook():
    """The 16 NormalFloat-4 levels, ascending, as float32.

    QLoRA's NormalFloat construction (Dettmers et al., 2023): quantiles of
    N(0, 1) taken asymmetrically so that zero is exactly representable --
    8 positive levels from probabilities evenly spaced from ``delta`` down to
    (but excluding) 1/2 in 9 points, 7 negative levels from ``delta`` down to
    (excluding) 1/2 in 8 points, plus 0 -- then divided by the largest
    magnitude so the ends are exactly -1 and +1.  ``delta`` is the midpoint
    offset 1 - (1/(2*15) + 1/(2*16)) / 2.
    """
    delta = 1.0 - 0.5 * (1.0 / (2 * 15) + 1.0 / (2 * 16))
    pos_p = np.linspace(delta, 0.5, 9)[:-1]
    neg_p = np.linspace(delta, 0.5, 8)[:-1]
    pos = [_std_normal_quantile(p) for p in pos_p]
    neg = [-_std_normal_quantile(p) for p in neg_p]
    top = max(pos)
    levels = sorted([v / top for v in pos] + [0.0] + [v / top for v in neg])
    return np.asarray(levels, dtype=np.float32)


def quantize_nf4(w, cb):
    """Quantise bf16-valued weights ``w`` (N, K) (float32 array) to NF4 codes.

    Returns ``(codes, absmax)``: codes 0..15 uint8 (N, K), unpacked, and
    float32 absmax (N, K/64).  ``cb``: 16 float32 levels.
    """
    w = np.asarray(w, dtype=np.float32)
    cb = np.asarray(cb, dtype=np.float32)
    assert w.ndim == 2 and w.shape[1] % QK_NF4 == 0 and cb.shape == (16,)
    n, k = w.shape
    wb = w.reshape(n, k // QK_NF4, QK_NF4)
    absmax = np.max(np.abs(wb), axis=2).astype(np.float32)  # exact
    zero = absmax == 0
    asafe = np.where(zero, np.float32(1.0), absmax)
    v = (wb / asafe[..., None]).astype(np.float32)          # IEEE fp32 div
    v = np.where(zero[..., None], np.float32(0.0), v)
    codes = np.empty(v.shape, dtype=np.uint8)
    # nearest level, distances in float32, lowest index on ties; done one
    # level at a time to keep the temporary small
    best = np.full(v.shape, np.inf, dtype=np.float32)
    for j in range(16):
        dist = np.abs((cb[j] - v).astype(np.float32))
        better = dist < best          # strict: an equal later level loses
        best = np.where(better, dist, best)
        codes = np.where(better, np.uint8(j), codes)
    return codes.reshape(n, k), absmax


def pack_nf4(codes):
    """Pack NF4 codes (N, K) two per byte, first element in the HIGH nibble."""
    c = np.asarray(codes, dtype=np.uint8)
    n, k = c.shape
    return ((c[:, 0::2] << 4) | c[:, 1::2]).astype(np.uint8)


def unpack_nf4(qs):
    """Inverse of ``pack_nf4``."""
    qs = np.asarray(qs, dtype=np.uint8)
    n, kh = qs.shape
    out = np.empty((n, kh * 2), dtype=np.uint8)
    out[:, 0::2] = qs >> 4
    out[:, 1::2] = qs & 0x0F
    return out


def dequantize_nf4(qs, absmax, cb):
    """Dequantised NF4 weights absmax * cb[code], float64 (N, K)."""
    c = unpack_nf4(qs)
    n, k = c.shape
    lv = np.asarray(cb, np.float32).astype(np.float64)[c]
    a = np.asarray(absmax, np.float32).astype(np.float64).reshape(n, k // QK_NF4, 1)
    return (lv.reshape(n, k // QK_NF4, QK_NF4) * a).reshape(n, k)


def dequantize_nf4_bf16(qs, absmax, cb):
    """bf16 bit patterns (uint16, (N, K)) of the dequantised NF4 weights.

    The dequantise-then-matrix-product path of bitsandbytes issue #1842
    ("Benchmark Data": dequantise + bf16 mm) materialises the weights in the
    model's bf16: each element is the IEEE float32 product absmax * cb[code]
    (the format's scale and level, both float32), rounded to bfloat16 to
    nearest even.
    """
    c = unpack_nf4(qs)
    n, k = c.shape
    lv = np.asarray(cb, np.float32)[c].reshape(n, k // QK_NF4, QK_NF4)
    a = np.asarray(absmax, np.float32).reshape(n, k // QK_NF4, 1)
    prod = (lv * a).astype(np.float32)          # float32 x float32 -> float32 (IEEE)
    return bf16_rn_bits(prod.reshape(n, k))


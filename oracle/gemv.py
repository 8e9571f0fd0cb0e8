"""Reference dot products, greedy argmax, read checksum and parity bound.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The operation throughout is the batch-1 decode matrix-vector product
y = W x of the batch1-cdna README ("Hand-written FP16 y = Wx, batch size
one"): each output element is one row of W dotted with the activation
vector.  With M activation columns it is done once per column.  Every sum is
accumulated in float64 (the README's correctness gate accumulates in
double precision), over exactly the operand values the device sees.
"""

import numpy as np

from .formats import QK4_0, QK8_0, QK_NF4, unpack_nf4, unpack_q4_0
from .numerics import ulp

_ROWS_PER_CHUNK = 1024


def _as_cols(x):
    x = np.asarray(x)
    return x[None, :] if x.ndim == 1 else x


def gemv_dense(w, x):
    """Y[m, n] = sum_k W[n, k] * X[m, k] in float64.

    ``w``: (N, K) exact operand values (fp16 / bf16-as-float32 / float32);
    ``x``: (K,) or (M, K).  Returns (M, N) float64.
    """
    w = np.asarray(w)
    x = _as_cols(x).astype(np.float64)
    n = w.shape[0]
    y = np.empty((x.shape[0], n), dtype=np.float64)
    for r0 in range(0, n, _ROWS_PER_CHUNK):
        wc = w[r0:r0 + _ROWS_PER_CHUNK].astype(np.float64)
        for m in range(x.shape[0]):
            y[m, r0:r0 + wc.shape[0]] = (wc * x[m]).sum(axis=1)
    return y


def abs_dot_dense(w, x):
    """sum_k |W[n, k] * X[m, k]| in float64, (M, N): the parity-bound scale."""
    return gemv_dense(np.abs(np.asarray(w, dtype=np.float64)),
                      np.abs(_as_cols(x).astype(np.float64)))


def q4_0_q8_1_blockdots(qs, q8):
    """Exact integer block dots sum_i (q4_i - 8) * q8_{m,i}, (M, N, K/32) int32.

    ``qs``: Q4_0 nibble plane (N, K/2); ``q8``: Q8_1 codes (M, K) int8.
    |sum| <= 32 * 8 * 127 = 32512, so int32 holds it exactly.
    """
    q4 = unpack_q4_0(qs).astype(np.int64) - 8
    q8 = _as_cols(q8).astype(np.int64)
    n, k = q4.shape
    m = q8.shape[0]
    nb = k // QK4_0
    out = np.empty((m, n, nb), dtype=np.int64)
    q8b = q8.reshape(m, nb, QK4_0)
    for r0 in range(0, n, _ROWS_PER_CHUNK):
        q4b = q4[r0:r0 + _ROWS_PER_CHUNK].reshape(-1, nb, QK4_0)
        for mm in range(m):
            out[mm, r0:r0 + q4b.shape[0]] = (q4b * q8b[mm]).sum(axis=2)
    assert np.all(np.abs(out) <= 32512)
    return out.astype(np.int32)


def gemv_q4_0_q8_1(qs, d4, q8, d8):
    """y[m, n] = sum_b d4[n, b] * d8[m, b] * sumi[m, n, b] in float64.

    ``d4``: fp16 weight scales (N, K/32); ``d8``: fp16 activation scales
    (M, K/32).  The integer sums are the exact block dots above; the scale
    product is the Q4_0 dequantisation times the Q8_1 dequantisation.
    """
    sumi = q4_0_q8_1_blockdots(qs, q8).astype(np.float64)
    a = np.asarray(d4, np.float16).astype(np.float64)
    b = _as_cols(np.asarray(d8, np.float16)).astype(np.float64)
    return (sumi * a[None, :, :] * b[:, None, :]).sum(axis=2)


def abs_dot_q4_0_q8_1(qs, d4, q8, d8):
    """sum_i |d4 (q4_i - 8)| * |d8 q8_i| in float64, (M, N)."""
    q4 = np.abs(unpack_q4_0(qs).astype(np.int64) - 8)
    q8 = np.abs(_as_cols(q8).astype(np.int64))
    n, k = q4.shape
    m = q8.shape[0]
    nb = k // QK4_0
    a = np.abs(np.asarray(d4, np.float16).astype(np.float64))
    b = np.abs(_as_cols(np.asarray(d8, np.float16)).astype(np.float64))
    out = np.empty((m, n), dtype=np.float64)
    q8b = q8.reshape(m, nb, QK4_0)
    for r0 in range(0, n, _ROWS_PER_CHUNK):
        q4b = q4[r0:r0 + _ROWS_PER_CHUNK].reshape(-1, nb, QK4_0)
        ac = a[r0:r0 + q4b.shape[0]]
        for mm in range(m):
            s = (q4b * q8b[mm]).sum(axis=2).astype(np.float64)
            out[mm, r0:r0 + q4b.shape[0]] = (s * ac * b[mm]).sum(axis=1)
    return out


def q8_0_q8_1_blockdots(qw, q8):
    """Exact integer block dots sum_i qw_i * q8_{m,i}, (M, N, K/32) int32.

    ``qw``: Q8_0 codes (N, K) int8; ``q8``: Q8_1 codes (M, K) int8.
    |sum| <= 32 * 127 * 127 = 516128, so int32 holds it exactly.
    """
    qw = np.asarray(qw, dtype=np.int8).astype(np.int64)
    q8 = _as_cols(q8).astype(np.int64)
    n, k = qw.shape
    m = q8.shape[0]
    nb = k // QK8_0
    out = np.empty((m, n, nb), dtype=np.int64)
    q8b = q8.reshape(m, nb, QK8_0)
    for r0 in range(0, n, _ROWS_PER_CHUNK):
        qb = qw[r0:r0 + _ROWS_PER_CHUNK].reshape(-1, nb, QK8_0)
        for mm in range(m):
            out[mm, r0:r0 + qb.shape[0]] = (qb * q8b[mm]).sum(axis=2)
    assert np.all(np.abs(out) <= 516128)
    return out.astype(np.int32)


def gemv_q8_0_q8_1(qw, dw, q8, d8):
    """y[m, n] = sum_b dw[n, b] * d8[m, b] * sumi[m, n, b] in float64.

    ``dw``: fp16 Q8_0 weight scales (N, K/32); ``d8``: fp16 Q8_1 activation
    scales (M, K/32); ``sumi``: the exact block dots above.
    """
    sumi = q8_0_q8_1_blockdots(qw, q8).astype(np.float64)
    a = np.asarray(dw, np.float16).astype(np.float64)
    b = _as_cols(np.asarray(d8, np.float16)).astype(np.float64)
    return (sumi * a[None, :, :] * b[:, None, :]).sum(axis=2)


def abs_dot_q8_0_q8_1(qw, dw, q8, d8):
    """sum_i |dw qw_i| * |d8 q8_i| in float64, (M, N)."""
    return gemv_q8_0_q8_1(np.abs(np.asarray(qw, np.int8).astype(np.int16)).astype(np.int8),
                          np.abs(np.asarray(dw, np.float16)),
                          np.abs(_as_cols(np.asarray(q8, np.int8)).astype(np.int16)).astype(np.int8),
                          np.abs(_as_cols(np.asarray(d8, np.float16))))


def gemv_nf4(qs, absmax, cb, x):
    """y[m, n] = sum_b absmax[n, b] * sum_i cb[code_{n,i}] * x[m, i], float64.

    ``qs``: NF4 code plane (N, K/2); ``absmax``: float32 (N, K/64);
    ``cb``: 16 float32 levels; ``x``: (K,) or (M, K) exact activation values.
    """
    codes = unpack_nf4(qs)
    n, k = codes.shape
    nb = k // QK_NF4
    lv = np.asarray(cb, np.float32).astype(np.float64)
    a = np.asarray(absmax, np.float32).astype(np.float64)
    x = _as_cols(x).astype(np.float64)
    y = np.empty((x.shape[0], n), dtype=np.float64)
    for r0 in range(0, n, _ROWS_PER_CHUNK):
        c = lv[codes[r0:r0 + _ROWS_PER_CHUNK]].reshape(-1, nb, QK_NF4)
        ac = a[r0:r0 + c.shape[0]]
        for m in range(x.shape[0]):
            inner = (c * x[m].reshape(nb, QK_NF4)).sum(axis=2)
            y[m, r0:r0 + c.shape[0]] = (ac * inner).sum(axis=1)
    return y


def abs_dot_nf4(qs, absmax, cb, x):
    """sum_i |absmax * cb[code_i]| * |x_i| in float64, (M, N)."""
    cba = np.abs(np.asarray(cb, np.float32))
    return gemv_nf4(qs, np.abs(np.asarray(absmax, np.float32)), cba,
                    np.abs(_as_cols(x).astype(np.float64)))


def argmax_rows(logits):
    """Greedy argmax of each row of ``logits`` (M, N): int64 (M,).

    The largest value wins; among equal values (-0.0 equals +0.0) the lowest
    index wins -- the reduction of the ArgCompare discussion ("[WIP]
    ArgCompare Benchmark Results and Performance Analysis", section
    "ArgMax/ArgMin Operations Analysis in real-world AI models": argmax over
    the vocabulary axis, f16/bf16/f32 in, i64 out).  Infinities are ordered
    like any other value (a masked logit is -inf); NaN is not allowed.
    """
    lg = _as_cols(np.asarray(logits))
    assert not np.any(np.isnan(lg)), "argmax_rows: NaN input"
    out = np.empty(lg.shape[0], dtype=np.int64)
    for m in range(lg.shape[0]):
        best = lg[m].max()
        out[m] = np.flatnonzero(lg[m] == best)[0]
    return out


def argmin_rows(values):
    """Argmin of each row of ``values`` (M, N): int64 (M,).

    The ArgCompare discussion covers argmin beside argmax (same page, the
    "Vector Quantization" and "Image Retrieval" rows: argmin over the last
    axis, f32 in, i64 out).  The smallest value wins; among equal values
    (-0.0 equals +0.0) the lowest index wins; infinities are ordered, NaN is
    not allowed.
    """
    v = _as_cols(np.asarray(values))
    assert not np.any(np.isnan(v)), "argmin_rows: NaN input"
    out = np.empty(v.shape[0], dtype=np.int64)
    for m in range(v.shape[0]):
        least = v[m].min()
        out[m] = np.flatnonzero(v[m] == least)[0]
    return out


def xor_words(buf):
    """XOR of all little-endian 32-bit words of a byte buffer (uint32).

    The streaming-read probe of the batch1-cdna README ("01-ceiling") folds
    every element it reads into one scalar so no load can be dropped; XOR
    is the fold used here, so the probe's result is checkable exactly.
    """
    b = np.ascontiguousarray(np.asarray(buf, dtype=np.uint8))
    assert b.size % 4 == 0
    return np.uint32(np.bitwise_xor.reduce(b.view('<u4'), dtype=np.uint32)
                     if b.size else 0)


def parity_bound(y_ref, abs_dot, out_fmt):
    """Allowed |y - y_ref|: 1e-3 * sum|w_i x_i| + one unit in the last place.

    The unit is taken at |y_ref| in the larger of binary16 and the output
    format (``'f16'``, ``'bf16'`` or ``'f32'``), so the bound is never
    tighter than one fp16 ulp and always admits the output's own rounding.
    """
    u = np.maximum(ulp(y_ref, "f16"), ulp(y_ref, out_fmt))
    return 1e-3 * np.asarray(abs_dot, np.float64) + u

"""Pins for the oracle's dot products and reductions (CPU only).

Brute force with exact rational arithmetic, closed forms, the hand-worked
2x64 example, and tie rules.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from golden_io import hexbytes, load, nf4_codebook_fixture


def _exact_dot(row, col):
    return sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(row, col))


@pytest.mark.parametrize("n,k,m", [(1, 8, 1), (2, 16, 3), (3, 64, 2), (7, 16, 1), (5, 8, 4)])
def test_dense_brute_force_fractions(n, k, m):
    rng = np.random.default_rng(100 + n * k + m)
    w = rng.standard_normal((n, k)).astype(np.float16)
    x = rng.standard_normal((m, k)).astype(np.float16)
    y = oracle.gemv_dense(w, x)
    assert y.shape == (m, n)
    for mm in range(m):
        for nn in range(n):
            ref = _exact_dot(w[nn], x[mm])
            assert abs(y[mm, nn] - float(ref)) <= 1e-13 * max(1.0, float(sum(
                abs(Fraction(float(a)) * Fraction(float(b))) for a, b in zip(w[nn], x[mm]))))
    a = oracle.abs_dot_dense(w, x)
    assert np.all(a >= np.abs(y) - 1e-12)


def test_dense_closed_forms():
    k = 64
    w = np.ones((3, k), np.float16)
    x = (np.arange(k) % 4).astype(np.float16)
    assert np.array_equal(oracle.gemv_dense(w, x)[0], np.full(3, 96.0))   # 1.5 K
    # identity: y = x exactly
    xi = np.random.default_rng(5).standard_normal(16).astype(np.float16)
    assert np.array_equal(oracle.gemv_dense(np.eye(16, dtype=np.float16), xi)[0], xi.astype(np.float64))
    # W[n, k] = n (non-square): a transposed operand would give K(K-1)/2 instead of n K
    n, k = 5, 12
    w = np.repeat(np.arange(n, dtype=np.float16)[:, None], k, axis=1)
    y = oracle.gemv_dense(w, np.ones(k, np.float16))[0]
    assert np.array_equal(y, np.arange(n) * float(k))


def test_q4_0_q8_1_h4_hand_example():
    g = load("q4_0_q8_1_h4.json")
    w = np.empty((2, 64), np.float32)
    w[0] = np.tile(np.array([-1.0, 0.5], np.float32), 32)
    w[1] = 0.5
    w[1, 0] = 1.0
    w[1, 32] = 1.0
    q4, d4 = oracle.quantize_q4_0(w)
    qs = oracle.pack_q4_0(q4)
    q8, d8, s8 = oracle.quantize_q8_1(np.ones((1, 64), np.float32))
    sumi = oracle.q4_0_q8_1_blockdots(qs, q8)
    assert sumi.dtype == np.int32
    assert np.array_equal(sumi[0], np.asarray(g["sumi"]))
    y = oracle.gemv_q4_0_q8_1(qs, d4, q8, d8)
    assert list(y[0]) == g["y"]                         # exact in binary
    # ~ the unquantised sum of w (quantisation error only)
    assert abs(y[0, 1] - w[1].sum()) < 0.01


def test_q4_0_q8_1_against_dequantised_fractions():
    rng = np.random.default_rng(200)
    n, k, m = 3, 96, 2
    w = (rng.standard_normal((n, k)) * 0.02).astype(np.float32)
    x = rng.standard_normal((m, k)).astype(np.float32)
    q4, d4 = oracle.quantize_q4_0(w)
    qs = oracle.pack_q4_0(q4)
    q8, d8, _ = oracle.quantize_q8_1(x)
    y = oracle.gemv_q4_0_q8_1(qs, d4, q8, d8)
    sumi = oracle.q4_0_q8_1_blockdots(qs, q8)
    # independent route: per element, dequantise both operands exactly and sum
    for mm in range(m):
        for nn in range(n):
            acc = Fraction(0)
            for kk in range(k):
                b = kk // 32
                wv = Fraction(float(d4[nn, b])) * (int(q4[nn, kk]) - 8)
                xv = Fraction(float(d8[mm, b])) * int(q8[mm, kk])
                acc += wv * xv
            assert abs(y[mm, nn] - float(acc)) <= 1e-12 * max(1.0, abs(float(acc)))
            for b in range(k // 32):
                s = sum((int(q4[nn, kk]) - 8) * int(q8[mm, kk]) for kk in range(32 * b, 32 * b + 32))
                assert sumi[mm, nn, b] == s
    ad = oracle.abs_dot_q4_0_q8_1(qs, d4, q8, d8)
    ref = np.abs(oracle.dequantize_q4_0(qs, d4)) @ np.abs(d8.astype(np.float64).repeat(32, 1) * q8).T
    assert np.allclose(ad, ref.T, rtol=1e-12)


def test_nf4_gemv_against_dequantised_fractions():
    cb = nf4_codebook_fixture()
    rng = np.random.default_rng(300)
    n, k = 4, 128
    import torch
    w = torch.from_numpy((rng.standard_normal((n, k)) * 0.02).astype(np.float32)).to(torch.bfloat16).float().numpy()
    x = torch.from_numpy(rng.standard_normal(k).astype(np.float32)).to(torch.bfloat16).float().numpy()
    codes, absmax = oracle.quantize_nf4(w, cb)
    qs = oracle.pack_nf4(codes)
    y = oracle.gemv_nf4(qs, absmax, cb, x)[0]
    for nn in range(n):
        acc = Fraction(0)
        for kk in range(k):
            acc += Fraction(float(absmax[nn, kk // 64])) * Fraction(float(cb[codes[nn, kk]])) * Fraction(float(x[kk]))
        assert abs(y[nn] - float(acc)) <= 1e-13 * max(1.0, abs(float(acc)))
    ad = oracle.abs_dot_nf4(qs, absmax, cb, x)[0]
    assert np.allclose(ad, np.abs(oracle.dequantize_nf4(qs, absmax, cb)) @ np.abs(x.astype(np.float64)))


def test_nf4_gemv_h5_block_with_unit_x():
    # the H5 block (levels in order, absmax 1) dotted with ones = 4 * sum(cb)
    cb = nf4_codebook_fixture()
    qs = hexbytes(load("nf4_h5.json")["qs_hex"])[None, :]
    y = oracle.gemv_nf4(qs, np.ones((1, 1), np.float32), cb, np.ones(64, np.float32))
    assert y[0, 0] == pytest.approx(4 * float(np.sum(cb.astype(np.float64))), abs=1e-12)


def test_argmax_h6():
    for case in load("argmax_h6.json")["cases"]:
        row = np.asarray(case["row"], dtype=np.float32)
        assert oracle.argmax_rows(row)[0] == case["argmax"], case["why"]


def test_argmax_rows_identical_columns_and_far_ties():
    rng = np.random.default_rng(7)
    base = rng.standard_normal(1000).astype(np.float32)
    base[0] = base[999] = base.max() + 1          # equal maxima at both ends
    lg = np.tile(base, (32, 1))
    assert np.all(oracle.argmax_rows(lg) == 0)


def test_xor_words_hand_cases():
    for case in load("xor_words.json")["cases"]:
        assert int(oracle.xor_words(hexbytes(case["bytes_hex"]))) == int(case["xor"], 16)


def test_xor_words_is_order_free_and_self_inverse():
    rng = np.random.default_rng(8)
    b = rng.integers(0, 256, 4096, dtype=np.uint8)
    x = int(oracle.xor_words(b))
    words = b.view('<u4')
    acc = 0
    for wv in words[::-1]:
        acc ^= int(wv)
    assert acc == x
    assert int(oracle.xor_words(np.concatenate([b, b]))) == 0


def _row(vals):
    return np.asarray([float(v) for v in vals], dtype=np.float32)


def test_argmin_hand_cases():
    for case in load("argmin_cases.json")["cases"]:
        assert oracle.argmin_rows(_row(case["row"]))[0] == case["argmin"], case["why"]


def test_argmax_infinities():
    for case in load("argmin_cases.json")["argmax_inf_cases"]:
        assert oracle.argmax_rows(_row(case["row"]))[0] == case["argmax"], case["why"]


def _scan(row, better):
    # a first-principles scan: keep the first element, replace it only by a
    # strictly better one, so the lowest index of the best value survives
    bi = 0
    for i in range(1, len(row)):
        if better(float(row[i]), float(row[bi])):
            bi = i
    return bi


def test_argmax_argmin_brute_force_with_many_ties():
    rng = np.random.default_rng(11)
    for n in (1, 2, 3, 7, 33, 100):
        # few distinct values (ties everywhere), signed zeros and infinities mixed in
        pool = np.asarray([-np.inf, -2.0, -0.0, 0.0, 1.5, 3.0, np.inf], np.float32)
        rows = pool[rng.integers(0, len(pool), size=(20, n))]
        amax, amin = oracle.argmax_rows(rows), oracle.argmin_rows(rows)
        for m in range(rows.shape[0]):
            assert amax[m] == _scan(rows[m], lambda a, b: a > b)
            assert amin[m] == _scan(rows[m], lambda a, b: a < b)


def test_argmin_is_argmax_of_the_negation():
    rng = np.random.default_rng(12)
    v = rng.integers(-5, 6, size=(64, 257)).astype(np.float32)   # many ties
    v[3, :] = 0.0
    v[3, 100] = -0.0                                               # -0 and +0 tie
    assert np.array_equal(oracle.argmin_rows(v), oracle.argmax_rows(-v))
    assert oracle.argmin_rows(v)[3] == 0


# ------------------------------------------------------------ Q8_0 x Q8_1

def _h8_inputs():
    h7 = load("q8_0_h7_h8.json")["h7"]["w"]
    w = np.zeros((2, 64), np.float32)
    w[0, :32] = h7
    w[0, 32:] = 1.0
    w[1, 32] = -1.0
    w[1, 33:] = 0.25
    return w


def test_q8_0_q8_1_h8_worked_example():
    from fractions import Fraction
    h = load("q8_0_h7_h8.json")["h8"]
    qw, dw = oracle.quantize_q8_0(_h8_inputs())
    q8, d8, _ = oracle.quantize_q8_1(np.ones((1, 64), np.float32))
    assert np.array_equal(oracle.q8_0_q8_1_blockdots(qw, q8)[0], np.asarray(h["sumi"]))
    assert dw.astype(np.float64).tolist() == h["dw"]
    y = oracle.gemv_q8_0_q8_1(qw, dw, q8, d8)[0]
    for n in range(2):
        num, den = h["y_num_den"][n]
        assert y[n] == float(Fraction(num, den))


def test_q8_0_q8_1_blockdots_brute_force():
    rng = np.random.default_rng(23)
    qw = rng.integers(-127, 128, size=(3, 96)).astype(np.int8)
    q8 = rng.integers(-127, 128, size=(2, 96)).astype(np.int8)
    got = oracle.q8_0_q8_1_blockdots(qw, q8)
    for m in range(2):
        for n in range(3):
            for b in range(3):
                s = 0
                for i in range(32):
                    s += int(qw[n, 32 * b + i]) * int(q8[m, 32 * b + i])
                assert got[m, n, b] == s


def test_q8_0_q8_1_closed_forms():
    # constant positive rows quantise to all-127 codes: against x = ones each
    # block dot is 32 * 127 * 127, and a transposed operand would break the
    # row-index pattern of the second check
    w = np.full((4, 128), 0.3, np.float32)
    qw, dw = oracle.quantize_q8_0(w)
    q8, d8, _ = oracle.quantize_q8_1(np.ones((1, 128), np.float32))
    assert np.all(oracle.q8_0_q8_1_blockdots(qw, q8) == 32 * 127 * 127)
    # unit scales: weights n * e_0 per row (amax n, d = n/127 exactly only for
    # n = 127) -- use codes directly: y = sum of row codes times x codes
    qw2 = np.zeros((5, 32), np.int8)
    for n in range(5):
        qw2[n, n] = n + 1
    x8 = np.arange(1, 33, dtype=np.int8)[None, :]
    y = oracle.gemv_q8_0_q8_1(qw2, np.ones((5, 1), np.float16), x8, np.ones((1, 1), np.float16))[0]
    assert y.tolist() == [float((n + 1) * (n + 1)) for n in range(5)]


def _abs_dot_q8_0_fraction(qw, dw, q8, d8, m, n):
    # sum over blocks b and lanes i of |dw[n, b] qw[n, i]| * |d8[m, b] q8[m, i]|,
    # term by term in exact rationals
    acc = Fraction(0)
    for kk in range(qw.shape[1]):
        b = kk // 32
        wv = Fraction(float(dw[n, b])) * int(qw[n, kk])
        xv = Fraction(float(d8[m, b])) * int(q8[m, kk])
        acc += abs(wv) * abs(xv)
    return acc


def _abs_dot_q8_0_signed_then_abs(qw, dw, q8, d8):
    # a plausible mistake planted in a copy of the oracle: |.| taken after
    # the signed dot instead of on every term
    return np.abs(oracle.gemv_q8_0_q8_1(qw, dw, q8, d8))


def _abs_dot_q8_0_scale_dropped(qw, dw, q8, d8):
    # the other plausible mistake: the weight scale's magnitude left out
    return oracle.gemv_q8_0_q8_1(np.abs(qw.astype(np.int16)).astype(np.int8), np.ones_like(dw),
                                 np.abs(q8.astype(np.int16)).astype(np.int8), np.abs(d8))


def _cancelling_q8_0_case():
    # signed terms that cancel inside each block (codes +c / -c against equal
    # activation codes) and negative scales: the signed dot is 0, the sum of
    # magnitudes is not
    rng = np.random.default_rng(41)
    n, k, m = 3, 96, 2
    half = rng.integers(1, 128, size=(n, k // 32, 16))
    qw = np.concatenate([half, -half], axis=2).reshape(n, k).astype(np.int8)
    q8 = np.ones((m, k), np.int8) * np.int8(5)
    q8[1] = -q8[1]
    dw = np.asarray([[0.5, -0.25, 2.0], [-1.0, 0.125, -0.5], [3.0, -3.0, 0.75]], np.float16)
    d8 = np.asarray([[0.25, -1.0, 0.5], [-0.125, 2.0, -4.0]], np.float16)
    return qw, dw, q8, d8


def test_q8_0_q8_1_abs_dot_fractions_random_and_cancelling():
    rng = np.random.default_rng(40)
    qw = rng.integers(-127, 128, size=(4, 96)).astype(np.int8)
    q8 = rng.integers(-127, 128, size=(3, 96)).astype(np.int8)
    dw = (rng.standard_normal((4, 3)) * 0.01).astype(np.float16)   # signed on purpose
    d8 = (rng.standard_normal((3, 3)) * 0.01).astype(np.float16)
    for case in ((qw, dw, q8, d8), _cancelling_q8_0_case()):
        a, b, c, d = case
        got = oracle.abs_dot_q8_0_q8_1(a, b, c, d)
        assert got.shape == (c.shape[0], a.shape[0])
        for mm in range(c.shape[0]):
            for nn in range(a.shape[0]):
                ref = _abs_dot_q8_0_fraction(a, b, c, d, mm, nn)
                assert abs(got[mm, nn] - float(ref)) <= 1e-13 * float(ref)
    # the cancelling case has a zero signed dot in every output
    a, b, c, d = _cancelling_q8_0_case()
    assert np.all(oracle.gemv_q8_0_q8_1(a, b, c, d) == 0.0)


def test_q8_0_q8_1_abs_dot_h8_worked_example():
    # x = 64 ones -> Q8_1 codes 127, d8 = 129/16384 in both blocks.  Row 0:
    # |h7 codes| sum 127+4+3+0+1+127+127 = 389 at dw = 1, then 32 codes 127 at
    # dw = 129/16384; row 1: block 0 zero, block 1 |-127| + 31 * 32 = 1119 at
    # dw = 129/16384
    qw, dw = oracle.quantize_q8_0(_h8_inputs())
    q8, d8, _ = oracle.quantize_q8_1(np.ones((1, 64), np.float32))
    s = Fraction(129, 16384)
    want = [389 * 127 * s + 32 * 127 * 127 * s * s, 1119 * 127 * s * s]
    got = oracle.abs_dot_q8_0_q8_1(qw, dw, q8, d8)[0]
    assert got.tolist() == [float(v) for v in want]


def test_q8_0_q8_1_abs_dot_pins_catch_planted_mistakes():
    a, b, c, d = _cancelling_q8_0_case()
    for bad in (_abs_dot_q8_0_signed_then_abs, _abs_dot_q8_0_scale_dropped):
        got = bad(a, b, c, d)
        ref = np.asarray([[float(_abs_dot_q8_0_fraction(a, b, c, d, mm, nn)) for nn in range(a.shape[0])]
                          for mm in range(c.shape[0])])
        assert not np.allclose(got, ref, rtol=1e-6)

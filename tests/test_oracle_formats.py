"""Pins for the oracle's quantised formats (CPU only).

Hand-worked fixtures under tests/golden/ fix the exact bits; invariants and
brute force cover random data.
"""
import numpy as np
import pytest

import oracle
from golden_io import hexbytes, load, nf4_codebook_fixture


# ------------------------------------------------------------------ Q8_1

def test_q8_1_h1_hand_example():
    g = load("q8_1_h1.json")
    x = np.asarray(g["x"], np.float32)[None, :]
    q, d16, s16 = oracle.quantize_q8_1(x)
    assert np.all(q == g["q"])
    assert d16.view(np.uint16)[0, 0] == int(g["d16_bits"], 16)
    assert float(d16[0, 0]) == g["d16_value"]
    assert s16.view(np.uint16)[0, 0] == int(g["s16_bits"], 16)
    blk = oracle.pack_q8_1(q, d16, s16)
    assert np.array_equal(blk[0], hexbytes(g["block_bytes_hex"]))
    q2, d2, s2 = oracle.unpack_q8_1(blk, 32)
    assert np.array_equal(q2, q) and np.array_equal(d2.view(np.uint16), d16.view(np.uint16))


def _rand_x(m, k, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((m, k)) * scale).astype(np.float32)


def test_q8_1_invariants_random():
    x = _rand_x(5, 4096, 10)
    x[0, :32] = 0.0                       # an all-zero block
    x[1, 32:64] = -3.0                    # constant negative block
    q, d16, s16 = oracle.quantize_q8_1(x)
    xb = x.reshape(5, -1, 32).astype(np.float64)
    qb = q.reshape(5, -1, 32).astype(np.float64)
    amax = np.abs(xb).max(axis=2)
    d = (amax.astype(np.float32) / np.float32(127)).astype(np.float64)
    # codes in range; the largest-magnitude element maps to +-127
    assert np.all(np.abs(qb) <= 127)
    nz = amax > 0
    i = np.argmax(np.abs(xb), axis=2)
    qmax = np.take_along_axis(qb, i[..., None], axis=2)[..., 0]
    assert np.all(np.abs(qmax[nz]) == 127)
    assert np.all(np.sign(qmax[nz]) == np.sign(np.take_along_axis(xb, i[..., None], 2)[..., 0][nz]))
    # reconstruction error at most half a step (plus float32 quotient rounding)
    err = np.abs(xb - d[..., None] * qb)
    assert np.all(err <= d[..., None] * (0.5 + 127 * 2.0 ** -23) + 1e-30)
    # zero block: d = 0, q = 0, s = 0
    assert float(d16[0, 0]) == 0.0 and np.all(qb[0, 0] == 0) and float(s16[0, 0]) == 0.0
    # sum field = d * sum(q), to within fp16 rounding of the float32 product
    sref = d * qb.sum(axis=2)
    tol = 0.5 * oracle.ulp(sref, "f16") + np.abs(sref) * 2.0 ** -23
    assert np.all(np.abs(s16.astype(np.float64) - sref) <= tol)
    # d16 is the RNE fp16 of the float32 scale
    assert np.all(np.abs(d16.astype(np.float64) - d) <= 0.5 * oracle.ulp(d, "f16"))


def test_q8_1_brute_force_small():
    x = _rand_x(2, 64, 11, scale=3.0)
    q, d16, s16 = oracle.quantize_q8_1(x)
    for m in range(2):
        for b in range(2):
            blk = [float(v) for v in x[m, 32 * b:32 * b + 32]]
            amax = max(abs(v) for v in blk)
            d = np.float32(np.float32(amax) / np.float32(127.0))
            for i, v in enumerate(blk):
                r = np.float32(np.float32(v) / d)
                want = int(np.floor(abs(float(r)) + 0.5)) * (1 if r >= 0 else -1)
                assert q[m, 32 * b + i] == want


# ------------------------------------------------------------------ Q4_0

def test_q4_0_h2_hand_examples():
    g = load("q4_0_h2.json")["cases"]
    w0 = np.tile(np.array(g[0]["pattern"], np.float32), 16)[None, :]
    q, d16 = oracle.quantize_q4_0(w0)
    assert d16.view(np.uint16)[0, 0] == int(g[0]["d16_bits"], 16)
    assert list(q[0, :4]) == [0, 12, 0, 12] and np.all(q[0, 0::2] == 0) and np.all(q[0, 1::2] == 12)
    qs = oracle.pack_q4_0(q)
    assert np.array_equal(qs[0], hexbytes(g[0]["qs_hex"]))
    assert np.array_equal(oracle.dequantize_q4_0(qs, d16), w0.astype(np.float64))

    w1 = np.full((1, 32), 0.5, np.float32)
    w1[0, 0] = 1.0
    q, d16 = oracle.quantize_q4_0(w1)
    assert d16.view(np.uint16)[0, 0] == int(g[1]["d16_bits"], 16)
    qs = oracle.pack_q4_0(q)
    assert np.array_equal(qs[0], hexbytes(g[1]["qs_hex"]))
    assert np.array_equal(oracle.dequantize_q4_0(qs, d16), w1.astype(np.float64))
    assert np.array_equal(oracle.unpack_q4_0(qs), q)


def test_q4_0_h3_ties():
    g = load("q4_0_h3_ties.json")
    w = np.zeros((1, 32), np.float32)
    w[0, :4] = g["w_head"]
    q, d16 = oracle.quantize_q4_0(w)
    assert d16.view(np.uint16)[0, 0] == int(g["d16_bits"], 16)
    assert list(q[0, :4]) == g["q_head"]
    assert np.all(q[0, 4:] == g["q_rest"])


def test_q4_0_invariants_random():
    rng = np.random.default_rng(20)
    w = (rng.standard_normal((64, 1024)) * 0.02).astype(np.float32)
    w[3, :32] = 0.0                         # zero block -> q = 8, d = 0
    w[4, 32:64] = 0.01                      # constant block
    q, d16 = oracle.quantize_q4_0(w)
    assert q.max() <= 15
    wb = w.reshape(64, -1, 32).astype(np.float64)
    qb = q.reshape(64, -1, 32).astype(np.int64)
    i = np.argmax(np.abs(wb), axis=2)
    assert np.all(np.take_along_axis(qb, i[..., None], 2)[..., 0][np.abs(wb).max(2) > 0] == 0)
    assert np.all(qb[3, 0] == 8) and float(d16[3, 0]) == 0.0
    amax = np.take_along_axis(wb, i[..., None], 2)[..., 0]
    d = (amax.astype(np.float32) / np.float32(-8)).astype(np.float64)
    deq_d = d[..., None] * (qb - 8)                     # with the float32 scale
    err = np.abs(wb - deq_d)
    ratio = wb / np.where(d == 0, 1, d)[..., None]
    clamped = ratio > 7.5
    assert np.all(err[~clamped] <= np.abs(d)[..., None].repeat(32, 2)[~clamped] * (0.5 + 2.0 ** -20))
    assert np.all(err[clamped] <= np.abs(d)[..., None].repeat(32, 2)[clamped] * (1 + 2.0 ** -20))
    # pack/unpack round trip, nibble order against a plain loop
    qs = oracle.pack_q4_0(q)
    for r in (0, 5, 63):
        for b in (0, 7, 31):
            for j in range(16):
                byte = qs[r, 16 * b + j]
                assert byte & 0xF == q[r, 32 * b + j] and byte >> 4 == q[r, 32 * b + j + 16]
    assert np.array_equal(oracle.unpack_q4_0(qs), q)


# ------------------------------------------------------------------- NF4

def test_nf4_codebook_structure_and_library_quantiles():
    import scipy.stats as st
    cb = oracle.nf4_codebook()
    assert cb.dtype == np.float32 and cb.shape == (16,)
    assert cb[0] == -1.0 and cb[15] == 1.0 and cb[7] == 0.0
    assert np.all(np.diff(cb) > 0)
    assert np.sum(cb < 0) == 7 and np.sum(cb > 0) == 8
    # the levels are normal quantiles: re-derive with scipy's inverse CDF
    delta = 1 - 0.5 * (1 / 30 + 1 / 32)
    top = st.norm.ppf(delta)
    pos = st.norm.ppf(np.linspace(delta, 0.5, 9)[:-1]) / top
    neg = -st.norm.ppf(np.linspace(delta, 0.5, 8)[:-1]) / top
    want = np.sort(np.concatenate([pos, [0.0], neg]))
    assert np.max(np.abs(cb.astype(np.float64) - want)) < 2e-7
    # two published NormalFloat-4 levels (QLoRA, appendix table of NF4 values)
    assert abs(float(cb[1]) - (-0.6961928)) < 1e-6
    assert abs(float(cb[14]) - 0.7229568) < 1e-6
    # and the frozen fixture is this codebook bit for bit
    assert np.array_equal(nf4_codebook_fixture().view(np.uint32), cb.view(np.uint32))


def _bf16_values(shape, seed, std):
    import torch
    g = torch.Generator().manual_seed(seed)
    w = (torch.randn(shape, generator=g) * std).to(torch.bfloat16).to(torch.float32)
    return w.numpy()


def test_nf4_h5_hand_example():
    g = load("nf4_h5.json")
    cb = nf4_codebook_fixture()
    import torch
    lv = torch.from_numpy(cb).to(torch.bfloat16).to(torch.float32).numpy()
    w = np.tile(lv, 4)[None, :]
    codes, absmax = oracle.quantize_nf4(w, cb)
    assert float(absmax[0, 0]) == g["absmax"]
    assert np.array_equal(codes[0], np.tile(np.arange(16), 4))
    qs = oracle.pack_nf4(codes)
    assert np.array_equal(qs[0], hexbytes(g["qs_hex"]))
    assert np.array_equal(oracle.unpack_nf4(qs), codes)


def test_nf4_invariants_and_brute_force():
    cb = nf4_codebook_fixture()
    w = _bf16_values((8, 512), 30, 0.02)
    w[2, :64] = 0.0
    codes, absmax = oracle.quantize_nf4(w, cb)
    wb = w.reshape(8, -1, 64).astype(np.float64)
    cbk = codes.reshape(8, -1, 64)
    assert np.array_equal(absmax.astype(np.float64), np.abs(wb).max(2))
    assert np.all(cbk[2, 0] == 7)                       # zero block -> exact-zero level
    i = np.argmax(np.abs(wb), axis=2)
    top = np.take_along_axis(cbk, i[..., None], 2)[..., 0]
    topw = np.take_along_axis(wb, i[..., None], 2)[..., 0]
    ok = np.abs(topw) > 0
    assert np.all(np.where(topw[ok] > 0, top[ok] == 15, top[ok] == 0))
    # brute force: every code is the nearest level (float32 distances, lowest on ties)
    for r in range(8):
        for kk in range(0, 512, 7):
            a = absmax[r, kk // 64]
            v = np.float32(w[r, kk] / a) if a != 0 else np.float32(0)
            dists = [abs(float(np.float32(c - v))) for c in cb]
            best = min(dists)
            assert codes[r, kk] == dists.index(best)
    # dequantisation error at most half the widest gap times absmax
    deq = oracle.dequantize_nf4(oracle.pack_nf4(codes), absmax, cb)
    halfgap = 0.5 * np.max(np.diff(cb.astype(np.float64)))
    assert np.all(np.abs(deq - w) <= np.repeat(absmax.astype(np.float64), 64, 1) * halfgap * (1 + 1e-6))


def test_nf4_nearest_tie_goes_to_lower_level():
    cb = np.array([-1, -0.5, 0, 0.5] + [1.0] * 12, dtype=np.float32)
    cb[4:] = np.linspace(0.6, 1.0, 12, dtype=np.float32)
    w = np.zeros((1, 64), np.float32)
    w[0, 0] = 1.0            # absmax = 1
    w[0, 1] = 0.25           # exactly between levels 2 (0) and 3 (0.5)
    w[0, 2] = -0.75          # exactly between levels 0 and 1
    codes, _ = oracle.quantize_nf4(w, cb)
    assert codes[0, 1] == 2 and codes[0, 2] == 0


# ------------------------------------------------------------------ Q8_0

def test_q8_0_h7_worked_block():
    h = load("q8_0_h7_h8.json")["h7"]
    q, d16 = oracle.quantize_q8_0(np.asarray([h["w"]], dtype=np.float32))
    assert q[0].tolist() == h["q"]
    assert float(d16[0, 0]) == h["d16"]


def test_q8_0_invariants_on_random_rows():
    rng = np.random.default_rng(21)
    w = (rng.standard_normal((40, 256)) * 0.02).astype(np.float32)
    w[3, :32] = 0.0                                   # a zero block
    q, d16 = oracle.quantize_q8_0(w)
    assert q.dtype == np.int8 and np.all(np.abs(q.astype(np.int32)) <= 127)
    wb = w.reshape(40, 8, 32)
    qb = q.reshape(40, 8, 32).astype(np.float64)
    amax = np.abs(wb).max(axis=2)
    for n in range(40):
        for b in range(8):
            if amax[n, b] == 0:
                assert np.all(qb[n, b] == 0) and float(d16[n, b]) == 0.0
                continue
            i = int(np.argmax(np.abs(wb[n, b])))
            assert abs(qb[n, b, i]) == 127 and np.sign(qb[n, b, i]) == np.sign(wb[n, b, i])
            d = float(np.float32(amax[n, b]) / np.float32(127.0))
            # each code is the nearest multiple of d, up to float32 rounding of the quotient
            assert np.all(np.abs(wb[n, b].astype(np.float64) - d * qb[n, b]) <= d / 2 * (1 + 2 ** -20))
    # dequantised weights stay within half an fp16 step plus the fp16 rounding of d
    deq = oracle.dequantize_q8_0(q, d16)
    dd = np.repeat(d16.astype(np.float64), 32, axis=1)
    assert np.all(np.abs(deq - w) <= dd * 0.5 + 127 * dd * 2 ** -11 + 1e-12)


def test_q8_0_codes_equal_q8_1_codes():
    # Q8_1 is Q8_0 plus a sum field: on the same numbers the codes and
    # scales agree (two oracle functions written separately)
    rng = np.random.default_rng(22)
    v = rng.standard_normal((5, 320)).astype(np.float32)
    q0, d0 = oracle.quantize_q8_0(v)
    q1, d1, _ = oracle.quantize_q8_1(v)
    assert np.array_equal(q0, q1) and np.array_equal(d0.view(np.uint16), d1.view(np.uint16))


# ------------------------------------------------- NF4 -> bf16 dequantisation

def _bf16_bits_by_torch(v32):
    """bf16 patterns of float32 values through torch's own conversion (RNE)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(v32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_nf4_bf16_dequant_h5_block_gives_the_levels_in_order():
    # the H5 block (levels 0..15 in order, four times) with absmax 1: each
    # element is bf16(level), in element order
    cb = nf4_codebook_fixture()
    qs = hexbytes(load("nf4_h5.json")["qs_hex"])[None, :]
    bits = oracle.dequantize_nf4_bf16(qs, np.ones((1, 1), np.float32), cb)
    assert np.array_equal(bits[0], np.tile(_bf16_bits_by_torch(cb), 4))


def test_nf4_bf16_dequant_against_exact_products_and_library_rounding():
    # two float32 factors have an exact float64 product (48 significant
    # bits); numpy's float64 -> float32 is RNE, torch's float32 -> bf16 is RNE
    cb = nf4_codebook_fixture()
    rng = np.random.default_rng(77)
    n, k = 6, 256
    codes = rng.integers(0, 16, size=(n, k))
    absmax = (rng.random((n, k // 64)) * np.exp(rng.uniform(-30, 30, (n, k // 64)))).astype(np.float32)
    absmax[1, 2] = 0.0
    bits = oracle.dequantize_nf4_bf16(oracle.pack_nf4(codes), absmax, cb)
    exact = cb.astype(np.float64)[codes] * np.repeat(absmax.astype(np.float64), 64, axis=1)
    want = _bf16_bits_by_torch(exact.astype(np.float32))
    assert np.array_equal(bits, want)
    # a power-of-two absmax scales the bf16 levels exactly
    a2 = np.full((1, 1), np.float32(2.0 ** -7), np.float32)
    b2 = oracle.dequantize_nf4_bf16(oracle.pack_nf4(np.arange(64)[None, :] % 16), a2, cb)
    lv = oracle.bf16_bits_to_f32(_bf16_bits_by_torch(cb)).astype(np.float64) * 2.0 ** -7
    assert np.array_equal(oracle.bf16_bits_to_f32(b2[0]).astype(np.float64), np.tile(lv, 4))
    # truncating instead of rounding to nearest would change some of them
    trunc = (exact.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    assert not np.array_equal(bits, trunc)

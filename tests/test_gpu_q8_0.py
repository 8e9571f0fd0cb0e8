"""Q8_0 weights on the GPU against the oracle: the quantiser bit for bit,
the Q8_0 x Q8_1 GEMV within the bound at 1 to 32 columns (ragged segments,
several launches past eight columns), exact integer outputs on unit-scale
inputs, the worked example, argmax, column symmetry, guard regions."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_split_gb300 as wobs
from golden_io import load
from parity import assert_within, dev, f16_to_dev, to_dev, w_x_fp32
from weight_only_bit_split_gb300 import synth

pytestmark = pytest.mark.gpu


def _case(n, k, m, copy=0):
    w, x = w_x_fp32(2, n, k, m, copy=copy)
    qw, dw = oracle.quantize_q8_0(w)
    q8, d8, s8 = oracle.quantize_q8_1(x)
    xq = oracle.pack_q8_1(q8, d8, s8)
    ref = oracle.gemv_q8_0_q8_1(qw, dw, q8, d8)
    ad = oracle.abs_dot_q8_0_q8_1(qw, dw, q8, d8)
    return (to_dev(qw), f16_to_dev(dw), to_dev(xq)), ref, ad


@pytest.mark.parametrize("n,k", [(1, 32), (37, 96), (300, 4096), (64, 14336), (5, 4128)])
def test_quantize_q8_0_bit_exact(n, k):
    w = synth.weights(2, (n, k))
    w[0, :32] = torch.tensor(load("q8_0_h7_h8.json")["h7"]["w"])     # halves and signed maxima
    if n > 1:
        w[1, :32] = 0.0                                                # a zero block
    qs, d = wobs.wobs_quantize_q8_0(w.to(dev()))
    qr, dr = oracle.quantize_q8_0(w.numpy())
    assert np.array_equal(qs.cpu().numpy(), qr)
    assert np.array_equal(d.cpu().numpy().view(np.uint16), dr.view(np.uint16))


@pytest.mark.parametrize("n,k", [(1, 256), (37, 768), (300, 2304), (1024, 4096), (33, 14336),
                                 (4100, 512)])
def test_gemv_q8_0_m1(n, k):
    (qs, d, xq), ref, ad = _case(n, k, 1)
    y, am = wobs.wobs_gemv_q8_0_q8_1(qs, d, xq, want_argmax=True)
    yn = y.cpu().numpy()
    assert_within(yn, ref, ad, "f32", f"q8_0 M=1 {n}x{k}")
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yn))


@pytest.mark.parametrize("m", [2, 3, 4, 5, 8, 9, 16, 17, 32])
def test_gemv_q8_0_multi_column(m):
    (qs, d, xq), ref, ad = _case(600, 2048, m, copy=m)
    y, am = wobs.wobs_gemv_q8_0_q8_1(qs, d, xq, want_argmax=True)
    yn = y.cpu().numpy()
    assert_within(yn, ref, ad, "f32", f"q8_0 M={m}")
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yn))


def _unit_scale_case(n, k, m, seed):
    """Random codes, every scale exactly 1: y is the integer sum of the block dots."""
    rng = np.random.default_rng(seed)
    qw = rng.integers(-127, 128, size=(n, k)).astype(np.int8)
    q8 = rng.integers(-127, 128, size=(m, k)).astype(np.int8)
    dw = np.ones((n, k // 32), np.float16)
    d8 = np.ones((m, k // 32), np.float16)
    s8 = q8.reshape(m, k // 32, 32).astype(np.int64).sum(axis=2).astype(np.float16)
    exact = oracle.q8_0_q8_1_blockdots(qw, q8).astype(np.int64).sum(axis=2)
    assert np.abs(exact).max() < 2 ** 24
    return (to_dev(qw), f16_to_dev(dw), to_dev(oracle.pack_q8_1(q8, d8, s8))), exact


@pytest.mark.parametrize("m", [1, 2, 7, 8, 12, 32])
@pytest.mark.parametrize("n,k", [(16, 256), (37, 1024), (300, 2048)])
def test_q8_0_block_dots_are_exact(n, k, m):
    # |y| < 2^24 with unit scales: every float step is exact, so equality
    (qs, d, xq), exact = _unit_scale_case(n, k, m, seed=7 * n + m)
    y, am = wobs.wobs_gemv_q8_0_q8_1(qs, d, xq, want_argmax=True)
    yn = y.cpu().numpy()
    assert np.array_equal(yn, exact.astype(np.float32))
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yn))


def test_q8_0_h8_worked_example_on_gpu():
    from fractions import Fraction
    h = load("q8_0_h7_h8.json")
    w = np.zeros((2, 256), np.float32)             # the 2x64 example, padded with zero blocks
    w[0, :32] = h["h7"]["w"]
    w[0, 32:64] = 1.0
    w[1, 32] = -1.0
    w[1, 33:64] = 0.25
    x = np.zeros((1, 256), np.float32)
    x[0, :64] = 1.0
    qs, d = wobs.wobs_quantize_q8_0(torch.from_numpy(w).to(dev()))
    xq = wobs.wobs_quantize_q8_1(torch.from_numpy(x).to(dev()))
    y, _ = wobs.wobs_gemv_q8_0_q8_1(qs, d, xq)
    for n in range(2):
        num, den = h["h8"]["y_num_den"][n]
        assert abs(float(y[0, n]) - float(Fraction(num, den))) <= 2e-6 * float(Fraction(num, den))


def test_q8_0_column_symmetry_and_determinism():
    (qs, d, _), _, _ = _case(1000, 4096, 1)
    x = synth.activations(2, (1, 4096)).to(dev())
    xq = wobs.wobs_quantize_q8_1(x.repeat(19, 1))
    y1, _ = wobs.wobs_gemv_q8_0_q8_1(qs, d, xq)
    y2, _ = wobs.wobs_gemv_q8_0_q8_1(qs, d, xq)
    assert torch.equal(y1, y2)
    for m in range(1, 19):
        assert torch.equal(y1[m], y1[0])


def test_q8_0_rejects_unsupported_shapes():
    qs = torch.zeros(4, 96, dtype=torch.int8, device=dev())
    d = torch.zeros(4, 3, dtype=torch.float16, device=dev())
    xq = torch.zeros(1, 3 * 36, dtype=torch.uint8, device=dev())
    with pytest.raises(wobs.WobsError, match="UNSUPPORTED_SHAPE"):
        wobs.wobs_gemv_q8_0_q8_1(qs, d, xq)


def test_q8_0_full_size_down_projection():
    # the 8B model's down projection (4096 x 14336) at one and eight columns,
    # every output checked
    for m in (1, 8):
        (qs, d, xq), ref, ad = _case(4096, 14336, m)
        y, am = wobs.wobs_gemv_q8_0_q8_1(qs, d, xq, want_argmax=True)
        yn = y.cpu().numpy()
        assert_within(yn, ref, ad, "f32", f"q8_0 4096x14336 M={m}")
        assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yn))

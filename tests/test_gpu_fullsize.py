"""Parity at the full decode workload sizes, in the launch configuration the
benchmark times (default dispatch, weights made by the library's own
quantisers where the benchmark does so).  Where the oracle cannot afford
every output, sampled rows are recomputed one by one; argmax indices are
checked exactly against the oracle's argmax of the GPU's own logits."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_split_gb300 as wobs
from parity import assert_within, dev, f16_to_dev, q4_inputs_from_oracle, to_dev, w_x_fp32
from weight_only_bit_split_gb300 import synth
from weight_only_bit_split_gb300.nf4_levels import normal_float_levels

pytestmark = pytest.mark.gpu


def _sample_rows(n, count, seed):
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, count)]))
    return rows


def test_fp16_4096x4096_full():
    n = k = 4096
    w = synth.weights(1, (n, k), dtype=torch.float16)
    x = synth.activations(1, (1, k), dtype=torch.float16)
    y = wobs.wobs_gemv_f16(w.to(dev()), x.to(dev())).cpu().float().numpy()
    err = assert_within(y, oracle.gemv_dense(w.numpy(), x.numpy()),
                        oracle.abs_dot_dense(w.numpy(), x.numpy()), "f16", "C1")
    assert err < 1e-4


@pytest.mark.parametrize("n,k", [(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336)])
def test_q4_0_m1_8b_shapes_full(n, k):
    w, x = w_x_fp32(2, n, k, 1)
    # the benchmark quantises on the GPU: those bytes must equal the oracle's
    qs_g, d_g = wobs.wobs_quantize_q4_0(torch.from_numpy(w).to(dev()))
    xq_g = wobs.wobs_quantize_q8_1(torch.from_numpy(x).to(dev()))
    qs, d4, q8, d8, xq = q4_inputs_from_oracle(w, x)
    assert np.array_equal(qs_g.cpu().numpy(), qs)
    assert np.array_equal(d_g.cpu().numpy().view(np.uint16), d4.view(np.uint16))
    assert np.array_equal(xq_g.cpu().numpy(), xq)
    y, am = wobs.wobs_gemv_q4_0_q8_1(qs_g, d_g, xq_g, want_argmax=True)
    yn = y.cpu().numpy()
    err = assert_within(yn, oracle.gemv_q4_0_q8_1(qs, d4, q8, d8),
                        oracle.abs_dot_q4_0_q8_1(qs, d4, q8, d8), "f32", f"C2 {n}x{k}")
    assert err < 1e-4
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yn))


@pytest.mark.parametrize("n,k", [(4096, 4096), (14336, 4096)])
@pytest.mark.parametrize("m", [1, 2, 4, 8, 12, 16, 24, 32])
def test_q4_0_m_sweep_full_sampled(n, k, m):
    wdev = synth.weights(4, (n, k), device=dev())
    xdev = synth.activations(4, (m, k), device=dev())
    qs_g, d_g = wobs.wobs_quantize_q4_0(wdev)
    xq_g = wobs.wobs_quantize_q8_1(xdev)
    y, am = wobs.wobs_gemv_q4_0_q8_1(qs_g, d_g, xq_g, want_argmax=True)
    yn = y.cpu().numpy()
    rows = _sample_rows(n, 192, 40 + m)
    wr = wdev[torch.from_numpy(rows).to(dev())].cpu().numpy()
    qs, d4, q8, d8, xq = q4_inputs_from_oracle(wr, xdev.cpu().numpy())
    assert np.array_equal(qs_g[torch.from_numpy(rows).to(dev())].cpu().numpy(), qs)
    assert np.array_equal(xq_g.cpu().numpy(), xq)
    assert_within(yn[:, rows], oracle.gemv_q4_0_q8_1(qs, d4, q8, d8),
                  oracle.abs_dot_q4_0_q8_1(qs, d4, q8, d8), "f32", f"C4 {n}x{k} M={m}")
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yn))


def test_nf4_28672x8192_full_sampled():
    n, k = 28672, 8192
    cb = normal_float_levels().numpy()
    wdev = synth.weights(3, (n, k), device=dev(), dtype=torch.bfloat16)
    x = synth.activations(3, (k,), device=dev(), dtype=torch.bfloat16)
    qs_g, am_g = wobs.wobs_quantize_nf4(wdev, cb)
    y, idx = wobs.wobs_gemv_nf4(qs_g, am_g, cb, x, want_argmax=True)
    yf = y.float().cpu().numpy()
    rows = _sample_rows(n, 256, 3)
    ridx = torch.from_numpy(rows).to(dev())
    wr = wdev[ridx].float().cpu().numpy()
    codes, absmax = oracle.quantize_nf4(wr, cb)
    qs = oracle.pack_nf4(codes)
    assert np.array_equal(qs_g[ridx].cpu().numpy(), qs)
    assert np.array_equal(am_g[ridx].cpu().numpy().view(np.uint32), absmax.view(np.uint32))
    xf = x.float().cpu().numpy()
    err = assert_within(yf[rows], oracle.gemv_nf4(qs, absmax, cb, xf)[0],
                        oracle.abs_dot_nf4(qs, absmax, cb, xf)[0], "bf16", "C3")
    assert err < 1e-2
    assert int(idx.item()) == int(oracle.argmax_rows(yf)[0])


@pytest.mark.parametrize("m", [1, 32])
def test_bf16_lm_head_128000x4096_full_sampled(m):
    n, k = 128000, 4096
    wdev = synth.weights(5, (n, k), device=dev(), dtype=torch.bfloat16)
    xdev = synth.activations(5, (m, k), device=dev(), dtype=torch.bfloat16)
    logits, am = wobs.wobs_gemv_bf16(wdev, xdev, want_argmax=True)
    lg = logits.cpu().numpy()
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(lg))
    rows = np.unique(np.concatenate([_sample_rows(n, 256, 5 + m), am.cpu().numpy()]))
    wr = wdev[torch.from_numpy(rows).to(dev())].float().cpu().numpy()
    xf = xdev.float().cpu().numpy()
    err = assert_within(lg[:, rows], oracle.gemv_dense(wr, xf), oracle.abs_dot_dense(wr, xf),
                        "f32", f"C5 M={m}")
    assert err < 1e-4

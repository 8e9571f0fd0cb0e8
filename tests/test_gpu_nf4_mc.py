"""NF4 with several activation columns and the dequantise-then-GEMM path on
the GPU, against the fp64 oracle.

The fused multi-column GEMV (wobs_gemv_nf4 with M > 1: the mma.sync kernel
for up to four columns, the tcgen05 kernel, or the CUDA-core kernel where
neither applies) is compared element by element with oracle.gemv_nf4 within
the bf16 parity bound, its argmax with the oracle's argmax of the returned
outputs; ragged row tiles, split K ranges, columns past the MMA width,
scaled inputs, columns of very different magnitudes, pitched activation
rows, the fallback kernel, identical columns, the full 70B MLP shape on
sampled rows and guard regions around every output are covered.  The dequantiser is bit-exact with
oracle.dequantize_nf4_bf16, and the dequantise-then-GEMM composition is
compared with the dense oracle on those bf16 weights.
"""
import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_split_gb300 as wobs
from golden_io import nf4_codebook_fixture
from parity import assert_within, dev, to_dev
from test_gpu_canaries import check_guards, guarded
from weight_only_bit_split_gb300 import synth
from weight_only_bit_split_gb300.nf4_levels import normal_float_levels

pytestmark = pytest.mark.gpu


def _planes(n, k, copy=0, cb=None):
    cb = nf4_codebook_fixture() if cb is None else cb
    w = synth.weights(3, (n, k), copy=copy, dtype=torch.bfloat16).float().numpy()
    codes, absmax = oracle.quantize_nf4(w, nf4_codebook_fixture())
    return cb, oracle.pack_nf4(codes), absmax


def _x(m, k, copy=0, mul=1.0):
    return (synth.activations(3, (m, k), copy=copy) * mul).to(torch.bfloat16)


def _ref(qs, absmax, cb, xb):
    xf = xb.float().numpy()
    return oracle.gemv_nf4(qs, absmax, cb, xf), oracle.abs_dot_nf4(qs, absmax, cb, xf)


@pytest.fixture(params=["mma", "tc", "cp"])
def mc_path(request, monkeypatch):
    """The default choice (mma.sync kernel for up to four columns, else the
    tensor-memory kernel), the tensor-memory kernel forced for every M, and
    the CUDA-core kernel (forced)."""
    monkeypatch.delenv("WOBS_NF4", raising=False)
    monkeypatch.delenv("WOBS_NF4_MC", raising=False)
    if request.param == "cp":
        monkeypatch.setenv("WOBS_NF4", "cp")
    elif request.param == "tc":
        monkeypatch.setenv("WOBS_NF4_MC", "tc")
    return request.param


@pytest.mark.parametrize("n,k,m", [(300, 1024, 2), (1000, 4096, 5), (129, 256, 16), (2000, 2048, 17),
                                   (640, 8192, 32), (4096, 1024, 32), (77, 512, 3), (1, 768, 9),
                                   (5003, 2048, 8), (1000, 8192, 4), (5003, 4096, 3), (64, 2048, 2),
                                   (4097, 1024, 4), (3000, 8192, 8), (777, 8192, 5), (130, 1024, 7),
                                   (9000, 8192, 6), (1, 1024, 2), (65, 2048, 3), (63, 8192, 4)])
def test_nf4_columns_match_the_oracle(n, k, m, mc_path):
    cb, qs, absmax = _planes(n, k)
    xb = _x(m, k)
    ref, ad = _ref(qs, absmax, cb, xb)
    y, am = wobs.wobs_gemv_nf4(to_dev(qs), to_dev(absmax), cb, xb.to(dev()), want_argmax=True)
    yf = y.float().cpu().numpy()
    assert y.shape == (m, n)
    err = assert_within(yf, ref, ad, "bf16", f"nf4 {m} columns {n}x{k} ({mc_path})")
    assert err < 1e-2
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yf))


@pytest.mark.parametrize("n,k,m", [(500, 320, 4), (130, 1088, 12), (64, 64, 2)])
def test_nf4_columns_fallback_shapes(n, k, m):
    """K not a multiple of 256: the CUDA-core kernel takes the call."""
    cb, qs, absmax = _planes(n, k, copy=1)
    xb = _x(m, k, copy=1)
    ref, ad = _ref(qs, absmax, cb, xb)
    y, am = wobs.wobs_gemv_nf4(to_dev(qs), to_dev(absmax), cb, xb.to(dev()), want_argmax=True)
    yf = y.float().cpu().numpy()
    assert_within(yf, ref, ad, "bf16", f"nf4 fallback {m} columns {n}x{k}")
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yf))


def test_nf4_columns_offset_rows_take_the_fallback():
    """Activation rows off the 16-byte grid (pitch K + 4): still correct."""
    n, k, m = 700, 1024, 6
    cb, qs, absmax = _planes(n, k, copy=2)
    xb = _x(m, k, copy=2)
    big = torch.zeros(m, k + 4, dtype=torch.bfloat16)
    big[:, 2:k + 2] = xb
    xv = big.to(dev())[:, 2:k + 2]
    ref, ad = _ref(qs, absmax, cb, xb)
    y, _ = wobs.wobs_gemv_nf4(to_dev(qs), to_dev(absmax), cb, xv)
    assert_within(y.float().cpu().numpy(), ref, ad, "bf16", "nf4 offset activation rows")


@pytest.mark.parametrize("m", [2, 3, 4])
def test_nf4_columns_pitched_rows(m, mc_path):
    """Activation rows 16-byte aligned with a pitch above K."""
    n, k = 900, 4096
    cb, qs, absmax = _planes(n, k, copy=2)
    xb = _x(m, k, copy=2)
    big = torch.zeros(m, k + 64, dtype=torch.bfloat16)
    big[:, :k] = xb
    xv = big.to(dev())[:, :k]
    ref, ad = _ref(qs, absmax, cb, xb)
    y, am = wobs.wobs_gemv_nf4(to_dev(qs), to_dev(absmax), cb, xv, want_argmax=True)
    yf = y.float().cpu().numpy()
    assert_within(yf, ref, ad, "bf16", f"nf4 {m} pitched columns ({mc_path})")
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yf))


@pytest.mark.parametrize("muls", [(2.0 ** 40, 2.0 ** -40), (1.0, 2.0 ** -60, 2.0 ** 30),
                                  (2.0 ** -30, 1.0, 2.0 ** 50, 3.0e-3),
                                  (1.0, 2.0 ** 40, 2.0 ** -40, 7.0, 2.0 ** -20, 2.0 ** 20, 0.1, 3.0e5)])
def test_nf4_columns_far_apart_magnitudes(muls, mc_path):
    """Columns whose magnitudes differ by many powers of two: each column's
    own scaling must keep every column within its bound."""
    n, k, m = 700, 8192, len(muls)
    cb, qs, absmax = _planes(n, k, copy=9)
    xb = torch.cat([_x(1, k, copy=10 + i, mul=mul) for i, mul in enumerate(muls)])
    ref, ad = _ref(qs, absmax, cb, xb)
    y, _ = wobs.wobs_gemv_nf4(to_dev(qs), to_dev(absmax), cb, xb.to(dev()))
    assert_within(y.float().cpu().numpy(), ref, ad, "bf16", f"nf4 column magnitudes {muls} ({mc_path})")


@pytest.mark.parametrize("xmul,cbmul", [(2.0 ** 40, 1.0), (2.0 ** -40, 1.0), (1.0, 1000.0),
                                        (3.0e-3, 2.0 ** -30)])
def test_nf4_columns_scaled_inputs(xmul, cbmul):
    """Magnitudes far from 1: the per-column and per-row powers of two of the
    tensor-memory kernel come back out exactly."""
    n, k, m = 300, 4096, 7
    cb = (nf4_codebook_fixture() * np.float32(cbmul)).astype(np.float32)
    _, qs, absmax = _planes(n, k, copy=3)
    xb = _x(m, k, copy=3, mul=xmul)
    ref, ad = _ref(qs, absmax, cb, xb)
    y, _ = wobs.wobs_gemv_nf4(to_dev(qs), to_dev(absmax), cb, xb.to(dev()))
    assert_within(y.float().cpu().numpy(), ref, ad, "bf16", f"nf4 columns x*{xmul} cb*{cbmul}")


@pytest.mark.parametrize("m", [4, 8, 24])
def test_nf4_identical_columns_give_identical_outputs(m, mc_path):
    n, k = 1000, 2048
    cb, qs, absmax = _planes(n, k, copy=4)
    xb = _x(1, k, copy=4).repeat(m, 1)
    y, am = wobs.wobs_gemv_nf4(to_dev(qs), to_dev(absmax), cb, xb.to(dev()), want_argmax=True)
    yi = y.view(torch.int16).cpu().numpy()
    assert np.all(yi == yi[0:1])
    assert np.all(am.cpu().numpy() == am.cpu().numpy()[0])


@pytest.mark.parametrize("m", [8, 32])
def test_nf4_columns_deterministic(m):
    n, k = 3000, 8192
    cb, qs, absmax = _planes(n, k, copy=5)
    xb = _x(m, k, copy=5).to(dev())
    qd, ad = to_dev(qs), to_dev(absmax)
    a, _ = wobs.wobs_gemv_nf4(qd, ad, cb, xb)
    b, _ = wobs.wobs_gemv_nf4(qd, ad, cb, xb)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("m", [2, 4, 8, 32])
def test_nf4_28672x8192_columns_full_sampled(m):
    n, k = 28672, 8192
    cb = normal_float_levels().numpy()
    wdev = synth.weights(3, (n, k), device=dev(), dtype=torch.bfloat16)
    xb = synth.activations(3, (m, k), copy=m, device=dev(), dtype=torch.bfloat16)
    qs_g, am_g = wobs.wobs_quantize_nf4(wdev, cb)
    y, idx = wobs.wobs_gemv_nf4(qs_g, am_g, cb, xb, want_argmax=True)
    yf = y.float().cpu().numpy()
    rng = np.random.default_rng(40 + m)
    rows = np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, 192), idx.cpu().numpy()]))
    ridx = torch.from_numpy(rows).to(dev())
    qs, absmax = qs_g[ridx].cpu().numpy(), am_g[ridx].cpu().numpy()
    ref, ad = _ref(qs, absmax, cb, xb.cpu())
    err = assert_within(yf[:, rows], ref, ad, "bf16", f"NF4 28672x8192 M={m}")
    assert err < 1e-2
    assert np.array_equal(idx.cpu().numpy(), oracle.argmax_rows(yf))


@pytest.mark.parametrize("n,k,m,path", [(1000, 4096, 32, "tc"), (333, 1024, 5, "tc"),
                                        (5003, 8192, 17, "tc"), (700, 1088, 6, "cp"),
                                        (2049, 8192, 2, "mma"), (333, 1024, 3, "mma"),
                                        (1000, 4096, 4, "mma"), (2049, 8192, 7, "mma"),
                                        (300, 4096, 8, "mma")])
def test_nf4_columns_stay_in_bounds(n, k, m, path, monkeypatch):
    if path == "cp":
        monkeypatch.setenv("WOBS_NF4", "cp")
    cb, qs, absmax = _planes(n, k, copy=6)
    xb = _x(m, k, copy=6)
    gy = guarded((m, n), torch.bfloat16)
    ga = guarded((m,), torch.int64)
    need = wobs.wobs_workspace_size(wobs.OP_GEMV_NF4, m, n, k)
    gw = guarded((need,), torch.uint8)
    gw[4].zero_()
    wobs.wobs_gemv_nf4(to_dev(qs), to_dev(absmax), cb, xb.to(dev()), y=gy[4], argmax=ga[4], ws=gw[4])
    torch.cuda.synchronize()
    check_guards(gy, "nf4 columns y")
    check_guards(ga, "nf4 columns argmax")
    check_guards(gw, "nf4 columns workspace")
    ref, ad = _ref(qs, absmax, cb, xb)
    yf = gy[4].float().cpu().numpy()
    assert_within(yf, ref, ad, "bf16", "guarded nf4 columns")
    # counters and keys are left zero for the next call
    assert int(gw[4][:min(need, wobs.WS_ZERO_BYTES)].sum().item()) == 0


def test_nf4_columns_dispatch(monkeypatch, capfd):
    monkeypatch.setenv("WOBS_DEBUG", "1")
    monkeypatch.delenv("WOBS_NF4", raising=False)
    monkeypatch.delenv("WOBS_NF4_MC", raising=False)
    for k, m in ((8192, 32), (4096, 2), (8192, 4), (2048, 5), (8192, 8), (8192, 9), (320, 4),
                 (512, 2)):
        cb, qs, absmax = _planes(256, k)
        wobs.wobs_gemv_nf4(to_dev(qs), to_dev(absmax), cb, _x(m, k).to(dev()))
    monkeypatch.setenv("WOBS_NF4_MC", "tc")
    cb, qs, absmax = _planes(256, 4096)
    wobs.wobs_gemv_nf4(to_dev(qs), to_dev(absmax), cb, _x(3, 4096).to(dev()))
    torch.cuda.synchronize()
    err = capfd.readouterr().err
    kernels = [ln.split("kernel=")[1].split()[0] for ln in err.splitlines() if ln.startswith("wobs: op=")]
    assert kernels == ["nf4_tc", "nf4_mma", "nf4_mma", "nf4_tc", "nf4_tc", "nf4_tc", "nf4_mn",
                       "nf4_tc", "nf4_tc"], kernels


# ------------------------------------------------------- dequantise -> GEMM

@pytest.mark.parametrize("n,k", [(1, 64), (300, 1024), (129, 8192), (4097, 320)])
def test_dequantize_nf4_bit_exact(n, k):
    cb, qs, absmax = _planes(n, k, copy=7)
    W = wobs.wobs_dequantize_nf4(to_dev(qs), to_dev(absmax), cb)
    got = W.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, oracle.dequantize_nf4_bf16(qs, absmax, cb))


def test_dequantize_nf4_pitched_output_stays_in_bounds():
    n, k = 200, 1024
    cb, qs, absmax = _planes(n, k, copy=8)
    g = guarded((n, k + 64), torch.bfloat16)
    W = g[4][:, :k]
    wobs.wobs_dequantize_nf4(to_dev(qs), to_dev(absmax), cb, W=W)
    torch.cuda.synchronize()
    check_guards(g, "dequantised W")
    assert np.array_equal(W.contiguous().view(torch.int16).cpu().numpy().view(np.uint16),
                          oracle.dequantize_nf4_bf16(qs, absmax, cb))


@pytest.mark.parametrize("pitch_extra", [2, 6, 8])
def test_dequantize_nf4_any_even_pitch(pitch_extra, monkeypatch, capfd):
    """Pitches that are not whole 16-byte pieces take the element kernel,
    those that are take the row kernel; both bit-exact and in bounds."""
    monkeypatch.setenv("WOBS_DEBUG", "1")
    n, k = 130, 2048
    cb, qs, absmax = _planes(n, k, copy=8)
    g = guarded((n, k + pitch_extra), torch.bfloat16)
    W = g[4][:, :k]
    wobs.wobs_dequantize_nf4(to_dev(qs), to_dev(absmax), cb, W=W)
    torch.cuda.synchronize()
    check_guards(g, "dequantised W")
    assert np.array_equal(W.contiguous().view(torch.int16).cpu().numpy().view(np.uint16),
                          oracle.dequantize_nf4_bf16(qs, absmax, cb))
    err = capfd.readouterr().err
    kernels = [ln.split("kernel=")[1].split()[0] for ln in err.splitlines() if ln.startswith("wobs: op=")]
    aligned = (k + pitch_extra) % 8 == 0 and W.data_ptr() % 16 == 0
    assert kernels == ["dequantize_nf4_rows" if aligned else "dequantize_nf4"], kernels


@pytest.mark.parametrize("n,k,m", [(1000, 4096, 1), (640, 2048, 40), (3000, 1024, 32)])
def test_nf4_dequant_gemm_path(n, k, m):
    cb, qs, absmax = _planes(n, k, copy=9)
    xb = _x(m, k, copy=9)
    logits, W = wobs.nf4_dequant_gemm(to_dev(qs), to_dev(absmax), cb, xb.to(dev()))
    wbits = oracle.dequantize_nf4_bf16(qs, absmax, cb)
    assert np.array_equal(W.view(torch.int16).cpu().numpy().view(np.uint16), wbits)
    wf = oracle.bf16_bits_to_f32(wbits)
    xf = xb.float().numpy()
    assert_within(logits.cpu().numpy(), oracle.gemv_dense(wf, xf), oracle.abs_dot_dense(wf, xf), "f32",
                  f"dequant + GEMM {m} columns")

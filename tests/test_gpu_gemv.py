"""GEMV parity on the GPU against the oracle, at sizes the oracle finishes in
seconds: several tiles, ragged tails, every kernel path, edge cases."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_split_gb300 as wobs
from golden_io import load, nf4_codebook_fixture
from parity import assert_within, dev, f16_to_dev, q4_inputs_from_oracle, to_dev, w_x_fp32
from weight_only_bit_split_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["cp", "ldg"])
def m1_path(request, monkeypatch):
    """Run an M = 1 test through the async-copy kernels and the direct-load ones."""
    if request.param == "ldg":
        monkeypatch.setenv("WOBS_M1", "ldg")
    else:
        monkeypatch.delenv("WOBS_M1", raising=False)
    return request.param


@pytest.fixture(params=["tc", "mma", "mc1", "mc4"])
def q4_mc_path(request, monkeypatch):
    """Run a multi-column Q4_0 test through the tcgen05 kernel (forced for 5..32
    columns wherever its plan applies) and with it disabled (mma.sync / few-
    column / CUDA-core kernels); "mc1" and "mc4" also run the 2..4-column
    kernel with one or four weight rows per warp instead of the default
    choice by shape."""
    monkeypatch.setenv("WOBS_Q4TC", "1" if request.param == "tc" else "0")
    if request.param in ("mc1", "mc4"):
        monkeypatch.setenv("WOBS_Q4MC", request.param[-1])
    else:
        monkeypatch.delenv("WOBS_Q4MC", raising=False)
    return request.param


@pytest.fixture(params=["tc", "mma"])
def mc_path(request, monkeypatch):
    """Run a multi-column dense test through the tcgen05 kernel and the mma.sync one."""
    if request.param == "mma":
        monkeypatch.setenv("WOBS_TC", "0")
    else:
        monkeypatch.delenv("WOBS_TC", raising=False)
    return request.param


# ----------------------------------------------------------------- dense

@pytest.mark.parametrize("n,k", [(1, 8), (37, 264), (300, 4096), (1000, 4104), (4096, 4096)])
def test_gemv_f16_m1(n, k, m1_path):
    w = synth.weights(1, (n, k), dtype=torch.float16)
    x = synth.activations(1, (1, k), dtype=torch.float16)
    y = wobs.wobs_gemv_f16(w.to(dev()), x.to(dev())).cpu().float().numpy()
    ref = oracle.gemv_dense(w.numpy(), x.numpy())
    assert_within(y, ref, oracle.abs_dot_dense(w.numpy(), x.numpy()), "f16", "gemv_f16 M=1")


@pytest.mark.parametrize("m,n,k", [(2, 300, 520), (3, 513, 1024), (8, 64, 4096)])
def test_gemv_f16_multi_column_strided(m, n, k, mc_path):
    w = synth.weights(1, (n, k + 8), dtype=torch.float16)[:, :k]       # pitch k+8
    x = synth.activations(1, (m, k + 16), dtype=torch.float16)[:, :k]
    y = wobs.wobs_gemv_f16(w.to(dev()), x.to(dev())).cpu().float().numpy()
    wn, xn = w.contiguous().numpy(), x.contiguous().numpy()
    assert_within(y, oracle.gemv_dense(wn, xn), oracle.abs_dot_dense(wn, xn), "f16", "gemv_f16 M>1")


@pytest.mark.parametrize("m,n,k", [(2, 1, 8), (9, 127, 72), (16, 129, 64), (17, 1000, 4104),
                                   (31, 300, 520), (32, 4100, 1024), (1, 19600, 136), (3, 19500, 200)])
def test_dense_multi_column_small_integers_exact(m, n, k, mc_path):
    # small integers: every product and partial sum is exact in fp32, so the
    # logits equal the integer result bit for bit whatever the summation order
    # (pins the K tail, padded columns and rows, and the operand layouts)
    rng = np.random.default_rng(m * 1000 + n)
    w = rng.integers(-8, 9, size=(n, k)).astype(np.float32)
    x = rng.integers(-8, 9, size=(m, k)).astype(np.float32)
    exact = (x.astype(np.float64) @ w.astype(np.float64).T).astype(np.float32)
    wt = torch.from_numpy(w).to(torch.bfloat16).to(dev())
    xt = torch.from_numpy(x).to(torch.bfloat16).to(dev())
    lg, am = wobs.wobs_gemv_bf16(wt, xt, want_argmax=True)
    lgn = lg.cpu().numpy()
    assert np.array_equal(lgn, exact)
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(lgn))
    y16 = wobs.wobs_gemv_f16(wt.to(torch.float16), xt.to(torch.float16)).cpu().float().numpy()
    ref16 = exact.astype(np.float16).astype(np.float32)
    assert np.array_equal(y16, ref16)


@pytest.mark.parametrize("m,n,k", [(1, 1, 8), (1, 5000, 1024), (1, 3001, 4104), (2, 777, 512),
                                   (5, 1200, 2048), (32, 2000, 4096)])
def test_gemv_bf16_logits_and_argmax(m, n, k, m1_path, mc_path):
    w = synth.weights(5, (n, k), dtype=torch.bfloat16)
    x = synth.activations(5, (m, k), dtype=torch.bfloat16)
    logits, am = wobs.wobs_gemv_bf16(w.to(dev()), x.to(dev()), want_argmax=True)
    lg = logits.cpu().numpy()
    wf, xf = w.float().numpy(), x.float().numpy()
    assert_within(lg, oracle.gemv_dense(wf, xf), oracle.abs_dot_dense(wf, xf), "f32", "gemv_bf16")
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(lg))


def test_m1_dispatch_coverage(monkeypatch, capfd):
    """The dispatch log names the kernel that ran (coverage, not assumption)."""
    monkeypatch.setenv("WOBS_DEBUG", "1")
    monkeypatch.delenv("WOBS_M1", raising=False)
    (qs, d, xq), _, _, _ = _q4_case(64, 4096, 1)
    wobs.wobs_gemv_q4_0_q8_1(qs, d, xq)
    (qs2, d2, xq2), _, _, _ = _q4_case(64, 4160, 1)
    wobs.wobs_gemv_q4_0_q8_1(qs2, d2, xq2)
    w = synth.weights(5, (64, 512), dtype=torch.bfloat16).to(dev())
    wobs.wobs_gemv_bf16(w, synth.activations(5, (1, 512), dtype=torch.bfloat16).to(dev()))
    wobs.wobs_gemv_bf16(w, synth.activations(5, (3, 512), dtype=torch.bfloat16).to(dev()))
    monkeypatch.setenv("WOBS_M1", "ldg")
    wobs.wobs_gemv_q4_0_q8_1(qs, d, xq)
    torch.cuda.synchronize()
    err = capfd.readouterr().err
    lines = [ln for ln in err.splitlines() if ln.startswith("wobs: op=")]
    kernels = [ln.split("kernel=")[1].split()[0] for ln in lines]
    assert kernels == ["q4_0_q8_1_m1_cp", "q4_0_q8_1_m1", "dense_m1_cp", "dense_tc",
                       "q4_0_q8_1_m1"], kernels


def test_gemv_bf16_argmax_ties_go_to_the_lowest_row():
    n, k = 6000, 256
    w = synth.weights(5, (n, k), dtype=torch.bfloat16)
    x = synth.activations(5, (2, k), dtype=torch.bfloat16)
    w[5900] = w[5900] * 4            # make row 5900 the winner for both columns
    w[100] = w[5900]                 # an identical earlier row, far away (other CTA)
    w[5999] = w[5900]
    logits, am = wobs.wobs_gemv_bf16(w.to(dev()), x.to(dev()), want_argmax=True)
    lg = logits.cpu().numpy()
    assert lg[0, 100] == lg[0, 5900] == lg[0, 5999]
    ref = oracle.argmax_rows(lg)
    assert np.array_equal(am.cpu().numpy(), ref)
    assert ref[0] == 100 or lg[0].max() > lg[0, 100]


def test_gemv_bf16_workspace_is_left_clean_and_reusable():
    n, k = 3000, 512
    w = synth.weights(5, (n, k), dtype=torch.bfloat16).to(dev())
    ws = torch.zeros(wobs.wobs_workspace_size(wobs.OP_GEMV_BF16, 4, n, k), dtype=torch.uint8, device=dev())
    for m in (1, 4):
        x = synth.activations(5, (m, k), copy=m, dtype=torch.bfloat16).to(dev())
        for _ in range(3):
            lg, am = wobs.wobs_gemv_bf16(w, x, want_argmax=True, ws=ws)
            assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(lg.cpu().numpy()))
            assert int(ws[:wobs.WS_ZERO_BYTES].count_nonzero()) == 0


@pytest.mark.parametrize("splits", ["2", "3", "7"])
def test_dense_forced_split_k(monkeypatch, splits):
    monkeypatch.setenv("WOBS_SPLITK", splits)
    for m in (1, 3):
        w = synth.weights(5, (700, 2048), dtype=torch.bfloat16)
        x = synth.activations(5, (m, 2048), dtype=torch.bfloat16)
        lg, am = wobs.wobs_gemv_bf16(w.to(dev()), x.to(dev()), want_argmax=True)
        lgn = lg.cpu().numpy()
        wf, xf = w.float().numpy(), x.float().numpy()
        assert_within(lgn, oracle.gemv_dense(wf, xf), oracle.abs_dot_dense(wf, xf), "f32", "split-K")
        assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(lgn))


# ------------------------------------------------------------------ Q4_0

def _q4_case(n, k, m, seed_copy=0):
    w, x = w_x_fp32(2, n, k, m, copy=seed_copy)
    qs, d4, q8, d8, xq = q4_inputs_from_oracle(w, x)
    ref = oracle.gemv_q4_0_q8_1(qs, d4, q8, d8)
    ad = oracle.abs_dot_q4_0_q8_1(qs, d4, q8, d8)
    return (to_dev(qs), f16_to_dev(d4), to_dev(xq)), ref, ad, (qs, q8)


@pytest.mark.parametrize("n,k", [(1, 32), (7, 64), (100, 4096), (33, 14336), (64, 4160),
                                 (1024, 4096), (300, 1024)])
def test_gemv_q4_0_m1(n, k, m1_path):
    (qs, d, xq), ref, ad, _ = _q4_case(n, k, 1)
    y, am = wobs.wobs_gemv_q4_0_q8_1(qs, d, xq, want_argmax=True)
    yn = y.cpu().numpy()
    assert_within(yn, ref, ad, "f32", f"q4_0 M=1 {n}x{k}")
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yn))


def test_blockdots_bit_exact():
    for (n, k, m) in [(5, 64, 1), (70, 1024, 3), (33, 4096, 32)]:
        (qs, d, xq), _, _, (qsn, q8) = _q4_case(n, k, m)
        got = wobs.wobs_q4_0_q8_1_blockdots(qs, xq).cpu().numpy()
        assert np.array_equal(got, oracle.q4_0_q8_1_blockdots(qsn, q8))


def test_q4_0_h4_worked_example_on_gpu():
    g = load("q4_0_q8_1_h4.json")
    w = np.empty((2, 64), np.float32)
    w[0] = np.tile(np.array([-1.0, 0.5], np.float32), 32)
    w[1] = 0.5
    w[1, 0] = w[1, 32] = 1.0
    qs, d4, q8, d8, xq = q4_inputs_from_oracle(w, np.ones((1, 64), np.float32))
    y, _ = wobs.wobs_gemv_q4_0_q8_1(to_dev(qs), f16_to_dev(d4), to_dev(xq))
    assert abs(float(y[0, 0]) - g["y"][0]) < 1e-5 and abs(float(y[0, 1]) - g["y"][1]) < 1e-5
    sumi = wobs.wobs_q4_0_q8_1_blockdots(to_dev(qs), to_dev(xq)).cpu().numpy()
    assert np.array_equal(sumi[0], np.asarray(g["sumi"]))


@pytest.mark.parametrize("m", [2, 4, 8, 12, 16, 24, 32])
def test_gemv_q4_0_multi_column(m, q4_mc_path):
    (qs, d, xq), ref, ad, _ = _q4_case(600, 2048, m)
    y, am = wobs.wobs_gemv_q4_0_q8_1(qs, d, xq, want_argmax=True)
    yn = y.cpu().numpy()
    assert_within(yn, ref, ad, "f32", f"q4_0 M={m}")
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yn))


def _q4_unit_scale_case(n, k, m, seed):
    """Random codes with every scale exactly 1: y is the integer sum of the block dots."""
    rng = np.random.default_rng(seed)
    q4 = rng.integers(0, 16, size=(n, k), dtype=np.uint8)
    q8 = rng.integers(-127, 128, size=(m, k)).astype(np.int8)
    qs = oracle.pack_q4_0(q4)
    d4 = np.ones((n, k // 32), np.float16)
    d8 = np.ones((m, k // 32), np.float16)
    s8 = q8.reshape(m, k // 32, 32).astype(np.int64).sum(axis=2).astype(np.float16)
    xq = oracle.pack_q8_1(q8, d8, s8)
    exact = oracle.q4_0_q8_1_blockdots(qs, q8).sum(axis=2)
    assert np.abs(exact).max() < 2 ** 24
    return (to_dev(qs), f16_to_dev(d4), to_dev(xq)), exact


@pytest.mark.parametrize("m", [2, 3, 8, 9, 16, 17, 24, 32])
@pytest.mark.parametrize("n,k", [(16, 256), (37, 1024), (300, 4096), (129, 14336)])
def test_q4_0_multi_column_block_dots_are_exact(n, k, m, q4_mc_path):
    # unit scales make every output an integer below 2^24, so any exact block
    # dot and any summation order give the same float: equality, not tolerance
    (qs, d, xq), exact = _q4_unit_scale_case(n, k, m, seed=n * 1000 + m)
    y, am = wobs.wobs_gemv_q4_0_q8_1(qs, d, xq, want_argmax=True)
    yn = y.cpu().numpy()
    assert np.array_equal(yn.astype(np.int64), exact) and np.array_equal(yn, exact.astype(np.float32))
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yn))


@pytest.mark.parametrize("m,n,k", [(2, 1, 256), (5, 15, 512), (7, 17, 768), (32, 4100, 4096),
                                   (12, 1000, 14336), (32, 333, 8192)])
def test_gemv_q4_0_multi_column_ragged(m, n, k, q4_mc_path):
    (qs, d, xq), ref, ad, _ = _q4_case(n, k, m)
    y, am = wobs.wobs_gemv_q4_0_q8_1(qs, d, xq, want_argmax=True)
    yn = y.cpu().numpy()
    assert_within(yn, ref, ad, "f32", f"q4_0 M={m} {n}x{k}")
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yn))


def test_q4_0_multi_column_paths_agree_exactly(monkeypatch, capfd):
    """Every multi-column kernel gives the exact integer answer on unit-scale
    inputs: the few-column whole-row kernel (M <= 8), the tensor-core kernel,
    and the CUDA-core fallback (K not a multiple of 256, or a scale plane
    that is only 2-byte aligned); the dispatch log names each kernel."""
    monkeypatch.setenv("WOBS_DEBUG", "1")
    expect = []
    for m, k, odd, kern in [(4, 2048, False, "q4_0_q8_1_mc_cp"), (2, 4096, False, "q4_0_q8_1_mc_cp"),
                            (3, 4096, False, "q4_0_q8_1_mc_cp"), (12, 2048, False, "q4_0_q8_1_mma"),
                            (6, 2048, False, "q4_0_q8_1_mma"),
                            (6, 2048, True, "q4_0_q8_1_mn"), (6, 2080, False, "q4_0_q8_1_mn")]:
        (qs, d, xq), exact = _q4_unit_scale_case(70, k, m, seed=m * 31 + k)
        if odd:
            buf = torch.empty(d.numel() + 8, dtype=torch.float16, device=d.device)
            d_odd = buf[1:1 + d.numel()].view(d.shape)
            d_odd.copy_(d)
            d = d_odd
        y, am = wobs.wobs_gemv_q4_0_q8_1(qs, d, xq, want_argmax=True)
        yn = y.cpu().numpy()
        assert np.array_equal(yn, exact.astype(np.float32)), kern
        assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yn)), kern
        expect.append(kern)
    err = capfd.readouterr().err
    kernels = [ln.split("kernel=")[1].split()[0] for ln in err.splitlines() if ln.startswith("wobs: op=")]
    assert kernels == expect, kernels


@pytest.mark.parametrize("m,n,k", [(17, 4096, 4096), (32, 6144, 4096), (32, 2048, 14336), (26, 19000, 2048),
                                   (32, 600, 768)])
def test_q4_0_tensor_memory_kernel_dispatch_and_parity(m, n, k, monkeypatch, capfd):
    """Shapes with 17..32 columns that fill the GPU take the tcgen05 kernel by
    default (K split into ranges of 1024 or 768 elements: 1, 2, 4 and 14
    splits here; 600 x 768 is forced); outputs within the bound, argmax exact,
    the workspace left zero."""
    if n * k < 1 << 20:
        monkeypatch.setenv("WOBS_Q4TC", "1")
    else:
        monkeypatch.delenv("WOBS_Q4TC", raising=False)
    monkeypatch.setenv("WOBS_DEBUG", "1")
    (qs, d, xq), ref, ad, _ = _q4_case(n, k, m)
    ws = wobs.workspace(wobs.OP_GEMV_Q4_0_Q8_1, m, n, k, dev())
    y, am = wobs.wobs_gemv_q4_0_q8_1(qs, d, xq, want_argmax=True, ws=ws)
    yn = y.cpu().numpy()
    err = assert_within(yn, ref, ad, "f32", f"q4_0 tc M={m} {n}x{k}")
    assert err < 1e-4
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yn))
    assert int(ws[:wobs.WS_ZERO_BYTES].count_nonzero()) == 0
    log = capfd.readouterr().err
    assert "kernel=q4_0_q8_1_tc" in log, log


def test_one_workspace_across_split_k_layouts(monkeypatch):
    """One workspace serves calls whose split-K layouts differ: the tcgen05
    kernel leaves its partials in place, and the next calls (other ops, other
    row counts) still find their counters zero and compute correct results."""
    n_big = 6144
    ws = torch.zeros(1 << 25, dtype=torch.uint8, device=dev())
    cases = [("tc", 32, n_big, 4096), ("mma", 8, 9000, 2048), ("tc", 27, 2048, 14336),
             ("mma", 12, 517, 2048), ("tc", 32, n_big, 4096)]
    for path, m, n, k in cases:
        monkeypatch.setenv("WOBS_Q4TC", "1" if path == "tc" else "0")
        assert wobs.wobs_workspace_size(wobs.OP_GEMV_Q4_0_Q8_1, m, n, k) <= ws.numel()
        (qs, d, xq), ref, ad, _ = _q4_case(n, k, m, seed_copy=m)
        y, am = wobs.wobs_gemv_q4_0_q8_1(qs, d, xq, want_argmax=True, ws=ws)
        yn = y.cpu().numpy()
        assert_within(yn, ref, ad, "f32", f"shared workspace {path} M={m} {n}x{k}")
        assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yn))
        assert int(ws[:wobs.WS_ZERO_BYTES].count_nonzero()) == 0
    lg, amb = wobs.wobs_gemv_bf16(synth.weights(5, (3000, 512), dtype=torch.bfloat16).to(dev()),
                                  synth.activations(5, (4, 512), copy=4, dtype=torch.bfloat16).to(dev()),
                                  want_argmax=True, ws=ws)
    assert np.array_equal(amb.cpu().numpy(), oracle.argmax_rows(lg.cpu().numpy()))
    assert int(ws[:wobs.WS_ZERO_BYTES].count_nonzero()) == 0


@pytest.mark.parametrize("splits", ["2", "5", "64"])
def test_gemv_q4_0_forced_split_k(monkeypatch, splits):
    monkeypatch.setenv("WOBS_SPLITK", splits)
    for m in (1, 6):
        (qs, d, xq), ref, ad, _ = _q4_case(517, 2048, m)
        y, am = wobs.wobs_gemv_q4_0_q8_1(qs, d, xq, want_argmax=True)
        yn = y.cpu().numpy()
        assert_within(yn, ref, ad, "f32", f"q4_0 split {splits} M={m}")
        assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yn))


def test_q4_0_column_symmetry_and_determinism(q4_mc_path):
    n, k = 1000, 4096
    w, x = w_x_fp32(4, n, k, 1)
    xs = np.repeat(x, 16, axis=0)
    qs, d4, q8, d8, xq = q4_inputs_from_oracle(w, xs)
    args = (to_dev(qs), f16_to_dev(d4), to_dev(xq))
    y1, _ = wobs.wobs_gemv_q4_0_q8_1(*args)
    y2, _ = wobs.wobs_gemv_q4_0_q8_1(*args)
    a = y1.cpu().numpy()
    assert np.array_equal(a, y2.cpu().numpy())                    # run to run
    assert all(np.array_equal(a[0], a[i]) for i in range(16))   # identical columns
    # a column permutation permutes the outputs bit for bit
    x2 = np.concatenate([xs[:1], x * 0.5], axis=0)
    _, _, _, _, xq2 = q4_inputs_from_oracle(w, x2)
    _, _, _, _, xq3 = q4_inputs_from_oracle(w, x2[::-1].copy())
    p, _ = wobs.wobs_gemv_q4_0_q8_1(args[0], args[1], to_dev(xq2))
    r, _ = wobs.wobs_gemv_q4_0_q8_1(args[0], args[1], to_dev(xq3))
    assert np.array_equal(p.cpu().numpy(), r.cpu().numpy()[::-1])


def test_q4_0_gpu_quantised_weights_match_oracle_path():
    # the product path (GPU quantisers) feeding the GEMV equals the oracle path
    n, k = 256, 4096
    w, x = w_x_fp32(2, n, k, 1)
    qs, d = wobs.wobs_quantize_q4_0(torch.from_numpy(w).to(dev()))
    xq = wobs.wobs_quantize_q8_1(torch.from_numpy(x).to(dev()))
    y, _ = wobs.wobs_gemv_q4_0_q8_1(qs, d, xq)
    qsn, d4, q8, d8, xqn = q4_inputs_from_oracle(w, x)
    assert np.array_equal(xq.cpu().numpy(), xqn)
    assert_within(y.cpu().numpy(), oracle.gemv_q4_0_q8_1(qsn, d4, q8, d8),
                  oracle.abs_dot_q4_0_q8_1(qsn, d4, q8, d8), "f32", "q4 product path")


# ------------------------------------------------------------------- NF4

def _nf4_case(n, k, copy=0):
    cb = nf4_codebook_fixture()
    w = synth.weights(3, (n, k), copy=copy, dtype=torch.bfloat16).float().numpy()
    x = synth.activations(3, (1, k), copy=copy, dtype=torch.bfloat16)
    codes, absmax = oracle.quantize_nf4(w, cb)
    qs = oracle.pack_nf4(codes)
    xf = x.float().numpy()
    ref = oracle.gemv_nf4(qs, absmax, cb, xf)[0]
    ad = oracle.abs_dot_nf4(qs, absmax, cb, xf)[0]
    return cb, to_dev(qs), to_dev(absmax), x.to(dev()).reshape(-1), ref, ad


@pytest.fixture(params=["mma", "cp", "ldg"])
def nf4_path(request, monkeypatch):
    """Run an NF4 test through the tensor-core kernel, the staged CUDA-core one
    and the plain-load one (shapes a kernel does not take fall through to the
    next)."""
    monkeypatch.delenv("WOBS_NF4", raising=False)
    monkeypatch.delenv("WOBS_M1", raising=False)
    if request.param == "cp":
        monkeypatch.setenv("WOBS_NF4", "cp")
    elif request.param == "ldg":
        monkeypatch.setenv("WOBS_M1", "ldg")
    return request.param


@pytest.mark.parametrize("n,k", [(1, 64), (31, 1024), (100, 8192), (33, 1088), (257, 4096),
                                 (70, 16384), (95, 2048), (1000, 8192), (3, 8192), (129, 6144)])
def test_gemv_nf4(n, k, nf4_path):
    cb, qs, am, x, ref, ad = _nf4_case(n, k)
    y, idx = wobs.wobs_gemv_nf4(qs, am, cb, x, want_argmax=True)
    yf = y.float().cpu().numpy()
    assert_within(yf, ref, ad, "bf16", f"nf4 {n}x{k}")
    assert int(idx.item()) == int(oracle.argmax_rows(yf)[0])


# more row tiles than the ring has stages in every CTA, and a ragged last tile
@pytest.mark.parametrize("n,k", [(5003, 8192), (60013, 1024)])
def test_gemv_nf4_stage_ring_wraps(n, k):
    cb, qs, am, x, ref, ad = _nf4_case(n, k, copy=1)
    y, idx = wobs.wobs_gemv_nf4(qs, am, cb, x, want_argmax=True)
    yf = y.float().cpu().numpy()
    assert_within(yf, ref, ad, "bf16", f"nf4 {n}x{k}")
    assert int(idx.item()) == int(oracle.argmax_rows(yf)[0])


# activation and codebook magnitudes far from 1: the tensor-core kernel's
# power-of-two scalings must come back out exactly
@pytest.mark.parametrize("xmul,cbmul", [(2.0 ** 40, 1.0), (2.0 ** -40, 1.0), (1.0, 1000.0),
                                        (3.0e-3, 2.0 ** -30)])
def test_gemv_nf4_scaled_inputs(xmul, cbmul):
    n, k = 300, 4096
    cb = (np.asarray(nf4_codebook_fixture(), np.float32) * np.float32(cbmul)).astype(np.float32)
    w = synth.weights(4, (n, k), dtype=torch.bfloat16).float().numpy()
    x = (synth.activations(4, (1, k)) * xmul).to(torch.bfloat16)
    codes, absmax = oracle.quantize_nf4(w, np.asarray(nf4_codebook_fixture(), np.float32))
    qs = oracle.pack_nf4(codes)
    xf = x.float().numpy()
    ref = oracle.gemv_nf4(qs, absmax, cb, xf)[0]
    ad = oracle.abs_dot_nf4(qs, absmax, cb, xf)[0]
    y, _ = wobs.wobs_gemv_nf4(to_dev(qs), to_dev(absmax), cb, x.to(dev()).reshape(-1))
    assert_within(y.float().cpu().numpy(), ref, ad, "bf16", f"nf4 x*{xmul} cb*{cbmul}")


def test_nf4_dispatch_coverage(monkeypatch, capfd):
    monkeypatch.setenv("WOBS_DEBUG", "1")
    monkeypatch.delenv("WOBS_M1", raising=False)
    monkeypatch.delenv("WOBS_NF4", raising=False)
    for k in (8192, 1088):
        cb, qs, am, x, _, _ = _nf4_case(40, k)
        wobs.wobs_gemv_nf4(qs, am, cb, x)
    # a codebook entry too small for f16 beside the others takes the float kernel
    cb, qs, am, x, ref, ad = _nf4_case(40, 8192)
    cb2 = np.asarray(cb, np.float32).copy()
    cb2[8] = np.float32(1e-12)
    wobs.wobs_gemv_nf4(qs, am, cb2, x)
    monkeypatch.setenv("WOBS_NF4", "cp")
    wobs.wobs_gemv_nf4(qs, am, cb, x)
    torch.cuda.synchronize()
    err = capfd.readouterr().err
    kernels = [ln.split("kernel=")[1].split()[0] for ln in err.splitlines() if ln.startswith("wobs: op=")]
    assert kernels == ["nf4_mma", "nf4_m1", "nf4_m1_cp", "nf4_m1_cp"], kernels


def test_gemv_nf4_deterministic():
    cb, qs, am, x, _, _ = _nf4_case(500, 8192)
    a, _ = wobs.wobs_gemv_nf4(qs, am, cb, x)
    b, _ = wobs.wobs_gemv_nf4(qs, am, cb, x)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


# ----------------------------------------------------------------- probe

@pytest.mark.parametrize("variant", [0, 1, 2, 3])
@pytest.mark.parametrize("nbytes", [16, 4112, 1 << 20, (32 << 20) + 48])
def test_bw_probe_reads_every_word(variant, nbytes):
    g = torch.Generator(device=dev()).manual_seed(nbytes + variant)
    buf = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, device=dev(), generator=g)
    for grid in (0, 3):
        out = wobs.wobs_bw_probe(buf, grid=grid, variant=variant)
        got = int(out.cpu().numpy().view(np.uint32)[0])
        assert got == int(oracle.xor_words(buf.cpu().numpy()))
    assert wobs.wobs_error_word() == 0


# ------------------------------------------------------------ step graph

def test_step_graph_replays_the_captured_calls():
    (qs, d, xq), ref, ad, _ = _q4_case(777, 4096, 1)
    n, k = 777, 4096
    xh = torch.from_numpy(synth.activations(2, (1, k), copy=9).numpy()).pin_memory()
    x = torch.empty(1, k, device=dev())
    xq2 = torch.empty_like(xq)
    y = torch.empty(1, n, device=dev())
    yh = torch.empty(1, n).pin_memory()

    def step():
        x.copy_(xh, non_blocking=True)
        wobs.wobs_quantize_q8_1(x, xq2)
        wobs.wobs_gemv_q4_0_q8_1(qs, d, xq2, y=y)
        yh.copy_(y, non_blocking=True)

    g = wobs.StepGraph(step)
    eager = yh.clone()
    for _ in range(3):
        yh.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(yh, eager)
    # new inputs written into the pinned buffer are picked up by the next replay
    xh.copy_(torch.from_numpy(synth.activations(2, (1, k), copy=10).numpy()))
    g.replay()
    torch.cuda.synchronize()
    step()
    torch.cuda.synchronize()
    again = yh.clone()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(yh, again) and not torch.equal(again, eager)

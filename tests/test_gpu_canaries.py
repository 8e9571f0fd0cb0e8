"""Out-of-bounds write checks without a sanitizer: every output (and the
workspace) of each kernel path is a view inside a larger buffer whose guard
regions hold a sentinel bit pattern, checked after the call; and the bounded-
wait failure path, forced by the library's self test, leaves the context
usable."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_split_gb300 as wobs
from parity import assert_within, dev, f16_to_dev, q4_inputs_from_oracle, to_dev, w_x_fp32
from golden_io import nf4_codebook_fixture
from weight_only_bit_split_gb300 import _lib, synth

pytestmark = pytest.mark.gpu

PAD = 4096                 # guard elements on each side
SENTINEL = 0x7FA5A5A5      # a NaN bit pattern as float32; any 4-byte dtype gets these bits


def guarded(shape, dtype):
    n = int(np.prod(shape))
    esize = torch.empty(0, dtype=dtype).element_size()
    words = (2 * PAD * esize + n * esize + 3) // 4 + 4
    raw = torch.full((words,), SENTINEL, dtype=torch.int32, device=dev())
    flat = raw.view(torch.uint8)
    start = PAD * esize
    view = flat[start:start + n * esize].view(dtype).view(shape)
    return raw, flat, start, n * esize, view


def check_guards(g, what):
    raw, flat, start, nbytes, _ = g
    ref = torch.full_like(raw, SENTINEL).view(torch.uint8)
    assert torch.equal(flat[:start], ref[:start]), f"{what}: write before the output"
    assert torch.equal(flat[start + nbytes:], ref[start + nbytes:]), f"{what}: write after the output"


def _q4(n, k, m):
    w, x = w_x_fp32(2, n, k, m)
    qs, d4, q8, d8, xq = q4_inputs_from_oracle(w, x)
    return (to_dev(qs), f16_to_dev(d4), to_dev(xq)), oracle.gemv_q4_0_q8_1(qs, d4, q8, d8), \
        oracle.abs_dot_q4_0_q8_1(qs, d4, q8, d8)


@pytest.mark.parametrize("m,n,k,env", [(1, 1000, 4096, None), (1, 333, 4160, None),
                                       (1, 1000, 4096, ("WOBS_M1", "ldg")), (3, 700, 2048, None),
                                       (12, 600, 2048, None), (6, 70, 2080, None),
                                       (6, 517, 2048, ("WOBS_SPLITK", "5")),
                                       (32, 1000, 4096, ("WOBS_Q4TC", "1")),
                                       (9, 333, 1280, ("WOBS_Q4TC", "1")),
                                       (28, 6000, 4096, None)])
def test_q4_0_outputs_and_workspace_stay_in_bounds(m, n, k, env, monkeypatch):
    if env:
        monkeypatch.setenv(*env)
    (qs, d, xq), ref, ad = _q4(n, k, m)
    gy = guarded((m, n), torch.float32)
    ga = guarded((m,), torch.int64)
    wsz = wobs.wobs_workspace_size(wobs.OP_GEMV_Q4_0_Q8_1, m, n, k)
    gw = guarded((max(wsz, 1),), torch.uint8)
    gw[4].zero_()
    ws = gw[4] if wsz > 0 else None
    y, am = wobs.wobs_gemv_q4_0_q8_1(qs, d, xq, y=gy[4], argmax=ga[4], ws=ws)
    torch.cuda.synchronize()
    for g, what in ((gy, "y"), (ga, "argmax"), (gw, "workspace")):
        check_guards(g, f"q4_0 M={m} {n}x{k} {what}")
    yn = y.cpu().numpy()
    assert_within(yn, ref, ad, "f32", "guarded q4_0")
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yn))
    if ws is not None:
        assert int(ws[:wobs.WS_ZERO_BYTES].count_nonzero()) == 0


@pytest.mark.parametrize("m,k", [(1, 4096), (3, 4096), (32, 2048)])
def test_quantize_q8_1_stays_in_bounds(m, k):
    x = synth.activations(2, (m, k)).to(dev())
    g = guarded((m, k // 32 * 36), torch.uint8)
    wobs.wobs_quantize_q8_1(x, g[4])
    torch.cuda.synchronize()
    check_guards(g, "xq")
    q8, d8, s8 = oracle.quantize_q8_1(x.cpu().numpy())
    assert np.array_equal(g[4].cpu().numpy(), oracle.pack_q8_1(q8, d8, s8))


@pytest.mark.parametrize("m,n,k,env", [(1, 777, 1024, None), (3, 777, 1024, None),
                                       (3, 700, 2048, ("WOBS_TC", "0")), (1, 19600, 136, None),
                                       (32, 300, 520, None), (1, 777, 1024, ("WOBS_M1", "ldg"))])
def test_dense_bf16_outputs_and_workspace_stay_in_bounds(m, n, k, env, monkeypatch):
    if env:
        monkeypatch.setenv(*env)
    w = synth.weights(5, (n, k), dtype=torch.bfloat16)
    x = synth.activations(5, (m, k), dtype=torch.bfloat16)
    gy = guarded((m, n), torch.float32)
    ga = guarded((m,), torch.int64)
    wsz = wobs.wobs_workspace_size(wobs.OP_GEMV_BF16, m, n, k)
    gw = guarded((max(wsz, 1),), torch.uint8)
    gw[4].zero_()
    lg, am = wobs.wobs_gemv_bf16(w.to(dev()), x.to(dev()), logits=gy[4], argmax=ga[4], ws=gw[4])
    torch.cuda.synchronize()
    for g, what in ((gy, "logits"), (ga, "argmax"), (gw, "workspace")):
        check_guards(g, f"bf16 M={m} {n}x{k} {what}")
    lgn = lg.cpu().numpy()
    wf, xf = w.float().numpy(), x.float().numpy()
    assert_within(lgn, oracle.gemv_dense(wf, xf), oracle.abs_dot_dense(wf, xf), "f32", "guarded bf16")
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(lgn))


@pytest.mark.parametrize("m,n,k", [(1, 513, 4096), (4, 513, 1024)])
def test_dense_f16_output_stays_in_bounds(m, n, k):
    w = synth.weights(1, (n, k), dtype=torch.float16)
    x = synth.activations(1, (m, k), dtype=torch.float16)
    gy = guarded((m, n), torch.float16)
    wobs.wobs_gemv_f16(w.to(dev()), x.to(dev()), Y=gy[4])
    torch.cuda.synchronize()
    check_guards(gy, f"f16 M={m}")


@pytest.mark.parametrize("n,k", [(100, 8192), (33, 1088), (95, 2048), (5003, 8192)])
def test_nf4_output_stays_in_bounds(n, k):
    cb = nf4_codebook_fixture()
    w = synth.weights(3, (n, k), dtype=torch.bfloat16).float().numpy()
    x = synth.activations(3, (1, k), dtype=torch.bfloat16)
    codes, absmax = oracle.quantize_nf4(w, cb)
    qs = oracle.pack_nf4(codes)
    gy = guarded((n,), torch.bfloat16)
    ga = guarded((1,), torch.int64)
    y, am = wobs.wobs_gemv_nf4(to_dev(qs), to_dev(absmax), cb, x.to(dev()).reshape(-1), y=gy[4],
                               argmax=ga[4])
    torch.cuda.synchronize()
    check_guards(gy, "nf4 y")
    check_guards(ga, "nf4 argmax")
    ref = oracle.gemv_nf4(qs, absmax, cb, x.float().numpy())[0]
    assert_within(y.float().cpu().numpy(), ref, oracle.abs_dot_nf4(qs, absmax, cb, x.float().numpy())[0],
                  "bf16", "guarded nf4")


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    assert wobs.wobs_error_word() == 0
    wobs.wobs_selftest_wait_timeout(2_000_000)          # about a millisecond
    assert wobs.wobs_error_word() == 3                   # recorded, then cleared by the read
    assert wobs.wobs_error_word() == 0
    # through the C ABI the read reports the timeout as its status
    lib = _lib.get()
    word = ctypes.c_int(-1)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    wobs.wobs_selftest_wait_timeout(2_000_000)
    assert lib.wobs_error_word(stream, ctypes.byref(word)) == wobs.ERR_DEVICE_TIMEOUT
    assert word.value == 3 and "gave up" in lib.wobs_last_error().decode()
    assert lib.wobs_error_word(stream, ctypes.byref(word)) == 0 and word.value == 0
    (qs, d, xq), ref, ad = _q4(300, 1024, 1)
    y, _ = wobs.wobs_gemv_q4_0_q8_1(qs, d, xq)
    assert_within(y.cpu().numpy(), ref, ad, "f32", "after the self test")
    assert wobs.wobs_error_word() == 0
    with pytest.raises(wobs.WobsError):
        wobs.wobs_selftest_wait_timeout(0)


@pytest.mark.parametrize("m,n,k", [(1, 1000, 4096), (3, 333, 2304), (8, 700, 1024), (13, 77, 512)])
def test_q8_0_outputs_and_workspace_stay_in_bounds(m, n, k):
    w, x = w_x_fp32(2, n, k, m)
    qw, dw = oracle.quantize_q8_0(w)
    q8, d8, s8 = oracle.quantize_q8_1(x)
    gy = guarded((m, n), torch.float32)
    ga = guarded((m,), torch.int64)
    wsz = wobs.wobs_workspace_size(wobs.OP_GEMV_Q8_0_Q8_1, m, n, k)
    gw = guarded((max(wsz, 1),), torch.uint8)
    gw[4].zero_()
    y, am = wobs.wobs_gemv_q8_0_q8_1(to_dev(qw), f16_to_dev(dw), to_dev(oracle.pack_q8_1(q8, d8, s8)),
                                     y=gy[4], argmax=ga[4], ws=gw[4])
    torch.cuda.synchronize()
    for g, what in ((gy, "y"), (ga, "argmax"), (gw, "workspace")):
        check_guards(g, f"q8_0 M={m} {n}x{k} {what}")
    yn = y.cpu().numpy()
    assert_within(yn, oracle.gemv_q8_0_q8_1(qw, dw, q8, d8), oracle.abs_dot_q8_0_q8_1(qw, dw, q8, d8),
                  "f32", "guarded q8_0")
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yn))
    assert int(gw[4][:wobs.WS_ZERO_BYTES].count_nonzero()) == 0


@pytest.mark.parametrize("m,n,splits", [(1, 131077, None), (5, 1000, "3"), (400, 300, None)])
def test_argcmp_output_and_workspace_stay_in_bounds(m, n, splits, monkeypatch):
    if splits:
        monkeypatch.setenv("WOBS_SPLITK", splits)
    x = synth.normal((m, n), 1.0, synth.seed_of(6, 2, 3))
    go = guarded((m,), torch.int64)
    wsz = wobs.wobs_workspace_size(wobs.OP_ARGCMP, m, n, 4)
    gw = guarded((max(wsz, 1),), torch.uint8)
    gw[4].zero_()
    out = wobs.wobs_argmax(x.to(dev()), out=go[4], ws=gw[4] if wsz else None)
    torch.cuda.synchronize()
    check_guards(go, "argmax out")
    check_guards(gw, "argmax workspace")
    assert np.array_equal(out.cpu().numpy(), oracle.argmax_rows(x.numpy()))
    assert int(gw[4][:wobs.WS_ZERO_BYTES].count_nonzero()) == 0

"""wobs_gemv_q4_0_f32 (Q8_1 quantisation of the fp32 activation vector fused
into the Q4_0 GEMV) on the GPU: outputs against the oracle's quantise-then-
GEMV, bit-identity with the two-call path of the library, the format's edge
cases (zero blocks, exact .5 quotients, the largest K), the benchmark's full
8B shapes, guard regions around every output, and argument rejection."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_split_gb300 as wobs
from parity import assert_within, dev, f16_to_dev, to_dev, w_x_fp32
from test_gpu_canaries import check_guards, guarded

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["32", "16", "auto"])
def variant(request, monkeypatch):
    """Both prologue shapes, forced: 32 warps and one CTA per SM, 16 warps
    and two CTAs per SM; and the library's own choice by shape."""
    if request.param == "auto":
        monkeypatch.delenv("WOBS_Q4F32", raising=False)
    else:
        monkeypatch.setenv("WOBS_Q4F32", request.param)
    return request.param


def _planes(w):
    q4, d4 = oracle.quantize_q4_0(w)
    return oracle.pack_q4_0(q4), d4


def _oracle_y(qs, d4, x):
    q8, d8, _ = oracle.quantize_q8_1(x.reshape(1, -1))
    return oracle.gemv_q4_0_q8_1(qs, d4, q8, d8), oracle.abs_dot_q4_0_q8_1(qs, d4, q8, d8)


def _two_call(qs_d, d_d, x_d, want_argmax):
    xq = wobs.wobs_quantize_q8_1(x_d.view(1, -1))
    return wobs.wobs_gemv_q4_0_q8_1(qs_d, d_d, xq, want_argmax=want_argmax)


@pytest.mark.parametrize("n,k", [(1, 256), (7, 512), (100, 4096), (305, 1024), (1000, 4096),
                                 (33, 14336), (4097, 2048), (64, 65536), (16, 104704)])
def test_fused_matches_oracle_and_the_two_call_path(n, k, variant):
    w, x = w_x_fp32(7, n, k, 1)
    qs, d4 = _planes(w)
    ref, ad = _oracle_y(qs, d4, x)
    qs_d, d_d, x_d = to_dev(qs), f16_to_dev(d4), to_dev(x.reshape(-1))
    xq_out = torch.full((k // 32 * 36,), 0xA5, dtype=torch.uint8, device=dev())
    y, am = wobs.wobs_gemv_q4_0_f32(qs_d, d_d, x_d, want_argmax=True, xq_out=xq_out)
    yn = y.cpu().numpy()
    assert_within(yn, ref, ad, "f32", f"q4_0 f32 {n}x{k}")
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yn))
    # the Q8_1 blocks it writes are the quantiser's, sum field included
    assert np.array_equal(xq_out.cpu().numpy(),
                          oracle.pack_q8_1(*oracle.quantize_q8_1(x.reshape(1, -1))).reshape(-1))
    y2, am2 = _two_call(qs_d, d_d, x_d, True)
    assert np.array_equal(yn.view(np.uint32), y2.cpu().numpy().view(np.uint32))
    assert int(am2.item()) == int(am.item())


def test_fused_quantisation_edge_cases(variant):
    """Zero blocks (d = 0), exact half quotients of both signs (round half away
    from zero), blocks whose maximum is negative, subnormal-sized values."""
    n, k = 300, 1024
    w, _ = w_x_fp32(7, n, k, 1)
    qs, d4 = _planes(w)
    x = np.zeros(k, np.float32)
    x[32:64] = np.arange(32, dtype=np.float32) - 15.5       # block 1: amax 15.5 -> many .5 ties
    x[64] = 127.0                                            # block 2: d = 1 exactly
    x[65:96] = (np.arange(31, dtype=np.float32) - 15.0) + 0.5
    x[96:128] = -np.linspace(0.0, 3.0, 32, dtype=np.float32)  # block 3: negative maximum
    x[128:160] = np.float32(1e-38) * (np.arange(32, dtype=np.float32) - 16)
    x[160:] = np.random.default_rng(5).standard_normal(k - 160).astype(np.float32)
    ref, ad = _oracle_y(qs, d4, x)
    qs_d, d_d, x_d = to_dev(qs), f16_to_dev(d4), to_dev(x)
    y, _ = wobs.wobs_gemv_q4_0_f32(qs_d, d_d, x_d)
    yn = y.cpu().numpy()
    assert_within(yn, ref, ad, "f32", "q4_0 f32 edge cases")
    y2, _ = _two_call(qs_d, d_d, x_d, False)
    assert np.array_equal(yn.view(np.uint32), y2.cpu().numpy().view(np.uint32))


def _near_tie_vector(k, seed):
    """Blocks whose quotients x / d sit on, or a few float32 steps either side
    of, the half-integers where rounding to the nearest code changes.  Three
    kinds of block in turn: the block maximum is 127 * 2^e (so d = 2^e
    exactly) and the other elements are (j + 1/2) * 2^e, nudged by -1, 0 or
    +1 ulp, of both signs; the block maximum is an arbitrary value (d not a
    power of two) and the other elements are float32((j + 1/2) * d) nudged
    by -3 ... +3 ulp, so the IEEE quotients land within a few ulp of the
    half-integers on both sides; plain Gaussian blocks."""
    rng = np.random.default_rng(seed)
    x = np.empty(k, np.float32)
    for b in range(k // 32):
        if b % 4 == 3:
            x[32 * b:32 * b + 32] = rng.standard_normal(32).astype(np.float32)
            continue
        e = np.float32(2.0) ** int(rng.integers(-20, 5))   # d and s = d * sum(q) stay finite in fp16
        sign = np.float32(rng.choice([-1, 1]))
        if b % 4 == 2:
            amax = np.float32(127.0 * float(e) * (1.0 + 0.99 * rng.random()))
            d = np.float32(amax) / np.float32(127.0)
            half = ((rng.integers(-127, 127, 31) + 0.5) * np.float64(d)).astype(np.float32)
            for _ in range(3):
                step = rng.integers(-1, 2, 31)
                half = np.where(step > 0, np.nextafter(half, np.float32(np.inf)),
                                np.where(step < 0, np.nextafter(half, np.float32(-np.inf)), half))
            blk = np.concatenate([[amax * sign], half])
        else:
            half = (rng.integers(-127, 127, 31).astype(np.float32) + np.float32(0.5)) * e
            nudge = rng.integers(-1, 2, 31)
            half = np.where(nudge > 0, np.nextafter(half, np.float32(np.inf)),
                            np.where(nudge < 0, np.nextafter(half, np.float32(-np.inf)), half))
            blk = np.concatenate([[np.float32(127.0) * e * sign], half])
        x[32 * b:32 * b + 32] = blk.astype(np.float32)[rng.permutation(32)]
    return x


@pytest.mark.parametrize("k", [1024, 14336])
def test_fused_codes_match_the_quantiser_at_rounding_boundaries(k, variant):
    """Every weight code is 0 (weights all equal, so q4 - 8 = -8 everywhere):
    a code of x off by one anywhere changes y, so bit-identity with the
    quantiser's path shows that every rounding decision agrees."""
    n = 48
    w = np.repeat(np.linspace(0.5, 2.0, n, dtype=np.float32)[:, None], k, axis=1)
    qs, d4 = _planes(w)
    x = _near_tie_vector(k, 11 + k)
    qs_d, d_d, x_d = to_dev(qs), f16_to_dev(d4), to_dev(x)
    xq_out = torch.empty(k // 32 * 36, dtype=torch.uint8, device=dev())
    y, _ = wobs.wobs_gemv_q4_0_f32(qs_d, d_d, x_d, xq_out=xq_out)
    y2, _ = _two_call(qs_d, d_d, x_d, False)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y2.cpu().numpy().view(np.uint32))
    want = oracle.pack_q8_1(*oracle.quantize_q8_1(x.reshape(1, -1)))
    assert np.array_equal(wobs.wobs_quantize_q8_1(x_d.view(1, -1)).cpu().numpy(), want)
    assert np.array_equal(xq_out.cpu().numpy(), want.reshape(-1))
    ref, ad = _oracle_y(qs, d4, x)
    assert_within(y.cpu().numpy(), ref, ad, "f32", "near-tie activations")


@pytest.mark.parametrize("n,k", [(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336)])
def test_fused_8b_shapes_full(n, k, variant):
    """The benchmark's shapes at full size: bit-identical to quantise + GEMV
    (itself checked against the oracle at these sizes), sampled rows against
    the oracle directly."""
    w, x = w_x_fp32(2, n, k, 1)
    qs_d, d_d = wobs.wobs_quantize_q4_0(torch.from_numpy(w).to(dev()))
    x_d = to_dev(x.reshape(-1))
    y, am = wobs.wobs_gemv_q4_0_f32(qs_d, d_d, x_d, want_argmax=True)
    y2, am2 = _two_call(qs_d, d_d, x_d, True)
    yn = y.cpu().numpy()
    assert np.array_equal(yn.view(np.uint32), y2.cpu().numpy().view(np.uint32))
    assert int(am.item()) == int(am2.item()) == int(oracle.argmax_rows(yn)[0])
    rows = np.unique(np.concatenate([[0, n - 1], np.random.default_rng(n + k).integers(0, n, 48)]))
    qs, d4 = _planes(w[rows])
    ref, ad = _oracle_y(qs, d4, x)
    assert_within(yn[:, rows], ref, ad, "f32", f"q4_0 f32 {n}x{k} sampled rows")


def test_fused_outputs_and_workspace_stay_in_bounds(variant):
    n, k = 1000, 4096
    w, x = w_x_fp32(7, n, k, 1)
    qs, d4 = _planes(w)
    ref, ad = _oracle_y(qs, d4, x)
    gy = guarded((1, n), torch.float32)
    ga = guarded((1,), torch.int64)
    wsz = wobs.wobs_workspace_size(wobs.OP_GEMV_Q4_0_F32, 1, n, k)
    gw = guarded((wsz,), torch.uint8)
    gw[4].zero_()
    gq = guarded((k // 32 * 36,), torch.uint8)
    y, am = wobs.wobs_gemv_q4_0_f32(to_dev(qs), f16_to_dev(d4), to_dev(x.reshape(-1)),
                                    y=gy[4], argmax=ga[4], ws=gw[4], xq_out=gq[4])
    torch.cuda.synchronize()
    for g, what in ((gy, "y"), (ga, "argmax"), (gw, "workspace"), (gq, "xq_out")):
        check_guards(g, f"q4_0 f32 {what}")
    assert np.array_equal(gq[4].cpu().numpy(),
                          oracle.pack_q8_1(*oracle.quantize_q8_1(x.reshape(1, -1))).reshape(-1))
    yn = y.cpu().numpy()
    assert_within(yn, ref, ad, "f32", "guarded q4_0 f32")
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yn))
    assert int(gw[4][:wobs.WS_ZERO_BYTES].count_nonzero()) == 0


def test_fused_rejects_unsupported_calls():
    n = 64
    w, x = w_x_fp32(7, n, 4160, 1)
    qs, d4 = _planes(w)
    with pytest.raises(wobs.WobsError, match="multiple of 256"):
        wobs.wobs_gemv_q4_0_f32(to_dev(qs), f16_to_dev(d4), to_dev(x.reshape(-1)))
    w, x = w_x_fp32(7, n, 1024, 1)
    qs, d4 = _planes(w)
    xb = torch.zeros(1025, dtype=torch.float32, device=dev())
    xb[1:].copy_(torch.from_numpy(x.reshape(-1)))
    with pytest.raises(wobs.WobsError, match="aligned"):
        wobs.wobs_gemv_q4_0_f32(to_dev(qs), f16_to_dev(d4), xb[1:])

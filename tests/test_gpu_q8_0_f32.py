"""wobs_gemv_q8_0_f32 (Q8_1 quantisation of the fp32 activation vector fused
into the Q8_0 GEMV) on the GPU: outputs against the oracle's quantise-then-
GEMV, bit-identity with the library's two-call path and with the quantiser's
Q8_1 blocks, rounding-boundary activations, the benchmark's 8B shapes, guard
regions, and argument rejection."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_split_gb300 as wobs
from parity import assert_within, dev, f16_to_dev, to_dev, w_x_fp32
from test_gpu_canaries import check_guards, guarded
from test_gpu_q4_f32 import _near_tie_vector

pytestmark = pytest.mark.gpu


def _oracle_y(qw, dw, x):
    q8, d8, _ = oracle.quantize_q8_1(x.reshape(1, -1))
    return oracle.gemv_q8_0_q8_1(qw, dw, q8, d8), oracle.abs_dot_q8_0_q8_1(qw, dw, q8, d8)


def _two_call(qs_d, d_d, x_d, want_argmax):
    xq = wobs.wobs_quantize_q8_1(x_d.view(1, -1))
    return wobs.wobs_gemv_q8_0_q8_1(qs_d, d_d, xq, want_argmax=want_argmax)


def _blocks(x):
    return oracle.pack_q8_1(*oracle.quantize_q8_1(x.reshape(1, -1))).reshape(-1)


@pytest.mark.parametrize("n,k", [(1, 256), (7, 512), (300, 4096), (1000, 2048), (33, 14336),
                                 (4097, 1024), (16, 65536), (8, 139264)])
def test_q8_0_fused_matches_oracle_and_the_two_call_path(n, k):
    w, x = w_x_fp32(8, n, k, 1)
    qw, dw = oracle.quantize_q8_0(w)
    ref, ad = _oracle_y(qw, dw, x)
    qs_d, d_d, x_d = to_dev(qw), f16_to_dev(dw), to_dev(x.reshape(-1))
    xq_out = torch.full((k // 32 * 36,), 0xA5, dtype=torch.uint8, device=dev())
    y, am = wobs.wobs_gemv_q8_0_f32(qs_d, d_d, x_d, want_argmax=True, xq_out=xq_out)
    yn = y.cpu().numpy()
    assert_within(yn, ref, ad, "f32", f"q8_0 f32 {n}x{k}")
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yn))
    assert np.array_equal(xq_out.cpu().numpy(), _blocks(x))
    y2, am2 = _two_call(qs_d, d_d, x_d, True)
    assert np.array_equal(yn.view(np.uint32), y2.cpu().numpy().view(np.uint32))
    assert int(am2.item()) == int(am.item())


@pytest.mark.parametrize("k", [1024, 14336])
def test_q8_0_fused_codes_match_the_quantiser_at_rounding_boundaries(k):
    """Weights all equal per row (every code 127): an activation code off by
    one anywhere changes y, so bit-identity with the quantiser's path shows
    that every rounding decision agrees."""
    n = 40
    w = np.repeat(np.linspace(0.5, 2.0, n, dtype=np.float32)[:, None], k, axis=1)
    qw, dw = oracle.quantize_q8_0(w)
    x = _near_tie_vector(k, 21 + k)
    qs_d, d_d, x_d = to_dev(qw), f16_to_dev(dw), to_dev(x)
    xq_out = torch.empty(k // 32 * 36, dtype=torch.uint8, device=dev())
    y, _ = wobs.wobs_gemv_q8_0_f32(qs_d, d_d, x_d, xq_out=xq_out)
    y2, _ = _two_call(qs_d, d_d, x_d, False)
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y2.cpu().numpy().view(np.uint32))
    assert np.array_equal(xq_out.cpu().numpy(), _blocks(x))
    ref, ad = _oracle_y(qw, dw, x)
    assert_within(y.cpu().numpy(), ref, ad, "f32", "q8_0 near-tie activations")


@pytest.mark.parametrize("n,k", [(4096, 4096), (1024, 4096), (14336, 4096), (4096, 14336)])
def test_q8_0_fused_8b_shapes_full(n, k):
    w, x = w_x_fp32(9, n, k, 1)
    qs_d, d_d = wobs.wobs_quantize_q8_0(torch.from_numpy(w).to(dev()))
    x_d = to_dev(x.reshape(-1))
    y, am = wobs.wobs_gemv_q8_0_f32(qs_d, d_d, x_d, want_argmax=True)
    y2, am2 = _two_call(qs_d, d_d, x_d, True)
    yn = y.cpu().numpy()
    assert np.array_equal(yn.view(np.uint32), y2.cpu().numpy().view(np.uint32))
    assert int(am.item()) == int(am2.item()) == int(oracle.argmax_rows(yn)[0])
    rows = np.unique(np.concatenate([[0, n - 1], np.random.default_rng(n + k).integers(0, n, 48)]))
    qw, dw = oracle.quantize_q8_0(w[rows])
    ref, ad = _oracle_y(qw, dw, x)
    assert_within(yn[:, rows], ref, ad, "f32", f"q8_0 f32 {n}x{k} sampled rows")


def test_q8_0_fused_outputs_and_workspace_stay_in_bounds():
    n, k = 1000, 4096
    w, x = w_x_fp32(8, n, k, 1)
    qw, dw = oracle.quantize_q8_0(w)
    ref, ad = _oracle_y(qw, dw, x)
    gy = guarded((1, n), torch.float32)
    ga = guarded((1,), torch.int64)
    wsz = wobs.wobs_workspace_size(wobs.OP_GEMV_Q8_0_F32, 1, n, k)
    gw = guarded((wsz,), torch.uint8)
    gw[4].zero_()
    gq = guarded((k // 32 * 36,), torch.uint8)
    y, am = wobs.wobs_gemv_q8_0_f32(to_dev(qw), f16_to_dev(dw), to_dev(x.reshape(-1)),
                                    y=gy[4], argmax=ga[4], ws=gw[4], xq_out=gq[4])
    torch.cuda.synchronize()
    for g, what in ((gy, "y"), (ga, "argmax"), (gw, "workspace"), (gq, "xq_out")):
        check_guards(g, f"q8_0 f32 {what}")
    yn = y.cpu().numpy()
    assert_within(yn, ref, ad, "f32", "guarded q8_0 f32")
    assert np.array_equal(am.cpu().numpy(), oracle.argmax_rows(yn))
    assert np.array_equal(gq[4].cpu().numpy(), _blocks(x))
    assert int(gw[4][:wobs.WS_ZERO_BYTES].count_nonzero()) == 0


def test_q8_0_fused_rejects_unsupported_calls():
    w, x = w_x_fp32(8, 64, 4160, 1)
    qw, dw = oracle.quantize_q8_0(w)
    with pytest.raises(wobs.WobsError, match="multiple of 256"):
        wobs.wobs_gemv_q8_0_f32(to_dev(qw), f16_to_dev(dw), to_dev(x.reshape(-1)))

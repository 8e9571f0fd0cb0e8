"""GPU quantisers vs the oracle: bit-exact (codes, scales, sum fields)."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_split_gb300 as wobs
from golden_io import load, nf4_codebook_fixture
from parity import dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("m,k", [(1, 32), (1, 4096), (3, 96), (32, 4096), (5, 14336)])
def test_quantize_q8_1_bit_exact(m, k):
    g = torch.Generator().manual_seed(1000 + m * 7 + k)
    x = torch.randn(m, k, generator=g)
    x[0, :32] = 0.0                                   # zero block
    if k >= 64:
        x[0, 32:64] = torch.tensor([0.5, -0.5] * 16)  # halves after scaling
    want = oracle.pack_q8_1(*oracle.quantize_q8_1(x.numpy()))
    got = wobs.wobs_quantize_q8_1(x.to(dev())).cpu().numpy()
    assert np.array_equal(got, want)


def test_quantize_q8_1_strided_rows_and_h1():
    h1 = load("q8_1_h1.json")
    x = torch.zeros(2, 128)
    x[:, :32] = 1.0
    big = torch.full((2, 160), 7.0)
    big[:, :128] = x
    got = wobs.wobs_quantize_q8_1(big.to(dev())[:, :128]).cpu().numpy()
    assert bytes(got[0, :36]).hex() == h1["block_bytes_hex"]
    assert np.array_equal(got, oracle.pack_q8_1(*oracle.quantize_q8_1(x.numpy())))


@pytest.mark.parametrize("n,k", [(1, 32), (7, 64), (33, 4096), (4, 14336)])
def test_quantize_q4_0_bit_exact(n, k):
    g = torch.Generator().manual_seed(2000 + n + k)
    w = torch.randn(n, k, generator=g) * 0.02
    w[0, :32] = 0.0
    if n > 1 and k >= 64:
        w[1, 32:64] = torch.tensor([-2.0, -0.375, 0.625, 0.375] + [0.0] * 28)   # the tie block
        w[1, 0:32] = torch.tensor([0.5] * 31 + [-0.5])                          # equal magnitudes
    q4, d4 = oracle.quantize_q4_0(w.numpy())
    qs_ref = oracle.pack_q4_0(q4)
    qs, d = wobs.wobs_quantize_q4_0(w.to(dev()))
    assert np.array_equal(qs.cpu().numpy(), qs_ref)
    assert np.array_equal(d.cpu().numpy().view(np.uint16), d4.view(np.uint16))


@pytest.mark.parametrize("n,k", [(1, 64), (5, 128), (17, 8192)])
def test_quantize_nf4_bit_exact(n, k):
    cb = nf4_codebook_fixture()
    g = torch.Generator().manual_seed(3000 + n + k)
    w = (torch.randn(n, k, generator=g) * 0.02).to(torch.bfloat16)
    w[0, :64] = 0.0
    if n > 1:
        w[1, :64] = torch.from_numpy(np.tile(cb, 4)).to(torch.bfloat16)
    codes, absmax = oracle.quantize_nf4(w.float().numpy(), cb)
    qs, am = wobs.wobs_quantize_nf4(w.to(dev()), cb)
    assert np.array_equal(qs.cpu().numpy(), oracle.pack_nf4(codes))
    assert np.array_equal(am.cpu().numpy().view(np.uint32), absmax.view(np.uint32))

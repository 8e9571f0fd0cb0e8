"""Standalone argmax / argmin on the GPU against the oracle: every element
type, both kernel shapes (a CTA per row slice, a warp per row), forced
slice counts with ties planted on slice boundaries, ragged tails, padded
pitches, signed zeros and infinities, and the real-world row shapes of the
ArgCompare discussion at full size.  Indices must match bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_split_gb300 as wobs
from parity import dev
from weight_only_bit_split_gb300 import synth

pytestmark = pytest.mark.gpu

DTYPES = [torch.float16, torch.bfloat16, torch.float32]


def rows(shape, seed, dtype, levels=None):
    """N(0, 1) rows (seeded); with ``levels``, rounded onto that many steps so
    that equal values are everywhere."""
    t = synth.normal(shape, 1.0, synth.seed_of(6, 2, seed))
    if levels:
        t = torch.round(t * (levels / 8.0))
    return t.to(dtype)


def ref(t, is_min):
    a = t.float().numpy().astype(np.float64)
    return oracle.argmin_rows(a) if is_min else oracle.argmax_rows(a)


def call(t, is_min, **kw):
    f = wobs.wobs_argmin if is_min else wobs.wobs_argmax
    return f(t.to(dev()), **kw).cpu().numpy()


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("is_min", [False, True])
@pytest.mark.parametrize("m,n", [(1, 1), (1, 7), (3, 64), (2, 1000), (1, 4097), (5, 131077),
                                 (33, 2050)])
def test_random_rows_with_ties(dtype, is_min, m, n):
    t = rows((m, n), 1, dtype, levels=6)
    assert np.array_equal(call(t, is_min), ref(t, is_min))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("splits", ["1", "2", "5", "64"])
def test_forced_slices_with_boundary_ties(dtype, splits, monkeypatch):
    monkeypatch.setenv("WOBS_SPLITK", splits)
    m, n = 4, 10000
    t = rows((m, n), 2, dtype)
    # the same maximum at both ends of a row, and a run of equal maxima
    # straddling every multiple of 64 (the slice granularity) in another
    big = torch.tensor(9.0, dtype=dtype)
    t[0, 0] = big; t[0, n - 1] = big
    for b in range(64, n, 64):
        t[1, b - 1] = big; t[1, b] = big
    t[2, :] = 0.0
    t[3, 5000] = big
    for is_min in (False, True):
        u = -t if is_min else t
        got = call(u, is_min)
        assert np.array_equal(got, ref(u, is_min))
    assert call(t, False)[0] == 0 and call(t, False)[1] == 63 and call(t, False)[2] == 0


@pytest.mark.parametrize("dtype", DTYPES)
def test_warp_per_row_path(dtype):
    # many short rows take the warp-per-row kernel
    t = rows((700, 300), 3, dtype, levels=4)
    for is_min in (False, True):
        assert np.array_equal(call(t, is_min), ref(t, is_min))


@pytest.mark.parametrize("dtype", DTYPES)
def test_padded_pitch(dtype):
    full = rows((9, 5000 + 24), 4, dtype, levels=10)
    view = full[:, :5000]                     # pitch 5024 elements, last columns ignored
    full[:, 5000:] = 100.0                    # would win if read
    for is_min in (False, True):
        got = (wobs.wobs_argmin if is_min else wobs.wobs_argmax)(view.to(dev()))
        u = view.contiguous()
        assert np.array_equal(got.cpu().numpy(), ref(u, is_min))
    dv = full.to(dev())[:, :5000]             # the same, strided on the device
    assert np.array_equal(wobs.wobs_argmax(dv).cpu().numpy(), ref(view.contiguous(), False))


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("offset", [1, 3, 5])
@pytest.mark.parametrize("splits", ["", "7"])
def test_rows_off_the_16_byte_grid(dtype, offset, splits, monkeypatch):
    # a row that starts `offset` elements past a 16-byte boundary, odd pitch
    if splits:
        monkeypatch.setenv("WOBS_SPLITK", splits)
    m, n, ld = 6, 3001, 3003
    flat = rows((m * ld + offset,), 10, dtype, levels=5)
    view = flat[offset:].view(m, ld)[:, :n]
    got = wobs.wobs_argmax(flat.to(dev())[offset:].view(m, ld)[:, :n]).cpu().numpy()
    assert np.array_equal(got, ref(view.contiguous(), False))
    got = wobs.wobs_argmin(flat.to(dev())[offset:].view(m, ld)[:, :n]).cpu().numpy()
    assert np.array_equal(got, ref(view.contiguous(), True))


@pytest.mark.parametrize("dtype", DTYPES)
def test_signed_zeros_infinities_and_constant_rows(dtype):
    n = 20000
    t = torch.full((6, n), -1.0, dtype=dtype)
    t[0, 7000] = -0.0; t[0, 9000] = 0.0          # argmax 7000
    t[1, :] = float("-inf")                       # fully masked: argmax 0
    t[2, 123] = float("inf"); t[2, 19999] = float("inf")
    t[3, :] = 2.5                                 # constant row
    t[4, 19999] = 0.0                             # the last element only
    t[5, 5] = float("-inf"); t[5, 6] = float("-inf")
    for is_min in (False, True):
        assert np.array_equal(call(t, is_min), ref(t, is_min))
    assert list(call(t, False)) == [7000, 0, 123, 0, 19999, 0]
    assert list(call(t, True)) == [0, 0, 0, 0, 0, 5]


def test_workspace_left_zero_and_reused():
    m, n = 3, 200000
    ws = torch.zeros(wobs.wobs_workspace_size(wobs.OP_ARGCMP, m, n, 4), dtype=torch.uint8,
                     device=dev())
    assert ws.numel() > 0
    for seed in (5, 6, 7):
        t = rows((m, n), seed, torch.float32)
        got = wobs.wobs_argmax(t.to(dev()), ws=ws).cpu().numpy()
        assert np.array_equal(got, ref(t, False))
        assert int(ws.count_nonzero()) == 0


def test_repeated_calls_are_identical():
    t = rows((32, 128000), 8, torch.bfloat16, levels=3).to(dev())
    a = wobs.wobs_argmax(t)
    for _ in range(5):
        assert torch.equal(wobs.wobs_argmax(t), a)


# the real-world row shapes (model table of the ArgCompare discussion)
FULL = [((1, 128000), torch.bfloat16, False), ((32, 128000), torch.bfloat16, False),
        ((1, 262144), torch.bfloat16, False), ((1, 256000), torch.bfloat16, False),
        ((8, 32768), torch.float16, False), ((1, 50257), torch.float32, False),
        ((32, 1024), torch.float32, False), ((4096, 8192), torch.float32, True),
        ((512, 30522), torch.float32, False),
        ((256, 131072), torch.float32, False), ((64, 1048576), torch.float32, False),
        ((32, 1048576), torch.float32, True)]


@pytest.mark.parametrize("shape,dtype,is_min", FULL, ids=lambda v: str(v))
def test_full_size_real_world_shapes(shape, dtype, is_min):
    t = rows(shape, 9, dtype)
    assert np.array_equal(call(t, is_min), ref(t, is_min))

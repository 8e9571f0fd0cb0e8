"""The allocation-free bf16 GEMV entry point, through the C ABI.

wobs_gemv_bf16_noalloc serves callers that may not allocate device memory
when they call the GEMV (an engine that reserved its whole memory budget up
front and owns every allocation, a plugin inside a host process that
accounts all device memory): its workspace is a fixed scratch array inside
the library.  Each shape is called twice in a row, so the second call runs
on whatever the first left in the shared scratch; both results are checked
against the fp64 oracle within the parity bound, their argmax against the
oracle's argmax of the returned logits, and both against the regular entry
point wobs_gemv_bf16 with a caller-provided workspace.  One shape splits K,
so the scratch's split-K partials and counters are exercised.  This file is
collected last and needs no state from other tests.
"""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_split_gb300 as wobs
from weight_only_bit_split_gb300 import _lib, synth

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _scratch_bytes():
    """WOBS_NOALLOC_SCRATCH_BYTES as the header defines it."""
    text = open(os.path.join(ROOT, "include", "wobs.h")).read()
    m = re.search(r"#define\s+WOBS_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "WOBS_NOALLOC_SCRATCH_BYTES not found in the header"
    return int(m.group(1)) << int(m.group(2))


def _noalloc(W, X, logits, argmax):
    lib = _lib.get()
    M, K = X.shape
    N = W.shape[0]
    rc = lib.wobs_gemv_bf16_noalloc(
        ctypes.c_void_p(W.data_ptr()), W.stride(0), ctypes.c_void_p(X.data_ptr()), X.stride(0), M,
        ctypes.c_void_p(logits.data_ptr()),
        ctypes.c_void_p(argmax.data_ptr()) if argmax is not None else None, N, K,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, lib.wobs_last_error().decode()


# (M, N, K, split-K expected): the last shape has too few 256-row tiles to
# fill the GPU, so K is split and the scratch holds partials past the counters
SHAPES = [(1, 5000, 1024, False), (4, 3000, 2048, False), (32, 2000, 4096, False),
          (4, 1000, 8192, True)]


@pytest.mark.parametrize("m,n,k,splits", SHAPES)
def test_noalloc_twice_against_the_oracle_and_the_workspace_entry_point(m, n, k, splits):
    dev = torch.device("cuda", 0)
    need = wobs.wobs_workspace_size(wobs.OP_GEMV_BF16, m, n, k)
    assert need <= _scratch_bytes()
    if splits:
        assert need > wobs.WS_ZERO_BYTES, "expected a split-K shape"
    W = synth.weights(5, (n, k), device=dev, dtype=torch.bfloat16)
    X = synth.activations(5, (m, k), copy=m, device=dev, dtype=torch.bfloat16)
    w64, x64 = W.float().cpu().numpy(), X.float().cpu().numpy()
    y_ref = oracle.gemv_dense(w64, x64)
    bound = oracle.parity_bound(y_ref, oracle.abs_dot_dense(w64, x64), "f32")
    ws_logits, ws_arg = wobs.wobs_gemv_bf16(W, X, want_argmax=True)
    ws_got = ws_logits.cpu().numpy().astype(np.float64)
    assert np.all(np.abs(ws_got - y_ref) <= bound)
    for _ in range(2):
        logits = torch.full((m, n), float("nan"), dtype=torch.float32, device=dev)
        arg = torch.full((m,), -1, dtype=torch.int64, device=dev)
        rc, msg = _noalloc(W, X, logits, arg)
        assert rc == 0, msg
        torch.cuda.synchronize()
        got = logits.cpu().numpy()
        assert np.all(np.abs(got.astype(np.float64) - y_ref) <= bound)
        # the same kernel and split order as the workspace entry point
        assert np.array_equal(got, ws_logits.cpu().numpy())
        a = arg.cpu().numpy()
        assert np.array_equal(a, oracle.argmax_rows(got))
        assert np.array_equal(a, ws_arg.cpu().numpy())


def test_noalloc_rejects_shapes_beyond_the_scratch():
    dev = torch.device("cuda", 0)
    m, n, k = 32, 8192, 4096
    assert wobs.wobs_workspace_size(wobs.OP_GEMV_BF16, m, n, k) > _scratch_bytes()
    W = torch.zeros(n, k, dtype=torch.bfloat16, device=dev)
    X = torch.zeros(m, k, dtype=torch.bfloat16, device=dev)
    logits = torch.empty(m, n, dtype=torch.float32, device=dev)
    rc, msg = _noalloc(W, X, logits, None)
    assert rc == -4 and "scratch" in msg          # WOBS_ERR_WORKSPACE_TOO_SMALL

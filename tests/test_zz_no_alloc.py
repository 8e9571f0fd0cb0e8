"""The allocation-free bf16 GEMV entry point against the regular one.

wobs_gemv_bf16_noalloc serves callers that may not allocate device memory
when they call the GEMV (inside a CUDA graph capture, or under an engine
that owns every device allocation): its workspace is a fixed scratch array
inside the library.  Here it is called through the C ABI directly, twice in
a row per shape, and its logits and argmax are checked against
wobs_gemv_bf16 with a caller-provided workspace.  This file is collected
last and needs no state from other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import weight_only_bit_split_gb300 as wobs
from weight_only_bit_split_gb300 import _lib, synth

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 4 << 20


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


@pytest.mark.parametrize("m,n,k", [(1, 5000, 1024), (4, 3000, 2048), (32, 2000, 4096)])
def test_noalloc_matches_workspace_entry_point_twice(m, n, k):
    dev = torch.device("cuda", 0)
    W = synth.weights(5, (n, k), device=dev, dtype=torch.bfloat16)
    X = synth.activations(5, (m, k), copy=m, device=dev, dtype=torch.bfloat16)
    assert wobs.wobs_workspace_size(wobs.OP_GEMV_BF16, m, n, k) <= SCRATCH_BYTES
    ref_logits, ref_arg = wobs.wobs_gemv_bf16(W, X, want_argmax=True)
    ref = ref_logits.cpu().numpy().astype(np.float64)
    absdot = oracle.abs_dot_dense(W.float().cpu().numpy(), X.float().cpu().numpy())
    bound = oracle.parity_bound(ref, absdot, "f32")
    for _ in range(2):
        logits = torch.full((m, n), float("nan"), dtype=torch.float32, device=dev)
        arg = torch.full((m,), -1, dtype=torch.int64, device=dev)
        rc, msg = _noalloc(W, X, logits, arg)
        assert rc == 0, msg
        got = logits.cpu().numpy().astype(np.float64)
        assert np.all(np.abs(got - ref) <= bound)
        assert np.array_equal(arg.cpu().numpy(), ref_arg.cpu().numpy())


def test_noalloc_rejects_shapes_beyond_the_scratch():
    dev = torch.device("cuda", 0)
    m, n, k = 32, 8192, 4096
    assert wobs.wobs_workspace_size(wobs.OP_GEMV_BF16, m, n, k) > SCRATCH_BYTES
    W = torch.zeros(n, k, dtype=torch.bfloat16, device=dev)
    X = torch.zeros(m, k, dtype=torch.bfloat16, device=dev)
    logits = torch.empty(m, n, dtype=torch.float32, device=dev)
    rc, msg = _noalloc(W, X, logits, None)
    assert rc == -4 and "scratch" in msg

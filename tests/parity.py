"""Shared helpers for the GPU parity tests: inputs through the oracle,
comparison against the oracle's bound, and small reporting."""
import numpy as np
import torch

import oracle
from weight_only_bit_split_gb300 import synth


def dev():
    return torch.device("cuda", 0)


def assert_within(y_gpu, y_ref, abs_dot, out_fmt, what=""):
    """|y - y_ref| <= 1e-3 * sum|w x| + 1 ulp, elementwise; returns max normalised error."""
    y = np.asarray(y_gpu, dtype=np.float64)
    bound = oracle.parity_bound(y_ref, abs_dot, out_fmt)
    err = np.abs(y - y_ref)
    bad = err > bound
    if bad.any():
        i = np.flatnonzero(bad.reshape(-1))[0]
        raise AssertionError(
            f"{what}: {bad.sum()} outputs outside the bound; first at flat index {i}: "
            f"gpu={y.reshape(-1)[i]!r} ref={y_ref.reshape(-1)[i]!r} bound={bound.reshape(-1)[i]!r}")
    scale = np.maximum(np.asarray(abs_dot, np.float64), 1e-30)
    return float(np.max(err / scale)) if err.size else 0.0


def q4_inputs_from_oracle(w32, x32):
    """Oracle-quantised Q4_0 planes and Q8_1 blocks (numpy), plus fields."""
    q4, d4 = oracle.quantize_q4_0(w32)
    qs = oracle.pack_q4_0(q4)
    q8, d8, s8 = oracle.quantize_q8_1(x32)
    xq = oracle.pack_q8_1(q8, d8, s8)
    return qs, d4, q8, d8, xq


def to_dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.to(dev())


def f16_to_dev(a16):
    return torch.from_numpy(np.ascontiguousarray(a16).view(np.int16)).view(torch.float16).to(dev())


def w_x_fp32(workload, n, k, m, copy=0):
    w = synth.weights(workload, (n, k), copy=copy).numpy()
    x = synth.activations(workload, (m, k), copy=copy).numpy()
    return w, x

"""The C ABI on the host: symbols, argument checks, workspace sizing (CPU only).

No call here launches a kernel; every call returns from the library's
argument checks before touching the GPU.
"""
import ctypes
import os
import re

import numpy as np
import pytest

from weight_only_bit_split_gb300 import _lib
from weight_only_bit_split_gb300.nf4_levels import normal_float_levels

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "wobs.h")


def declared_symbols():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"WOBS_API\s+[\w\s\*]+?\b(wobs_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ["wobs_bw_probe", "wobs_gemv_f16", "wobs_gemv_bf16", "wobs_quantize_q8_1",
                     "wobs_gemv_q4_0_q8_1", "wobs_gemv_nf4", "wobs_workspace_size",
                     "wobs_q4_0_q8_1_blockdots", "wobs_error_word", "wobs_last_error"]:
        assert required in names


def test_library_loads_and_exports_every_declared_symbol():
    lib = _lib.get()
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"{name} has no ctypes signature"
    # and nothing the binding declares is missing from the header
    assert set(_lib.SIGNATURES) == set(declared_symbols())


def test_version_and_empty_error():
    lib = _lib.get()
    assert lib.wobs_version() >= 1
    assert isinstance(lib.wobs_last_error(), bytes)


def _status(name, *args):
    lib = _lib.get()
    rc = getattr(lib, name)(*args)
    return rc, lib.wobs_last_error().decode()


FAKE16 = ctypes.c_void_p(0x10000)      # never dereferenced: checks fail first
FAKE_ODD = ctypes.c_void_p(0x10001)


def test_null_pointers_are_invalid_args():
    rc, msg = _status("wobs_gemv_f16", None, 64, FAKE16, 64, 1, FAKE16, 8, 64, None, 0, None)
    assert rc == -1 and "null" in msg
    rc, _ = _status("wobs_gemv_q4_0_q8_1", FAKE16, None, FAKE16, 1, FAKE16, None, 8, 64, None, 0, None)
    assert rc == -1
    rc, _ = _status("wobs_bw_probe", None, 16, 0, 0, FAKE16, None)
    assert rc == -1


def test_shape_checks():
    # K not a multiple of 32 for Q4_0 / Q8_1, of 64 for NF4, of 8 for dense
    rc, _ = _status("wobs_gemv_q4_0_q8_1", FAKE16, FAKE16, FAKE16, 1, FAKE16, None, 8, 48, None, 0, None)
    assert rc == -3
    rc, _ = _status("wobs_quantize_q8_1", FAKE16, 48, 1, 48, FAKE16, None)
    assert rc == -3
    cb = (ctypes.c_float * 16)()
    rc, _ = _status("wobs_gemv_nf4", FAKE16, FAKE16, cb, FAKE16, 96, 1, FAKE16, None, 8, 96, None, 0, None)
    assert rc == -3
    rc, _ = _status("wobs_dequantize_nf4", FAKE16, FAKE16, cb, 8, 96, FAKE16, 96, None)
    assert rc == -3
    # NF4 columns: M outside 1..32, activation pitch below K
    rc, _ = _status("wobs_gemv_nf4", FAKE16, FAKE16, cb, FAKE16, 128, 33, FAKE16, None, 8, 128, None, 0, None)
    assert rc == -1
    rc, _ = _status("wobs_gemv_nf4", FAKE16, FAKE16, cb, FAKE16, 64, 2, FAKE16, None, 8, 128, None, 0, None)
    assert rc == -1
    rc, _ = _status("wobs_gemv_f16", FAKE16, 12, FAKE16, 12, 1, FAKE16, 8, 12, None, 0, None)
    assert rc == -3
    # M outside 1..32
    rc, _ = _status("wobs_gemv_bf16", FAKE16, 64, FAKE16, 64, 33, FAKE16, None, 8, 64, None, 0, None)
    assert rc == -1
    rc, _ = _status("wobs_gemv_bf16", FAKE16, 64, FAKE16, 64, 0, FAKE16, None, 8, 64, None, 0, None)
    assert rc == -1


def test_alignment_checks():
    rc, _ = _status("wobs_gemv_f16", FAKE_ODD, 64, FAKE16, 64, 1, FAKE16, 8, 64, None, 0, None)
    assert rc == -2
    rc, _ = _status("wobs_gemv_f16", FAKE16, 60, FAKE16, 64, 1, FAKE16, 8, 56, None, 0, None)
    assert rc == -2                       # pitch of 60 halves breaks 16-byte rows
    rc, _ = _status("wobs_bw_probe", FAKE16, 24, 0, 0, FAKE16, None)
    assert rc == -2                       # byte count not a multiple of 16
    rc, _ = _status("wobs_gemv_q4_0_q8_1", FAKE_ODD, FAKE16, FAKE16, 1, FAKE16, None, 8, 64, None, 0, None)
    assert rc == -2


def test_argmax_needs_a_workspace():
    rc, msg = _status("wobs_gemv_bf16", FAKE16, 64, FAKE16, 64, 1, FAKE16, FAKE16, 8, 64, None, 0, None)
    assert rc == -1 and "workspace" in msg
    rc, _ = _status("wobs_gemv_bf16", FAKE16, 64, FAKE16, 64, 1, FAKE16, FAKE16, 8, 64, FAKE16, 16, None)
    assert rc == -4


def test_workspace_size_rules():
    lib = _lib.get()
    assert lib.wobs_workspace_size(99, 1, 64, 64) == 0
    assert lib.wobs_workspace_size(3, 0, 64, 64) == 0
    assert lib.wobs_workspace_size(3, 33, 64, 64) == 0
    for op in (1, 2, 3, 4):
        s = lib.wobs_workspace_size(op, 1, 4096, 4096)
        assert s >= 8 + 8 * 32 and s % 256 == 0


def test_workspace_grows_with_forced_split(monkeypatch):
    lib = _lib.get()
    base = lib.wobs_workspace_size(3, 4, 1000, 4096)
    monkeypatch.setenv("WOBS_SPLITK", "8")
    forced = lib.wobs_workspace_size(3, 4, 1000, 4096)
    assert forced >= base + 4 * 4 * 4 * 1000


def test_product_codebook_equals_oracle_fixture():
    from golden_io import nf4_codebook_fixture
    a = normal_float_levels().numpy()
    b = nf4_codebook_fixture()
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_argcmp_argument_checks():
    out = FAKE16
    for name in ("wobs_argmax", "wobs_argmin"):
        rc, _ = _status(name, 2, None, 64, 1, 64, out, None, 0, None)
        assert rc == -1                   # null X
        rc, _ = _status(name, 7, FAKE16, 64, 1, 64, out, None, 0, None)
        assert rc == -1                   # unknown dtype
        rc, _ = _status(name, 2, FAKE16, 64, 0, 64, out, None, 0, None)
        assert rc == -1                   # M = 0
        rc, _ = _status(name, 2, FAKE16, 64, 1, 0, out, None, 0, None)
        assert rc == -3                   # N = 0
        rc, _ = _status(name, 2, FAKE16, 32, 2, 64, out, None, 0, None)
        assert rc == -1                   # ldx < N
        rc, _ = _status(name, 2, FAKE_ODD, 64, 1, 64, out, None, 0, None)
        assert rc == -2                   # bf16 X at an odd address
        rc, _ = _status(name, 3, ctypes.c_void_p(0x10002), 64, 1, 64, out, None, 0, None)
        assert rc == -2                   # fp32 X not 4-byte aligned
        rc, _ = _status(name, 3, FAKE16, 64, 1, 64, ctypes.c_void_p(0x10004), None, 0, None)
        assert rc == -2                   # out not 8-byte aligned


def test_argcmp_workspace_rules(monkeypatch):
    lib = _lib.get()
    assert lib.wobs_workspace_size(5, 1, 1000, 3) == 0        # element size must be 2 or 4
    assert lib.wobs_workspace_size(5, 0, 1000, 2) == 0
    # a single long row is split, so it needs its key and counter
    assert lib.wobs_workspace_size(5, 1, 131072, 2) == 16
    # forcing one slice a row removes the workspace; forcing several adds it
    monkeypatch.setenv("WOBS_SPLITK", "1")
    assert lib.wobs_workspace_size(5, 1, 131072, 2) == 0
    monkeypatch.setenv("WOBS_SPLITK", "3")
    assert lib.wobs_workspace_size(5, 10, 1000, 4) == (12 * 10 + 15) // 16 * 16
    # and the call refuses a missing or short workspace before any launch
    rc, msg = _status("wobs_argmax", 3, FAKE16, 1000, 10, 1000, FAKE16, None, 0, None)
    assert rc == -1 and "workspace" in msg
    rc, _ = _status("wobs_argmax", 3, FAKE16, 1000, 10, 1000, FAKE16, FAKE16, 64, None)
    assert rc == -4


def test_q8_0_argument_checks():
    rc, _ = _status("wobs_quantize_q8_0", None, 64, 1, 64, FAKE16, FAKE16, None)
    assert rc == -1
    rc, _ = _status("wobs_quantize_q8_0", FAKE16, 64, 1, 48, FAKE16, FAKE16, None)
    assert rc == -3                        # K not a multiple of 32
    rc, _ = _status("wobs_quantize_q8_0", FAKE16, 64, 1, 64, FAKE16, FAKE_ODD, None)
    assert rc == -2                        # fp16 scales at an odd address
    g = "wobs_gemv_q8_0_q8_1"
    rc, _ = _status(g, FAKE16, None, FAKE16, 1, FAKE16, None, 8, 256, None, 0, None)
    assert rc == -1
    rc, _ = _status(g, FAKE16, FAKE16, FAKE16, 33, FAKE16, None, 8, 256, None, 0, None)
    assert rc == -1                        # M above 32
    rc, _ = _status(g, FAKE16, FAKE16, FAKE16, 1, FAKE16, None, 8, 96, None, 0, None)
    assert rc == -3                        # K not a multiple of 256
    rc, _ = _status(g, FAKE16, ctypes.c_void_p(0x10008), FAKE16, 1, FAKE16, None, 8, 256, None, 0, None)
    assert rc == -2                        # scale plane not 16-byte aligned
    rc, msg = _status(g, FAKE16, FAKE16, FAKE16, 1, FAKE16, FAKE16, 8, 256, None, 0, None)
    assert rc == -1 and "workspace" in msg  # argmax without a workspace
    lib = _lib.get()
    assert lib.wobs_workspace_size(6, 1, 4096, 4096) >= 8 + 8 * 32
    assert lib.wobs_workspace_size(6, 33, 4096, 4096) == 0


def test_q4_0_f32_argument_checks():
    g = "wobs_gemv_q4_0_f32"
    rc, _ = _status(g, FAKE16, FAKE16, None, None, FAKE16, None, 8, 256, None, 0, None)
    assert rc == -1                        # no activation vector
    rc, msg = _status(g, FAKE16, FAKE16, FAKE16, None, FAKE16, None, 8, 4160, None, 0, None)
    assert rc == -3 and "256" in msg       # K not a multiple of 256
    rc, _ = _status(g, FAKE16, FAKE16, FAKE16, None, FAKE16, None, 0, 256, None, 0, None)
    assert rc == -3                        # no rows
    rc, _ = _status(g, FAKE16, ctypes.c_void_p(0x10008), FAKE16, None, FAKE16, None, 8, 256, None, 0, None)
    assert rc == -2                        # scale plane not 16-byte aligned
    rc, _ = _status(g, FAKE16, FAKE16, ctypes.c_void_p(0x10004), None, FAKE16, None, 8, 256, None, 0, None)
    assert rc == -2                        # x not 16-byte aligned
    rc, msg = _status(g, FAKE16, FAKE16, FAKE16, None, FAKE16, None, 8, 131072, None, 0, None)
    assert rc == -3 and "shared-memory" in msg
    rc, msg = _status(g, FAKE16, FAKE16, FAKE16, None, FAKE16, None, 8, 104960, None, 0, None)
    assert rc == -3 and "shared-memory" in msg   # one 256-block past the largest K, 104704
    rc, msg = _status(g, FAKE16, FAKE16, FAKE16, None, FAKE16, FAKE16, 8, 256, None, 0, None)
    assert rc == -1 and "workspace" in msg  # argmax without a workspace
    rc, _ = _status(g, FAKE16, FAKE16, FAKE16, FAKE_ODD, FAKE16, None, 8, 256, None, 0, None)
    assert rc == -2                        # xq_out not 4-byte aligned
    lib = _lib.get()
    assert lib.wobs_workspace_size(7, 1, 4096, 4096) == lib.wobs_workspace_size(3, 1, 4096, 4096)


def test_q8_0_f32_argument_checks():
    g = "wobs_gemv_q8_0_f32"
    rc, _ = _status(g, FAKE16, FAKE16, None, None, FAKE16, None, 8, 256, None, 0, None)
    assert rc == -1
    rc, msg = _status(g, FAKE16, FAKE16, FAKE16, None, FAKE16, None, 8, 4160, None, 0, None)
    assert rc == -3 and "256" in msg
    rc, _ = _status(g, FAKE16, ctypes.c_void_p(0x10008), FAKE16, None, FAKE16, None, 8, 256, None, 0, None)
    assert rc == -2
    rc, _ = _status(g, FAKE16, FAKE16, FAKE16, FAKE_ODD, FAKE16, None, 8, 256, None, 0, None)
    assert rc == -2
    rc, msg = _status(g, FAKE16, FAKE16, FAKE16, None, FAKE16, FAKE16, 8, 256, None, 0, None)
    assert rc == -1 and "workspace" in msg


def test_workspace_counter_region_and_split_k_row_limit(monkeypatch):
    """Split-K partials start past a fixed counter region of WOBS_WS_ZERO_BYTES,
    so no call's counters can fall on another call's partials; split-K calls
    beyond 2^20 rows are refused before any launch."""
    lib = _lib.get()
    src = open(HEADER).read()
    zero = int(re.search(r"#define WOBS_WS_ZERO_BYTES (\d+)", src).group(1))
    from weight_only_bit_split_gb300 import WS_ZERO_BYTES
    assert zero == WS_ZERO_BYTES == 264 + 4 * 65536
    monkeypatch.setenv("WOBS_SPLITK", "2")
    assert lib.wobs_workspace_size(3, 1, 4096, 4096) >= zero + 4 * 2 * 4096
    n = (1 << 20) + 16
    rc, msg = _status("wobs_gemv_q4_0_q8_1", FAKE16, FAKE16, FAKE16, 1, FAKE16, None, n, 4096,
                      FAKE16, 1 << 30, None)
    assert rc == -3 and "rows" in msg

"""weight_only_bit_split_gb300 -- weight-only low-bit decode GEMV for GB300.

A thin Python binding over the C ABI of ``libwobs.so`` (declared in
``include/wobs.h``).  Each function here has the name of the C entry point
it calls and only marshals arguments: it checks tensor devices, dtypes and
shapes, passes raw pointers and the current CUDA stream, and turns a
negative status into ``WobsError``.  Every step of the computation runs in
the library's CUDA kernels; there is no CPU fallback.

PyTorch supplies device memory and streams only.
"""
import ctypes

import torch

from . import _lib

OP_GEMV_F16 = 1
OP_GEMV_BF16 = 2
OP_GEMV_Q4_0_Q8_1 = 3
OP_GEMV_NF4 = 4
OP_ARGCMP = 5
OP_GEMV_Q8_0_Q8_1 = 6
OP_GEMV_Q4_0_F32 = 7
OP_GEMV_Q8_0_F32 = 8
ERR_DEVICE_TIMEOUT = -7
# leading workspace bytes that hold counters and keys: zero between calls
WS_ZERO_BYTES = 262408
DTYPE_CODES = {torch.float16: 1, torch.bfloat16: 2, torch.float32: 3}
MAX_M = 32
Q8_1_BLOCK_BYTES = 36

STATUS = {0: "OK", -1: "INVALID_ARG", -2: "MISALIGNED", -3: "UNSUPPORTED_SHAPE",
          -4: "WORKSPACE_TOO_SMALL", -5: "LAUNCH_FAILED", -6: "CUDA", -7: "DEVICE_TIMEOUT"}


class WobsError(RuntimeError):
    def __init__(self, code, message):
        super().__init__(f"{STATUS.get(code, code)}: {message}")
        self.code = code


def _check(rc, lib):
    if rc != 0:
        raise WobsError(rc, lib.wobs_last_error().decode(errors="replace"))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, name, dtype=None, ndim=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor (the library has no CPU path)")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype}, expected {dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name}: {t.dim()} dims, expected {ndim}")
    if device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if t.dim() >= 1 and t.stride(-1) != 1:
        raise ValueError(f"{name}: last dimension must be contiguous")


def _rows(t):
    """Row pitch in elements of a 2-D tensor with a contiguous last dim."""
    return t.stride(0) if t.dim() == 2 else t.shape[-1]


def _codebook(cb):
    vals = [float(v) for v in (cb.tolist() if hasattr(cb, "tolist") else cb)]
    if len(vals) != 16:
        raise ValueError("codebook: 16 levels expected")
    return (ctypes.c_float * 16)(*vals)


# ----------------------------------------------------------- step graph

class StepGraph:
    """A fixed sequence of library calls, replayed as one CUDA graph.

    Decode loops make the same calls with the same shapes and buffers for
    every token.  ``fn`` (any mix of ``wobs_*`` calls and tensor copies) runs
    once eagerly on ``stream``, which also sizes the cached workspaces, and is
    then captured; ``replay()`` launches the whole sequence with one graph
    launch on the current stream.  Every buffer the calls touch must stay
    alive and in place while the graph is used; host buffers of copies must
    be pinned.
    """

    def __init__(self, fn, stream=None):
        self.stream = stream if stream is not None else torch.cuda.Stream()
        with torch.cuda.stream(self.stream):
            fn()
        self.stream.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph, stream=self.stream):
            fn()

    def replay(self):
        self.graph.replay()


# ------------------------------------------------------------ workspace

_ws_cache = {}

# Workspace bytes of the argmax state alone (counter, keys, alignment).  A
# larger wobs_workspace_size() means the call splits K and needs the
# workspace even without an argmax.
_WS_HEADER_BYTES = 512


def _auto_ws(op, M, N, K, device, argmax):
    if argmax is None and wobs_workspace_size(op, M, N, K) <= _WS_HEADER_BYTES:
        return None
    return workspace(op, M, N, K, device)


def workspace(op, M, N, K, device=None):
    """A zero-filled workspace for (op, M, N, K) on the current stream.

    Cached per (device, stream) and grown as needed; the library leaves its
    counter region (the first WS_ZERO_BYTES bytes) zero after every
    successful call and overwrites split-K partials before reading them, so
    it is reused as is.  Calls
    that may overlap on the GPU should run on different streams.
    """
    device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    need = wobs_workspace_size(op, M, N, K)
    if need == 0:
        return None
    key = (device.index, torch.cuda.current_stream(device).cuda_stream)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < need:
        buf = torch.zeros(max(need, 4096), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def wobs_workspace_size(op, M, N, K):
    lib = _lib.get()
    return int(lib.wobs_workspace_size(int(op), int(M), int(N), int(K)))


def wobs_version():
    return int(_lib.get().wobs_version())


def wobs_last_error():
    return _lib.get().wobs_last_error().decode(errors="replace")


# ------------------------------------------------------------ entry points

def wobs_bw_probe(buf, grid=0, variant=1, xor_out=None):
    """Streaming read of ``buf`` (uint8 CUDA tensor); returns the uint32 XOR tensor."""
    lib = _lib.get()
    _need(buf, "buf")
    if xor_out is None:
        xor_out = torch.zeros(1, dtype=torch.int32, device=buf.device)
    rc = lib.wobs_bw_probe(_ptr(buf), buf.numel() * buf.element_size(), int(grid), int(variant),
                           _ptr(xor_out), _stream(buf.device))
    _check(rc, lib)
    return xor_out


def wobs_gemv_f16(W, X, Y=None, ws=None):
    """Y[M, N] (fp16) = X[M, K] @ W[N, K]^T with fp32 accumulation."""
    lib = _lib.get()
    _need(W, "W", torch.float16, 2)
    X2 = X if X.dim() == 2 else X.view(1, -1)
    _need(X2, "X", torch.float16, 2, W.device)
    M, K = X2.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError("W and X disagree on K")
    if Y is None:
        Y = torch.empty(M, N, dtype=torch.float16, device=W.device)
    _need(Y, "Y", torch.float16, None, W.device)
    if ws is None:
        ws = _auto_ws(OP_GEMV_F16, M, N, K, W.device, None)
    rc = lib.wobs_gemv_f16(_ptr(W), _rows(W), _ptr(X2), _rows(X2), M, _ptr(Y), N, K, _ptr(ws),
                           ws.numel() if ws is not None else 0, _stream(W.device))
    _check(rc, lib)
    return Y


def wobs_gemv_bf16(W, X, logits=None, argmax=None, want_argmax=False, ws=None):
    """logits[M, N] (fp32) = X[M, K] @ W[N, K]^T; optional fused argmax[M] (int64)."""
    lib = _lib.get()
    _need(W, "W", torch.bfloat16, 2)
    X2 = X if X.dim() == 2 else X.view(1, -1)
    _need(X2, "X", torch.bfloat16, 2, W.device)
    M, K = X2.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError("W and X disagree on K")
    if logits is None:
        logits = torch.empty(M, N, dtype=torch.float32, device=W.device)
    _need(logits, "logits", torch.float32, None, W.device)
    if argmax is None and want_argmax:
        argmax = torch.empty(M, dtype=torch.int64, device=W.device)
    if ws is None:
        ws = _auto_ws(OP_GEMV_BF16, M, N, K, W.device, argmax)
    rc = lib.wobs_gemv_bf16(_ptr(W), _rows(W), _ptr(X2), _rows(X2), M, _ptr(logits), _ptr(argmax),
                            N, K, _ptr(ws), ws.numel() if ws is not None else 0, _stream(W.device))
    _check(rc, lib)
    return logits, argmax


def wobs_gemv_bf16_noalloc(W, X, logits=None, argmax=None, want_argmax=False):
    """wobs_gemv_bf16 with the library's fixed scratch in place of a workspace.

    For callers that may not allocate device memory at call time (an engine
    that reserved its memory budget up front and owns every allocation, a
    plugin whose host process accounts all device memory).  Pass
    preallocated ``logits`` / ``argmax`` to allocate nothing here either.
    Calls that may overlap on the GPU share the scratch and must not be issued.
    """
    lib = _lib.get()
    _need(W, "W", torch.bfloat16, 2)
    X2 = X if X.dim() == 2 else X.view(1, -1)
    _need(X2, "X", torch.bfloat16, 2, W.device)
    M, K = X2.shape
    N = W.shape[0]
    if W.shape[1] != K:
        raise ValueError("W and X disagree on K")
    if logits is None:
        logits = torch.empty(M, N, dtype=torch.float32, device=W.device)
    _need(logits, "logits", torch.float32, None, W.device)
    if argmax is None and want_argmax:
        argmax = torch.empty(M, dtype=torch.int64, device=W.device)
    rc = lib.wobs_gemv_bf16_noalloc(_ptr(W), _rows(W), _ptr(X2), _rows(X2), M, _ptr(logits),
                                    _ptr(argmax), N, K, _stream(W.device))
    _check(rc, lib)
    return logits, argmax


def wobs_quantize_q8_1(X, xq=None):
    """Q8_1 blocks of fp32 activations X[M, K]: uint8 [M, K/32*36]."""
    lib = _lib.get()
    X2 = X if X.dim() == 2 else X.view(1, -1)
    _need(X2, "X", torch.float32, 2)
    M, K = X2.shape
    if xq is None:
        xq = torch.empty(M, (K // 32) * Q8_1_BLOCK_BYTES, dtype=torch.uint8, device=X2.device)
    _need(xq, "xq", torch.uint8, None, X2.device)
    rc = lib.wobs_quantize_q8_1(_ptr(X2), _rows(X2), M, K, _ptr(xq), _stream(X2.device))
    _check(rc, lib)
    return xq


def wobs_quantize_q4_0(W, qs=None, d=None):
    """Q4_0 planes of fp32 weights W[N, K]: (qs uint8 [N, K/2], d fp16 [N, K/32])."""
    lib = _lib.get()
    _need(W, "W", torch.float32, 2)
    N, K = W.shape
    if qs is None:
        qs = torch.empty(N, K // 2, dtype=torch.uint8, device=W.device)
    if d is None:
        d = torch.empty(N, K // 32, dtype=torch.float16, device=W.device)
    _need(qs, "qs", torch.uint8, 2, W.device)
    _need(d, "d", torch.float16, 2, W.device)
    rc = lib.wobs_quantize_q4_0(_ptr(W), _rows(W), N, K, _ptr(qs), _ptr(d), _stream(W.device))
    _check(rc, lib)
    return qs, d


def wobs_quantize_nf4(W, codebook, qs=None, absmax=None):
    """NF4 planes of bf16 weights W[N, K]: (qs uint8 [N, K/2], absmax fp32 [N, K/64])."""
    lib = _lib.get()
    _need(W, "W", torch.bfloat16, 2)
    N, K = W.shape
    if qs is None:
        qs = torch.empty(N, K // 2, dtype=torch.uint8, device=W.device)
    if absmax is None:
        absmax = torch.empty(N, K // 64, dtype=torch.float32, device=W.device)
    _need(qs, "qs", torch.uint8, 2, W.device)
    _need(absmax, "absmax", torch.float32, 2, W.device)
    rc = lib.wobs_quantize_nf4(_ptr(W), _rows(W), N, K, _codebook(codebook), _ptr(qs),
                               _ptr(absmax), _stream(W.device))
    _check(rc, lib)
    return qs, absmax


def wobs_gemv_q4_0_q8_1(qs, d, xq, y=None, argmax=None, want_argmax=False, ws=None):
    """y[M, N] (fp32) from Q4_0 planes (qs [N, K/2], d [N, K/32]) and Q8_1 blocks xq [M, ...]."""
    lib = _lib.get()
    _need(qs, "qs", torch.uint8, 2)
    _need(d, "d", torch.float16, 2, qs.device)
    xq2 = xq if xq.dim() == 2 else xq.view(1, -1)
    _need(xq2, "xq", torch.uint8, 2, qs.device)
    N, K = qs.shape[0], qs.shape[1] * 2
    M = xq2.shape[0]
    if xq2.shape[1] != (K // 32) * Q8_1_BLOCK_BYTES or not xq2.is_contiguous():
        raise ValueError("xq must be contiguous [M, K/32*36]")
    if not (qs.is_contiguous() and d.is_contiguous()) or d.shape != (N, K // 32):
        raise ValueError("qs/d must be contiguous planes [N, K/2] and [N, K/32]")
    if y is None:
        y = torch.empty(M, N, dtype=torch.float32, device=qs.device)
    _need(y, "y", torch.float32, None, qs.device)
    if argmax is None and want_argmax:
        argmax = torch.empty(M, dtype=torch.int64, device=qs.device)
    if ws is None:
        ws = _auto_ws(OP_GEMV_Q4_0_Q8_1, M, N, K, qs.device, argmax)
    rc = lib.wobs_gemv_q4_0_q8_1(_ptr(qs), _ptr(d), _ptr(xq2), M, _ptr(y), _ptr(argmax), N, K,
                                 _ptr(ws), ws.numel() if ws is not None else 0,
                                 _stream(qs.device))
    _check(rc, lib)
    return y, argmax


def wobs_gemv_q4_0_f32(qs, d, x, y=None, argmax=None, want_argmax=False, ws=None, xq_out=None):
    """y[1, N] (fp32) from Q4_0 planes and one fp32 activation vector x [K] (or [1, K]),
    quantised to Q8_1 inside the GEMV kernel; the Q8_1 blocks are also written to
    ``xq_out`` (uint8, K/32*36 bytes) when it is given."""
    lib = _lib.get()
    _need(qs, "qs", torch.uint8, 2)
    _need(d, "d", torch.float16, 2, qs.device)
    x1 = x.reshape(-1) if x.dim() == 2 and x.shape[0] == 1 else x
    _need(x1, "x", torch.float32, 1, qs.device)
    N, K = qs.shape[0], qs.shape[1] * 2
    if x1.shape[0] != K or not x1.is_contiguous():
        raise ValueError("x must be a contiguous fp32 vector of K elements")
    if not (qs.is_contiguous() and d.is_contiguous()) or d.shape != (N, K // 32):
        raise ValueError("qs/d must be contiguous planes [N, K/2] and [N, K/32]")
    if y is None:
        y = torch.empty(1, N, dtype=torch.float32, device=qs.device)
    _need(y, "y", torch.float32, None, qs.device)
    if argmax is None and want_argmax:
        argmax = torch.empty(1, dtype=torch.int64, device=qs.device)
    if xq_out is not None:
        _need(xq_out, "xq_out", torch.uint8, None, qs.device)
        if xq_out.numel() < (K // 32) * Q8_1_BLOCK_BYTES or not xq_out.is_contiguous():
            raise ValueError("xq_out must be a contiguous uint8 buffer of K/32*36 bytes")
    if ws is None:
        ws = _auto_ws(OP_GEMV_Q4_0_F32, 1, N, K, qs.device, argmax)
    rc = lib.wobs_gemv_q4_0_f32(_ptr(qs), _ptr(d), _ptr(x1), _ptr(xq_out), _ptr(y), _ptr(argmax), N, K,
                                _ptr(ws), ws.numel() if ws is not None else 0, _stream(qs.device))
    _check(rc, lib)
    return y, argmax


def wobs_quantize_q8_0(W, qs=None, d=None):
    """Q8_0 planes of fp32 weights W[N, K]: (qs int8 [N, K], d fp16 [N, K/32])."""
    lib = _lib.get()
    _need(W, "W", torch.float32, 2)
    N, K = W.shape
    if qs is None:
        qs = torch.empty(N, K, dtype=torch.int8, device=W.device)
    if d is None:
        d = torch.empty(N, K // 32, dtype=torch.float16, device=W.device)
    _need(qs, "qs", torch.int8, 2, W.device)
    _need(d, "d", torch.float16, 2, W.device)
    rc = lib.wobs_quantize_q8_0(_ptr(W), _rows(W), N, K, _ptr(qs), _ptr(d), _stream(W.device))
    _check(rc, lib)
    return qs, d


def wobs_gemv_q8_0_q8_1(qs, d, xq, y=None, argmax=None, want_argmax=False, ws=None):
    """y[M, N] (fp32) from Q8_0 planes (qs int8 [N, K], d [N, K/32]) and Q8_1 blocks xq [M, ...]."""
    lib = _lib.get()
    _need(qs, "qs", torch.int8, 2)
    _need(d, "d", torch.float16, 2, qs.device)
    xq2 = xq if xq.dim() == 2 else xq.view(1, -1)
    _need(xq2, "xq", torch.uint8, 2, qs.device)
    N, K = qs.shape
    M = xq2.shape[0]
    if xq2.shape[1] != (K // 32) * Q8_1_BLOCK_BYTES or not xq2.is_contiguous():
        raise ValueError("xq must be contiguous [M, K/32*36]")
    if not (qs.is_contiguous() and d.is_contiguous()) or d.shape != (N, K // 32):
        raise ValueError("qs/d must be contiguous planes [N, K] and [N, K/32]")
    if y is None:
        y = torch.empty(M, N, dtype=torch.float32, device=qs.device)
    _need(y, "y", torch.float32, None, qs.device)
    if argmax is None and want_argmax:
        argmax = torch.empty(M, dtype=torch.int64, device=qs.device)
    if ws is None:
        ws = _auto_ws(OP_GEMV_Q8_0_Q8_1, M, N, K, qs.device, argmax)
    rc = lib.wobs_gemv_q8_0_q8_1(_ptr(qs), _ptr(d), _ptr(xq2), M, _ptr(y), _ptr(argmax), N, K,
                                 _ptr(ws), ws.numel() if ws is not None else 0,
                                 _stream(qs.device))
    _check(rc, lib)
    return y, argmax


def wobs_gemv_q8_0_f32(qs, d, x, y=None, argmax=None, want_argmax=False, ws=None, xq_out=None):
    """y[1, N] (fp32) from Q8_0 planes (qs int8 [N, K], d [N, K/32]) and one fp32 activation
    vector x [K] (or [1, K]), quantised to Q8_1 inside the GEMV kernel; the Q8_1 blocks are
    also written to ``xq_out`` (uint8, K/32*36 bytes) when it is given."""
    lib = _lib.get()
    _need(qs, "qs", torch.int8, 2)
    _need(d, "d", torch.float16, 2, qs.device)
    x1 = x.reshape(-1) if x.dim() == 2 and x.shape[0] == 1 else x
    _need(x1, "x", torch.float32, 1, qs.device)
    N, K = qs.shape
    if x1.shape[0] != K or not x1.is_contiguous():
        raise ValueError("x must be a contiguous fp32 vector of K elements")
    if not (qs.is_contiguous() and d.is_contiguous()) or d.shape != (N, K // 32):
        raise ValueError("qs/d must be contiguous planes [N, K] and [N, K/32]")
    if y is None:
        y = torch.empty(1, N, dtype=torch.float32, device=qs.device)
    _need(y, "y", torch.float32, None, qs.device)
    if argmax is None and want_argmax:
        argmax = torch.empty(1, dtype=torch.int64, device=qs.device)
    if xq_out is not None:
        _need(xq_out, "xq_out", torch.uint8, None, qs.device)
        if xq_out.numel() < (K // 32) * Q8_1_BLOCK_BYTES or not xq_out.is_contiguous():
            raise ValueError("xq_out must be a contiguous uint8 buffer of K/32*36 bytes")
    if ws is None:
        ws = _auto_ws(OP_GEMV_Q8_0_F32, 1, N, K, qs.device, argmax)
    rc = lib.wobs_gemv_q8_0_f32(_ptr(qs), _ptr(d), _ptr(x1), _ptr(xq_out), _ptr(y), _ptr(argmax), N, K,
                                _ptr(ws), ws.numel() if ws is not None else 0, _stream(qs.device))
    _check(rc, lib)
    return y, argmax


def wobs_gemv_nf4(qs, absmax, codebook, x, y=None, argmax=None, want_argmax=False, ws=None):
    """NF4 GEMV: bf16 y from NF4 planes (qs [N, K/2], absmax [N, K/64]).

    ``x`` is bf16 [K] (one column; y is [N]) or [M, K] (M columns, 1 <= M <=
    32; y is [M, N]); ``argmax`` is int64 [M].
    """
    lib = _lib.get()
    _need(qs, "qs", torch.uint8, 2)
    _need(absmax, "absmax", torch.float32, 2, qs.device)
    one = x.dim() == 1
    X2 = x.view(1, -1) if one else x
    _need(X2, "x", torch.bfloat16, 2, qs.device)
    N, K = qs.shape[0], qs.shape[1] * 2
    M = X2.shape[0]
    if X2.shape[1] != K or not (qs.is_contiguous() and absmax.is_contiguous()):
        raise ValueError("x must have K elements per column; planes must be contiguous")
    if y is None:
        y = torch.empty((N,) if one else (M, N), dtype=torch.bfloat16, device=qs.device)
    _need(y, "y", torch.bfloat16, None, qs.device)
    if y.numel() != M * N or not y.is_contiguous():
        raise ValueError("y must be a contiguous [M, N] bf16 tensor")
    if argmax is None and want_argmax:
        argmax = torch.empty(M, dtype=torch.int64, device=qs.device)
    if ws is None:
        ws = _auto_ws(OP_GEMV_NF4, M, N, K, qs.device, argmax)
    rc = lib.wobs_gemv_nf4(_ptr(qs), _ptr(absmax), _codebook(codebook), _ptr(X2), _rows(X2), M,
                           _ptr(y), _ptr(argmax), N, K, _ptr(ws), ws.numel() if ws is not None else 0,
                           _stream(qs.device))
    _check(rc, lib)
    return y, argmax


def wobs_dequantize_nf4(qs, absmax, codebook, W=None):
    """bf16 W [N, K] = absmax * codebook[code] (fp32 product, rounded to bf16)."""
    lib = _lib.get()
    _need(qs, "qs", torch.uint8, 2)
    _need(absmax, "absmax", torch.float32, 2, qs.device)
    N, K = qs.shape[0], qs.shape[1] * 2
    if not (qs.is_contiguous() and absmax.is_contiguous()):
        raise ValueError("planes must be contiguous")
    if W is None:
        W = torch.empty(N, K, dtype=torch.bfloat16, device=qs.device)
    _need(W, "W", torch.bfloat16, 2, qs.device)
    rc = lib.wobs_dequantize_nf4(_ptr(qs), _ptr(absmax), _codebook(codebook), N, K, _ptr(W), _rows(W),
                                 _stream(qs.device))
    _check(rc, lib)
    return W


def nf4_dequant_gemm(qs, absmax, codebook, X, W=None, logits=None):
    """The dequantise-then-GEMM path: wobs_dequantize_nf4 into ``W`` (bf16
    [N, K], allocated if not given), then the dense bf16 GEMV
    (wobs_gemv_bf16) over the columns of X (bf16 [M, K]) in calls of at most
    32 columns.  Returns fp32 logits [M, N] and W."""
    W = wobs_dequantize_nf4(qs, absmax, codebook, W)
    X2 = X.view(1, -1) if X.dim() == 1 else X
    _need(X2, "X", torch.bfloat16, 2, qs.device)
    M = X2.shape[0]
    N = W.shape[0]
    if logits is None:
        logits = torch.empty(M, N, dtype=torch.float32, device=qs.device)
    for m0 in range(0, M, MAX_M):
        m1 = min(M, m0 + MAX_M)
        wobs_gemv_bf16(W, X2[m0:m1], logits=logits[m0:m1])
    return logits, W


def _argcmp(name, X, out, ws):
    lib = _lib.get()
    X2 = X if X.dim() == 2 else X.view(1, -1)
    _need(X2, "X", None, 2)
    if X2.dtype not in DTYPE_CODES:
        raise TypeError(f"X: dtype {X2.dtype}, expected float16, bfloat16 or float32")
    M, N = X2.shape
    if out is None:
        out = torch.empty(M, dtype=torch.int64, device=X2.device)
    _need(out, "out", torch.int64, None, X2.device)
    if ws is None:
        need = wobs_workspace_size(OP_ARGCMP, M, N, X2.element_size())
        ws = workspace(OP_ARGCMP, M, N, X2.element_size(), X2.device) if need else None
    rc = getattr(lib, name)(DTYPE_CODES[X2.dtype], _ptr(X2), _rows(X2), M, N, _ptr(out), _ptr(ws),
                            ws.numel() if ws is not None else 0, _stream(X2.device))
    _check(rc, lib)
    return out


def wobs_argmax(X, out=None, ws=None):
    """int64 [M]: index of the largest element of each row of X [M, N] (lowest on ties)."""
    return _argcmp("wobs_argmax", X, out, ws)


def wobs_argmin(X, out=None, ws=None):
    """int64 [M]: index of the smallest element of each row of X [M, N] (lowest on ties)."""
    return _argcmp("wobs_argmin", X, out, ws)


def wobs_q4_0_q8_1_blockdots(qs, xq):
    """Exact int32 block dots [M, N, K/32] (test export)."""
    lib = _lib.get()
    _need(qs, "qs", torch.uint8, 2)
    xq2 = xq if xq.dim() == 2 else xq.view(1, -1)
    _need(xq2, "xq", torch.uint8, 2, qs.device)
    N, K = qs.shape[0], qs.shape[1] * 2
    M = xq2.shape[0]
    out = torch.empty(M, N, K // 32, dtype=torch.int32, device=qs.device)
    rc = lib.wobs_q4_0_q8_1_blockdots(_ptr(qs), _ptr(xq2), M, N, K, _ptr(out), _stream(qs.device))
    _check(rc, lib)
    return out


def wobs_selftest_wait_timeout(limit_cycles=1_000_000, device=None):
    """Launch the failure-path self test (a wait that gives up); returns nothing."""
    lib = _lib.get()
    device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    _check(lib.wobs_selftest_wait_timeout(int(limit_cycles), _stream(device)), lib)


def wobs_error_word(device=None):
    """Read and clear the device error word (synchronises the current stream)."""
    lib = _lib.get()
    device = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    v = ctypes.c_int(0)
    rc = lib.wobs_error_word(_stream(device), ctypes.byref(v))
    if rc != ERR_DEVICE_TIMEOUT:       # a recorded timeout is the value asked for
        _check(rc, lib)
    return v.value

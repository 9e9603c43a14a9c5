"""Thin Python binding of libbq.so (the C ABI declared in include/bq.h).

Argument marshalling only: every function checks the torch tensors it is
given, passes their device pointers, sizes and the current CUDA stream to
the C entry point of the same name, and raises ``BqError`` on a non-OK
status.  All arithmetic runs in the library's CUDA kernels; there is no
CPU fallback -- if the library is not built, importing the binding works
but every call raises.
"""

from __future__ import annotations

import ctypes
import os
import re

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libbq.so")
HEADER = os.path.join(os.path.dirname(PKG_DIR), "include", "bq.h")

BQ_OK, BQ_ERR_INVALID_ARG, BQ_ERR_UNSUPPORTED, BQ_ERR_ALIGNMENT, BQ_ERR_CUDA, BQ_ERR_TIMEOUT = range(6)
BQ_F16, BQ_F32 = 0, 1
LAYOUT_PLAIN, LAYOUT_INTERLEAVED = 0, 1
ROUND_F32DIV, ROUND_BMINF_HALF = 0, 1
LAYOUTS = {"plain": LAYOUT_PLAIN, "interleaved": LAYOUT_INTERLEAVED}
ACT_NONE, ACT_RELU, ACT_GELU = 0, 1, 2
ACTIVATIONS = {"none": ACT_NONE, "relu": ACT_RELU, "gelu": ACT_GELU}

_c_i64 = ctypes.c_int64
_vp = ctypes.c_void_p

_SIGNATURES = {
    "bq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "bq_quantize_sym": (ctypes.c_int, [_vp, ctypes.c_int, _c_i64, _c_i64, _c_i64, ctypes.c_int, ctypes.c_int,
                                       _vp, _vp, _vp]),
    "bq_packed_size": (ctypes.c_size_t, [_c_i64, _c_i64, ctypes.c_int, ctypes.c_int]),
    "bq_pack_weights": (ctypes.c_int, [_vp, _c_i64, _c_i64, ctypes.c_int, ctypes.c_int, _vp, _vp]),
    "bq_gemm_i8xi8": (ctypes.c_int, [_vp, _vp, _c_i64, _c_i64, _c_i64, _vp, _vp, _vp, _vp]),
    "bq_gemm_i8xi4": (ctypes.c_int, [_vp, _vp, ctypes.c_int, _c_i64, _c_i64, _c_i64, _vp, _vp, _vp, _vp]),
    "bq_gemm_i8xi2": (ctypes.c_int, [_vp, _vp, ctypes.c_int, _c_i64, _c_i64, _c_i64, _vp, _vp, _vp, _vp]),
    "bq_gemm_f16xi4": (ctypes.c_int, [_vp, _vp, ctypes.c_int, _c_i64, _c_i64, _c_i64, _vp, _vp, _vp]),
    "bq_gemm_i8xi8_act": (ctypes.c_int, [_vp, _vp, _c_i64, _c_i64, _c_i64, _vp, _vp, ctypes.c_int, _vp, _vp]),
    "bq_gemm_i8xi4_act": (ctypes.c_int, [_vp, _vp, ctypes.c_int, _c_i64, _c_i64, _c_i64, _vp, _vp, ctypes.c_int,
                                         _vp, _vp]),
    "bq_gemm_i8xi2_act": (ctypes.c_int, [_vp, _vp, ctypes.c_int, _c_i64, _c_i64, _c_i64, _vp, _vp, ctypes.c_int,
                                         _vp, _vp]),
    "bq_gemm_f16xi4_act": (ctypes.c_int, [_vp, _vp, ctypes.c_int, _c_i64, _c_i64, _c_i64, _vp, ctypes.c_int, _vp,
                                          _vp]),
    "bq_gemm_i8xi8_batched": (ctypes.c_int, [_vp, _c_i64, _vp, _c_i64, _c_i64, _c_i64, _c_i64, _c_i64, _vp, _c_i64,
                                             _vp, _c_i64, ctypes.c_int, _vp, _c_i64, _vp]),
    "bq_gemm_i8xi4_batched": (ctypes.c_int, [_vp, _c_i64, _vp, _c_i64, ctypes.c_int, _c_i64, _c_i64, _c_i64, _c_i64,
                                             _vp, _c_i64, _vp, _c_i64, ctypes.c_int, _vp, _c_i64, _vp]),
    "bq_gemm_i8xi2_batched": (ctypes.c_int, [_vp, _c_i64, _vp, _c_i64, ctypes.c_int, _c_i64, _c_i64, _c_i64, _c_i64,
                                             _vp, _c_i64, _vp, _c_i64, ctypes.c_int, _vp, _c_i64, _vp]),
    "bq_gemm_f16xi4_batched": (ctypes.c_int, [_vp, _c_i64, _vp, _c_i64, ctypes.c_int, _c_i64, _c_i64, _c_i64, _c_i64,
                                              _vp, _c_i64, ctypes.c_int, _vp, _c_i64, _vp]),
    "bq_quantized_linear": (ctypes.c_int, [_vp, _c_i64, _c_i64, _vp, ctypes.c_int, ctypes.c_int, _c_i64, _vp,
                                           ctypes.c_int, _vp, _vp, _vp]),
    "bq_gemm_f16xu4_zp": (ctypes.c_int, [_vp, _vp, ctypes.c_int, _c_i64, _c_i64, _c_i64, _vp, _vp, ctypes.c_int,
                                         _vp, _vp, _vp]),
    "bq_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int), ctypes.c_int]),
    "bq_set_wait_timeout_ns": (_c_i64, [_c_i64]),
}

_lib = None


class BqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {bq_status_string(status)} ({status})")


def lib() -> ctypes.CDLL:
    """Load libbq.so once; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libbq.so is not built ({LIB_PATH}); run quantized_mixed_precision_gb300.build")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def header_functions() -> list[str]:
    """Names of the functions include/bq.h declares."""
    with open(HEADER, encoding="utf-8") as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\*?\s+\*?(bq_\w+)\s*\(", text, re.M)))


def bq_status_string(status: int) -> str:
    return lib().bq_status_string(status).decode()


def _check(status: int, where: str):
    if status != BQ_OK:
        raise BqError(status, where)


# ----------------------------------------------------------------------------
# torch marshalling helpers
# ----------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _stream(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name, ndim=None):
    torch = _torch()
    if t is None:
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _layout(layout):
    return LAYOUTS[layout] if isinstance(layout, str) else int(layout)


def _activation(activation):
    return ACTIVATIONS[activation] if isinstance(activation, str) else int(activation)


# ----------------------------------------------------------------------------
# Entry points
# ----------------------------------------------------------------------------
def bq_quantize_sym(x, bits=8, mode=ROUND_F32DIV, q=None, scale=None, stream=None):
    """Per-row symmetric quantisation of a 2-D fp16/fp32 CUDA tensor -> (int8 codes, fp16 scale)."""
    torch = _torch()
    if x.dim() != 2 or x.stride(1) != 1:
        raise ValueError("x must be 2-D with unit column stride")
    xtype = {torch.float16: BQ_F16, torch.float32: BQ_F32}[x.dtype]
    rows, cols = x.shape
    if q is None:
        q = torch.empty((rows, cols), dtype=torch.int8, device=x.device)
    if scale is None:
        scale = torch.empty((rows,), dtype=torch.float16, device=x.device)
    _need(q, torch.int8, "q", 2)
    _need(scale, torch.float16, "scale", 1)
    st = lib().bq_quantize_sym(_ptr(x), xtype, rows, cols, x.stride(0), int(bits), int(mode), _ptr(q),
                               _ptr(scale), _stream(stream))
    _check(st, "bq_quantize_sym")
    return q, scale


def bq_packed_size(n, k, bits, layout=LAYOUT_INTERLEAVED) -> int:
    return int(lib().bq_packed_size(int(n), int(k), int(bits), _layout(layout)))


def bq_pack_weights(q, bits, layout=LAYOUT_INTERLEAVED, out=None, stream=None):
    """Pack int8 codes (n, k) into (n, k*bits/8) bytes."""
    torch = _torch()
    _need(q, torch.int8, "q", 2)
    n, k = q.shape
    lay = _layout(layout)
    if out is None:
        out = torch.empty((n, k * bits // 8), dtype=torch.uint8, device=q.device)
    _need(out, torch.uint8, "out")
    st = lib().bq_pack_weights(_ptr(q), n, k, int(bits), lay, _ptr(out), _stream(stream))
    _check(st, "bq_pack_weights")
    return out


def _gemm_out(M, N, scaled, out, device):
    torch = _torch()
    dtype = torch.float16 if scaled else torch.int32
    if out is None:
        out = torch.empty((M, N), dtype=dtype, device=device)
    _need(out, dtype, "out", 2)
    return out


def bq_gemm_i8xi8(A, B, row_scale=None, col_scale=None, out=None, stream=None):
    torch = _torch()
    _need(A, torch.int8, "A", 2)
    _need(B, torch.int8, "B", 2)
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K:
        raise ValueError("K mismatch")
    out = _gemm_out(M, N, col_scale is not None, out, A.device)
    st = lib().bq_gemm_i8xi8(_ptr(A), _ptr(B), M, N, K, _ptr(row_scale), _ptr(col_scale), _ptr(out),
                             _stream(stream))
    _check(st, "bq_gemm_i8xi8")
    return out


def _gemm_packed(fn_name, bits, A, Bp, layout, row_scale, col_scale, out, stream):
    torch = _torch()
    _need(A, torch.int8, "A", 2)
    _need(Bp, torch.uint8, "Bp", 2)
    M, K = A.shape
    N = Bp.shape[0]
    if Bp.shape[1] * 8 != K * bits:
        raise ValueError("packed width does not match K")
    out = _gemm_out(M, N, col_scale is not None, out, A.device)
    st = getattr(lib(), fn_name)(_ptr(A), _ptr(Bp), _layout(layout), M, N, K, _ptr(row_scale), _ptr(col_scale),
                                 _ptr(out), _stream(stream))
    _check(st, fn_name)
    return out


def bq_gemm_i8xi4(A, Bp, layout=LAYOUT_INTERLEAVED, row_scale=None, col_scale=None, out=None, stream=None):
    return _gemm_packed("bq_gemm_i8xi4", 4, A, Bp, layout, row_scale, col_scale, out, stream)


def bq_gemm_i8xi2(A, Bp, layout=LAYOUT_INTERLEAVED, row_scale=None, col_scale=None, out=None, stream=None):
    return _gemm_packed("bq_gemm_i8xi2", 2, A, Bp, layout, row_scale, col_scale, out, stream)


def bq_gemm_f16xi4(X, Wp, col_scale, layout=LAYOUT_INTERLEAVED, out=None, stream=None):
    torch = _torch()
    _need(X, torch.float16, "X", 2)
    _need(Wp, torch.uint8, "Wp", 2)
    _need(col_scale, torch.float16, "col_scale", 1)
    M, K = X.shape
    N = Wp.shape[0]
    if Wp.shape[1] * 2 != K:
        raise ValueError("packed width does not match K")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=X.device)
    _need(out, torch.float16, "out", 2)
    st = lib().bq_gemm_f16xi4(_ptr(X), _ptr(Wp), _layout(layout), M, N, K, _ptr(col_scale), _ptr(out),
                              _stream(stream))
    _check(st, "bq_gemm_f16xi4")
    return out


def bq_gemm_i8xi8_act(A, B, activation, row_scale=None, col_scale=None, out=None, stream=None):
    """int8 x int8 GEMM with the fp16 dequantisation and a fused activation ("none", "relu", "gelu")."""
    torch = _torch()
    _need(A, torch.int8, "A", 2)
    _need(B, torch.int8, "B", 2)
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K:
        raise ValueError("K mismatch")
    out = _gemm_out(M, N, col_scale is not None, out, A.device)
    st = lib().bq_gemm_i8xi8_act(_ptr(A), _ptr(B), M, N, K, _ptr(row_scale), _ptr(col_scale),
                                 _activation(activation), _ptr(out), _stream(stream))
    _check(st, "bq_gemm_i8xi8_act")
    return out


def _gemm_packed_act(fn_name, bits, A, Bp, layout, activation, row_scale, col_scale, out, stream):
    torch = _torch()
    _need(A, torch.int8, "A", 2)
    _need(Bp, torch.uint8, "Bp", 2)
    M, K = A.shape
    N = Bp.shape[0]
    if Bp.shape[1] * 8 != K * bits:
        raise ValueError("packed width does not match K")
    out = _gemm_out(M, N, col_scale is not None, out, A.device)
    st = getattr(lib(), fn_name)(_ptr(A), _ptr(Bp), _layout(layout), M, N, K, _ptr(row_scale), _ptr(col_scale),
                                 _activation(activation), _ptr(out), _stream(stream))
    _check(st, fn_name)
    return out


def bq_gemm_i8xi4_act(A, Bp, activation, layout=LAYOUT_INTERLEAVED, row_scale=None, col_scale=None, out=None,
                      stream=None):
    return _gemm_packed_act("bq_gemm_i8xi4_act", 4, A, Bp, layout, activation, row_scale, col_scale, out, stream)


def bq_gemm_i8xi2_act(A, Bp, activation, layout=LAYOUT_INTERLEAVED, row_scale=None, col_scale=None, out=None,
                      stream=None):
    return _gemm_packed_act("bq_gemm_i8xi2_act", 2, A, Bp, layout, activation, row_scale, col_scale, out, stream)


def bq_gemm_f16xi4_act(X, Wp, col_scale, activation, layout=LAYOUT_INTERLEAVED, out=None, stream=None):
    torch = _torch()
    _need(X, torch.float16, "X", 2)
    _need(Wp, torch.uint8, "Wp", 2)
    _need(col_scale, torch.float16, "col_scale", 1)
    M, K = X.shape
    N = Wp.shape[0]
    if Wp.shape[1] * 2 != K:
        raise ValueError("packed width does not match K")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=X.device)
    _need(out, torch.float16, "out", 2)
    st = lib().bq_gemm_f16xi4_act(_ptr(X), _ptr(Wp), _layout(layout), M, N, K, _ptr(col_scale),
                                  _activation(activation), _ptr(out), _stream(stream))
    _check(st, "bq_gemm_f16xi4_act")
    return out


def _batch_stride(t, batch, name):
    """Element stride between the batch items of an operand whose first
    dimension is its batch; a batch of 1 is shared by every item (stride 0)."""
    lead = t.shape[0]
    if lead not in (1, batch):
        raise ValueError(f"{name}: batch dimension {lead} is neither 1 nor {batch}")
    return 0 if lead == 1 else t[0].numel()


def _scale_stride(t, batch, name):
    """Scales are (n,) -- shared by every item -- or (batch or 1, n)."""
    if t is None or t.dim() == 1:
        return 0
    return _batch_stride(t, batch, name)


def _batched(fn_name, A, Bw, bits, layout, row_scale, col_scale, activation, out, stream, act_type):
    torch = _torch()
    _need(A, act_type, "A", 3)
    _need(Bw, torch.int8 if bits == 8 else torch.uint8, "B", 3)
    batch = max(A.shape[0], Bw.shape[0])
    M, K = A.shape[1], A.shape[2]
    N = Bw.shape[1]
    if Bw.shape[2] * 8 != K * bits:
        raise ValueError("weight width does not match K")
    for t, nm in ((row_scale, "row_scale"), (col_scale, "col_scale")):
        if t is not None:
            _need(t, torch.float16, nm)
    scaled = col_scale is not None
    dtype = torch.float16 if scaled else torch.int32
    if out is None:
        out = torch.empty((batch, M, N), dtype=dtype, device=A.device)
    _need(out, dtype, "out", 3)
    sa = _batch_stride(A, batch, "A")
    sb = _batch_stride(Bw, batch, "B")
    srs = _scale_stride(row_scale, batch, "row_scale")
    scs = _scale_stride(col_scale, batch, "col_scale")
    sc = M * N
    f = getattr(lib(), fn_name)
    if fn_name == "bq_gemm_f16xi4_batched":
        st = f(_ptr(A), sa, _ptr(Bw), sb, _layout(layout), batch, M, N, K, _ptr(col_scale), scs,
               _activation(activation), _ptr(out), sc, _stream(stream))
    elif fn_name == "bq_gemm_i8xi8_batched":
        st = f(_ptr(A), sa, _ptr(Bw), sb, batch, M, N, K, _ptr(row_scale), srs, _ptr(col_scale), scs,
               _activation(activation), _ptr(out), sc, _stream(stream))
    else:
        st = f(_ptr(A), sa, _ptr(Bw), sb, _layout(layout), batch, M, N, K, _ptr(row_scale), srs, _ptr(col_scale),
               scs, _activation(activation), _ptr(out), sc, _stream(stream))
    _check(st, fn_name)
    return out


def bq_gemm_i8xi8_batched(A, B, row_scale=None, col_scale=None, activation="none", out=None, stream=None):
    """A (Ba, M, K) int8, B (Bb, N, K) int8 with Ba, Bb in {1, batch} (1 = shared by every item);
    scales (batch or 1, M / N) or (M,) / (N,); out (batch, M, N)."""
    return _batched("bq_gemm_i8xi8_batched", A, B, 8, LAYOUT_PLAIN, row_scale, col_scale, activation, out, stream,
                    _torch().int8)


def bq_gemm_i8xi4_batched(A, Bp, layout=LAYOUT_INTERLEAVED, row_scale=None, col_scale=None, activation="none",
                          out=None, stream=None):
    return _batched("bq_gemm_i8xi4_batched", A, Bp, 4, layout, row_scale, col_scale, activation, out, stream,
                    _torch().int8)


def bq_gemm_i8xi2_batched(A, Bp, layout=LAYOUT_INTERLEAVED, row_scale=None, col_scale=None, activation="none",
                          out=None, stream=None):
    return _batched("bq_gemm_i8xi2_batched", A, Bp, 2, layout, row_scale, col_scale, activation, out, stream,
                    _torch().int8)


def bq_gemm_f16xi4_batched(X, Wp, col_scale, layout=LAYOUT_INTERLEAVED, activation="none", out=None, stream=None):
    return _batched("bq_gemm_f16xi4_batched", X, Wp, 4, layout, None, col_scale, activation, out, stream,
                    _torch().float16)


def bq_quantized_linear(X, W, bits, w_scale, layout=LAYOUT_INTERLEAVED, activation="none", out=None,
                        x_scale=None, stream=None):
    """Fused quantised linear: X fp16 (M, K) quantised per row to int8 inside the
    GEMM against weights W (N, K) (int8 codes, or packed 4- / 2-bit codes in
    ``layout``) with per-column fp16 ``w_scale``.  Returns (Y fp16 (M, N),
    x_scale fp16 (M,))."""
    torch = _torch()
    _need(X, torch.float16, "X", 2)
    _need(W, torch.int8 if bits == 8 else torch.uint8, "W", 2)
    _need(w_scale, torch.float16, "w_scale", 1)
    M, K = X.shape
    N = W.shape[0]
    if W.shape[1] * 8 != K * bits:
        raise ValueError("weight width does not match K")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=X.device)
    if x_scale is None:
        x_scale = torch.empty((M,), dtype=torch.float16, device=X.device)
    _need(out, torch.float16, "out", 2)
    _need(x_scale, torch.float16, "x_scale", 1)
    st = lib().bq_quantized_linear(_ptr(X), M, K, _ptr(W), int(bits), _layout(layout), N, _ptr(w_scale),
                                   _activation(activation), _ptr(x_scale), _ptr(out), _stream(stream))
    _check(st, "bq_quantized_linear")
    return out, x_scale


def bq_gemm_f16xu4_zp(X, Wp, col_scale, zero_point, layout=LAYOUT_INTERLEAVED, activation="none", out=None,
                      row_sum=None, stream=None):
    """fp16 X (M, K) times unsigned 4-bit weights Wp (N, K // 2 bytes) with a
    per-column fp16 scale and zero point.  Returns (Y fp16 (M, N), row_sum
    fp32 (M,))."""
    torch = _torch()
    _need(X, torch.float16, "X", 2)
    _need(Wp, torch.uint8, "Wp", 2)
    _need(col_scale, torch.float16, "col_scale", 1)
    _need(zero_point, torch.float16, "zero_point", 1)
    M, K = X.shape
    N = Wp.shape[0]
    if Wp.shape[1] * 2 != K:
        raise ValueError("packed width does not match K")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float16, device=X.device)
    if row_sum is None:
        row_sum = torch.empty((M,), dtype=torch.float32, device=X.device)
    _need(out, torch.float16, "out", 2)
    _need(row_sum, torch.float32, "row_sum", 1)
    st = lib().bq_gemm_f16xu4_zp(_ptr(X), _ptr(Wp), _layout(layout), M, N, K, _ptr(col_scale), _ptr(zero_point),
                                 _activation(activation), _ptr(row_sum), _ptr(out), _stream(stream))
    _check(st, "bq_gemm_f16xu4_zp")
    return out, row_sum


def bq_device_status(reset=True) -> int:
    v = ctypes.c_int(0)
    _check(lib().bq_device_status(ctypes.byref(v), 1 if reset else 0), "bq_device_status")
    return v.value


def bq_set_wait_timeout_ns(ns: int) -> int:
    return int(lib().bq_set_wait_timeout_ns(int(ns)))

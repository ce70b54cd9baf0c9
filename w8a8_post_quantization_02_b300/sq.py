"""Thin Python binding of the C ABI in ``include/sq.h`` (ctypes + torch).

Argument marshalling only: every step of the path runs in the CUDA
library ``libsq_b300.so``.  torch provides device memory and the current
stream.  There is no fallback: if the library is missing or the device is
not sm_103, the calls raise.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsq_b300.so")

(SQ_OK, SQ_ERR_INVALID_ARG, SQ_ERR_NONFINITE, SQ_ERR_CUDA, SQ_ERR_UNSUPPORTED, SQ_ERR_WORKSPACE,
 SQ_ERR_TIMEOUT) = range(7)
SQ_GEMM_MAX_K = 133136
SQ_FLAG_NONFINITE, SQ_FLAG_TIMEOUT = 1, 2
SQ_F32, SQ_BF16 = 0, 1
SQ_CODES_I8, SQ_CODES_BF16 = 0, 1
(SQ_OP_CALIBRATE, SQ_OP_SMOOTH, SQ_OP_FOLD_QUANTIZE, SQ_OP_QUANT_ACT, SQ_OP_GEMM, SQ_OP_STATIC_SCALE,
 SQ_OP_QUANT_ACT_STATIC, SQ_OP_FOLD_NORM_GAIN, SQ_OP_RMSNORM_QUANT_ACT, SQ_OP_ROTATE_ACT,
 SQ_OP_ROTATE_WEIGHT) = range(11)

# name -> (restype, argtypes), mirroring include/sq.h
_P, _I64, _I32, _F, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_size_t


class LinearBuffers(ctypes.Structure):
    """sq_linear_buffers: the caller's device buffers for sq_linear_host."""
    _fields_ = [(name, _P) for name in ("x", "w", "amax_x", "amax_w", "s", "s_inv", "wq", "w_scale",
                                        "xq", "x_scale", "y", "workspace")] + [("ws_bytes", _SZ)]


SIGNATURES = {
    "sq_calibrate_absmax": (_I32, [_P, _I32, _I64, _I64, _I64, _I32, _I32, _P, _P]),
    "sq_smooth_factors": (_I32, [_P, _P, _I64, _F, _P, _P, _P, _P]),
    "sq_fold_quantize_weight": (_I32, [_P, _I32, _I64, _I64, _I64, _P, _P, _I32, _P, _P, _P, _SZ, _P]),
    "sq_fold_quantize_weight_noalloc": (_I32, [_P, _I32, _I64, _I64, _I64, _P, _P, _I32, _P, _P, _P]),
    "sq_quant_act": (_I32, [_P, _I32, _I64, _I64, _I64, _P, _P, _I32, _P, _P, _P]),
    "sq_static_act_scale": (_I32, [_P, _P, _I64, _P, _P, _P]),
    "sq_fold_norm_gain": (_I32, [_P, _P, _I64, _P, _P]),
    "sq_rotate_quant_act": (_I32, [_P, _I32, _I64, _I64, _I64, _P, _I32, _I32, _P, _I32, _P, _P, _P]),
    "sq_rotate_fold_quantize_weight": (_I32, [_P, _I32, _I64, _I64, _I64, _P, _I32, _I32, _P, _I32, _P,
                                              _P, _P, _SZ, _P]),
    "sq_rmsnorm_quant_act": (_I32, [_P, _I32, _I64, _I64, _I64, _P, _F, _P, _I32, _P, _P, _P]),
    "sq_quant_act_static": (_I32, [_P, _I32, _I64, _I64, _I64, _P, _P, _P, _I32, _P, _P, _P, _P]),
    "sq_w8a8_gemm": (_I32, [_P, _P, _P, _P, _I32, _I64, _I64, _I64, _P, _P, _P, _P, _SZ, _P]),
    "sq_workspace_bytes": (_SZ, [_I32, _I64, _I64, _I64, _I32]),
    "sq_kernel_count": (_I32, [_I32, _I32, _I64, _I64, _I64, _I64, _I32, _I32]),
    "sq_act_quant_error": (_I32, [_P, _I32, _I64, _I64, _I64, _P, _P, _I32, _P, _P, _P]),
    "sq_weight_quant_error": (_I32, [_P, _I32, _I64, _I64, _I64, _P, _P, _I32, _P, _P, _P]),
    "sq_layer_error": (_I32, [_P, _P, _I32, _I64, _I64, _I64, _I64, _I64, _P, _P, _I32, _P, _P]),
    "sq_channel_stats": (_I32, [_P, _P, _I64, _P, _P]),
    "sq_linear_host": (_I32, [_P, _P, _I32, _I64, _I64, _I64, _F, _I32, _P, ctypes.POINTER(LinearBuffers),
                              _P, _P]),
    "sq_read_device_flags": (_I32, [_P, _I32, ctypes.POINTER(ctypes.c_int32), _P]),
    "sq_test_w8a8_gemm_stalled": (_I32, [_P, _P, _P, _P, _I32, _I64, _I64, _I64, _P, _P, ctypes.c_uint64, _P]),
    "sq_test_w8a8_gemm_stalled_ws": (_I32, [_P, _P, _P, _P, _I32, _I64, _I64, _I64, _P, _P, _P, _SZ,
                                            ctypes.c_uint64, _P]),
    "sq_test_quant_act_stalled": (_I32, [_P, _I32, _I64, _I64, _I64, _P, _P, _I32, _P, _P, ctypes.c_uint64,
                                         _P]),
    "sq_status_string": (ctypes.c_char_p, [_I32]),
    "sq_check_device": (_I32, [_I32]),
}


class SqError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} failed: {text} (status {status})")
        self.status = status


_lib = None


def load_library():
    """Load libsq_b300.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        _lib = lib
    return _lib


def _check(fn: str, status: int):
    if status != SQ_OK:
        raise SqError(fn, status, load_library().sq_status_string(status).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return SQ_F32
    if t.dtype == torch.bfloat16:
        return SQ_BF16
    raise TypeError(f"unsupported input dtype {t.dtype}")


def _codes_fmt(codes: str) -> int:
    return {"i8": SQ_CODES_I8, "bf16": SQ_CODES_BF16}[codes]


def _codes_dtype(codes: str):
    return {"i8": torch.int8, "bf16": torch.bfloat16}[codes]


def _check_cuda_2d(t: torch.Tensor, name: str):
    if not t.is_cuda or t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D CUDA tensor with unit column stride")


def check_device(device: int = 0) -> None:
    _check("sq_check_device", load_library().sq_check_device(device))


def workspace_bytes(op: int, m: int, n: int, k: int, codes: str = "i8") -> int:
    return int(load_library().sq_workspace_bytes(op, m, n, k, _codes_fmt(codes)))


def kernel_count(op: int, dtype: int, m: int, n: int, k: int, ld: int = 0, axis: int = 0,
                 accumulate: bool = False) -> int:
    """Kernels one call of ``op`` enqueues for these sizes (see include/sq.h)."""
    return int(load_library().sq_kernel_count(op, dtype, m, n, k, ld, axis, int(accumulate)))


def calibrate_absmax(a: torch.Tensor, axis: int, out: torch.Tensor | None = None,
                     accumulate: bool = False, stream=None) -> torch.Tensor:
    """Step 1: per-channel max|a| over rows (axis 0) or columns (axis 1)."""
    _check_cuda_2d(a, "a")
    rows, cols = a.shape
    if out is None:
        if accumulate:
            raise ValueError("accumulate needs an existing `out`")
        out = torch.empty(cols if axis == 0 else rows, device=a.device, dtype=torch.float32)
    st = load_library().sq_calibrate_absmax(_ptr(a), _dtype_code(a), rows, cols, a.stride(0), axis,
                                            int(accumulate), _ptr(out), _stream(stream))
    _check("sq_calibrate_absmax", st)
    return out


def smooth_factors(amax_x: torch.Tensor, amax_w: torch.Tensor, alpha: float,
                   flags: torch.Tensor | None = None, stream=None):
    """Step 2: (s, s_inv) with s_j = amax_x^alpha / amax_w^(1-alpha)."""
    cin = amax_x.numel()
    s = torch.empty(cin, device=amax_x.device, dtype=torch.float32)
    s_inv = torch.empty_like(s)
    st = load_library().sq_smooth_factors(_ptr(amax_x), _ptr(amax_w), cin, float(alpha), _ptr(s),
                                          _ptr(s_inv), _ptr(flags), _stream(stream))
    _check("sq_smooth_factors", st)
    return s, s_inv


def fold_quantize_weight(w: torch.Tensor, s: torch.Tensor, codes: str = "i8",
                         flags: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                         stream=None):
    """Step 3: W [Cin x Cout] -> (wq [Cout x Cin] codes, w_scale [Cout])."""
    _check_cuda_2d(w, "w")
    cin, cout = w.shape
    wq = torch.empty(cout, cin, device=w.device, dtype=_codes_dtype(codes))
    w_scale = torch.empty(cout, device=w.device, dtype=torch.float32)
    nbytes = workspace_bytes(SQ_OP_FOLD_QUANTIZE, 0, cout, cin, codes)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 1), device=w.device, dtype=torch.uint8)
    st = load_library().sq_fold_quantize_weight(
        _ptr(w), _dtype_code(w), cin, cout, w.stride(0), _ptr(s), _ptr(wq), _codes_fmt(codes),
        _ptr(w_scale), _ptr(flags), _ptr(workspace), workspace.numel(), _stream(stream))
    _check("sq_fold_quantize_weight", st)
    return wq, w_scale


def quant_act(x: torch.Tensor, s_inv: torch.Tensor, codes: str = "i8",
              flags: torch.Tensor | None = None, out=None, stream=None):
    """Step 4: X [tokens x Cin] -> (xq codes [tokens x Cin], x_scale [tokens])."""
    _check_cuda_2d(x, "x")
    tokens, cin = x.shape
    if out is None:
        xq = torch.empty(tokens, cin, device=x.device, dtype=_codes_dtype(codes))
        x_scale = torch.empty(tokens, device=x.device, dtype=torch.float32)
    else:
        xq, x_scale = out
    st = load_library().sq_quant_act(_ptr(x), _dtype_code(x), tokens, cin, x.stride(0), _ptr(s_inv),
                                     _ptr(xq), _codes_fmt(codes), _ptr(x_scale), _ptr(flags),
                                     _stream(stream))
    _check("sq_quant_act", st)
    return xq, x_scale


def static_act_scale(amax_x: torch.Tensor, s_inv: torch.Tensor, flags: torch.Tensor | None = None,
                     out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Step 4, static variant: the one calibrated scale d (a 1-element tensor)."""
    d = out if out is not None else torch.empty(1, device=amax_x.device, dtype=torch.float32)
    st = load_library().sq_static_act_scale(_ptr(amax_x), _ptr(s_inv), amax_x.numel(), _ptr(d),
                                            _ptr(flags), _stream(stream))
    _check("sq_static_act_scale", st)
    return d


def quant_act_static(x: torch.Tensor, s_inv: torch.Tensor, d: torch.Tensor, codes: str = "i8",
                     clipped: torch.Tensor | None = None, flags: torch.Tensor | None = None,
                     out=None, stream=None):
    """Step 4 with the calibrated scale d: (xq codes, x_scale filled with d)."""
    _check_cuda_2d(x, "x")
    tokens, cin = x.shape
    if out is None:
        xq = torch.empty(tokens, cin, device=x.device, dtype=_codes_dtype(codes))
        x_scale = torch.empty(tokens, device=x.device, dtype=torch.float32)
    else:
        xq, x_scale = out
    st = load_library().sq_quant_act_static(_ptr(x), _dtype_code(x), tokens, cin, x.stride(0),
                                            _ptr(s_inv), _ptr(d), _ptr(xq), _codes_fmt(codes),
                                            _ptr(x_scale), _ptr(clipped), _ptr(flags), _stream(stream))
    _check("sq_quant_act_static", st)
    return xq, x_scale


def fold_norm_gain(gamma: torch.Tensor, s_inv: torch.Tensor, stream=None) -> torch.Tensor:
    """Offline: the normalization gain with S^-1 folded in, gamma * (1/s)."""
    out = torch.empty_like(gamma)
    st = load_library().sq_fold_norm_gain(_ptr(gamma), _ptr(s_inv), gamma.numel(), _ptr(out),
                                          _stream(stream))
    _check("sq_fold_norm_gain", st)
    return out


def rmsnorm_quant_act(h: torch.Tensor, gamma_folded: torch.Tensor, eps: float, codes: str = "i8",
                      flags: torch.Tensor | None = None, out=None, stream=None):
    """RMS normalization with the folded gain fused into the per-token quantizer."""
    _check_cuda_2d(h, "h")
    tokens, cin = h.shape
    if out is None:
        xq = torch.empty(tokens, cin, device=h.device, dtype=_codes_dtype(codes))
        x_scale = torch.empty(tokens, device=h.device, dtype=torch.float32)
    else:
        xq, x_scale = out
    st = load_library().sq_rmsnorm_quant_act(_ptr(h), _dtype_code(h), tokens, cin, h.stride(0),
                                             _ptr(gamma_folded), float(eps), _ptr(xq), _codes_fmt(codes),
                                             _ptr(x_scale), _ptr(flags), _stream(stream))
    _check("sq_rmsnorm_quant_act", st)
    return xq, x_scale


def rotate_quant_act(x: torch.Tensor, s_inv: torch.Tensor | None, rotate: bool = True, qmax: int = 7,
                     codes: str = "i8", flags: torch.Tensor | None = None, stream=None):
    """Smooth Rotation, activation side: codes of (X S^-1) H per token with
    grid +-qmax; x_scale carries 2^-log2(cin) when rotated."""
    _check_cuda_2d(x, "x")
    tokens, cin = x.shape
    xq = torch.empty(tokens, cin, device=x.device, dtype=_codes_dtype(codes))
    x_scale = torch.empty(tokens, device=x.device, dtype=torch.float32)
    st = load_library().sq_rotate_quant_act(_ptr(x), _dtype_code(x), tokens, cin, x.stride(0), _ptr(s_inv),
                                            int(rotate), int(qmax), _ptr(xq), _codes_fmt(codes),
                                            _ptr(x_scale), _ptr(flags), _stream(stream))
    _check("sq_rotate_quant_act", st)
    return xq, x_scale


def rotate_fold_quantize_weight(w: torch.Tensor, s: torch.Tensor | None, rotate: bool = True,
                                qmax: int = 7, codes: str = "i8", flags: torch.Tensor | None = None,
                                workspace: torch.Tensor | None = None, stream=None):
    """Smooth Rotation, weight side: codes of H^T S W per output channel."""
    _check_cuda_2d(w, "w")
    cin, cout = w.shape
    wq = torch.empty(cout, cin, device=w.device, dtype=_codes_dtype(codes))
    w_scale = torch.empty(cout, device=w.device, dtype=torch.float32)
    nbytes = workspace_bytes(SQ_OP_ROTATE_WEIGHT, 0, cout, cin, codes)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), device=w.device, dtype=torch.uint8)
    st = load_library().sq_rotate_fold_quantize_weight(
        _ptr(w), _dtype_code(w), cin, cout, w.stride(0), _ptr(s), int(rotate), int(qmax), _ptr(wq),
        _codes_fmt(codes), _ptr(w_scale), _ptr(flags), _ptr(workspace), workspace.numel(), _stream(stream))
    _check("sq_rotate_fold_quantize_weight", st)
    return wq, w_scale


def w8a8_gemm(xq: torch.Tensor, x_scale: torch.Tensor, wq: torch.Tensor, w_scale: torch.Tensor,
              want_acc: bool = False, flags: torch.Tensor | None = None,
              workspace: torch.Tensor | None = None, out=None, stream=None):
    """Step 5: y = bf16(acc * x_scale * w_scale); returns y or (y, acc)."""
    _check_cuda_2d(xq, "xq")
    _check_cuda_2d(wq, "wq")
    if xq.dtype != wq.dtype:
        raise TypeError("xq and wq must use the same code format")
    codes = "bf16" if xq.dtype == torch.bfloat16 else "i8"
    m, k = xq.shape
    n = wq.shape[0]
    y = out if out is not None else torch.empty(m, n, device=xq.device, dtype=torch.bfloat16)
    acc = torch.empty(m, n, device=xq.device, dtype=torch.int32) if want_acc else None
    nbytes = workspace_bytes(SQ_OP_GEMM, m, n, k, codes)
    if workspace is None and nbytes:
        workspace = torch.empty(nbytes, device=xq.device, dtype=torch.uint8)
    st = load_library().sq_w8a8_gemm(
        _ptr(xq), _ptr(x_scale), _ptr(wq), _ptr(w_scale), _codes_fmt(codes), m, n, k, _ptr(y),
        _ptr(acc), _ptr(flags), _ptr(workspace), 0 if workspace is None else workspace.numel(),
        _stream(stream))
    _check("sq_w8a8_gemm", st)
    return (y, acc) if want_acc else y


# ------------------------------------------------------------------ diagnostics
def act_quant_error(x: torch.Tensor, s_inv: torch.Tensor, xq: torch.Tensor, x_scale: torch.Tensor,
                    stream=None) -> torch.Tensor:
    """Per-token squared reconstruction error of the activation codes (float64)."""
    _check_cuda_2d(x, "x")
    tokens, cin = x.shape
    err = torch.empty(tokens, device=x.device, dtype=torch.float64)
    codes = "bf16" if xq.dtype == torch.bfloat16 else "i8"
    st = load_library().sq_act_quant_error(_ptr(x), _dtype_code(x), tokens, cin, x.stride(0), _ptr(s_inv),
                                           _ptr(xq), _codes_fmt(codes), _ptr(x_scale), _ptr(err),
                                           _stream(stream))
    _check("sq_act_quant_error", st)
    return err


def weight_quant_error(w: torch.Tensor, s: torch.Tensor, wq: torch.Tensor, w_scale: torch.Tensor,
                       stream=None) -> torch.Tensor:
    """Per-output-channel squared reconstruction error of the folded weight (float64)."""
    _check_cuda_2d(w, "w")
    cin, cout = w.shape
    err = torch.empty(cout, device=w.device, dtype=torch.float64)
    codes = "bf16" if wq.dtype == torch.bfloat16 else "i8"
    st = load_library().sq_weight_quant_error(_ptr(w), _dtype_code(w), cin, cout, w.stride(0), _ptr(s),
                                              _ptr(wq), _codes_fmt(codes), _ptr(w_scale), _ptr(err),
                                              _stream(stream))
    _check("sq_weight_quant_error", st)
    return err


def layer_error(x: torch.Tensor, w: torch.Tensor, y: torch.Tensor, rows: torch.Tensor,
                stream=None) -> torch.Tensor:
    """Per sampled token: sum_n ((X W) - Y)^2 against the unquantized product (float64)."""
    _check_cuda_2d(x, "x")
    _check_cuda_2d(w, "w")
    tokens, cin = x.shape
    cout = w.shape[1]
    if tuple(y.shape) != (tokens, cout) or y.dtype != torch.bfloat16:
        raise ValueError(f"y must be bf16 [{tokens} x {cout}], got {y.dtype} {tuple(y.shape)}")
    rows = rows.to(device=x.device, dtype=torch.int32).contiguous()
    if rows.numel() and (int(rows.min()) < 0 or int(rows.max()) >= tokens):
        raise ValueError(f"sampled rows must lie in [0, {tokens})")
    err = torch.empty(rows.numel(), device=x.device, dtype=torch.float64)
    st = load_library().sq_layer_error(_ptr(x), _ptr(w), _dtype_code(x), tokens, cin, cout, x.stride(0),
                                       w.stride(0), _ptr(y.contiguous()), _ptr(rows), rows.numel(),
                                       _ptr(err), _stream(stream))
    _check("sq_layer_error", st)
    return err


def read_device_flags(flags: torch.Tensor, clear: bool = False, stream=None):
    """Synchronize `stream`, read the device flag word (optionally zeroing
    it) and return (status, raw word): SQ_ERR_TIMEOUT, SQ_ERR_NONFINITE or
    SQ_OK."""
    out = ctypes.c_int32(0)
    st = load_library().sq_read_device_flags(_ptr(flags), int(clear), ctypes.byref(out), _stream(stream))
    if st in (SQ_ERR_INVALID_ARG, SQ_ERR_CUDA):
        _check("sq_read_device_flags", st)
    return st, out.value


def channel_stats(amax: torch.Tensor, scale: torch.Tensor | None = None, stream=None):
    """(mean, population std) of the channel magnitudes (times scale if given), float64."""
    out = torch.empty(2, device=amax.device, dtype=torch.float64)
    st = load_library().sq_channel_stats(_ptr(amax), _ptr(scale), amax.numel(), _ptr(out),
                                         _stream(stream))
    _check("sq_channel_stats", st)
    return out


def smoothquant_linear(x: torch.Tensor, w: torch.Tensor, alpha: float, codes: str = "i8",
                       flags: torch.Tensor | None = None, want_acc: bool = False):
    """Steps 1-5 on one layer: calibrate on X, smooth, fold + quantize W,
    quantize X, GEMM.  Returns a dict of every intermediate."""
    amax_x = calibrate_absmax(x, 0)
    amax_w = calibrate_absmax(w, 1)
    s, s_inv = smooth_factors(amax_x, amax_w, alpha, flags)
    wq, w_scale = fold_quantize_weight(w, s, codes, flags)
    xq, x_scale = quant_act(x, s_inv, codes, flags)
    r = w8a8_gemm(xq, x_scale, wq, w_scale, want_acc=want_acc, flags=flags)
    y, acc = r if want_acc else (r, None)
    return dict(amax_x=amax_x, amax_w=amax_w, s=s, s_inv=s_inv, wq=wq, w_scale=w_scale, xq=xq,
                x_scale=x_scale, y=y, acc=acc)


def linear_buffers(bufs: dict, workspace: torch.Tensor) -> LinearBuffers:
    """Pack device tensors (keys as in sq_linear_buffers) for sq_linear_host."""
    b = LinearBuffers()
    for name, _ in LinearBuffers._fields_[:-2]:
        setattr(b, name, bufs[name].data_ptr())
    b.workspace = workspace.data_ptr()
    b.ws_bytes = workspace.numel() * workspace.element_size()
    return b


def linear_host(x_host: torch.Tensor, w_host: torch.Tensor, alpha: float, codes: str,
                y_host: torch.Tensor, dev: LinearBuffers, flags: torch.Tensor | None = None,
                stream=None) -> None:
    """The whole path on host tensors (pinned for asynchronous copies):
    X and W copied in, steps 1-5 on the device buffers `dev`, Y copied out
    into y_host, all enqueued on `stream`."""
    for t, name in ((x_host, "x_host"), (w_host, "w_host"), (y_host, "y_host")):
        if t.is_cuda or not t.is_contiguous() or t.dim() != 2:
            raise ValueError(f"{name} must be a contiguous 2-D host tensor")
    if y_host.dtype != torch.bfloat16:
        raise ValueError("y_host must be bfloat16")
    if w_host.dtype != x_host.dtype:
        raise ValueError("x_host and w_host must have the same dtype")
    tokens, cin = x_host.shape
    cout = w_host.shape[1]
    if w_host.shape[0] != cin or tuple(y_host.shape) != (tokens, cout):
        raise ValueError(f"shapes do not chain: x {tuple(x_host.shape)}, w {tuple(w_host.shape)}, "
                         f"y {tuple(y_host.shape)}")
    _check("sq_linear_host", load_library().sq_linear_host(
        _ptr(x_host), _ptr(w_host), _dtype_code(x_host), tokens, cin, cout, alpha, _codes_fmt(codes),
        _ptr(y_host), ctypes.byref(dev), _ptr(flags), _stream(stream)))

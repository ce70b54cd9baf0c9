"""One SmoothQuant W8A8 linear layer with preallocated device buffers.

``Layer.step()`` runs the five steps of the path in order on the current
stream through the C ABI (calibrate X and W, smoothing factors, fold +
quantize W, quantize X, GEMM) without allocating, so it can be timed and
captured into a CUDA graph.  The benchmark and the full-size parity tests
use this same object, so they exercise identical launches.
"""
from __future__ import annotations

import ctypes

import torch

from . import sq

# Above this token count the library runs 1-byte codes on the tensor cores
# (widened to fp16 in the GEMM's workspace first), at or below it on the
# weight-streaming and mma.sync kernels.
I8_TENSOR_MIN_TOKENS = 64


def choose_codes(tokens: int) -> str:
    """The layer's code storage when the caller names none: one byte per
    code, the method's W8A8 storage, at every token count.  Storing the same
    integers as bf16 values ("bf16") lets the tensor-core GEMM read them
    without the widening pass: about 8 % faster per prefill step, at twice
    the weight and activation code memory."""
    del tokens
    return "i8"


class Layer:
    def __init__(self, tokens: int, cin: int, cout: int, dtype: str, alpha: float,
                 codes: str | None = None, device="cuda", act_scale: str = "dynamic",
                 gemm_workspace: bool = True):
        if act_scale not in ("dynamic", "static", "norm"):
            raise ValueError("act_scale is 'dynamic' (per token), 'static' (one calibrated scale) or "
                             "'norm' (RMS normalization with S^-1 folded into its gain, then per token)")
        self.tokens, self.cin, self.cout = tokens, cin, cout
        self.dtype = dtype
        self.alpha = float(alpha)
        self.act_scale = act_scale
        self.codes = codes or choose_codes(tokens)
        tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
        cdt = torch.bfloat16 if self.codes == "bf16" else torch.int8
        dv = torch.device(device)
        self.x = torch.empty(tokens, cin, dtype=tdt, device=dv)
        self.w = torch.empty(cin, cout, dtype=tdt, device=dv)
        self.amax_x = torch.empty(cin, dtype=torch.float32, device=dv)
        self.amax_w = torch.empty(cin, dtype=torch.float32, device=dv)
        self.s = torch.empty(cin, dtype=torch.float32, device=dv)
        self.s_inv = torch.empty(cin, dtype=torch.float32, device=dv)
        self.wq = torch.empty(cout, cin, dtype=cdt, device=dv)
        self.w_scale = torch.empty(cout, dtype=torch.float32, device=dv)
        self.xq = torch.empty(tokens, cin, dtype=cdt, device=dv)
        self.x_scale = torch.empty(tokens, dtype=torch.float32, device=dv)
        self.y = torch.empty(tokens, cout, dtype=torch.bfloat16, device=dv)
        self.acc = torch.empty(tokens, cout, dtype=torch.int32, device=dv)
        self.flags = torch.zeros(1, dtype=torch.int32, device=dv)
        self.d = torch.empty(1, dtype=torch.float32, device=dv)          # static scale
        self.clipped = torch.zeros(1, dtype=torch.int32, device=dv)      # static clip count
        # 'norm' mode: x holds the normalization's input h, gamma its gain
        self.gamma = torch.ones(cin, dtype=torch.float32, device=dv)
        self.gamma_f = torch.empty(cin, dtype=torch.float32, device=dv)
        self.eps = 1e-5
        fmt = sq._codes_fmt(self.codes)
        self._fmt = fmt
        ws_fold = sq.workspace_bytes(sq.SQ_OP_FOLD_QUANTIZE, 0, cout, cin, self.codes)
        # without the GEMM's workspace, 1-byte codes above 64 tokens run the
        # kernel that widens them in shared memory as it goes
        ws_gemm = sq.workspace_bytes(sq.SQ_OP_GEMM, tokens, cout, cin, self.codes) if gemm_workspace else 0
        self.gemm_workspace = bool(gemm_workspace)
        self.ws_fold = torch.empty(max(ws_fold, 256), dtype=torch.uint8, device=dv)
        self.ws_gemm = torch.empty(max(ws_gemm, 256), dtype=torch.uint8, device=dv)
        self._lib = sq.load_library()

    @classmethod
    def for_case(cls, case, codes: str | None = None, act_scale: str = "dynamic",
                 gemm_workspace: bool = True) -> "Layer":
        return cls(case.tokens, case.cin, case.cout, case.dtype, case.alpha, codes,
                   act_scale=act_scale, gemm_workspace=gemm_workspace)

    def load(self, x: torch.Tensor, w: torch.Tensor) -> None:
        self.x.copy_(x)
        self.w.copy_(w)

    # bytes one step moves through HBM by definition of each step (the
    # algorithmic traffic used for the roofline figures): every INT8 code
    # counts one byte, whatever format stores it
    def algorithmic_bytes(self) -> dict:
        return self._bytes(code_bytes=1)

    # bytes each step moves with the codes in their storage format (two bytes
    # per code when they are stored as bf16 values)
    def storage_bytes(self) -> dict:
        return self._bytes(code_bytes=2 if self.codes == "bf16" else 1)

    def _bytes(self, code_bytes: int) -> dict:
        eb = 2 if self.dtype == "bf16" else 4
        cb = code_bytes
        T, K, N = self.tokens, self.cin, self.cout
        return {
            "calibrate_x": T * K * eb + K * 4,
            "calibrate_w": K * N * eb + K * 4,
            "smooth": K * 4 * 4,
            "fold_quantize": K * N * eb + N * K * cb + N * 4,
            "quant_act": T * K * eb + T * K * cb + T * 4 + K * 4,
            "static_scale": K * 4 * 2 + 4,
            "fold_norm_gain": K * 4 * 3,
            "rmsnorm_quant_act": T * K * eb + T * K * cb + T * 4 + K * 4,
            "quant_act_static": T * K * eb + T * K * cb + T * 4 + K * 4,
            "gemm": (T + N) * K * cb + T * N * 2 + (T + N) * 4,
        }

    def gemm_ops(self) -> int:
        return 2 * self.tokens * self.cin * self.cout

    def stages(self, want_acc: bool = False):
        """The path as (name, launches, fn(stream)) in execution order; ``launches``
        counts the library kernels one call enqueues."""
        counts = self.kernel_counts()
        L, P = self._lib, ctypes.c_void_p
        dt = sq._dtype_code(self.x)
        T, K, N = self.tokens, self.cin, self.cout
        ck = sq._check
        ptr = lambda t: P(t.data_ptr())  # noqa: E731
        flags = ptr(self.flags)

        def calibrate_x(st):
            ck("sq_calibrate_absmax", L.sq_calibrate_absmax(ptr(self.x), dt, T, K, K, 0, 0, ptr(self.amax_x), st))

        def calibrate_w(st):
            ck("sq_calibrate_absmax", L.sq_calibrate_absmax(ptr(self.w), dt, K, N, N, 1, 0, ptr(self.amax_w), st))

        def smooth(st):
            ck("sq_smooth_factors", L.sq_smooth_factors(ptr(self.amax_x), ptr(self.amax_w), K, self.alpha,
                                                        ptr(self.s), ptr(self.s_inv), flags, st))

        def fold_quantize(st):
            ck("sq_fold_quantize_weight", L.sq_fold_quantize_weight(
                ptr(self.w), dt, K, N, N, ptr(self.s), ptr(self.wq), self._fmt, ptr(self.w_scale), flags,
                ptr(self.ws_fold), self.ws_fold.numel(), st))

        def quant_act(st):
            ck("sq_quant_act", L.sq_quant_act(ptr(self.x), dt, T, K, K, ptr(self.s_inv), ptr(self.xq),
                                              self._fmt, ptr(self.x_scale), flags, st))

        def gemm(st):
            ck("sq_w8a8_gemm", L.sq_w8a8_gemm(
                ptr(self.xq), ptr(self.x_scale), ptr(self.wq), ptr(self.w_scale), self._fmt, T, N, K,
                ptr(self.y), ptr(self.acc) if want_acc else None, flags, ptr(self.ws_gemm),
                self.ws_gemm.numel(), st))

        def static_scale(st):
            ck("sq_static_act_scale", L.sq_static_act_scale(ptr(self.amax_x), ptr(self.s_inv), K,
                                                            ptr(self.d), flags, st))

        def quant_act_static(st):
            ck("sq_quant_act_static", L.sq_quant_act_static(
                ptr(self.x), dt, T, K, K, ptr(self.s_inv), ptr(self.d), ptr(self.xq), self._fmt,
                ptr(self.x_scale), ptr(self.clipped), flags, st))

        def fold_norm_gain(st):
            ck("sq_fold_norm_gain", L.sq_fold_norm_gain(ptr(self.gamma), ptr(self.s_inv), K,
                                                        ptr(self.gamma_f), st))

        def rmsnorm_quant_act(st):
            ck("sq_rmsnorm_quant_act", L.sq_rmsnorm_quant_act(
                ptr(self.x), dt, T, K, K, ptr(self.gamma_f), self.eps, ptr(self.xq), self._fmt,
                ptr(self.x_scale), flags, st))

        act = {"dynamic": [("quant_act", quant_act)],
               "static": [("static_scale", static_scale), ("quant_act_static", quant_act_static)],
               "norm": [("fold_norm_gain", fold_norm_gain), ("rmsnorm_quant_act", rmsnorm_quant_act)],
               }[self.act_scale]
        fns = ([("calibrate_x", calibrate_x), ("calibrate_w", calibrate_w), ("smooth", smooth),
                ("fold_quantize", fold_quantize)] + act + [("gemm", gemm)])
        return [(name, counts[name], fn) for name, fn in fns]

    def kernel_counts(self) -> dict:
        """Library kernels each stage of one step enqueues (the library's own count)."""
        dt = sq.SQ_BF16 if self.dtype == "bf16" else sq.SQ_F32
        T, K, N = self.tokens, self.cin, self.cout
        return {
            "calibrate_x": sq.kernel_count(sq.SQ_OP_CALIBRATE, dt, T, K, 0, K, 0, False),
            "calibrate_w": sq.kernel_count(sq.SQ_OP_CALIBRATE, dt, K, N, 0, N, 1, False),
            "smooth": sq.kernel_count(sq.SQ_OP_SMOOTH, dt, 0, 0, K),
            "fold_quantize": sq.kernel_count(sq.SQ_OP_FOLD_QUANTIZE, dt, 0, N, K, N),
            "quant_act": sq.kernel_count(sq.SQ_OP_QUANT_ACT, dt, T, 0, K, K),
            "static_scale": sq.kernel_count(sq.SQ_OP_STATIC_SCALE, dt, 0, 0, K),
            "quant_act_static": sq.kernel_count(sq.SQ_OP_QUANT_ACT_STATIC, dt, T, 0, K, K),
            "fold_norm_gain": sq.kernel_count(sq.SQ_OP_FOLD_NORM_GAIN, dt, 0, 0, K),
            "rmsnorm_quant_act": sq.kernel_count(sq.SQ_OP_RMSNORM_QUANT_ACT, dt, T, 0, K, K),
            # the library counts with the workspace it asks for; without it the
            # 1-byte GEMM is its one on-chip-widening kernel
            "gemm": (sq.kernel_count(sq.SQ_OP_GEMM, dt, T, N, K, 0, sq._codes_fmt(self.codes))
                     if self.gemm_workspace else 1),
        }

    def kernel_count(self) -> int:
        """Library kernels one step enqueues."""
        counts = self.kernel_counts()
        return sum(counts[name] for name, _, _ in self.stages())

    def linear_buffers(self) -> "sq.LinearBuffers":
        """This layer's device buffers as the C ABI's sq_linear_buffers."""
        names = ("x", "w", "amax_x", "amax_w", "s", "s_inv", "wq", "w_scale", "xq", "x_scale", "y")
        # the fold and the GEMM run one after the other on the call's stream:
        # one buffer, the larger of the two workspaces, serves both
        ws = self.ws_gemm if self.ws_gemm.numel() > self.ws_fold.numel() else self.ws_fold
        return sq.linear_buffers({n: getattr(self, n) for n in names}, ws)

    def run_host(self, x_host: torch.Tensor, w_host: torch.Tensor, y_host: torch.Tensor,
                 stream=None, bufs: "sq.LinearBuffers | None" = None) -> None:
        """One step from host memory through the C ABI's sq_linear_host: X and
        W copied in, the whole path (dynamic per-token scale), Y copied out."""
        if self.act_scale != "dynamic":
            raise ValueError("sq_linear_host runs the dynamic per-token activation scale")
        # the device buffers are this layer's: the host tensors must match them
        if (tuple(x_host.shape) != tuple(self.x.shape) or tuple(w_host.shape) != tuple(self.w.shape)
                or x_host.dtype != self.x.dtype or w_host.dtype != self.w.dtype):
            raise ValueError("x_host / w_host do not match this layer's shapes and dtype")
        sq.linear_host(x_host, w_host, self.alpha, self.codes, y_host,
                       bufs if bufs is not None else self.linear_buffers(), self.flags, stream)

    def _enqueue(self, fns: dict, main, side) -> None:
        """Enqueue steps 1-4 on two streams.  The X side (absmax of X, then
        the activation codes) runs on ``side`` beside the W side (absmax of W,
        then the fold); they meet at the smoothing factors, which need both
        absmax vectors, and again before the GEMM.  Same kernels and work as
        the serial order, fewer idle SMs in the small kernels and tails."""
        act = [n for n in fns if n not in ("calibrate_x", "calibrate_w", "smooth", "fold_quantize", "gemm")]
        fork, x_done, s_done, act_done = (torch.cuda.Event() for _ in range(4))
        fork.record(main)
        side.wait_event(fork)
        fns["calibrate_x"](sq._stream(side))
        x_done.record(side)
        fns["calibrate_w"](sq._stream(main))
        main.wait_event(x_done)
        fns["smooth"](sq._stream(main))
        s_done.record(main)
        side.wait_event(s_done)
        for name in act:
            fns[name](sq._stream(side))
        act_done.record(side)
        fns["fold_quantize"](sq._stream(main))
        main.wait_event(act_done)

    def _side_stream(self):
        if getattr(self, "_side", None) is None:
            self._side = torch.cuda.Stream(device=self.x.device)
        return self._side

    def step(self, want_acc: bool = False, stream=None) -> None:
        main = stream if stream is not None else torch.cuda.current_stream()
        fns = {name: fn for name, _, fn in self.stages(want_acc)}
        self._enqueue(fns, main, self._side_stream())
        fns["gemm"](sq._stream(main))

    def capture(self, want_acc: bool = False):
        """Two CUDA graphs of one step: steps 1-4 (calibration through the
        activation codes, forked over two streams and joined) and the GEMM,
        replayed with ``graph.replay()`` on the current stream.  Call
        ``step()`` once first, outside capture, so the library's one-time
        set-up (kernel attributes) is done."""
        fns = {name: fn for name, _, fn in self.stages(want_acc)}
        side = self._side_stream()
        g_pre, g_gemm = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_pre):
            self._enqueue(fns, torch.cuda.current_stream(), side)
        with torch.cuda.graph(g_gemm):
            fns["gemm"](sq._stream())
        return g_pre, g_gemm


def available_codes():
    """Code formats the library's GEMM runs."""
    return ["i8", "bf16"]


def diagnose(layer: "Layer", rows=None) -> dict:
    """Quantization diagnostics of a layer after ``step()`` (float64 sums):
    activation and weight reconstruction errors, the layer error on sampled
    tokens (default: up to 64 evenly spaced), the channel-magnitude spread
    ("quantization difficulty") of X before and after smoothing and of the
    folded W, and the static-scale clip count when that mode ran."""
    if rows is None:
        n = min(64, layer.tokens)
        rows = torch.linspace(0, layer.tokens - 1, n).round().to(torch.int32)
    rows = torch.as_tensor(rows, dtype=torch.int32)
    act = sq.act_quant_error(layer.x, layer.s_inv, layer.xq, layer.x_scale)
    wgt = sq.weight_quant_error(layer.w, layer.s, layer.wq, layer.w_scale)
    lay = sq.layer_error(layer.x, layer.w, layer.y, rows)
    x_before = sq.channel_stats(layer.amax_x)
    x_after = sq.channel_stats(layer.amax_x, layer.s_inv)
    w_before = sq.channel_stats(layer.amax_w)
    w_after = sq.channel_stats(layer.amax_w, layer.s)
    out = {
        "alpha": layer.alpha,
        "act_error": float(act.sum()), "weight_error": float(wgt.sum()),
        "layer_error": float(lay.sum()), "layer_error_rows": rows.numel(),
        "x_difficulty": float(x_before[1]), "x_difficulty_smoothed": float(x_after[1]),
        "w_difficulty": float(w_before[1]), "w_difficulty_smoothed": float(w_after[1]),
    }
    if layer.act_scale == "static":
        out["clipped"] = int(layer.clipped.item())
    return out


def alpha_sweep(x: torch.Tensor, w: torch.Tensor, alphas, codes: str | None = None,
                act_scale: str = "dynamic", rows=None) -> list:
    """Run the whole path at each smoothing strength and return the
    diagnostics of each (the pages select the strength on calibration or
    development data; this gives the measurements to select by)."""
    tokens, cin = x.shape
    cout = w.shape[1]
    dtype = "bf16" if x.dtype == torch.bfloat16 else "f32"
    results = []
    for a in alphas:
        layer = Layer(tokens, cin, cout, dtype, float(a), codes, device=x.device, act_scale=act_scale)
        layer.load(x, w)
        layer.step()
        results.append(diagnose(layer, rows))
    torch.cuda.synchronize()
    return results


def smooth_rotation_study(x: torch.Tensor, w: torch.Tensor, alpha: float = 0.5, qmax: int = 7,
                          codes: str = "bf16", rows=None) -> dict:
    """The four preprocessing choices the Smooth Rotation review compares,
    each quantized to +-qmax codes on both operands (qmax = 7: W4A4) and run
    through the same GEMM: 'original', 'smooth', 'rotate', 'smooth_rotate'.
    Returns each one's layer error (sum over the sampled tokens of the
    squared difference to the unquantized X W) and its activation-scale
    maximum.  Cin must be a power of two for the rotated variants."""
    tokens, cin = x.shape
    if rows is None:
        n = min(64, tokens)
        rows = torch.linspace(0, tokens - 1, n).round().to(torch.int32)
    rows = torch.as_tensor(rows, dtype=torch.int32)
    amax_x = sq.calibrate_absmax(x, 0)
    amax_w = sq.calibrate_absmax(w, 1)
    s, s_inv = sq.smooth_factors(amax_x, amax_w, alpha)
    out = {}
    for name, smooth, rotate in (("original", False, False), ("smooth", True, False),
                                 ("rotate", False, True), ("smooth_rotate", True, True)):
        xq, xs = sq.rotate_quant_act(x, s_inv if smooth else None, rotate, qmax, codes)
        wq, ws = sq.rotate_fold_quantize_weight(w, s if smooth else None, rotate, qmax, codes)
        y = sq.w8a8_gemm(xq, xs, wq, ws)
        err = sq.layer_error(x, w, y, rows)
        out[name] = {"layer_error": float(err.sum()), "x_scale_max": float(xs.max())}
    torch.cuda.synchronize()
    return out

"""CPU oracle for the SmoothQuant W8A8 linear-layer path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports or runs
this module: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may.  It shares
no code with the CUDA library; both sides only consume the seeded inputs
of ``w8a8_post_quantization_02_b300.synth``.

Each function is the plain definition of one step, written with numpy
float32 arithmetic (IEEE-754 binary32, round-to-nearest-even, no fused
multiply-add), one library primitive per step where one is used, and no
blocking or reordering.  Sources (page title, then the passage):

* "Move activation scale without changing the real linear map"
  (study.greatitself.com, activation outliers and smoothing), paragraph 1:
  with X [tokens x Cin] and W [Cin x Cout], Y = XW equals (X S^-1)(S W)
  for a positive invertible diagonal S; scaling the other dimension of W
  is a different map; the factors must be finite and nonzero.
  Paragraph 3: an explicit runtime step multiplying activations by S^-1,
  and one compensation shared by every consumer of an activation.
* pith.science review of arXiv 2506.01967 ("Smooth Rotation"),
  ``key_machinery``: s_j = sqrt(max|X_j| / max|W_j|) from per-channel
  maxima of activations and weights; ``core_discovery``: symmetric
  round-to-nearest quantization.
* learn-kernels.com "Quantization", paragraph 2: both operands of the
  matmul quantized to INT8, the transform applied offline before serving.

Readings where the pages are silent:

1. general smoothing strength: s_j = max|X_j|^a / max|W_j|^(1-a); a = 0.5
   is the printed case.  Each power is the correctly rounded binary32
   value of the real power (computed here with 256-bit mpmath), 1 - a is
   a binary32 subtraction, the quotient one binary32 division.
2. "finite and nonzero": statistics are floored at 1e-5 before the powers,
   and s is clamped to [1e-5, 1e5]; non-finite statistics raise the
   non-finite flag and give s = 1.
3. the runtime scaling multiplies by S^-1, i.e. X'[t,j] = X[t,j] * (1/s_j)
   with 1/s_j one binary32 division; the fold multiplies W's rows (input
   channels) by s_j.
4. symmetric INT8 quantizer (the review's ``core_discovery``: symmetric
   round-to-nearest) with scale d = amax / 127 (binary32 division; d = 1
   when amax == 0) and codes clamp(rne(v / d), -127, 127), v / d one
   binary32 division (the plain definition of round(v / step)); per output
   channel for W, per token (dynamic) for X.
5. the GEMM accumulates exactly (int64 here) and its epilogue rounds
   acc * x_scale * w_scale, evaluated in float64, once to bf16 (RNE).
"""
from __future__ import annotations

import math

import numpy as np

try:
    import mpmath
except ImportError:  # pragma: no cover - mpmath ships with sympy in this image
    mpmath = None

F32 = np.float32
STAT_FLOOR = F32(1e-5)
S_MIN = F32(1e-5)
S_MAX = F32(1e5)
QMAX = 127


# --------------------------------------------------------------------------
# step 1: calibration statistics
# --------------------------------------------------------------------------
def calibrate_absmax(a, axis: int, prev=None) -> np.ndarray:
    """Per-channel max |a| (Smooth Rotation review, ``key_machinery``).

    ``axis=0`` reduces over rows (X [tokens x Cin] -> [Cin]); ``axis=1``
    reduces over columns (W [Cin x Cout] -> [Cin]).  ``prev`` gives a
    running maximum over calibration batches (the SmoothQuant glossary
    page: statistics are collected on a small calibration set).  NaN
    propagates, so a NaN anywhere makes that channel's statistic NaN.
    """
    a32 = np.asarray(a, dtype=F32)
    m = np.max(np.abs(a32), axis=axis).astype(F32)
    if prev is not None:
        m = np.maximum(np.asarray(prev, dtype=F32), m).astype(F32)
    return m


# --------------------------------------------------------------------------
# step 2: smoothing factors
# --------------------------------------------------------------------------
def rn32_pow(x, y) -> np.float32:
    """Correctly rounded binary32 value of x**y for finite x > 0 (reading 1)."""
    x = F32(x)
    y = F32(y)
    assert np.isfinite(x) and x > 0 and np.isfinite(y)
    if y == 0:
        return F32(1.0)
    if y == 1:
        return x
    with mpmath.workprec(256):
        v = mpmath.power(mpmath.mpf(float(x)), mpmath.mpf(float(y)))
        f = F32(float(v))
        cands = (np.nextafter(f, F32(0)), f, np.nextafter(f, F32(np.inf)))

        def key(c):
            return (abs(mpmath.mpf(float(c)) - v), int(np.asarray(c, F32).view(np.uint32)) & 1)

        return F32(min(cands, key=key))


def smooth_factors(amax_x, amax_w, alpha):
    """s_j = max|X_j|^a / max|W_j|^(1-a), clamped finite and nonzero.

    Smooth Rotation review (``key_machinery``) prints the a = 0.5 case;
    the first page (paragraph 1) requires finite, nonzero factors.
    Returns ``(s, s_inv, nonfinite)`` where ``s_inv = 1/s`` (one binary32
    division each) is the S^-1 that the runtime step multiplies by.
    """
    ax_all = np.asarray(amax_x, dtype=F32)
    aw_all = np.asarray(amax_w, dtype=F32)
    a = F32(alpha)
    b = F32(F32(1.0) - a)
    s = np.empty(ax_all.shape[0], dtype=F32)
    nonfinite = False
    with np.errstate(over="ignore"):
        for j in range(ax_all.shape[0]):
            ax, aw = ax_all[j], aw_all[j]
            if not (np.isfinite(ax) and np.isfinite(aw)):
                s[j] = F32(1.0)
                nonfinite = True
                continue
            ax = max(ax, STAT_FLOOR)
            aw = max(aw, STAT_FLOOR)
            p = rn32_pow(ax, a)
            q = rn32_pow(aw, b)
            sj = F32(p / q)
            s[j] = min(max(sj, S_MIN), S_MAX)
    s_inv = (F32(1.0) / s).astype(F32)
    return s, s_inv, nonfinite


# --------------------------------------------------------------------------
# shared quantizer definition (reading 4)
# --------------------------------------------------------------------------
def _scale(amax: np.ndarray):
    """d = amax / 127 (one binary32 division), 1 where amax == 0; and
    whether any amax is non-finite."""
    amax = np.asarray(amax, dtype=F32)
    nonfinite = bool((~np.isfinite(amax)).any())
    with np.errstate(invalid="ignore", over="ignore"):
        d = (amax / F32(QMAX)).astype(F32)
        d = np.where(amax == 0, F32(1.0), d).astype(F32)
    return d, nonfinite


def _quotients(v: np.ndarray, d: np.ndarray) -> np.ndarray:
    """v / d, one IEEE binary32 division per element."""
    with np.errstate(invalid="ignore", over="ignore", divide="ignore"):
        return (np.asarray(v, F32) / np.asarray(d, F32)).astype(F32)


def _codes(v: np.ndarray, d: np.ndarray) -> np.ndarray:
    """clamp(rne(v / d), -127, 127); a NaN quotient gives code 0."""
    t = _quotients(v, d)
    with np.errstate(invalid="ignore", over="ignore"):
        r = np.rint(t)             # round half to even
        r = np.clip(r, -QMAX, QMAX)
        r = np.where(np.isnan(r), 0, r)
    return r.astype(np.int8)


# --------------------------------------------------------------------------
# step 3: offline fold + per-output-channel weight quantization
# --------------------------------------------------------------------------
def fold_quantize_weight(w, s, return_folded: bool = False):
    """Fold diag(s) into W's rows, then quantize each output channel.

    First page, paragraph 1: S multiplies W on the input-channel side
    (rows of the [Cin x Cout] weight).  learn-kernels "Quantization",
    paragraph 2: the transform is applied offline and W is quantized to
    INT8.  Returns ``wq`` int8 [Cout x Cin] (each output channel's codes
    contiguous), ``w_scale`` float32 [Cout] and the non-finite flag; with
    ``return_folded`` also the binary32 folded weight W' [Cin x Cout].
    """
    w32 = np.asarray(w, dtype=F32)
    s32 = np.asarray(s, dtype=F32)
    with np.errstate(over="ignore", invalid="ignore"):
        wf = (s32[:, None] * w32).astype(F32)
    amax = np.max(np.abs(wf), axis=0).astype(F32)
    d, nonfinite = _scale(amax)
    q = _codes(wf, d[None, :])
    wq = np.ascontiguousarray(q.T)
    if return_folded:
        return wq, d, nonfinite, wf
    return wq, d, nonfinite


# --------------------------------------------------------------------------
# step 4: runtime X * S^-1 fused with dynamic per-token quantization
# --------------------------------------------------------------------------
def quant_act(x, s_inv, return_scaled: bool = False):
    """X' = X * (1/s) per channel, then per-token symmetric INT8 codes.

    First page, paragraph 3 (the runtime scaling step multiplying by S^-1);
    learn-kernels "Quantization", paragraph 2 (activations to INT8).
    Returns ``xq`` int8 [tokens x Cin], ``x_scale`` float32 [tokens] and
    the non-finite flag; with ``return_scaled`` also X' in binary32.
    """
    x32 = np.asarray(x, dtype=F32)
    si = np.asarray(s_inv, dtype=F32)
    with np.errstate(over="ignore", invalid="ignore"):
        xs = (x32 * si[None, :]).astype(F32)
    amax = np.max(np.abs(xs), axis=1).astype(F32) if xs.shape[1] else np.zeros(xs.shape[0], F32)
    d, nonfinite = _scale(amax)
    q = _codes(xs, d[:, None])
    if return_scaled:
        return q, d, nonfinite, xs
    return q, d, nonfinite


# --------------------------------------------------------------------------
# step 4, static variant: one calibrated scale per activation tensor
# --------------------------------------------------------------------------
def static_act_scale(amax_x, s_inv):
    """Per-tensor activation scale from the calibration statistics.

    SmoothQuant glossary (dataterminology.com): the method is
    calibration-based, its statistics come from a small calibration set.
    Reading: the activation scale may be fixed from those statistics too,
    d = max over the tensor of |X'| / 127 with X' = X * (1/s).  Because a
    binary32 multiply by a fixed positive factor is monotone in |x|, the
    largest |X'[t, j]| over tokens is RN(max_t |X[t, j]| * s_inv[j]), so d
    follows from the per-channel maxima alone.  Returns ``(d, nonfinite)``.
    """
    ax = np.asarray(amax_x, dtype=F32)
    si = np.asarray(s_inv, dtype=F32)
    with np.errstate(over="ignore", invalid="ignore"):
        v = (ax * si).astype(F32)          # one binary32 multiply per channel
    m = F32(np.max(v)) if v.size else F32(0)
    if np.isnan(v).any():
        m = F32(np.nan)
    d, nonfinite = _scale(np.array([m], dtype=F32))
    return F32(d[0]), nonfinite


def quant_act_static(x, s_inv, d):
    """X' = X * (1/s), codes with one fixed scale d for every token.

    Same quantizer as ``quant_act`` (reading 4) with the per-token scale
    replaced by the calibrated d: codes clamp(rne(X' / d), -127, 127).
    Runtime activations may exceed the calibration maximum, so the clamp
    can act; ``clipped`` counts the elements it changed (a quotient that
    overflows to infinity, like a non-finite X', saturates uncounted).
    Returns ``(xq, x_scale, clipped)`` with x_scale = d for every token, so
    the GEMM's epilogue is unchanged.
    """
    x32 = np.asarray(x, dtype=F32)
    si = np.asarray(s_inv, dtype=F32)
    d = F32(d)
    with np.errstate(over="ignore", invalid="ignore"):
        xs = (x32 * si[None, :]).astype(F32)
    t = _quotients(xs, np.full((xs.shape[0], 1), d, dtype=F32))
    r = np.rint(t)
    clipped = int(np.count_nonzero(np.isfinite(r) & (np.abs(r) > QMAX)))
    q = _codes(xs, np.full((xs.shape[0], 1), d, dtype=F32))
    return q, np.full(xs.shape[0], d, dtype=F32), clipped


# --------------------------------------------------------------------------
# step 4 folded into the preceding normalization
# --------------------------------------------------------------------------
def fold_norm_gain(gamma, s_inv):
    """gamma'_j = RN32(gamma_j * (1/s_j)).

    First page, paragraph 3: instead of an extra runtime scaling kernel the
    inverse factors may be folded into the preceding operation, provided
    every consumer keeps its compensation (one s shared by all consumers of
    the normalized activation).  Reading: the preceding operation is an RMS
    normalization with a per-channel gain (LLaMA-style layers), whose gain
    absorbs S^-1.
    """
    return (np.asarray(gamma, F32) * np.asarray(s_inv, F32)).astype(F32)


def sum_squares_f32(row) -> np.float32:
    """The exact sum of the squares of a binary32 row, rounded once to
    binary32 (nearest, ties to even).

    math.fsum gives the float64 rounding of the exact sum; rounding that
    to binary32 equals rounding the exact sum directly unless the float64
    value is itself a binary32 midpoint, in which case the exact sum (as an
    integer multiple of 2^-300) decides.
    """
    import math
    vals = np.asarray(row, F32)
    s64 = math.fsum((vals.astype(np.float64) ** 2).tolist())   # squares exact in float64
    f = F32(s64)
    if float(f) == s64 or not np.isfinite(f):
        return f
    nb = np.nextafter(f, F32(np.inf) if s64 > float(f) else F32(0))
    mid = (float(f) + float(nb)) / 2.0                        # exact: both binary32
    if s64 != mid:
        return f
    # exact: h = m * 2^(e - 150), h^2 * 2^300 = m^2 * 2^(2e)
    bits = vals.view(np.uint32) & np.uint32(0x7FFFFFFF)
    total = 0
    for b in bits.tolist():
        e = b >> 23
        m = (b & 0x7FFFFF) | (0x800000 if e else 0)
        total += (m * m) << (2 * max(e, 1))
    from fractions import Fraction
    exact = Fraction(total, 2 ** 300)
    mid_f = Fraction(mid)
    if exact > mid_f:
        return F32(max(float(f), float(nb)))
    if exact < mid_f:
        return F32(min(float(f), float(nb)))
    return f if (int(np.asarray(f).view(np.uint32)) & 1) == 0 else nb


def rms_inverse(h, eps):
    """Per token r_t = RN(1 / RN(sqrt(RN(RN(S / K) + eps)))) in binary32,
    where S is the exact sum of squares rounded once to binary32
    (``sum_squares_f32``) and every step is one IEEE binary32 operation."""
    h32 = np.asarray(h, F32)
    K = F32(h32.shape[1])
    e32 = F32(eps)
    out = np.empty(h32.shape[0], F32)
    with np.errstate(over="ignore", divide="ignore", invalid="ignore"):
        for t in range(h32.shape[0]):
            s = sum_squares_f32(h32[t])
            ms = F32(F32(s / K) + e32)
            out[t] = F32(F32(1.0) / np.sqrt(ms))
    return out


def rmsnorm_quant_act(h, gamma_folded, eps, return_scaled=False):
    """X' = RN32(RN32(h * r_t) * gamma'_j), then the dynamic per-token
    quantizer of step 4 (reading 4) on X'.  Returns ``(xq, x_scale,
    nonfinite)`` (and X' with ``return_scaled``)."""
    h32 = np.asarray(h, F32)
    r = rms_inverse(h32, eps)
    with np.errstate(over="ignore", invalid="ignore"):
        xs = ((h32 * r[:, None]).astype(F32) * np.asarray(gamma_folded, F32)[None, :]).astype(F32)
    amax = np.max(np.abs(xs), axis=1).astype(F32) if xs.shape[1] else np.zeros(xs.shape[0], F32)
    d, nonfinite = _scale(amax)
    q = _codes(xs, d[:, None])
    if return_scaled:
        return q, d, nonfinite, xs
    return q, d, nonfinite


# --------------------------------------------------------------------------
# step 5: INT8 x INT8 -> exact accumulators -> bf16 epilogue
# --------------------------------------------------------------------------
def int_accumulate(xq, wq, rows=None) -> np.ndarray:
    """acc[t, n] = sum_j xq[t, j] * wq[n, j], exactly (int64 result).

    The library primitive is a float64 matmul on integer-valued operands:
    every product is at most 127^2 and every partial sum an integer far
    below 2^53, so each float64 operation is exact whatever the order.
    ``rows`` restricts the result to those tokens.
    """
    a = np.asarray(xq)
    if rows is not None:
        a = a[np.asarray(rows)]
    acc = a.astype(np.float64) @ np.asarray(wq).astype(np.float64).T
    acc = acc.astype(np.int64)
    assert np.abs(acc).max(initial=0) < 2 ** 31
    return acc


def bf16_rne_bits(v: np.ndarray) -> np.ndarray:
    """Round float64 values to bfloat16 with round-half-to-even (uint16 bits).

    Handles zeros, normals and values below bf16's normal range (which
    round on bf16's subnormal grid); |v| beyond bf16's largest finite
    value becomes infinity.
    """
    v = np.ascontiguousarray(v, dtype=np.float64)
    sign = (np.signbit(v)).astype(np.uint16) << np.uint16(15)
    a = np.abs(v)
    out = np.zeros(v.shape, dtype=np.uint16)
    # exponent of each |v| (2^e <= |v| < 2^(e+1)); grid spacing 2^(e-7),
    # but never finer than the subnormal spacing 2^-133.
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0))).astype(np.int64)
    # correct a possible off-by-one of floor(log2) near powers of two
    e = np.where(np.ldexp(1.0, e) > a, e - 1, e)
    e = np.where(np.ldexp(1.0, e + 1) <= a, e + 1, e)
    q = np.maximum(e - 7, -133)
    m = np.ldexp(a, -q)            # exact scaling by a power of two
    r = np.rint(m)                 # RNE on the bf16 grid
    val = np.ldexp(r, q)           # exact value, representable in bf16
    with np.errstate(over="ignore"):
        f32 = val.astype(np.float32)   # exact (bf16 grid is a subset of f32)
    bits = (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    big = val > 3.3895313892515355e38  # largest finite bf16
    bits = np.where(big, np.uint16(0x7F80), bits)
    out = np.where(a > 0, bits, np.uint16(0)) | sign
    nan = np.isnan(v)
    out = np.where(nan, np.uint16(0x7FC0), out)
    return out.astype(np.uint16)


def w8a8_gemm(xq, x_scale, wq, w_scale, rows=None):
    """Y = bf16(acc * x_scale[t] * w_scale[n]) with exact int accumulators.

    learn-kernels "Quantization", paragraph 2 (the matmul runs on INT8
    operands).  Returns ``(acc int64 [t x n], y bf16 bits uint16)``;
    ``rows`` limits the work to a subset of tokens.
    """
    acc = int_accumulate(xq, wq, rows)
    xs = np.asarray(x_scale, dtype=F32)
    if rows is not None:
        xs = xs[np.asarray(rows)]
    ws = np.asarray(w_scale, dtype=F32)
    y = acc.astype(np.float64) * xs.astype(np.float64)[:, None] * ws.astype(np.float64)[None, :]
    return acc, bf16_rne_bits(y)


# --------------------------------------------------------------------------
# diagnostics: the second half of the validation order
# --------------------------------------------------------------------------
F64 = np.float64


def act_quant_error(x, s_inv, xq, x_scale):
    """Per token: sum_j (X'[t, j] - xq[t, j] * x_scale[t])^2 in float64.

    First page, paragraph 4: after the unquantized rewrite checks out,
    quantize and measure activation error and clipping separately.  X' is
    the binary32 X * (1/s) the quantizer saw; each difference is exact in
    float64, the squares and the sum are rounded in float64.
    """
    xs = (np.asarray(x, F32) * np.asarray(s_inv, F32)[None, :]).astype(F32).astype(F64)
    deq = np.asarray(xq).astype(F64) * np.asarray(x_scale, F32).astype(F64)[:, None]
    return ((xs - deq) ** 2).sum(axis=1)


def weight_quant_error(w, s, wq, w_scale):
    """Per output channel: sum_j (W'[j, n] - wq[n, j] * w_scale[n])^2 in float64
    (first page, paragraph 4: weight reconstruction error).  W' is the
    binary32 fold s_j * W[j, n]."""
    wf = (np.asarray(s, F32)[:, None] * np.asarray(w, F32)).astype(F32).astype(F64)
    deq = np.asarray(wq).astype(F64).T * np.asarray(w_scale, F32).astype(F64)[None, :]
    return ((wf - deq) ** 2).sum(axis=0)


def layer_error(x, w, y_bits, rows):
    """Per sampled token t: sum_n ((X W)[t, n] - Y[t, n])^2 in float64.

    Smooth Rotation review (referee report summary): the layer-wise squared
    Frobenius quantization error; here against the layer's bf16 output Y
    (bit patterns of the whole [tokens x Cout] output; the rows listed are
    used), with X W formed in float64 from the unquantized inputs.
    """
    rows = np.asarray(rows)
    ref = np.asarray(x, F32)[rows].astype(F64) @ np.asarray(w, F32).astype(F64)
    yb = np.asarray(y_bits, np.uint16)[rows]          # Y is the whole output [tokens x Cout]
    y = (yb.astype(np.uint32) << np.uint32(16)).view(np.float32)
    return ((ref - y.astype(F64)) ** 2).sum(axis=1)


def channel_stats(amax, scale=None):
    """(mean, population standard deviation) of the per-channel magnitudes
    max|X_j| (times ``scale`` in binary32 when given, i.e. after smoothing).
    Smooth Rotation review: "quantization difficulty" is the standard
    deviation of channel magnitudes."""
    v = np.asarray(amax, F32)
    if scale is not None:
        v = (v * np.asarray(scale, F32)).astype(F32)
    v = v.astype(F64)
    mean = v.sum() / v.size
    return mean, float(np.sqrt(((v - mean) ** 2).sum() / v.size))


# --------------------------------------------------------------------------
# Smooth Rotation: smoothing, then a Hadamard rotation, low-bit codes
# --------------------------------------------------------------------------
def fwht(v):
    """Unnormalized fast Walsh-Hadamard transform along the last axis
    (length a power of two), Sylvester ordering: stages h = 1, 2, 4, ...,
    each butterfly (a, b) -> (a + b, a - b) one binary32 addition and one
    subtraction.  Equals v @ H_d with H_d the Sylvester Hadamard matrix."""
    x = np.array(v, dtype=F32, copy=True)
    d = x.shape[-1]
    assert d >= 1 and d & (d - 1) == 0, "length must be a power of two"
    lead = x.shape[:-1]
    h = 1
    while h < d:
        y = x.reshape(lead + (d // (2 * h), 2, h))
        a, b = y[..., 0, :], y[..., 1, :]
        x = np.stack(((a + b).astype(F32), (a - b).astype(F32)), axis=-2).reshape(lead + (d,))
        h *= 2
    return x


def _rows_quantized(z, qmax):
    """Per-row symmetric quantization with codes in [-qmax, qmax]: the
    quantizer of reading 4 with 127 replaced by qmax."""
    z = np.asarray(z, F32)
    amax = np.max(np.abs(z), axis=1).astype(F32)
    nonfinite = bool((~np.isfinite(amax)).any())
    with np.errstate(invalid="ignore", over="ignore"):
        d = (amax / F32(qmax)).astype(F32)
        d = np.where(amax == 0, F32(1.0), d).astype(F32)
    t = _quotients(z, d[:, None])
    with np.errstate(invalid="ignore", over="ignore"):
        r = np.clip(np.rint(t), -qmax, qmax)
        r = np.where(np.isnan(r), 0, r)
    return r.astype(np.int8), d, nonfinite


def rotate_quant_act(x, s_inv, rotate: bool, qmax: int):
    """Smooth Rotation review (key_machinery): X S^-1 R with R = H_d / sqrt(d)
    (entries +-1/sqrt(d)), then per-token symmetric codes with ``qmax``
    (7 for 4 bits).  Z = fwht(X S^-1) is quantized unnormalized; the 1/d
    of R R^T = H H^T / d is carried on the activation scale as the exact
    power of two 2^-log2(d), so x_scale = RN(max|Z| / qmax) * 2^-log2(d)
    and the GEMM epilogue is unchanged.  ``s_inv`` None: no smoothing;
    ``rotate`` False: no rotation (and no 2^-log2(d))."""
    x32 = np.asarray(x, F32)
    xs = x32 if s_inv is None else (x32 * np.asarray(s_inv, F32)[None, :]).astype(F32)
    z = fwht(xs) if rotate else xs
    q, d, nonfinite = _rows_quantized(z, qmax)
    if rotate:
        d = np.ldexp(d, -int(round(math.log2(xs.shape[1])))).astype(F32)
    return q, d, nonfinite


def rotate_fold_quantize_weight(w, s, rotate: bool, qmax: int):
    """R^T S W per output channel: the folded W'[j, n] = RN(s_j W[j, n]),
    then for each output channel n the transform over j (fwht of the row n
    of W'^T) and per-channel codes with ``qmax``.  Returns ``wq`` [Cout x
    Cin], ``w_scale`` [Cout] (no power of two here: it rides on the
    activation scale) and the non-finite flag."""
    w32 = np.asarray(w, F32)
    wf = w32 if s is None else (np.asarray(s, F32)[:, None] * w32).astype(F32)
    zt = fwht(np.ascontiguousarray(wf.T)) if rotate else np.ascontiguousarray(wf.T)
    return _rows_quantized(zt, qmax)


# --------------------------------------------------------------------------
# the whole path on one layer
# --------------------------------------------------------------------------
def run_path(x, w, alpha, rows=None):
    """Steps 1-5 in order on X [tokens x Cin] and W [Cin x Cout]."""
    amax_x = calibrate_absmax(x, axis=0)
    amax_w = calibrate_absmax(w, axis=1)
    s, s_inv, nf_s = smooth_factors(amax_x, amax_w, alpha)
    wq, w_scale, nf_w = fold_quantize_weight(w, s)
    xq, x_scale, nf_x = quant_act(x, s_inv)
    acc, y = w8a8_gemm(xq, x_scale, wq, w_scale, rows=rows)
    return dict(amax_x=amax_x, amax_w=amax_w, s=s, s_inv=s_inv, wq=wq, w_scale=w_scale,
                xq=xq, x_scale=x_scale, acc=acc, y=y, nonfinite=nf_s or nf_w or nf_x)


def bf16_ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """|ordinal(a) - ordinal(b)| for bf16 bit patterns (sign-magnitude order)."""
    def ordinal(b):
        b = np.asarray(b, dtype=np.uint16).astype(np.int64)
        mag = b & 0x7FFF
        return np.where(b & 0x8000, -mag, mag)
    return np.abs(ordinal(a_bits) - ordinal(b_bits))


__all__ = [
    "calibrate_absmax", "rn32_pow", "smooth_factors", "fold_quantize_weight", "quant_act",
    "static_act_scale", "quant_act_static", "act_quant_error", "weight_quant_error",
    "layer_error", "channel_stats", "fold_norm_gain", "sum_squares_f32", "rms_inverse",
    "rmsnorm_quant_act", "fwht", "rotate_quant_act", "rotate_fold_quantize_weight",
    "int_accumulate", "bf16_rne_bits", "w8a8_gemm", "run_path", "bf16_ulp_distance",
    "STAT_FLOOR", "S_MIN", "S_MAX", "QMAX",
]

if mpmath is None:  # pragma: no cover
    raise ImportError("the oracle needs mpmath for correctly rounded powers")


"""Seeded synthetic inputs for the SmoothQuant W8A8 linear-layer path.

This module only draws numbers. It holds none of the method's arithmetic
(no statistics, smoothing, folding, quantization or matmul), so both the
CUDA path and the CPU oracle may consume what it produces.

Generator
---------
Counter-based SplitMix64 (Steele, Lea & Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014): element ``i`` of stream
``(seed, tensor_id)`` is ``mix64(key + (i + 1) * GAMMA)`` with
``key = mix64(seed * 2**32 + tensor_id + GAMMA)``.  Uniforms take the top
53 bits, ``u = (z >> 11 + 0.5) * 2**-53``, in (0, 1).  Normals use the
Box-Muller cosine branch on the uniform pair ``(u[2i], u[2i+1])``.
Values are formed in float64 and rounded once to the tensor dtype with
round-half-to-even (bf16) or numpy's float32 cast (also RNE).

Workloads
---------
The five linear-layer shapes (tokens x Cin x Cout) stand in for the
LLaMA-7B-class activations and weights the pages study; no dataset or
trained weight is read.  ``make_case`` builds one of them, or any small
case with the same outlier structure for parity tests.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

# tensor ids (one independent stream per drawn tensor)
TID_X, TID_W, TID_XCH, TID_XFAC, TID_TOK, TID_SIGN, TID_W2, TID_W3 = range(1, 9)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, tid: int) -> np.uint64:
    with np.errstate(over="ignore"):
        base = np.array([(seed << 32) + tid], dtype=np.uint64) + GAMMA
        return _mix64(base)[0]


def raw_u64(seed: int, tid: int, start: int, count: int) -> np.ndarray:
    """Counter-based SplitMix64 outputs for positions [start, start+count)."""
    key = _key(seed, tid)
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(key + idx * GAMMA)


def uniform(seed: int, tid: int, count: int, start: int = 0) -> np.ndarray:
    z = raw_u64(seed, tid, start, count)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normal(seed: int, tid: int, count: int, std: float = 1.0) -> np.ndarray:
    """``count`` float64 draws of N(0, std^2), generated in chunks."""
    out = np.empty(count, dtype=np.float64)
    for s in range(0, count, _CHUNK):
        n = min(_CHUNK, count - s)
        u = uniform(seed, tid, 2 * n, start=2 * s)
        u1, u2 = u[0::2], u[1::2]
        out[s:s + n] = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2) * std
    return out


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round float64 to bfloat16 (RNE), returned as uint16 bit patterns.

    Valid for finite values whose magnitude lies in bf16's normal range
    (the generator never draws anything else; asserted).
    """
    v = np.ascontiguousarray(v, dtype=np.float64)
    a = np.abs(v)
    ok = np.isfinite(v) & ((a == 0) | ((a >= 2.0 ** -126) & (a < 3.3e38)))
    assert ok.all(), "value outside the bf16 normal range"
    b = v.view(np.uint64).copy()
    drop = np.uint64(45)  # 52 - 7 explicit mantissa bits
    lsb = (b >> drop) & np.uint64(1)
    b = b + (np.uint64((1 << 44) - 1) + lsb)
    b = b & ~np.uint64((1 << 45) - 1)
    f32 = b.view(np.float64).astype(np.float32)  # exact: <= 8 significant bits
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass
class Case:
    """One linear layer's synthetic inputs.

    ``x``/``w`` hold the raw storage: uint16 bf16 bit patterns when
    ``dtype == "bf16"``, float32 arrays when ``dtype == "f32"``.
    ``x`` is [tokens x cin] row-major, ``w`` is [cin x cout] row-major
    (input channels index the rows of W).  ``splits`` lists the widths of
    the output-channel blocks that share one activation (Q/K/V) and sum to
    ``cout``.
    """
    name: str
    dtype: str
    tokens: int
    cin: int
    cout: int
    alpha: float
    x: np.ndarray
    w: np.ndarray
    splits: tuple = ()

    def x_f32(self) -> np.ndarray:
        return bf16_bits_to_f32(self.x) if self.dtype == "bf16" else self.x

    def w_f32(self) -> np.ndarray:
        return bf16_bits_to_f32(self.w) if self.dtype == "bf16" else self.w


def _to_dtype(v: np.ndarray, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return f64_to_bf16_bits(v)
    return v.astype(np.float32)


def _pick(seed: int, tid: int, n: int, k: int, exclude=()) -> np.ndarray:
    """k distinct indices in [0, n) by a seeded permutation, skipping ``exclude``."""
    order = np.argsort(uniform(seed, tid, n), kind="stable")
    ex = set(int(e) for e in exclude)
    return np.array([int(i) for i in order if int(i) not in ex][:k], dtype=np.int64)


def make_case(name: str, tokens: int, cin: int, cout, *, dtype: str = "bf16",
              x_std: float = 1.0, w_std: float = 0.02, alpha: float = 0.5,
              outlier_frac: float = 0.0, outlier_lo: float = 20.0,
              outlier_hi: float = 100.0, fixed_channels=(), fixed_factor: float = 1.0,
              massive_tokens: int = 0, massive_channels: int = 0,
              massive_value: float = 1000.0, seed: int = 0) -> Case:
    """Draw X [tokens x cin] and W [cin x sum(cout)] with the pages' outlier structure.

    * channel outliers: ``floor(outlier_frac * cin)`` seeded channels are
      multiplied by per-channel factors drawn from U(outlier_lo, outlier_hi);
    * ``fixed_channels`` are multiplied by ``fixed_factor`` (config 1 and
      the two x60 channels of the down_proj case, whose indices are then
      drawn when given as an int count);
    * massive token outliers: ``massive_tokens`` seeded tokens get
      |x| = ``massive_value`` (seeded sign) in ``massive_channels`` seeded
      channels distinct from the scaled ones.
    ``cout`` may be a tuple of widths (shared-activation Q/K/V), drawn as
    independent streams and concatenated along the output channels.
    """
    couts = tuple(cout) if isinstance(cout, (tuple, list)) else (int(cout),)
    n_out = int(sum(couts))
    x = normal(seed, TID_X, tokens * cin, x_std).reshape(tokens, cin)
    scaled = []
    n_out_ch = int(math.floor(outlier_frac * cin))
    if n_out_ch:
        ch = _pick(seed, TID_XCH, cin, n_out_ch)
        fac = outlier_lo + (outlier_hi - outlier_lo) * uniform(seed, TID_XFAC, n_out_ch)
        x[:, ch] *= fac[None, :]
        scaled.extend(ch.tolist())
    if isinstance(fixed_channels, int):
        fixed_channels = _pick(seed, TID_XCH + 100, cin, fixed_channels, scaled).tolist()
    if len(fixed_channels):
        fc = np.asarray(fixed_channels, dtype=np.int64)
        x[:, fc] *= fixed_factor
        scaled.extend(fc.tolist())
    if massive_tokens:
        toks = _pick(seed, TID_TOK, tokens, massive_tokens)
        mch = _pick(seed, TID_XCH + 200, cin, massive_channels, scaled)
        sg = np.where(uniform(seed, TID_SIGN, massive_tokens * massive_channels) < 0.5, -1.0, 1.0)
        x[np.ix_(toks, mch)] = massive_value * sg.reshape(massive_tokens, massive_channels)
    ws = []
    for i, c in enumerate(couts):
        tid = (TID_W, TID_W2, TID_W3)[i] if i < 3 else 100 + i
        ws.append(normal(seed, tid, cin * c, w_std).reshape(cin, c))
    w = ws[0] if len(ws) == 1 else np.concatenate(ws, axis=1)
    return Case(name=name, dtype=dtype, tokens=tokens, cin=cin, cout=n_out, alpha=alpha,
                x=_to_dtype(x, dtype), w=_to_dtype(w, dtype),
                splits=couts if len(couts) > 1 else ())


# The five workloads (tokens x Cin x Cout), with their outlier recipes.
WORKLOADS = {
    "single_linear_64x512x512": dict(
        tokens=64, cin=512, cout=512, dtype="f32", x_std=1.0, w_std=0.02, alpha=0.5,
        fixed_channels=(3, 97, 250, 411), fixed_factor=50.0),
    "decode_7b_16x4096x4096": dict(
        tokens=16, cin=4096, cout=4096, dtype="bf16", x_std=1.0, w_std=0.02, alpha=0.5,
        outlier_frac=0.005, outlier_lo=20.0, outlier_hi=100.0),
    "prefill_upgate_2048x4096x11008": dict(
        tokens=2048, cin=4096, cout=11008, dtype="bf16", x_std=1.0, w_std=0.02, alpha=0.5,
        outlier_frac=0.005, outlier_lo=20.0, outlier_hi=100.0),
    "down_proj_2048x11008x4096": dict(
        tokens=2048, cin=11008, cout=4096, dtype="bf16", x_std=0.5, w_std=0.02, alpha=0.85,
        fixed_channels=2, fixed_factor=60.0, massive_tokens=4, massive_channels=2,
        massive_value=1000.0),
    "qkv_shared_8192x8192x10240": dict(
        tokens=8192, cin=8192, cout=(8192, 1024, 1024), dtype="bf16", x_std=1.0,
        w_std=0.015, alpha=0.8, outlier_frac=0.003, outlier_lo=30.0, outlier_hi=120.0),
}
WORKLOAD_ORDER = list(WORKLOADS)


def workload(name: str, seed: int = 0) -> Case:
    return make_case(name, seed=seed, **WORKLOADS[name])


def workload_dims(name: str):
    p = WORKLOADS[name]
    c = p["cout"]
    return p["tokens"], p["cin"], int(sum(c)) if isinstance(c, tuple) else int(c)

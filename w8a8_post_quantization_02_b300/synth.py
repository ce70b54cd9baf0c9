"""Seeded synthetic inputs for the SmoothQuant W8A8 linear-layer path.

This module only draws numbers. It holds none of the method's arithmetic
(no statistics, smoothing, folding, quantization or matmul), so both the
CUDA path and the CPU oracle may consume what it produces.

Generator
---------
numpy's PCG64 bit generator seeded with ``SeedSequence([seed, tensor_id])``,
one independent stream per drawn tensor; normals from its
``standard_normal`` and uniforms from ``random``.  Values are formed in
float64 and rounded once to the tensor dtype with round-half-to-even
(bf16, below) or numpy's float32 cast (also RNE).  Inputs are generated
once on the host and handed, bit for bit, to both the CUDA path and the
oracle.

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

_CHUNK = 1 << 20

# tensor ids (one independent stream per drawn tensor)
TID_X, TID_W, TID_XCH, TID_XFAC, TID_TOK, TID_SIGN, TID_W2, TID_W3 = range(1, 9)


def _gen(seed: int, tid: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tid])))


def uniform(seed: int, tid: int, count: int) -> np.ndarray:
    """``count`` float64 draws of U(0, 1) from stream (seed, tid)."""
    return _gen(seed, tid).random(count)


def normal(seed: int, tid: int, count: int, std: float = 1.0) -> np.ndarray:
    """``count`` float64 draws of N(0, std^2) from stream (seed, tid)."""
    out = _gen(seed, tid).standard_normal(count)
    if std != 1.0:
        out *= std
    return out


def f64_to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round float64 to bfloat16 (RNE), returned as uint16 bit patterns.

    Valid for finite values whose magnitude lies in bf16's normal range
    (the generator never draws anything else; asserted).
    """
    shape = np.shape(v)
    v = np.ascontiguousarray(v, dtype=np.float64).ravel()
    out = np.empty(v.shape, dtype=np.uint16)
    drop = np.uint64(45)  # 52 - 7 explicit mantissa bits
    half = np.uint64((1 << 44) - 1)
    keep = ~np.uint64((1 << 45) - 1)
    for s in range(0, v.size, _CHUNK):
        a = v[s:s + _CHUNK]
        m = np.abs(a)
        assert np.isfinite(m).all() and (m[m > 0].min(initial=1.0) >= 2.0 ** -126) \
            and m.max(initial=0.0) < 3.3e38, "value outside the bf16 normal range"
        b = a.view(np.uint64).copy()
        lsb = (b >> drop) & np.uint64(1)
        b += half
        b += lsb
        b &= keep
        f32 = b.view(np.float64).astype(np.float32)  # exact: <= 8 significant bits
        out[s:s + _CHUNK] = (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    return out.reshape(shape)


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

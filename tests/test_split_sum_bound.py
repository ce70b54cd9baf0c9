"""The error bound behind the RMS-normalizing quantizer's split sum of squares.

For bf16 rows the kernel sums each thread's squares on the floating-point
pipe: with U = 2^(2 (e - 127)) for the thread's largest exponent field e,
every square is split on the grid 2^-16 U by an add of sigma = 192 U, the
high parts are summed exactly and the low parts in binary32, and the two
sums are turned into a 128-bit fixed-point integer in units of 2^(2e - 362).
The kernel trusts that integer to within 2^-32.6 U of the thread's exact sum
(that is what lets the row's bound check decide the binary32 rounding).

This test restates those binary32 steps with exact rational arithmetic (each
fused multiply-add rounded once, each add by numpy's IEEE binary32) and
checks on adversarial threads that the high sums are exact, the low parts
exact, and the result within the bound.  It does not use the library or the
oracle.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

F32 = np.float32
FAST_LO, FAST_HI = 72, 187


def rn32(v: Fraction) -> float:
    """v rounded once to binary32 (nearest, ties to even; subnormals kept)."""
    if v == 0:
        return 0.0
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    q = max(e - 23, -149)
    n, rem = divmod(a / Fraction(2) ** q, 1)
    n = int(n)
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    r = float(Fraction(n) * Fraction(2) ** q)
    assert abs(r) < 3.4028234663852886e38
    return -r if v < 0 else r


def fma32(a, b, c) -> F32:
    return F32(rn32(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c))))


def f32_from_bits(b: int) -> F32:
    return np.array([b], np.uint32).view(F32)[0]


def split_sum(h: np.ndarray):
    """The kernel's per-thread sum: (fixed-point integer, e, pieces)."""
    bits = h.view(np.uint32) & np.uint32(0x7FFFFFFF)
    et = max(1, int(bits.max()) >> 23)
    assert FAST_LO <= et <= FAST_HI
    sigma = f32_from_bits(((2 * et - 120) << 23) | 0x400000)
    sh, sl = [F32(0), F32(0)], [F32(0), F32(0)]
    his = []
    for k, x in enumerate(h):
        t = fma32(x, x, sigma)
        hi = F32(t - sigma)
        lo = fma32(x, x, -hi)
        # the low part is exact: h^2 = hi + lo
        assert Fraction(float(x)) ** 2 == Fraction(float(hi)) + Fraction(float(lo)) or \
            abs(Fraction(float(x)) ** 2 - Fraction(float(lo))) <= Fraction(2) ** -150
        his.append(hi)
        sh[k & 1] = F32(sh[k & 1] + hi)
        sl[k & 1] = F32(sl[k & 1] + lo)
    s_hi = F32(sh[0] + sh[1])
    s_lo = F32(sl[0] + sl[1])
    U = Fraction(2) ** (2 * (et - 127))
    assert Fraction(float(s_hi)) == sum(Fraction(float(v)) for v in his)  # exact
    H = F32(s_hi * f32_from_bits((397 - 2 * et) << 23))
    assert float(H) == int(H) and 0 <= H <= 2 ** 23
    r = F32(s_lo * f32_from_bits((381 - 2 * et) << 23))
    L = int(np.rint(np.float64(F32(r * F32(2.0 ** 68)))))
    assert abs(L) <= 2 ** 56
    return (int(H) << 92) + (L << 40), et, U


def thread_error(h: np.ndarray) -> float:
    """|fixed-point result - exact sum| / U for one thread."""
    I, et, U = split_sum(h)
    unit = Fraction(2) ** (2 * et - 362)
    exact = sum(Fraction(float(x)) ** 2 for x in h)
    return float(abs(I * unit - exact) / U)


def bf16(v) -> np.ndarray:
    b = np.asarray(v, F32).view(np.uint32)
    b = (b + np.uint32(0x7FFF) + ((b >> 16) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return b.view(F32)


def in_fast_range(h) -> bool:
    et = max(1, int((h.view(np.uint32) & np.uint32(0x7FFFFFFF)).max()) >> 23)
    return FAST_LO <= et <= FAST_HI


def threads():
    rng = np.random.default_rng(2024)
    out = []
    for trial in range(120):
        kind = trial % 6
        if kind == 0:
            v = rng.standard_normal(32)
        elif kind == 1:                      # wide spread inside one thread
            v = rng.standard_normal(32) * np.exp2(rng.integers(-40, 40, 32))
        elif kind == 2:                      # squares just under the split grid
            v = np.exp2(rng.integers(-150, 0, 32).astype(float)) * rng.choice([-1.0, 1.0], 32)
            v[0] = 1.5
        elif kind == 3:                      # bottom of the fast range, tiny neighbours
            v = rng.standard_normal(32) * np.exp2(rng.integers(-140, 0, 32).astype(float)) * 2.0 ** -55
            v[trial % 32] = 1.25 * 2.0 ** -55
        elif kind == 4:                      # top of the fast range
            v = rng.standard_normal(32) * np.exp2(rng.integers(-60, 0, 32).astype(float)) * 2.0 ** 60
            v[trial % 32] = 1.75 * 2.0 ** 60
        else:                                # all values in one binade: many equal grid roundings
            v = (1.0 + rng.random(32)) * 2.0 ** int(rng.integers(-50, 50))
        h = bf16(v.astype(F32))
        if in_fast_range(h):
            out.append(h)
    return out


def test_split_sum_within_bound():
    worst = 0.0
    cases = threads()
    assert len(cases) >= 80
    for h in cases:
        worst = max(worst, thread_error(h))
    assert worst <= 2.0 ** -32.6, math.log2(worst)


@pytest.mark.parametrize("n", [2, 8, 16, 32])
def test_split_sum_short_threads(n):
    rng = np.random.default_rng(n)
    for _ in range(10):
        h = bf16((rng.standard_normal(n) * np.exp2(rng.integers(-30, 30, n))).astype(F32))
        if in_fast_range(h):
            assert thread_error(h) <= 2.0 ** -32.6

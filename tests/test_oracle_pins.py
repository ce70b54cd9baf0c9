"""Pins for the CPU oracle against facts fixed outside the oracle itself.

Each test checks the oracle against the pages' identity and examples,
closed forms, exact rational arithmetic or a library routine the oracle
does not use, so that a dropped term, a wrong sign or index, or a
transposed operand in the oracle fails one of them.
"""
import json
import math
import os
from fractions import Fraction as Fr

import numpy as np
import pytest

from oracle import sq_oracle as O
from w8a8_post_quantization_02_b300 import synth

F32 = np.float32
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- exact helpers
def rn_bin(v: Fr, p: int, emin: int = -126) -> Fr:
    """Round a rational to a binary format with a p-bit significand (RNE)."""
    if v == 0:
        return Fr(0)
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fr(2) ** e > a:
        e -= 1
    elif Fr(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    ulp = Fr(2) ** (e - (p - 1))
    r = round(a / ulp) * ulp  # Fraction.__round__ is half-to-even
    return r if v > 0 else -r


def rn32(v: Fr) -> Fr:
    return rn_bin(v, 24)


def rn_sqrt32(a: Fr) -> Fr:
    """Correctly rounded binary32 sqrt by exact comparison with midpoints."""
    f = F32(math.sqrt(float(a)))
    for _ in range(4):
        lo, hi = np.nextafter(f, F32(0)), np.nextafter(f, F32(np.inf))
        m_lo = (Fr(float(lo)) + Fr(float(f))) / 2
        m_hi = (Fr(float(f)) + Fr(float(hi))) / 2
        if m_lo * m_lo > a:
            f = lo
        elif m_hi * m_hi < a:
            f = hi
        else:
            return Fr(float(f))
    raise AssertionError("sqrt candidate search did not settle")


def bf16_from_fraction(v: Fr) -> int:
    r = rn_bin(v, 8)
    f = F32(float(r))
    return int(f.view(np.uint32) >> 16)


def brute_path(x, w, alpha_kind):
    """Independent exact-rational restatement of steps 1-5 on tiny inputs."""
    T, K = x.shape
    N = w.shape[1]
    X = [[Fr(float(v)) for v in row] for row in x]
    W = [[Fr(float(v)) for v in row] for row in w]
    amax_x = [max(abs(X[t][j]) for t in range(T)) for j in range(K)]
    amax_w = [max(abs(W[j][n]) for n in range(N)) for j in range(K)]
    floor = Fr(float(F32(1e-5)))
    smin, smax = floor, Fr(float(F32(1e5)))
    s = []
    for j in range(K):
        ax, aw = max(amax_x[j], floor), max(amax_w[j], floor)
        if alpha_kind == "half":
            p, q = rn_sqrt32(ax), rn_sqrt32(aw)
        elif alpha_kind == "one":
            p, q = ax, Fr(1)
        else:  # "zero"
            p, q = Fr(1), aw
        s.append(min(max(rn32(p / q), smin), smax))
    s_inv = [rn32(1 / sj) for sj in s]

    def quant(vals):
        amax = max(abs(v) for v in vals)
        d = Fr(1) if amax == 0 else rn32(amax / 127)
        codes = [max(-127, min(127, round(rn32(v / d)))) for v in vals]
        return codes, d

    wf = [[rn32(s[j] * W[j][n]) for n in range(N)] for j in range(K)]
    wq, wsc = [], []
    for n in range(N):
        c, d = quant([wf[j][n] for j in range(K)])
        wq.append(c)
        wsc.append(d)
    xq, xsc = [], []
    for t in range(T):
        c, d = quant([rn32(X[t][j] * s_inv[j]) for j in range(K)])
        xq.append(c)
        xsc.append(d)
    acc = [[sum(xq[t][j] * wq[n][j] for j in range(K)) for n in range(N)] for t in range(T)]
    y = [[bf16_from_fraction(acc[t][n] * xsc[t] * wsc[n]) for n in range(N)] for t in range(T)]
    return dict(amax_x=amax_x, amax_w=amax_w, s=s, s_inv=s_inv, wq=wq, w_scale=wsc,
                xq=xq, x_scale=xsc, acc=acc, y=y)


def _f(a):
    return [Fr(float(v)) for v in np.asarray(a).ravel()]


# ---------------------------------------------------------------- identity / orientation
def _small_case(seed=0, T=48, K=96, N=96, alpha=0.5, dtype="f32"):
    return synth.make_case("pin", T, K, N, dtype=dtype, alpha=alpha, outlier_frac=0.05,
                           outlier_lo=20.0, outlier_hi=100.0, seed=seed)


@pytest.mark.parametrize("alpha", [0.5, 0.85])
def test_identity_unquantized_rewrite(alpha):
    """(X S^-1)(S W) == X W to <= 1e-5 relative in float64, using the oracle's
    own binary32 X' and W' (first page, paragraph 1)."""
    c = _small_case(alpha=alpha)
    x, w = c.x_f32().astype(np.float64), c.w_f32().astype(np.float64)
    ax, aw = O.calibrate_absmax(c.x_f32(), 0), O.calibrate_absmax(c.w_f32(), 1)
    s, s_inv, nf = O.smooth_factors(ax, aw, alpha)
    assert not nf
    _, _, _, wf = O.fold_quantize_weight(c.w_f32(), s, return_folded=True)
    _, _, _, xs = O.quant_act(c.x_f32(), s_inv, return_scaled=True)
    y = x @ w
    y2 = xs.astype(np.float64) @ wf.astype(np.float64)
    rel = np.linalg.norm(y2 - y) / np.linalg.norm(y)
    assert rel <= 1e-5
    # the exact-arithmetic version of the same identity with the oracle's s
    s64 = s.astype(np.float64)
    rel_exact = np.linalg.norm((x / s64) @ (s64[:, None] * w) - y) / np.linalg.norm(y)
    assert rel_exact <= 1e-12


def test_wrong_dimension_is_a_different_map():
    """Scaling W's columns instead of its rows breaks the identity (first page, paragraph 1)."""
    c = _small_case(K=96, N=96)
    x, w = c.x_f32().astype(np.float64), c.w_f32().astype(np.float64)
    s, _, _ = O.smooth_factors(O.calibrate_absmax(c.x_f32(), 0),
                               O.calibrate_absmax(c.w_f32(), 1), 0.5)
    s64 = s.astype(np.float64)
    y = x @ w
    wrong = (x / s64) @ (w * s64[None, :])
    assert np.linalg.norm(wrong - y) / np.linalg.norm(y) > 1e-2
    # and the oracle's fold really scales rows: W'[j, :] == RN32(s_j * W[j, :])
    _, _, _, wf = O.fold_quantize_weight(c.w_f32(), s, return_folded=True)
    j = int(np.argmax(s))
    assert np.array_equal(wf[j], (s[j] * c.w_f32()[j]).astype(F32))
    assert not np.array_equal(wf[:, j], (s[j] * c.w_f32()[:, j]).astype(F32))


def test_matrix_lab_example():
    """diag(0.25, 1): determinant 0.25, e1 -> e1/4, e2 fixed, weight row 0 x4."""
    g = json.load(open(os.path.join(GOLDEN, "matrix_lab.json")))
    # statistics chosen so that alpha = 0.5 gives s = (4, 1)
    s, s_inv, nf = O.smooth_factors(np.array([16.0, 1.0], F32), np.array([1.0, 1.0], F32), 0.5)
    assert not nf
    assert s.tolist() == g["compensating_weight_scale"]
    m = np.diag(s_inv.astype(np.float64))
    assert m.tolist() == g["matrix"]
    assert np.linalg.det(m) == pytest.approx(g["determinant"], abs=0)
    _, _, _, xs = O.quant_act(np.eye(2, dtype=F32), s_inv, return_scaled=True)
    assert xs[0].tolist() == g["image_e1"] and xs[1].tolist() == g["image_e2"]
    w = np.array([[0.5, -1.0, 2.0], [3.0, 0.25, -0.75]], F32)
    _, _, _, wf = O.fold_quantize_weight(w, s, return_folded=True)
    assert wf[0].tolist() == (4 * w[0]).tolist() and wf[1].tolist() == w[1].tolist()


def test_lone_outlier_becomes_geometric_mean():
    """alpha = 0.5: a lone spike o in channel j becomes sqrt(|o| max|W_j|)
    (Smooth Rotation review, key_machinery and load_bearing_attack)."""
    rng_x = synth.normal(3, 1, 32 * 64, 0.01).reshape(32, 64).astype(F32)
    w = synth.normal(3, 2, 64 * 48, 0.02).reshape(64, 48).astype(F32)
    j, t, o = 17, 5, F32(-750.0)
    rng_x[t, j] = o
    ax, aw = O.calibrate_absmax(rng_x, 0), O.calibrate_absmax(w, 1)
    s, s_inv, _ = O.smooth_factors(ax, aw, 0.5)
    _, _, _, xs = O.quant_act(rng_x, s_inv, return_scaled=True)
    want = math.sqrt(abs(float(o)) * float(aw[j]))
    got = float(np.max(np.abs(xs[:, j])))
    assert abs(got - want) <= 4 * float(np.spacing(F32(want)))
    # the weight row grows by the same factor: max|W'_j| = sqrt(|o| max|W_j|) as well
    _, _, _, wf = O.fold_quantize_weight(w, s, return_folded=True)
    assert abs(float(np.max(np.abs(wf[j]))) - want) <= 4 * float(np.spacing(F32(want)))


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("alpha_kind,alpha", [("half", 0.5), ("one", 1.0), ("zero", 0.0)])
def test_brute_force_tiny(seed, alpha_kind, alpha):
    T, K, N = 1 + seed % 4, 2 + (3 * seed) % 7, 1 + (5 * seed) % 4
    x = synth.normal(seed, 11, T * K, 1.0).reshape(T, K).astype(F32)
    w = synth.normal(seed, 12, K * N, 0.02).reshape(K, N).astype(F32)
    if seed % 3 == 0:
        x[:, 0] *= F32(60.0)
    if seed == 4:
        x[0, :] = 0.0  # an all-zero token
        w[:, 0] = 0.0  # an all-zero output channel
    ref = brute_path(x, w, alpha_kind)
    got = O.run_path(x, w, alpha)
    assert _f(got["amax_x"]) == ref["amax_x"]
    assert _f(got["amax_w"]) == ref["amax_w"]
    assert _f(got["s"]) == ref["s"]
    assert _f(got["s_inv"]) == ref["s_inv"]
    assert got["wq"].tolist() == ref["wq"]
    assert _f(got["w_scale"]) == ref["w_scale"]
    assert got["xq"].tolist() == ref["xq"]
    assert _f(got["x_scale"]) == ref["x_scale"]
    assert got["acc"].tolist() == ref["acc"]
    assert got["y"].tolist() == ref["y"]


# ---------------------------------------------------------------- closed forms
def test_calibrate_matches_loops():
    a = synth.normal(1, 1, 37 * 53, 1.0).reshape(37, 53).astype(F32)
    a[3, 4] = -9.0
    col = [max(abs(float(a[t, j])) for t in range(37)) for j in range(53)]
    row = [max(abs(float(a[t, j])) for j in range(53)) for t in range(37)]
    assert O.calibrate_absmax(a, 0).tolist() == col
    assert O.calibrate_absmax(a, 1).tolist() == row
    prev = np.full(53, 2.5, F32)
    assert O.calibrate_absmax(a, 0, prev).tolist() == [max(2.5, v) for v in col]
    b = a.copy()
    b[7, 9] = np.nan
    assert np.isnan(O.calibrate_absmax(b, 0)[9]) and np.isnan(O.calibrate_absmax(b, 1)[7])


def test_rne_ties_and_clamp():
    # s = 1, row absmax 127 -> scale 1 and codes are rne(x) exactly
    x = np.array([[2.5, 3.5, -2.5, 0.5, 1.5, -127.0, 127.0, 126.5, -0.5]], F32)
    q, d, nf = O.quant_act(x, np.ones(x.shape[1], F32))
    assert d.tolist() == [1.0] and not nf
    assert q.tolist() == [[2, 4, -2, 0, 2, -127, 127, 126, 0]]


def division_split_cases(qmax, count, seed, amax_fixed=None):
    """Tuples (amax, v, code, reciprocal code) with |v| < amax where the
    code of v under the scale d = RN(amax / qmax), rne(RN(v / d)), differs
    from the code a reciprocal would give, rne(RN(v * RN(1 / d))).  Found
    and decided in exact rational arithmetic (no binary32 division is used),
    next to half-integer multiples of d, where the two roundings can part.
    ``amax_fixed`` keeps one maximum (one scale) for every case."""
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(100000):
        if len(out) >= count:
            break
        amax = F32(amax_fixed) if amax_fixed is not None else F32(rng.uniform(0.5, 100.0))
        d = rn32(Fr(float(amax)) / qmax)
        inv = rn32(1 / d)
        k = int(rng.integers(0, qmax)) + Fr(1, 2)
        v0 = F32(float(k * d))
        for step in range(-3, 4):
            v = v0
            for _ in range(abs(step)):
                v = np.nextafter(v, F32(np.inf) if step > 0 else F32(-np.inf))
            if not abs(v) < amax:
                continue
            by_div = round(rn32(Fr(float(v)) / d))
            by_rcp = round(rn32(Fr(float(v)) * inv))
            if by_div != by_rcp:
                sign = -1 if len(out) % 2 else 1
                out.append((amax, F32(sign * v), sign * by_div, sign * by_rcp))
                break
    assert len(out) == count, "too few crafted cases found"
    return out


def test_codes_divide_by_the_scale():
    """The quantizer's code is rne(v / d) with v / d one IEEE binary32
    division (the review's core_discovery: symmetric round-to-nearest, i.e.
    round(v / step)), not v times a rounded reciprocal: crafted elements
    whose two codes differ take the division's, for the per-token
    activation quantizer, the per-channel weight quantizer, the static
    scale and the low-bit rows of the rotated quantizer."""
    cases = division_split_cases(127, 8, seed=11)
    for amax, v, want, other in cases:
        assert want != other
        x = np.array([[amax, v]], F32)
        q, d, _ = O.quant_act(x, np.ones(2, F32))
        assert Fr(float(d[0])) == rn32(Fr(float(amax)) / 127)
        assert q.tolist() == [[127, want]]
        wq, _, _ = O.fold_quantize_weight(x.T.copy(), np.ones(2, F32))
        assert wq.tolist() == [[127, want]]
        qs, _, clipped = O.quant_act_static(x, np.ones(2, F32), d[0])
        assert qs.tolist() == [[127, want]] and clipped == 0
    for amax, v, want, other in division_split_cases(7, 6, seed=12):
        q, _, _ = O.rotate_quant_act(np.array([[amax, v]], F32), None, False, 7)
        assert q.tolist() == [[7, want]]


def test_absmax_element_maps_to_127():
    c = _small_case(seed=5)
    s, s_inv, _ = O.smooth_factors(O.calibrate_absmax(c.x_f32(), 0),
                                   O.calibrate_absmax(c.w_f32(), 1), 0.5)
    xq, _, _, xs = O.quant_act(c.x_f32(), s_inv, return_scaled=True)
    arg = np.argmax(np.abs(xs), axis=1)
    assert np.array_equal(np.abs(xq[np.arange(xq.shape[0]), arg]), np.full(xq.shape[0], 127))
    wq, _, _, wf = O.fold_quantize_weight(c.w_f32(), s, return_folded=True)
    argw = np.argmax(np.abs(wf), axis=0)
    assert np.array_equal(np.abs(wq[np.arange(wq.shape[0]), argw]), np.full(wq.shape[0], 127))
    assert xq.min() >= -127 and wq.min() >= -127


def test_zero_rows_and_columns():
    x = np.zeros((3, 8), F32)
    x[1] = np.arange(8, dtype=F32) - 3
    q, d, _ = O.quant_act(x, np.ones(8, F32))
    assert d[0] == 1.0 and d[2] == 1.0 and (q[0] == 0).all() and (q[2] == 0).all()
    w = np.ones((8, 4), F32)
    w[:, 2] = 0
    wq, ws, _ = O.fold_quantize_weight(w, np.ones(8, F32))
    assert ws[2] == 1.0 and (wq[2] == 0).all() and (wq[0] == 127).all()
    # a zero statistic is floored, giving a finite nonzero factor
    s, s_inv, nf = O.smooth_factors(np.array([0.0], F32), np.array([0.0], F32), 0.5)
    assert not nf and s[0] == 1.0 and s_inv[0] == 1.0


def test_nonfinite_statistics_flagged():
    s, _, nf = O.smooth_factors(np.array([np.nan, 2.0], F32), np.array([1.0, np.inf], F32), 0.5)
    assert nf and s.tolist() == [1.0, 1.0]
    _, _, nfx = O.quant_act(np.array([[np.inf, 1.0]], F32), np.ones(2, F32))
    assert nfx


def test_factor_clamp_range():
    s, _, _ = O.smooth_factors(np.array([1e30], F32), np.array([1e-30], F32), 1.0)
    assert s[0] == F32(1e5)
    s, _, _ = O.smooth_factors(np.array([1e-30], F32), np.array([1e30], F32), 0.0)
    assert s[0] == F32(1e-5)


@pytest.mark.parametrize("x,y,want", [
    (16.0, 0.5, 4.0), (4.0, 0.5, 2.0), (0.25, 0.5, 0.5), (16.0, 0.75, 8.0),
    (2.0 ** 20, 0.25, 32.0), (5.0, 1.0, 5.0), (5.0, 0.0, 1.0), (2.0 ** -20, 0.5, 2.0 ** -10)])
def test_pow_exact_cases(x, y, want):
    assert O.rn32_pow(x, y) == F32(want)


def test_pow_half_is_correctly_rounded_sqrt():
    xs = np.abs(synth.normal(7, 1, 400, 30.0)).astype(F32) + F32(1e-3)
    for x in xs:
        assert O.rn32_pow(x, 0.5) == np.sqrt(F32(x))  # IEEE sqrt is correctly rounded


def test_pow_matches_libm_double_away_from_midpoints():
    """The float64 libm pow decides the binary32 rounding whenever it is far
    (relative 1e-14) from a binary32 midpoint; the oracle must agree."""
    xs = np.concatenate([np.abs(synth.normal(9, 1, 300, 50.0)),
                         np.abs(synth.normal(9, 2, 100, 0.02))]).astype(F32) + F32(1e-4)
    checked = 0
    for y in (0.85, 0.15, 0.8, 0.2, 0.3, 0.7, 0.65):
        yf = F32(y)
        for x in xs:
            d = math.pow(float(x), float(yf))
            f = F32(d)
            lo, hi = np.nextafter(f, F32(0)), np.nextafter(f, F32(np.inf))
            m_lo, m_hi = (float(lo) + float(f)) / 2, (float(f) + float(hi)) / 2
            if not (m_lo * (1 + 1e-14) < d < m_hi * (1 - 1e-14)):
                continue
            assert O.rn32_pow(x, yf) == f
            checked += 1
    assert checked > 2700


def test_smoothing_formula_general_alpha():
    """s = x^a / w^(1-a) with a binary32 quotient of the two powers."""
    ax = np.array([3.0, 120.0, 0.5], F32)
    aw = np.array([0.05, 0.02, 0.1], F32)
    s, s_inv, _ = O.smooth_factors(ax, aw, 0.85)
    for j in range(3):
        p = F32(math.pow(float(ax[j]), float(F32(0.85))))
        q = F32(math.pow(float(aw[j]), float(F32(F32(1) - F32(0.85)))))
        assert s[j] == F32(p / q)
        assert s_inv[j] == F32(F32(1) / s[j])


# ---------------------------------------------------------------- GEMM + epilogue
def test_gemm_accumulators_exact():
    rng = np.random.default_rng(0)
    xq = rng.integers(-127, 128, size=(9, 200), dtype=np.int64).astype(np.int8)
    wq = rng.integers(-127, 128, size=(7, 200), dtype=np.int64).astype(np.int8)
    want = xq.astype(np.int64) @ wq.astype(np.int64).T  # integer matmul
    assert np.array_equal(O.int_accumulate(xq, wq), want)
    # the largest magnitude the widest layer can reach (all +-127, K = 11008)
    k = 11008
    a = np.full((2, k), 127, np.int8)
    a[1] = -127
    b = np.full((3, k), 127, np.int8)
    acc = O.int_accumulate(a, b)
    assert acc[0, 0] == 127 * 127 * k and acc[1, 2] == -127 * 127 * k


def test_epilogue_rounding():
    xq = np.array([[1], [1], [1], [3]], np.int8)
    wq = np.array([[1]], np.int8)
    xs = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, 0.5], F32)
    acc, y = O.w8a8_gemm(xq, xs, wq, np.array([1.0], F32))
    assert y[:, 0].tolist() == [0x3F80, 0x3F80, 0x3F82, 0x3FC0]
    for t in range(4):
        assert y[t, 0] == bf16_from_fraction(Fr(int(acc[t, 0])) * Fr(float(xs[t])))


def test_bf16_rounding_matches_exact_rationals():
    v = np.concatenate([synth.normal(2, 3, 2000, 1.0), synth.normal(2, 4, 200, 1e-30),
                        [0.0, -0.0, 1e-39, -3e-40, 2.0 ** -133]])
    bits = O.bf16_rne_bits(v)
    for a, b in zip(v, bits):
        want = bf16_from_fraction(Fr(float(a)))
        if a < 0 or (a == 0 and math.copysign(1, a) < 0):
            want |= 0x8000
        assert int(b) == want, (a, hex(int(b)), hex(want))


def test_ulp_distance_helper():
    a = np.array([0x3F80, 0x3F80, 0x8001, 0x0000], np.uint16)
    b = np.array([0x3F81, 0x3F80, 0x0001, 0x8000], np.uint16)
    assert O.bf16_ulp_distance(a, b).tolist() == [1, 0, 2, 0]



# ---------------------------------------------------------------- static activation scale
def test_static_scale_is_the_tensor_maximum():
    """d from the per-channel maxima equals max|X'| / 127 over every element
    (brute force over the tensor), for mixed signs and outlier channels."""
    c = synth.make_case("st", 97, 160, 8, dtype="bf16", outlier_frac=0.05, seed=3)
    x = c.x_f32()
    si = (0.1 + 3.0 * synth.uniform(5, 50, 160)).astype(F32)
    d, nf = O.static_act_scale(O.calibrate_absmax(x, 0), si)
    brute = max(abs(float(F32(F32(v) * F32(s)))) for row in x for v, s in zip(row, si))
    assert not nf and d == F32(F32(brute) / F32(127))


def test_static_codes_reduce_to_dynamic_for_one_token():
    """With one token calibrated on itself the static scale is that token's
    dynamic scale, so the codes are identical."""
    c = synth.make_case("st1", 1, 256, 8, dtype="bf16", outlier_frac=0.02, seed=4)
    x = c.x_f32()
    si = (0.5 + synth.uniform(6, 51, 256)).astype(F32)
    d, _ = O.static_act_scale(O.calibrate_absmax(x, 0), si)
    qs, xs_s, clipped = O.quant_act_static(x, si, d)
    qd, xs_d, _ = O.quant_act(x, si)
    assert clipped == 0 and np.array_equal(qs, qd) and xs_s[0] == xs_d[0]


def test_static_codes_clip_beyond_calibration():
    """Runtime values past the calibrated maximum saturate at +-127 and are
    counted; a value at exactly 127.5 steps rounds to 128 (half to even)
    and is clipped, 127.25 steps is not."""
    d = F32(1.0)
    si = np.ones(6, F32)
    x = np.array([[127.25, 127.5, -300.0, 254.0, 0.5, -1.5]], F32)
    q, xs, clipped = O.quant_act_static(x, si, d)
    assert q[0].tolist() == [127, 127, -127, 127, 0, -2]
    assert clipped == 3 and xs[0] == F32(1.0)



# ---------------------------------------------------------------- diagnostics
def test_quant_errors_match_exact_rationals():
    """Activation and weight reconstruction errors against the definition in
    exact rational arithmetic on a tiny layer."""
    x = synth.normal(7, 1, 3 * 8, 1.0).reshape(3, 8).astype(F32)
    w = synth.normal(7, 2, 8 * 5, 0.02).reshape(8, 5).astype(F32)
    r = O.run_path(x, w, 0.5)
    ea = O.act_quant_error(x, r["s_inv"], r["xq"], r["x_scale"])
    ew = O.weight_quant_error(w, r["s"], r["wq"], r["w_scale"])
    for t in range(3):
        exact = sum((Fr(float(F32(x[t, j] * r["s_inv"][j]))) - int(r["xq"][t, j]) * Fr(float(r["x_scale"][t]))) ** 2
                    for j in range(8))
        assert abs(Fr(float(ea[t])) - exact) <= exact * Fr(1, 10 ** 12)
    for n in range(5):
        exact = sum((Fr(float(F32(r["s"][j] * w[j, n]))) - int(r["wq"][n, j]) * Fr(float(r["w_scale"][n]))) ** 2
                    for j in range(8))
        assert abs(Fr(float(ew[n])) - exact) <= exact * Fr(1, 10 ** 12)


def test_quant_error_bounds():
    """Round to nearest: every element is off by at most half a step, so the
    error of a row is at most K * (d / 2)^2, and a row that is already a
    multiple of its step has error 0."""
    c = synth.make_case("eb", 40, 96, 24, dtype="bf16", outlier_frac=0.05, seed=9)
    r = O.run_path(c.x_f32(), c.w_f32(), 0.5)
    ea = O.act_quant_error(c.x_f32(), r["s_inv"], r["xq"], r["x_scale"])
    assert (ea <= 96 * (r["x_scale"].astype(np.float64) / 2) ** 2).all() and (ea > 0).all()
    ew = O.weight_quant_error(c.w_f32(), r["s"], r["wq"], r["w_scale"])
    assert (ew <= 96 * (r["w_scale"].astype(np.float64) / 2) ** 2).all()
    grid = np.arange(-127, 128, dtype=F32)[None, :]      # max 127: step exactly 1
    q, d, _ = O.quant_act(grid, np.ones(255, F32))
    assert d[0] == 1.0 and O.act_quant_error(grid, np.ones(255, F32), q, d)[0] == 0.0


def test_layer_error_definition():
    """The layer error of the exact product rounded to bf16 is the rounding
    alone (tiny, bounded by half a bf16 ulp per element), and the error of
    a quantized layer matches a float64 loop."""
    x = synth.normal(8, 1, 4 * 16, 1.0).reshape(4, 16).astype(F32)
    w = synth.normal(8, 2, 16 * 6, 0.1).reshape(16, 6).astype(F32)
    exact = x.astype(np.float64) @ w.astype(np.float64)
    e0 = O.layer_error(x, w, O.bf16_rne_bits(exact), np.arange(4))
    assert (e0 <= 6 * (np.abs(exact).max(axis=1) * 2.0 ** -8) ** 2).all()
    r = O.run_path(x, w, 0.5)
    e = O.layer_error(x, w, r["y"], [1, 3])
    yf = (r["y"].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    loop = [sum((sum(float(x[t, j]) * float(w[j, n]) for j in range(16)) - yf[t, n]) ** 2 for n in range(6))
            for t in (1, 3)]
    assert np.allclose(e, loop, rtol=1e-12, atol=0)


def test_channel_stats_against_statistics_module():
    import statistics
    amax = np.abs(synth.normal(9, 3, 300, 1.0)).astype(F32)
    amax[[5, 77]] *= F32(60.0)
    scale = (0.5 + synth.uniform(9, 4, 300)).astype(F32)
    m, sd = O.channel_stats(amax)
    assert m == pytest.approx(statistics.fmean(amax.astype(float)), rel=1e-13)
    assert sd == pytest.approx(statistics.pstdev(amax.astype(float)), rel=1e-12)
    m2, sd2 = O.channel_stats(amax, scale)
    v = [float(F32(a * b)) for a, b in zip(amax, scale)]
    assert sd2 == pytest.approx(statistics.pstdev(v), rel=1e-12)



# ---------------------------------------------------------------- RMSNorm fold
def test_rms_inverse_against_high_precision():
    """r_t is within 2 binary32 ulps of 1/sqrt(mean(h^2) + eps) computed with
    200-bit arithmetic (five roundings of at most half an ulp each), and a
    constant row of 2 with eps = 0 gives exactly 0.5."""
    import mpmath
    h = synth.normal(11, 1, 6 * 40, 1.0).reshape(6, 40).astype(F32)
    h[2, :] = F32(-3.0)
    h[4, 7] = F32(250.0)
    eps = F32(1e-6)
    r = O.rms_inverse(h, eps)
    with mpmath.workprec(200):
        for t in range(6):
            ss = sum(mpmath.mpf(float(v)) ** 2 for v in h[t])
            exact = float(1 / mpmath.sqrt(ss / 40 + mpmath.mpf(float(eps))))
            assert abs(float(r[t]) - exact) <= 2 * float(np.spacing(F32(exact)))
    assert O.rms_inverse(np.full((1, 64), 2.0, F32), F32(0.0))[0] == F32(0.5)


def test_sum_of_squares_rounds_the_exact_sum():
    """1 + 2^-24 + 2^-80: the float64 sum is the binary32 midpoint 1 + 2^-24
    (ties to even would give 1), but the exact sum lies above it, so the
    correctly rounded binary32 sum is 1 + 2^-23; the exact tie 1 + 2^-24
    itself rounds to even (1)."""
    row = np.array([1.0, 2.0 ** -12, 2.0 ** -40], F32)
    assert O.sum_squares_f32(row) == F32(1.0 + 2.0 ** -23)
    assert O.sum_squares_f32(np.array([1.0, 2.0 ** -12], F32)) == F32(1.0)
    assert O.sum_squares_f32(np.array([3.0, -4.0], F32)) == F32(25.0)


def test_sum_of_squares_sees_terms_below_float64():
    """A square far below float64's reach still decides a tie: 1 + 2^-24 +
    2^-120 (and with the tiny element negative, or several of them) rounds
    up to 1 + 2^-23, while subnormal squares that flush to nothing in binary32
    (2^-130 squared) also count; just below the tie (1 + 2^-24 - 2^-46 +
    2^-70, from 2^-12 (1 - 2^-23) in place of 2^-12) rounds down.  Checked
    against the exact rational sum."""
    from fractions import Fraction
    up = F32(1.0 + 2.0 ** -23)
    for tail in ([2.0 ** -60], [-(2.0 ** -60)], [2.0 ** -70] * 5, [2.0 ** -130], [2.0 ** -149]):
        row = np.array([1.0, 2.0 ** -12] + tail, F32)
        exact = sum(Fraction(float(v)) ** 2 for v in row)
        assert exact > Fraction(1) + Fraction(1, 2 ** 24)
        assert O.sum_squares_f32(row) == up
    below = np.array([1.0, 2.0 ** -12 * (1.0 - 2.0 ** -23)], F32)
    exact = sum(Fraction(float(v)) ** 2 for v in below)
    assert Fraction(1) < exact < Fraction(1) + Fraction(1, 2 ** 24)
    assert O.sum_squares_f32(below) == F32(1.0)


def test_folded_gain_matches_unfolded_path():
    """Folding S^-1 into the gain changes only roundings: X' from the fold
    is within 2 fp32 ulps of RMSNorm-then-X*S^-1, and in exact arithmetic
    the folded layer equals the original X W (first page, paragraph 3)."""
    c = synth.make_case("nf", 24, 64, 32, dtype="f32", outlier_frac=0.05, seed=12)
    h = c.x_f32()
    gamma = (0.5 + synth.uniform(12, 60, 64)).astype(F32)
    eps = F32(1e-5)
    r = O.rms_inverse(h, eps)
    x = ((h * r[:, None]).astype(F32) * gamma[None, :]).astype(F32)      # RMSNorm output
    ax, aw = O.calibrate_absmax(x, 0), O.calibrate_absmax(c.w_f32(), 1)
    s, s_inv, _ = O.smooth_factors(ax, aw, 0.5)
    _, _, _, xs_fold = O.rmsnorm_quant_act(h, O.fold_norm_gain(gamma, s_inv), eps, return_scaled=True)
    _, _, _, xs_plain = O.quant_act(x, s_inv, return_scaled=True)
    ulps = np.abs(xs_fold.view(np.int32).astype(np.int64) - xs_plain.view(np.int32).astype(np.int64))
    assert ulps.max() <= 2
    h64, g64, s64 = h.astype(np.float64), gamma.astype(np.float64), s.astype(np.float64)
    rr = 1.0 / np.sqrt((h64 * h64).mean(axis=1) + float(eps))
    y = ((h64 * rr[:, None]) * g64[None, :]) @ c.w_f32().astype(np.float64)
    y_fold = ((h64 * rr[:, None]) * (g64 / s64)[None, :]) @ (s64[:, None] * c.w_f32().astype(np.float64))
    assert np.linalg.norm(y_fold - y) / np.linalg.norm(y) <= 1e-12



# ---------------------------------------------------------------- Smooth Rotation
def test_fwht_is_the_sylvester_hadamard_product():
    """On integer vectors every butterfly is exact, so the transform equals
    v @ H (scipy's Sylvester Hadamard matrix, integer arithmetic) exactly;
    applying it twice gives d * v; on random floats it matches the float64
    product within the rounding of log2(d) stages."""
    from scipy.linalg import hadamard
    for d in (1, 2, 8, 64, 256):
        v = (np.floor(synth.uniform(d, 70, 3 * d) * 200) - 100).reshape(3, d).astype(F32)
        H = hadamard(d).astype(np.int64)
        assert np.array_equal(O.fwht(v).astype(np.int64), v.astype(np.int64) @ H)
        assert np.array_equal(O.fwht(O.fwht(v)), (d * v).astype(F32))
    d = 1024
    v = synth.normal(5, 71, 4 * d, 1.0).reshape(4, d).astype(F32)
    ref = v.astype(np.float64) @ hadamard(d).astype(np.float64)
    assert np.abs(O.fwht(v) - ref).max() <= 10 * 2.0 ** -24 * np.abs(v).sum(axis=1).max()


def test_rotation_keeps_the_linear_map():
    """(X S^-1 R)(R^T S W) == X W to <= 1e-12 relative in float64 with
    R = H / sqrt(d) orthogonal (Smooth Rotation review, key_machinery)."""
    from scipy.linalg import hadamard
    c = _small_case(K=64, N=32, alpha=0.5)
    x, w = c.x_f32().astype(np.float64), c.w_f32().astype(np.float64)
    s, _, _ = O.smooth_factors(O.calibrate_absmax(c.x_f32(), 0), O.calibrate_absmax(c.w_f32(), 1), 0.5)
    R = hadamard(64).astype(np.float64) / 8.0
    s64 = s.astype(np.float64)
    y2 = ((x / s64) @ R) @ (R.T @ (s64[:, None] * w))
    assert np.linalg.norm(y2 - x @ w) / np.linalg.norm(x @ w) <= 1e-12
    assert np.allclose(R @ R.T, np.eye(64), atol=1e-15)


def test_rotated_lone_outlier_maxima():
    """A token that is zero except one outlier o: rotation spreads it to
    +-o/sqrt(d) everywhere (review Eq (8) with one outlier); after smoothing
    at alpha = 0.5 the outlier is sqrt(|o| max|W_j|) and the rotated maximum
    is sqrt(|o| max|W_j|)/sqrt(d) -- the sqrt(d) denominator, not the
    printed d of Eq (9) (the referee's correction)."""
    d, j, o = 256, 37, F32(-900.0)
    x = np.zeros((1, d), F32)
    x[0, j] = o
    z = O.fwht(x) / F32(16.0)
    assert np.all(np.abs(z) == abs(o) / 16.0)
    w = synth.normal(6, 72, d * 8, 0.02).reshape(d, 8).astype(F32)
    aw = O.calibrate_absmax(w, 1)
    ax = np.full(d, F32(1e-3))
    ax[j] = abs(o)
    s, s_inv, _ = O.smooth_factors(ax, aw, 0.5)
    zs = O.fwht((x * s_inv[None, :]).astype(F32)) / F32(16.0)
    want = math.sqrt(abs(float(o)) * float(aw[j])) / math.sqrt(d)
    assert abs(float(np.abs(zs).max()) - want) <= 4 * float(np.spacing(F32(want)))


def test_rotated_w4a4_codes_and_scales():
    """4-bit codes stay in [-7, 7], each row's largest element maps to +-7,
    the activation scale carries exactly 2^-log2(d), and a layer's codes
    reproduce X W through the unchanged epilogue up to quantization error."""
    c = synth.make_case("sr", 32, 128, 48, dtype="bf16", x_std=0.5, fixed_channels=2, fixed_factor=60.0,
                        massive_tokens=3, massive_channels=2, seed=13)
    x, w = c.x_f32(), c.w_f32()
    s, s_inv, _ = O.smooth_factors(O.calibrate_absmax(x, 0), O.calibrate_absmax(w, 1), 0.5)
    xq, xs, nf1 = O.rotate_quant_act(x, s_inv, True, 7)
    wq, ws, nf2 = O.rotate_fold_quantize_weight(w, s, True, 7)
    assert not (nf1 or nf2)
    assert np.abs(xq).max() == 7 and np.abs(wq).max() == 7
    assert all(np.abs(r).max() == 7 for r in xq) and all(np.abs(r).max() == 7 for r in wq)
    z = O.fwht((x * s_inv[None, :]).astype(F32))
    d_unscaled = (np.max(np.abs(z), axis=1) / F32(7)).astype(F32)
    assert np.array_equal(xs, (d_unscaled / F32(128)).astype(F32))
    acc, _ = O.w8a8_gemm(xq, xs, wq, ws)
    yq = acc * xs.astype(np.float64)[:, None] * ws.astype(np.float64)[None, :]
    y = x.astype(np.float64) @ w.astype(np.float64)
    assert np.linalg.norm(yq - y) / np.linalg.norm(y) < 0.25

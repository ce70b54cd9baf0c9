"""Plant plausible mistakes in the CPU oracle and check that its pins catch
each one.

Every mutation below replaces one oracle function (or helper) with a copy
carrying a single typical slip: a transposed operand, a swapped exponent, a
wrong reduction axis, a different rounding, a dropped factor.  The pins of
tests/test_oracle_pins.py are then run; at least one of them must fail, or
the oracle could carry that mistake unnoticed.  Runs on the CPU only.
"""
import numpy as np
import pytest

from oracle import sq_oracle as O
from tests import test_oracle_pins as P

F32 = np.float32


def _pins():
    calls = [
        lambda: P.test_identity_unquantized_rewrite(0.5),
        lambda: P.test_identity_unquantized_rewrite(0.85),
        P.test_wrong_dimension_is_a_different_map,
        P.test_matrix_lab_example,
        P.test_lone_outlier_becomes_geometric_mean,
        P.test_calibrate_matches_loops,
        P.test_rne_ties_and_clamp,
        P.test_codes_divide_by_the_scale,
        P.test_absmax_element_maps_to_127,
        P.test_zero_rows_and_columns,
        P.test_nonfinite_statistics_flagged,
        P.test_factor_clamp_range,
        P.test_smoothing_formula_general_alpha,
        P.test_gemm_accumulators_exact,
        P.test_epilogue_rounding,
        P.test_static_scale_is_the_tensor_maximum,
        P.test_static_codes_reduce_to_dynamic_for_one_token,
        P.test_static_codes_clip_beyond_calibration,
        P.test_quant_errors_match_exact_rationals,
        P.test_quant_error_bounds,
        P.test_layer_error_definition,
        P.test_channel_stats_against_statistics_module,
        P.test_rms_inverse_against_high_precision,
        P.test_sum_of_squares_rounds_the_exact_sum,
        P.test_fwht_is_the_sylvester_hadamard_product,
        P.test_rotation_keeps_the_linear_map,
        P.test_rotated_lone_outlier_maxima,
        P.test_rotated_w4a4_codes_and_scales,
        P.test_folded_gain_matches_unfolded_path,
    ]
    for seed in range(6):
        for kind, alpha in (("half", 0.5), ("one", 1.0), ("zero", 0.0)):
            calls.append(lambda s=seed, k=kind, a=alpha: P.test_brute_force_tiny(s, k, a))
    return calls


def _some_pin_fails():
    for call in _pins():
        try:
            call()
        except Exception:  # an assertion, or the slip breaking a shape
            return True
    return False


# ---------------------------------------------------------------- the slips
def fold_scales_columns(w, s, return_folded=False):
    w32, s32 = np.asarray(w, F32), np.asarray(s, F32)
    k = min(w32.shape)
    wf = w32.copy()
    wf[:, :k] = (w32[:, :k] * s32[None, :k]).astype(F32)   # columns, not rows
    amax = np.max(np.abs(wf), axis=0).astype(F32)
    d, nf = O._scale(amax)
    q = O._codes(wf, d[None, :])
    wq = np.ascontiguousarray(q.T)
    return (wq, d, nf, wf) if return_folded else (wq, d, nf)


def exponents_swapped(amax_x, amax_w, alpha):
    return ORIG["smooth_factors"](amax_w, amax_x, alpha)


def calibrate_wrong_axis(a, axis, prev=None):
    return ORIG["calibrate_absmax"](a, 1 - axis, prev)


def codes_round_half_up(v, d):
    t = O._quotients(v, d)
    with np.errstate(invalid="ignore", over="ignore"):
        r = np.floor(t + F32(0.5))
        r = np.clip(r, -O.QMAX, O.QMAX)
        r = np.where(np.isfinite(r), r, 0)
    return r.astype(np.int8)


def codes_clamp_128(v, d):
    t = O._quotients(v, d)
    with np.errstate(invalid="ignore", over="ignore"):
        r = np.clip(np.rint(t), -128, 127)
        r = np.where(np.isfinite(r), r, 0)
    return r.astype(np.int8)


def scale_divides_by_128(amax):
    amax = np.asarray(amax, F32)
    with np.errstate(invalid="ignore", over="ignore"):
        d = np.where(amax == 0, F32(1.0), (amax / F32(128))).astype(F32)
    return d, bool((~np.isfinite(amax)).any())


def quotients_by_reciprocal(v, d):
    inv = (F32(1.0) / np.asarray(d, F32)).astype(F32)
    with np.errstate(invalid="ignore", over="ignore"):
        return (np.asarray(v, F32) * inv).astype(F32)             # v * RN(1/d), not RN(v/d)


def act_scale_per_channel(x, s_inv, return_scaled=False):
    x32, si = np.asarray(x, F32), np.asarray(s_inv, F32)
    xs = (x32 * si[None, :]).astype(F32)
    amax = np.max(np.abs(xs), axis=0).astype(F32)           # over tokens, not channels
    d, nf = O._scale(amax)
    q = O._codes(xs, d[None, :])
    tok = np.full(xs.shape[0], d.max(initial=F32(1.0)), F32)
    return (q, tok, nf, xs) if return_scaled else (q, tok, nf)


def epilogue_drops_w_scale(xq, x_scale, wq, w_scale, rows=None):
    return ORIG["w8a8_gemm"](xq, x_scale, wq, np.ones_like(np.asarray(w_scale, F32)), rows)


def s_inv_not_inverted(amax_x, amax_w, alpha):
    s, _, nf = ORIG["smooth_factors"](amax_x, amax_w, alpha)
    return s, s.copy(), nf


def static_scale_ignores_smoothing(amax_x, s_inv):
    return ORIG["static_act_scale"](amax_x, np.ones_like(np.asarray(s_inv, F32)))


def act_error_unscaled(x, s_inv, xq, x_scale):
    return ORIG["act_quant_error"](x, np.ones_like(np.asarray(s_inv, F32)), xq, x_scale)


def weight_error_transposed_scale(w, s, wq, w_scale):
    w32 = np.asarray(w, F32)
    wf = (np.asarray(s, F32)[:, None] * w32).astype(F32).astype(np.float64)
    ws = np.asarray(w_scale, F32).astype(np.float64)
    k = min(wf.shape[0], ws.shape[0])
    deq = np.asarray(wq).astype(np.float64).T.copy()
    deq[:k, :] *= ws[:k, None]                                  # rows, not columns
    return ((wf - deq) ** 2).sum(axis=0)


def stats_sample_std(amax, scale=None):
    v = np.asarray(amax, F32)
    if scale is not None:
        v = (v * np.asarray(scale, F32)).astype(F32)
    v = v.astype(np.float64)
    return v.mean(), float(v.std(ddof=1))


def rms_without_mean(h, eps):
    h32 = np.asarray(h, F32).astype(np.float64)
    return (1.0 / np.sqrt((h32 * h32).sum(axis=1) + float(F32(eps)))).astype(F32)   # sum, not mean


def squares_rounded_through_float64(row):
    import math
    return F32(math.fsum((np.asarray(row, F32).astype(np.float64) ** 2).tolist()))  # double rounding


def gain_folded_by_s(gamma, s_inv):
    return (np.asarray(gamma, F32) / np.asarray(s_inv, F32)).astype(F32)           # times s


def fwht_swapped_butterfly(v):
    x = np.array(v, dtype=F32, copy=True)
    d = x.shape[-1]
    lead = x.shape[:-1]
    h = 1
    while h < d:
        y = x.reshape(lead + (d // (2 * h), 2, h))
        a, b = y[..., 0, :], y[..., 1, :]
        x = np.stack(((a - b).astype(F32), (a + b).astype(F32)), axis=-2).reshape(lead + (d,))
        h *= 2
    return x


def rotate_act_without_power_of_two(x, s_inv, rotate, qmax):
    x32 = np.asarray(x, F32)
    xs = x32 if s_inv is None else (x32 * np.asarray(s_inv, F32)[None, :]).astype(F32)
    return O._rows_quantized(O.fwht(xs) if rotate else xs, qmax)


def rows_quantized_qmax_plus_one(z, qmax):
    return ORIG["_rows_quantized"](z, qmax + 1)


ORIG = {name: getattr(O, name) for name in (
    "fold_quantize_weight", "smooth_factors", "calibrate_absmax", "_codes", "_scale", "_quotients",
    "quant_act", "w8a8_gemm", "static_act_scale", "act_quant_error", "weight_quant_error",
    "channel_stats", "_rows_quantized")}

MUTATIONS = {
    "fold scales W's columns": ("fold_quantize_weight", fold_scales_columns),
    "alpha exponents swapped": ("smooth_factors", exponents_swapped),
    "calibration reduces the other axis": ("calibrate_absmax", calibrate_wrong_axis),
    "codes round half up": ("_codes", codes_round_half_up),
    "codes clamp to [-128, 127]": ("_codes", codes_clamp_128),
    "scale = amax / 128": ("_scale", scale_divides_by_128),
    "codes multiply by a rounded reciprocal": ("_quotients", quotients_by_reciprocal),
    "activation scale per channel": ("quant_act", act_scale_per_channel),
    "epilogue drops w_scale": ("w8a8_gemm", epilogue_drops_w_scale),
    "s_inv not inverted": ("smooth_factors", s_inv_not_inverted),
    "static scale ignores s^-1": ("static_act_scale", static_scale_ignores_smoothing),
    "activation error ignores s^-1": ("act_quant_error", act_error_unscaled),
    "weight error scales rows": ("weight_quant_error", weight_error_transposed_scale),
    "difficulty uses the sample std": ("channel_stats", stats_sample_std),
    "rms uses the sum of squares": ("rms_inverse", rms_without_mean),
    "sum of squares rounded twice": ("sum_squares_f32", squares_rounded_through_float64),
    "butterfly outputs swapped": ("fwht", fwht_swapped_butterfly),
    "rotation drops 1/d": ("rotate_quant_act", rotate_act_without_power_of_two),
    "low-bit grid off by one": ("_rows_quantized", rows_quantized_qmax_plus_one),
    "gain folded by s instead of 1/s": ("fold_norm_gain", gain_folded_by_s),
}


def test_unmutated_oracle_passes_every_pin():
    assert not _some_pin_fails()


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_each_planted_mistake_fails_a_pin(monkeypatch, name):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(O, attr, fn)
    assert _some_pin_fails(), f"no pin catches: {name}"

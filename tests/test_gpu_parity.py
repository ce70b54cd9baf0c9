"""GPU parity: every step of the CUDA path against the CPU oracle.

Each step is fed the oracle's own inputs for that step, so a mismatch
points at one kernel.  Integer work (statistics bits, factors, codes,
scales, accumulators) must match bit for bit; the bf16 outputs within one
bf16 ulp.  Small cases span several tiles and ragged tails; the five
workloads run at full size in the launch configuration the benchmark times,
with all codes compared and the GEMM output compared on sampled tokens.
"""
import numpy as np
import pytest
import torch

from oracle import sq_oracle as O
from w8a8_post_quantization_02_b300 import synth

pytestmark = pytest.mark.gpu
F32 = np.float32


@pytest.fixture(scope="module")
def sq():
    from tests._lib_util import ensure_built
    ensure_built()
    from w8a8_post_quantization_02_b300 import sq as sqmod
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sqmod.check_device(torch.cuda.current_device())
    return sqmod


# ------------------------------------------------------------------ helpers
def dev(a: np.ndarray, dtype: str):
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def f32bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy().astype(F32).view(np.uint32)


def npbits(a) -> np.ndarray:
    return np.asarray(a, F32).view(np.uint32)


def codes_np(t: torch.Tensor) -> np.ndarray:
    """int8 codes from either code format (bf16 codes must be exact integers)."""
    if t.dtype == torch.bfloat16:
        f = t.float().cpu().numpy()
        assert np.array_equal(f, np.rint(f)) and np.abs(f).max(initial=0) <= 127
        return f.astype(np.int8)
    return t.cpu().numpy()


def y_bits(t: torch.Tensor) -> np.ndarray:
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def flags_tensor():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


SMALL = [
    dict(name="single_linear", **synth.WORKLOADS["single_linear_64x512x512"]),
    dict(name="ragged_bf16", tokens=37, cin=80, cout=300, dtype="bf16", outlier_frac=0.05),
    dict(name="ragged_f32", tokens=129, cin=528, cout=33, dtype="f32", outlier_frac=0.02),
    dict(name="one_token", tokens=1, cin=256, cout=264, dtype="bf16", outlier_frac=0.02),
    dict(name="tall_narrow", tokens=300, cin=64, cout=17, dtype="bf16", x_std=0.5, alpha=0.85,
         fixed_channels=2, fixed_factor=60.0, massive_tokens=3, massive_channels=2),
    dict(name="multi_tile", tokens=200, cin=1040, cout=520, dtype="bf16", outlier_frac=0.01,
         alpha=0.8, outlier_lo=30.0, outlier_hi=120.0),
]


def make_small(p):
    p = dict(p)
    name = p.pop("name")
    return synth.make_case(name, **p)


def division_rows(cases, cin, seed):
    """Rows [amax, v, small filler...]: each row's maximum is amax (so its
    scale is RN(amax / qmax)) and v a crafted element whose division and
    reciprocal codes differ."""
    rng = np.random.default_rng(seed)
    x = (rng.uniform(-0.25, 0.25, size=(len(cases), cin)) * np.array([c[0] for c in cases])[:, None]).astype(F32)
    for t, (amax, v, _, _) in enumerate(cases):
        x[t, 0] = amax
        x[t, 1 + t % (cin - 1)] = v
    return x


@pytest.mark.parametrize("codes", ["i8", "bf16"])
def test_codes_divide_by_the_scale(sq, codes):
    """Crafted elements whose code under rne(RN(v / d)) differs from
    rne(RN(v * RN(1/d))): every quantizer (per token, per output channel in
    the single-pass and the two-pass fold, static scale, low-bit rows) gives
    the division's code."""
    from tests.test_oracle_pins import division_split_cases
    cases = division_split_cases(127, 96, seed=31)
    x = division_rows(cases, 48, seed=1)
    ones = torch.ones(48, device="cuda")
    xq_ref, xs_ref, _ = O.quant_act(x, np.ones(48, F32))
    for t, (_, v, want, _) in enumerate(cases):
        assert xq_ref[t, 1 + t % 47] == want
    xq, xs = sq.quant_act(dev(x, "f32"), ones, codes)
    assert np.array_equal(codes_np(xq), xq_ref) and np.array_equal(f32bits(xs), npbits(xs_ref))
    # the fold quantizes the same values per output channel (W = X^T)
    w = np.ascontiguousarray(x.T)
    wq_ref, ws_ref, _ = O.fold_quantize_weight(w, np.ones(48, F32))
    assert np.array_equal(wq_ref, xq_ref)
    wq, ws = sq.fold_quantize_weight(dev(w, "f32"), ones, codes)
    assert np.array_equal(codes_np(wq), wq_ref) and np.array_equal(f32bits(ws), npbits(ws_ref))
    # two-pass fold: a row stride that is not a multiple of 16 bytes
    wpad = torch.zeros(48, 97, device="cuda")
    wpad[:, :96] = dev(w, "f32")
    wq2, ws2 = sq.fold_quantize_weight(wpad[:, :96], ones, codes)
    assert np.array_equal(codes_np(wq2), wq_ref) and np.array_equal(f32bits(ws2), npbits(ws_ref))
    # static scale: one maximum for every row
    scases = division_split_cases(127, 64, seed=32, amax_fixed=37.25)
    xs_rows = division_rows(scases, 48, seed=2)
    d = torch.tensor([np.float32(37.25) / np.float32(127)], device="cuda")
    qs_ref, _, clipped_ref = O.quant_act_static(xs_rows, np.ones(48, F32), d.item())
    clipped = torch.zeros(1, dtype=torch.int32, device="cuda")
    qs, _ = sq.quant_act_static(dev(xs_rows, "f32"), ones, d, codes, clipped)
    assert np.array_equal(codes_np(qs), qs_ref) and int(clipped.item()) == clipped_ref == 0
    # low-bit rows (no smoothing, no rotation) with 7 and 127 levels
    for qmax, seed in ((7, 33), (127, 34)):
        rc = division_split_cases(qmax, 64, seed=seed)
        xr = division_rows(rc, 64, seed=seed)
        q_ref, s_ref, _ = O.rotate_quant_act(xr, None, False, qmax)
        q, sc = sq.rotate_quant_act(dev(xr, "f32"), None, False, qmax, codes)
        assert np.array_equal(codes_np(q), q_ref) and np.array_equal(f32bits(sc), npbits(s_ref))


# ------------------------------------------------------------------ per-step parity
@pytest.mark.parametrize("p", SMALL, ids=[p["name"] for p in SMALL])
def test_calibrate_bit_exact(sq, p):
    c = make_small(p)
    x, w = dev(c.x, c.dtype), dev(c.w, c.dtype)
    ax = sq.calibrate_absmax(x, 0)
    aw = sq.calibrate_absmax(w, 1)
    assert np.array_equal(f32bits(ax), npbits(O.calibrate_absmax(c.x_f32(), 0)))
    assert np.array_equal(f32bits(aw), npbits(O.calibrate_absmax(c.w_f32(), 1)))
    # column and row reductions of the other matrix too (both axes on both)
    assert np.array_equal(f32bits(sq.calibrate_absmax(w, 0)), npbits(O.calibrate_absmax(c.w_f32(), 0)))
    assert np.array_equal(f32bits(sq.calibrate_absmax(x, 1)), npbits(O.calibrate_absmax(c.x_f32(), 1)))


@pytest.mark.parametrize("p", SMALL, ids=[p["name"] for p in SMALL])
def test_smooth_factors_bit_exact(sq, p):
    c = make_small(p)
    ax, aw = O.calibrate_absmax(c.x_f32(), 0), O.calibrate_absmax(c.w_f32(), 1)
    s_ref, si_ref, nf = O.smooth_factors(ax, aw, c.alpha)
    flags = flags_tensor()
    s, si = sq.smooth_factors(torch.from_numpy(ax).cuda(), torch.from_numpy(aw).cuda(), c.alpha, flags)
    assert np.array_equal(f32bits(s), npbits(s_ref))
    assert np.array_equal(f32bits(si), npbits(si_ref))
    assert int(flags.item()) == 0 and not nf


@pytest.mark.parametrize("codes", ["i8", "bf16"])
@pytest.mark.parametrize("p", SMALL, ids=[p["name"] for p in SMALL])
def test_fold_quantize_bit_exact(sq, p, codes):
    c = make_small(p)
    s_ref, _, _ = O.smooth_factors(O.calibrate_absmax(c.x_f32(), 0), O.calibrate_absmax(c.w_f32(), 1), c.alpha)
    wq_ref, ws_ref, _ = O.fold_quantize_weight(c.w_f32(), s_ref)
    wq, ws = sq.fold_quantize_weight(dev(c.w, c.dtype), torch.from_numpy(s_ref).cuda(), codes)
    assert np.array_equal(codes_np(wq), wq_ref)
    assert np.array_equal(f32bits(ws), npbits(ws_ref))


@pytest.mark.parametrize("codes", ["i8", "bf16"])
@pytest.mark.parametrize("p", SMALL, ids=[p["name"] for p in SMALL])
def test_quant_act_bit_exact(sq, p, codes):
    c = make_small(p)
    _, si_ref, _ = O.smooth_factors(O.calibrate_absmax(c.x_f32(), 0), O.calibrate_absmax(c.w_f32(), 1), c.alpha)
    xq_ref, xs_ref, _ = O.quant_act(c.x_f32(), si_ref)
    flags = flags_tensor()
    xq, xs = sq.quant_act(dev(c.x, c.dtype), torch.from_numpy(si_ref).cuda(), codes, flags)
    assert np.array_equal(codes_np(xq), xq_ref)
    assert np.array_equal(f32bits(xs), npbits(xs_ref))
    assert int(flags.item()) == 0


def gemm_codes(sq, xq_ref, xs_ref, wq_ref, ws_ref, codes):
    if codes == "bf16":
        xq = torch.from_numpy(xq_ref.astype(F32)).to(torch.bfloat16).cuda()
        wq = torch.from_numpy(wq_ref.astype(F32)).to(torch.bfloat16).cuda()
    else:
        xq, wq = torch.from_numpy(xq_ref).cuda(), torch.from_numpy(wq_ref).cuda()
    return sq.w8a8_gemm(xq, torch.from_numpy(xs_ref).cuda(), wq, torch.from_numpy(ws_ref).cuda(),
                        want_acc=True, flags=flags_tensor())


def gemm_code_formats():
    return ["i8", "bf16"]


@pytest.mark.parametrize("codes", gemm_code_formats())
@pytest.mark.parametrize("p", SMALL, ids=[p["name"] for p in SMALL])
def test_gemm_exact_acc_and_ulp(sq, p, codes):
    c = make_small(p)
    r = O.run_path(c.x_f32(), c.w_f32(), c.alpha)
    y, acc = gemm_codes(sq, r["xq"], r["x_scale"], r["wq"], r["w_scale"], codes)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), r["acc"])
    d = O.bf16_ulp_distance(y_bits(y), r["y"])
    assert d.max() <= 1


@pytest.mark.parametrize("p", SMALL[:3], ids=[p["name"] for p in SMALL[:3]])
def test_whole_path_through_binding(sq, p):
    c = make_small(p)
    ref = O.run_path(c.x_f32(), c.w_f32(), c.alpha)
    for codes in gemm_code_formats():
        got = sq.smoothquant_linear(dev(c.x, c.dtype), dev(c.w, c.dtype), c.alpha, codes, want_acc=True)
        for key in ("amax_x", "amax_w", "s", "s_inv", "w_scale", "x_scale"):
            assert np.array_equal(f32bits(got[key]), npbits(ref[key])), key
        assert np.array_equal(codes_np(got["wq"]), ref["wq"])
        assert np.array_equal(codes_np(got["xq"]), ref["xq"])
        assert np.array_equal(got["acc"].cpu().numpy().astype(np.int64), ref["acc"])
        assert O.bf16_ulp_distance(y_bits(got["y"]), ref["y"]).max() <= 1


# ------------------------------------------------------------------ edge cases
def test_zero_channel_and_zero_token(sq):
    c = synth.make_case("z", 24, 64, 40, dtype="bf16", outlier_frac=0.05)
    x, w = c.x.copy(), c.w.copy()
    x[:, 5] = 0
    x[7, :] = 0
    w[:, 3] = 0   # output channel 3 all zero
    w[9, :] = 0   # input channel 9 all zero in W
    xf, wf = synth.bf16_bits_to_f32(x), synth.bf16_bits_to_f32(w)
    ref = O.run_path(xf, wf, 0.5)
    got = sq.smoothquant_linear(dev(x, "bf16"), dev(w, "bf16"), 0.5, "i8", want_acc=True)
    for key in ("s", "s_inv", "w_scale", "x_scale"):
        assert np.array_equal(f32bits(got[key]), npbits(ref[key])), key
    assert np.array_equal(codes_np(got["xq"]), ref["xq"])
    assert np.array_equal(codes_np(got["wq"]), ref["wq"])
    assert f32bits(got["x_scale"])[7] == npbits([1.0])[0]
    assert (codes_np(got["wq"])[3] == 0).all()


def test_rne_ties_and_clamp_on_gpu(sq):
    row = np.array([127.0, 2.5, 3.5, -2.5, 0.5, 1.5, -0.5, 126.5, -127.0] + [0.0] * 7, F32)
    x = torch.from_numpy(row[None, :].copy()).cuda()
    xq, xs = sq.quant_act(x, torch.ones(16, device="cuda"), "i8")
    assert xs.item() == 1.0
    assert codes_np(xq)[0, :9].tolist() == [127, 2, 4, -2, 0, 2, 0, 126, -127]


def test_nonfinite_flags(sq):
    x = torch.randn(8, 32, device="cuda").to(torch.bfloat16)
    x[3, 4] = float("nan")
    ax = sq.calibrate_absmax(x, 0)
    assert torch.isnan(ax[4]) and not torch.isnan(ax[:4]).any()
    flags = flags_tensor()
    s, si = sq.smooth_factors(ax, torch.ones(32, device="cuda"), 0.5, flags)
    assert int(flags.item()) & 1 and s[4].item() == 1.0 and si[4].item() == 1.0
    flags = flags_tensor()
    x2 = torch.ones(4, 32, device="cuda")
    x2[2, 7] = float("inf")
    sq.quant_act(x2, torch.ones(32, device="cuda"), "i8", flags)
    assert int(flags.item()) & 1


def test_calibration_running_max_and_shared_qkv(sq):
    c1 = synth.make_case("b1", 40, 96, 16, dtype="bf16", outlier_frac=0.05, seed=1)
    c2 = synth.make_case("b2", 40, 96, 16, dtype="bf16", outlier_frac=0.05, seed=2)
    out = sq.calibrate_absmax(dev(c1.x, "bf16"), 0)
    sq.calibrate_absmax(dev(c2.x, "bf16"), 0, out=out, accumulate=True)
    ref = O.calibrate_absmax(c2.x_f32(), 0, O.calibrate_absmax(c1.x_f32(), 0))
    assert np.array_equal(f32bits(out), npbits(ref))
    # one statistic over Q, K and V: running row max over the three weights
    qkv = synth.make_case("qkv", 8, 64, (48, 16, 16), dtype="bf16", w_std=0.015)
    w = qkv.w_f32()
    parts = [w[:, :48], w[:, 48:64], w[:, 64:]]
    aw = None
    for part in parts:
        t = torch.from_numpy(np.ascontiguousarray(part)).cuda()
        aw = sq.calibrate_absmax(t, 1) if aw is None else sq.calibrate_absmax(t, 1, out=aw, accumulate=True)
    assert np.array_equal(f32bits(aw), npbits(O.calibrate_absmax(w, 1)))


@pytest.mark.parametrize("codes", gemm_code_formats())
def test_gemm_saturated_widest_k(sq, codes):
    """All codes at +-127 with K = 11008: |acc| = 127^2 * 11008 exactly."""
    k = 11008
    xq = np.full((3, k), 127, np.int8)
    xq[1] = -127
    xq[2, ::2] = -127
    wq = np.full((5, k), 127, np.int8)
    wq[4, 1::2] = -127
    xs = np.array([1e-3, 2.5e-4, 1.0], F32)
    ws = np.array([1e-4, 3e-4, 1.0, 2.0, 1e-2], F32)
    y, acc = gemm_codes(sq, xq, xs, wq, ws, codes)
    ref_acc, ref_y = O.w8a8_gemm(xq, xs, wq, ws)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), ref_acc)
    assert ref_acc[0, 0] == 127 * 127 * k
    assert O.bf16_ulp_distance(y_bits(y), ref_y).max() <= 1


@pytest.mark.parametrize("codes", gemm_code_formats())
@pytest.mark.parametrize("m,n,k", [
    (1, 8, 16), (1, 1, 4096), (17, 9, 48), (130, 257, 1040), (256, 256, 2048),
    # tensor-core tiles: CTA pairs with output-channel tiles of 240 and 256
    # (chosen by the library per shape), a pair whose second CTA has no
    # valid rows (M = 300), K tails inside a k-block and several
    # 1024-product chunks
    (129, 72, 80), (520, 3080, 272), (777, 3464, 1040), (777, 4040, 2064), (2048, 2168, 208),
    (300, 1000, 3088),
    # one-CTA tensor-core tiles (64 < M <= 128): K tail, several chunks
    (65, 300, 2064), (100, 520, 1040), (128, 264, 64),
    # weight-streaming decode kernel (M <= 16): one or two token tiles, a
    # ragged channel block, K tails inside a stage and a k-block, more than
    # 1024 products per warp (the fp32 -> int32 flush)
    (8, 4096, 4096), (16, 100, 2064), (3, 33, 16), (16, 4096, 11008), (9, 72, 560),
    # more than 8192 codes of K per CTA: several exact fp32 chunks per CTA
    (16, 24, 66048), (3, 200, 70000),
    # more tiles than CTA pairs (or CTAs), a partial last wave: a K tail, a
    # ragged M, several chunks per tile, one-CTA tiles
    (2048, 5120, 1040), (520, 8192, 2048), (300, 20000, 3088), (64, 40000, 256),
    # int8 codes: weight rows staged in shared memory up to K = 12288 (a
    # ragged last block of rows, M in each of the 16/32/64-token tilings),
    # the register-fed kernel beyond it
    (16, 4104, 4096), (33, 40, 12288), (5, 24, 12304)])
def test_gemm_shapes_random_codes(sq, codes, m, n, k):
    u = synth.uniform(m + n + k, 5, (m + n) * k)
    codes_all = np.clip(np.floor(u * 255.0) - 127.0, -127, 127).astype(np.int8)
    xq, wq = codes_all[: m * k].reshape(m, k), codes_all[m * k:].reshape(n, k)
    xs = (0.001 + synth.uniform(1, 6, m)).astype(F32)
    ws = (0.0001 + synth.uniform(1, 7, n) * 0.01).astype(F32)
    y, acc = gemm_codes(sq, xq, xs, wq, ws, codes)
    ref_acc, ref_y = O.w8a8_gemm(xq, xs, wq, ws)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), ref_acc)
    assert O.bf16_ulp_distance(y_bits(y), ref_y).max() <= 1




@pytest.mark.parametrize("codes", gemm_code_formats())
@pytest.mark.parametrize("m,n,k", [(130, 264, 1040), (100, 520, 1040), (300, 2000, 2064)])
@pytest.mark.parametrize("offset", [2, 8])
def test_gemm_y_alignment_no_acc(sq, codes, m, n, k, offset):
    """Y written into a buffer 4 bytes (offset 2) or 16 bytes (offset 8) past
    an allocation, with no accumulators requested: the epilogue's TMA-store
    path needs N % 8 == 0 and a 16-byte aligned Y, and takes direct stores
    otherwise.  The bytes around Y stay untouched."""
    u = synth.uniform(m + n + k + offset, 9, (m + n) * k)
    codes_all = np.clip(np.floor(u * 255.0) - 127.0, -127, 127).astype(np.int8)
    xq, wq = codes_all[: m * k].reshape(m, k), codes_all[m * k:].reshape(n, k)
    xs = (0.001 + synth.uniform(1, 10, m)).astype(F32)
    ws = (0.0001 + synth.uniform(1, 11, n) * 0.01).astype(F32)
    if codes == "bf16":
        xt = torch.from_numpy(xq.astype(F32)).to(torch.bfloat16).cuda()
        wt = torch.from_numpy(wq.astype(F32)).to(torch.bfloat16).cuda()
    else:
        xt, wt = torch.from_numpy(xq).cuda(), torch.from_numpy(wq).cuda()
    sentinel = torch.tensor(-12345.0, dtype=torch.bfloat16)
    buf = torch.full((m * n + offset + 8,), float(sentinel), dtype=torch.bfloat16, device="cuda")
    y = buf[offset: offset + m * n].view(m, n)
    assert y.data_ptr() % 16 == (0 if offset == 8 else 4)
    sq.w8a8_gemm(xt, torch.from_numpy(xs).cuda(), wt, torch.from_numpy(ws).cuda(),
                 flags=flags_tensor(), out=y)
    _, ref_y = O.w8a8_gemm(xq, xs, wq, ws)
    assert O.bf16_ulp_distance(y_bits(y), ref_y).max() <= 1
    rest = torch.cat([buf[:offset], buf[offset + m * n:]]).cpu()
    assert torch.all(rest == sentinel)


@pytest.mark.parametrize("m,n,k", [(65, 300, 2064), (130, 257, 1040), (520, 3080, 272), (300, 1000, 3088)])
def test_gemm_i8_without_workspace(sq, m, n, k):
    """1-byte codes above 64 tokens given a workspace too small for the
    widened operands: the kernel that widens the codes in shared memory as
    it goes (the default, with the workspace, widens them in one pass
    first).  Both are exact."""
    u = synth.uniform(m + n + k, 12, (m + n) * k)
    codes_all = np.clip(np.floor(u * 255.0) - 127.0, -127, 127).astype(np.int8)
    xq, wq = codes_all[: m * k].reshape(m, k), codes_all[m * k:].reshape(n, k)
    xs = (0.001 + synth.uniform(1, 13, m)).astype(F32)
    ws = (0.0001 + synth.uniform(1, 14, n) * 0.01).astype(F32)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    y, acc = sq.w8a8_gemm(torch.from_numpy(xq).cuda(), torch.from_numpy(xs).cuda(), torch.from_numpy(wq).cuda(),
                          torch.from_numpy(ws).cuda(), want_acc=True, flags=flags_tensor(), workspace=small)
    ref_acc, ref_y = O.w8a8_gemm(xq, xs, wq, ws)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), ref_acc)
    assert O.bf16_ulp_distance(y_bits(y), ref_y).max() <= 1

def carrier_adversarial_codes(m, n, k, seed):
    """Codes built against the fp32 carrier of the tensor-core GEMM.

    Within each group of 16 products (one MMA's K) fifteen are +-127 * 127
    and one is +-1, so every 1024-product chunk sums to within 2^20 of its
    largest possible magnitude 1024 * 127^2 (just under 2^24) while carrying
    unit terms an adder keeping fewer than 24 bits would drop; the sign of
    whole chunks flips at chunk edges (rows by one pattern, columns by
    another), the odd position of the unit term moves from group to group,
    and a share of rows and columns alternates sign product by product."""
    rng = np.random.default_rng(seed)
    kk = np.arange(k)
    unit_pos = (kk // 16 * 7) % 16 == kk % 16            # one position per group of 16
    a = np.where(unit_pos, 1, 127)[None, :] * np.ones((m, 1), np.int64)
    b = np.where(unit_pos, 1, 127)[None, :] * np.ones((n, 1), np.int64)
    chunk = kk // 1024
    a *= np.where((chunk[None, :] + np.arange(m)[:, None]) % 2 == 0, 1, -1)   # row chunk signs
    b *= np.where((chunk[None, :] * (np.arange(n)[:, None] % 3)) % 2 == 0, 1, -1)
    unit_sign = rng.choice([-1, 1], size=(m, k))
    a = np.where(unit_pos[None, :], a * unit_sign, a)
    alt = rng.random(m) < 0.25                             # rows alternating product by product
    a[alt] *= np.where(kk % 2 == 0, 1, -1)[None, :]
    altb = rng.random(n) < 0.25
    b[altb] *= np.where(kk % 3 == 0, -1, 1)[None, :]
    return a.astype(np.int8), b.astype(np.int8)


@pytest.mark.parametrize("codes", gemm_code_formats())
@pytest.mark.parametrize("m,n,k", [(256, 256, 2048 + 64), (100, 264, 3072), (300, 240, 1040),
                                   (16, 256, 16384 + 64), (7, 40, 2048)])
def test_gemm_fp32_carrier_adversarial(sq, codes, m, n, k):
    """Exact accumulators on codes built against the fp32 carrier (chunk sums
    near 2^24 with unit products in every MMA group, sign flips at chunk
    edges)."""
    xq, wq = carrier_adversarial_codes(m, n, k, seed=m + n + k)
    ref_acc = O.int_accumulate(xq, wq)
    chunk_max = np.abs(xq[:, :1024].astype(np.int64) @ wq[:, :1024].astype(np.int64).T).max()
    assert chunk_max > 15 * 127 * 127 * 64 - 64 * 1 and chunk_max < 2 ** 24
    xs = np.full(m, 1e-3, F32)
    ws = np.full(n, 1e-4, F32)
    y, acc = gemm_codes(sq, xq, xs, wq, ws, codes)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), ref_acc)
    _, ref_y = O.w8a8_gemm(xq, xs, wq, ws)
    assert O.bf16_ulp_distance(y_bits(y), ref_y).max() <= 1


# ------------------------------------------------------------------ launch-shape coverage
# Weight shapes that reach every single-pass fold configuration: clusters of
# 1, 2, 4 and 8 CTAs of at most 1536 rows (Cin up to 1536, 3072, 6144,
# 12288), a cluster whose last CTA owns no rows (Cin = 6160 with 8 x
# 896-row CTAs), strips cut short by Cout, fp32 weights, and Cin beyond the
# single-pass limit (the two-pass path).
FOLD_SHAPES = [
    (768, 40, "bf16"), (1536, 96, "bf16"), (1552, 40, "bf16"), (4096, 264, "bf16"), (6144, 136, "bf16"),
    (6160, 72, "bf16"), (12288, 32, "bf16"), (12304, 24, "bf16"), (2048, 20, "f32"),
    (48, 1000, "f32"),
    # whole 64-channel strips of bf16 W: clusters of 1-8 CTAs with ragged last CTAs, and a box
    # running past the last row
    (4096, 128, "bf16"), (1040, 64, "bf16"), (48, 64, "bf16"), (2064, 192, "bf16"), (8192, 320, "bf16"),
]


@pytest.mark.parametrize("codes", ["i8", "bf16"])
@pytest.mark.parametrize("cin,cout,dtype", FOLD_SHAPES)
def test_fold_launch_shapes(sq, cin, cout, dtype, codes):
    c = synth.make_case("fold", 1, cin, cout, dtype=dtype, w_std=0.02, seed=cin + cout)
    s = (0.25 + 4.0 * synth.uniform(cin, 41, cin)).astype(F32)
    w = c.w.copy()
    w[:, cout // 2] = 0   # one all-zero output channel: that strip takes the clamped path
    wf = synth.bf16_bits_to_f32(w) if dtype == "bf16" else w
    wq_ref, ws_ref, _ = O.fold_quantize_weight(wf, s)
    flags = flags_tensor()
    wq, ws = sq.fold_quantize_weight(dev(w, dtype), torch.from_numpy(s).cuda(), codes, flags)
    assert int(flags.item()) == 0
    assert np.array_equal(f32bits(ws), npbits(ws_ref))
    assert np.array_equal(codes_np(wq), wq_ref)


# Activation shapes that reach every block size (128-1024 threads), 1-4
# vectors per thread, s^-1 in registers and re-read through L1, the largest
# row (64 KiB), and many rows per CTA (the shared-memory ring wraps).
ACT_SHAPES = [
    (1000, 16, "bf16"), (700, 4112, "bf16"), (300, 11008, "bf16"), (40, 32768, "bf16"),
    (3000, 512, "f32"), (9, 16384, "f32"), (4099, 64, "bf16"),
]


@pytest.mark.parametrize("codes", ["i8", "bf16"])
@pytest.mark.parametrize("tokens,cin,dtype", ACT_SHAPES)
def test_quant_act_launch_shapes(sq, tokens, cin, dtype, codes):
    c = synth.make_case("act", tokens, cin, 16, dtype=dtype, outlier_frac=0.01, seed=tokens + cin)
    x = c.x.copy()
    x[tokens // 3, :] = 0   # an all-zero token takes the clamped path
    xf = synth.bf16_bits_to_f32(x) if dtype == "bf16" else x
    si = (0.25 + 4.0 * synth.uniform(cin, 42, cin)).astype(F32)
    xq_ref, xs_ref, _ = O.quant_act(xf, si)
    flags = flags_tensor()
    xq, xs = sq.quant_act(dev(x, dtype), torch.from_numpy(si).cuda(), codes, flags)
    assert int(flags.item()) == 0
    assert np.array_equal(f32bits(xs), npbits(xs_ref))
    assert np.array_equal(codes_np(xq), xq_ref)


# Column-maxima shapes for the strip kernel: clusters of 1-8 CTAs, a last
# CTA with a partial box, strips cut short by the column count, rings that
# wrap many times (5000 rows), wide rows, running maxima over two batches,
# and a row stride that is not 16-byte aligned (the atomic path).
COLMAX_SHAPES = [
    (16, 4096, "bf16"), (2048, 4096, "bf16"), (300, 64, "bf16"), (1000, 40, "f32"),
    (129, 528, "f32"), (5000, 96, "bf16"), (77, 300, "bf16"), (3, 4096, "bf16"),
    (40, 32768, "bf16"), (24, 12288, "f32"), (6, 40000, "bf16"),
]


@pytest.mark.parametrize("rows,cols,dtype", COLMAX_SHAPES)
def test_colmax_launch_shapes(sq, rows, cols, dtype):
    c1 = synth.make_case("cm1", rows, cols, 8, dtype=dtype, outlier_frac=0.05, seed=rows)
    c2 = synth.make_case("cm2", rows, cols, 8, dtype=dtype, outlier_frac=0.05, seed=rows + 1)
    out = sq.calibrate_absmax(dev(c1.x, dtype), 0)
    assert np.array_equal(f32bits(out), npbits(O.calibrate_absmax(c1.x_f32(), 0)))
    sq.calibrate_absmax(dev(c2.x, dtype), 0, out=out, accumulate=True)
    ref = O.calibrate_absmax(c2.x_f32(), 0, O.calibrate_absmax(c1.x_f32(), 0))
    assert np.array_equal(f32bits(out), npbits(ref))

# ------------------------------------------------------------------ full-size workloads
FULL = synth.WORKLOAD_ORDER[1:]


def sample_rows(case, k=48):
    """Every token for layers of up to 2048 tokens (the oracle's float64 BLAS
    forms those accumulators in seconds); otherwise k spread tokens plus
    every massive-outlier token."""
    if case.tokens <= 2048:
        return np.arange(case.tokens)
    rows = set(np.linspace(0, case.tokens - 1, min(k, case.tokens)).astype(int).tolist())
    big = np.nonzero(np.abs(case.x_f32()).max(axis=1) >= 500)[0]
    rows.update(big.tolist())
    return np.array(sorted(rows))


# the default (1-byte codes) on every workload, and the bf16-stored codes
# where the tensor-core GEMM reads them
FULL_CODES = [(n, None) for n in FULL] + [(n, "bf16") for n in FULL if synth.WORKLOADS[n]["tokens"] > 64]


@pytest.mark.parametrize("name,codes", FULL_CODES, ids=[f"{n}-{c or 'auto'}" for n, c in FULL_CODES])
def test_full_workload_parity(sq, name, codes):
    from w8a8_post_quantization_02_b300 import pipeline
    c = synth.workload(name)
    ref_ax = O.calibrate_absmax(c.x_f32(), 0)
    ref_aw = O.calibrate_absmax(c.w_f32(), 1)
    s_ref, si_ref, _ = O.smooth_factors(ref_ax, ref_aw, c.alpha)
    wq_ref, ws_ref, _ = O.fold_quantize_weight(c.w_f32(), s_ref)
    xq_ref, xs_ref, _ = O.quant_act(c.x_f32(), si_ref)
    rows = sample_rows(c)
    acc_ref, y_ref = O.w8a8_gemm(xq_ref, xs_ref, wq_ref, ws_ref, rows=rows)

    layer = pipeline.Layer.for_case(c, codes=codes)
    layer.load(dev(c.x, c.dtype), dev(c.w, c.dtype))
    layer.step(want_acc=True)
    torch.cuda.synchronize()
    assert int(layer.flags.item()) == 0
    assert np.array_equal(f32bits(layer.amax_x), npbits(ref_ax))
    assert np.array_equal(f32bits(layer.amax_w), npbits(ref_aw))
    assert np.array_equal(f32bits(layer.s), npbits(s_ref))
    assert np.array_equal(f32bits(layer.s_inv), npbits(si_ref))
    assert np.array_equal(codes_np(layer.wq), wq_ref)
    assert np.array_equal(f32bits(layer.w_scale), npbits(ws_ref))
    assert np.array_equal(codes_np(layer.xq), xq_ref)
    assert np.array_equal(f32bits(layer.x_scale), npbits(xs_ref))
    rows_t = torch.from_numpy(rows).cuda()
    assert np.array_equal(layer.acc.index_select(0, rows_t).cpu().numpy().astype(np.int64), acc_ref)
    y = y_bits(layer.y.index_select(0, rows_t))
    assert O.bf16_ulp_distance(y, y_ref).max() <= 1


# ------------------------------------------------------------------ whole path from host memory
@pytest.mark.parametrize("name,codes", [("single_linear_64x512x512", None), ("single_linear_64x512x512", "bf16"),
                                        ("decode_7b_16x4096x4096", None), ("decode_7b_16x4096x4096", "bf16"),
                                        ("prefill_upgate_2048x4096x11008", None)])
def test_linear_host_parity(sq, name, codes):
    """sq_linear_host: pinned host X and W in, host Y out, through the C ABI;
    every intermediate bit-exact against the oracle, Y within 1 bf16 ulp.
    The prefill case with 1-byte codes has the fold and the GEMM share one
    workspace large enough for the GEMM's widened operands."""
    from w8a8_post_quantization_02_b300 import pipeline
    c = synth.workload(name)
    ref_ax = O.calibrate_absmax(c.x_f32(), 0)
    ref_aw = O.calibrate_absmax(c.w_f32(), 1)
    s_ref, si_ref, _ = O.smooth_factors(ref_ax, ref_aw, c.alpha)
    wq_ref, ws_ref, _ = O.fold_quantize_weight(c.w_f32(), s_ref)
    xq_ref, xs_ref, _ = O.quant_act(c.x_f32(), si_ref)
    _, y_ref = O.w8a8_gemm(xq_ref, xs_ref, wq_ref, ws_ref)

    layer = pipeline.Layer.for_case(c, codes=codes)
    x_host = dev(c.x, c.dtype).cpu().pin_memory()
    w_host = dev(c.w, c.dtype).cpu().pin_memory()
    y_host = torch.empty(c.tokens, c.cout, dtype=torch.bfloat16).pin_memory()
    stream = torch.cuda.Stream()
    layer.run_host(x_host, w_host, y_host, stream=stream)
    stream.synchronize()
    assert int(layer.flags.item()) == 0
    assert np.array_equal(f32bits(layer.amax_x), npbits(ref_ax))
    assert np.array_equal(f32bits(layer.amax_w), npbits(ref_aw))
    assert np.array_equal(f32bits(layer.s), npbits(s_ref))
    assert np.array_equal(codes_np(layer.wq), wq_ref)
    assert np.array_equal(f32bits(layer.w_scale), npbits(ws_ref))
    assert np.array_equal(codes_np(layer.xq), xq_ref)
    assert np.array_equal(f32bits(layer.x_scale), npbits(xs_ref))
    assert O.bf16_ulp_distance(y_bits(y_host), y_ref).max() <= 1
    # the device copy of Y is the one that was copied out
    assert torch.equal(layer.y.cpu().view(torch.int16), y_host.view(torch.int16))


# ------------------------------------------------------------------ static activation scale
# Calibrate on X, then quantize a runtime batch whose tokens are scaled by
# up to 1.6x (so some codes clip): scale, codes and clip count bit-exact.
STATIC_SHAPES = [
    (64, 512, "f32"), (37, 80, "bf16"), (300, 11008, "bf16"), (9, 16384, "f32"), (4099, 64, "bf16"),
    (700, 4112, "bf16"), (1, 256, "bf16"),
]


@pytest.mark.parametrize("codes", ["i8", "bf16"])
@pytest.mark.parametrize("tokens,cin,dtype", STATIC_SHAPES)
def test_static_scale_and_codes_bit_exact(sq, tokens, cin, dtype, codes):
    c = synth.make_case("st", tokens, cin, 16, dtype=dtype, outlier_frac=0.02, seed=tokens + 3 * cin)
    cal = c.x_f32()
    si = (0.25 + 4.0 * synth.uniform(cin, 43, cin)).astype(F32)
    ax = O.calibrate_absmax(cal, 0)
    d_ref, nf = O.static_act_scale(ax, si)
    flags = flags_tensor()
    d = sq.static_act_scale(torch.from_numpy(ax).cuda(), torch.from_numpy(si).cuda(), flags)
    assert f32bits(d)[0] == npbits([d_ref])[0] and not nf
    gain = (1.0 + 0.6 * synth.uniform(tokens, 44, tokens)).astype(F32)
    run = (cal * gain[:, None]).astype(F32)
    if dtype == "bf16":
        bits = synth.f64_to_bf16_bits(run.astype(np.float64))
        run = synth.bf16_bits_to_f32(bits)
        run_dev = dev(bits, "bf16")
    else:
        run_dev = dev(run, "f32")
    q_ref, xs_ref, clip_ref = O.quant_act_static(run, si, d_ref)
    clipped = torch.zeros(1, dtype=torch.int32, device="cuda")
    xq, xs = sq.quant_act_static(run_dev, torch.from_numpy(si).cuda(), d, codes, clipped, flags)
    assert int(flags.item()) == 0
    assert np.array_equal(codes_np(xq), q_ref)
    assert np.array_equal(f32bits(xs), npbits(xs_ref))
    assert int(clipped.item()) == clip_ref


def test_static_nonfinite_codes_and_flag(sq):
    x = torch.ones(3, 32, device="cuda")
    x[1, 5] = float("nan")
    x[2, 7] = float("inf")
    x[2, 8] = -float("inf")
    d = torch.tensor([1.0 / 127.0], device="cuda")
    flags, clipped = flags_tensor(), torch.zeros(1, dtype=torch.int32, device="cuda")
    xq, _ = sq.quant_act_static(x, torch.ones(32, device="cuda"), d, "i8", clipped, flags)
    q = codes_np(xq)
    assert int(flags.item()) & 1
    assert q[1, 5] == 0 and q[2, 7] == 127 and q[2, 8] == -127
    ref, _, clip_ref = O.quant_act_static(x.cpu().numpy(), np.ones(32, F32), F32(1.0 / 127.0))
    assert np.array_equal(q, ref) and int(clipped.item()) == clip_ref


@pytest.mark.parametrize("name", ["prefill_upgate_2048x4096x11008", "qkv_shared_8192x8192x10240"])
def test_full_workload_static_parity(sq, name):
    from w8a8_post_quantization_02_b300 import pipeline
    c = synth.workload(name)
    ax = O.calibrate_absmax(c.x_f32(), 0)
    s_ref, si_ref, _ = O.smooth_factors(ax, O.calibrate_absmax(c.w_f32(), 1), c.alpha)
    d_ref, _ = O.static_act_scale(ax, si_ref)
    xq_ref, xs_ref, clip_ref = O.quant_act_static(c.x_f32(), si_ref, d_ref)
    wq_ref, ws_ref, _ = O.fold_quantize_weight(c.w_f32(), s_ref)
    rows = sample_rows(c)
    acc_ref, y_ref = O.w8a8_gemm(xq_ref, xs_ref, wq_ref, ws_ref, rows=rows)
    layer = pipeline.Layer.for_case(c, act_scale="static")
    layer.load(dev(c.x, c.dtype), dev(c.w, c.dtype))
    layer.step(want_acc=True)
    torch.cuda.synchronize()
    assert int(layer.flags.item()) == 0
    assert f32bits(layer.d)[0] == npbits([d_ref])[0]
    assert int(layer.clipped.item()) == clip_ref == 0   # calibrated on the same X
    assert np.array_equal(codes_np(layer.xq), xq_ref)
    assert np.array_equal(f32bits(layer.x_scale), npbits(xs_ref))
    rows_t = torch.from_numpy(rows).cuda()
    assert np.array_equal(layer.acc.index_select(0, rows_t).cpu().numpy().astype(np.int64), acc_ref)
    assert O.bf16_ulp_distance(y_bits(layer.y.index_select(0, rows_t)), y_ref).max() <= 1


# ------------------------------------------------------------------ diagnostics
def _rel_close(got, want, rel, floor=0.0):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    return np.all(np.abs(got - want) <= rel * np.abs(want) + floor)


@pytest.mark.parametrize("codes", ["i8", "bf16"])
@pytest.mark.parametrize("p", SMALL, ids=[p["name"] for p in SMALL])
def test_diagnostics_match_oracle(sq, p, codes):
    c = make_small(p)
    if (c.cin * (2 if c.dtype == "bf16" else 4)) % 16:
        pytest.skip("activation rows must be 16-byte aligned")
    xf, wf = c.x_f32(), c.w_f32()
    r = O.run_path(xf, wf, c.alpha)
    x_t, w_t = dev(c.x, c.dtype), dev(c.w, c.dtype)
    si, s = torch.from_numpy(r["s_inv"]).cuda(), torch.from_numpy(r["s"]).cuda()
    cdt = torch.bfloat16 if codes == "bf16" else torch.int8
    xq = torch.from_numpy(r["xq"].astype(F32 if codes == "bf16" else np.int8)).to(cdt).cuda()
    wq = torch.from_numpy(r["wq"].astype(F32 if codes == "bf16" else np.int8)).to(cdt).cuda()
    xs, ws = torch.from_numpy(r["x_scale"]).cuda(), torch.from_numpy(r["w_scale"]).cuda()
    ea = sq.act_quant_error(x_t, si, xq, xs).cpu().numpy()
    assert _rel_close(ea, O.act_quant_error(xf, r["s_inv"], r["xq"], r["x_scale"]), 1e-12)
    ew = sq.weight_quant_error(w_t, s, wq, ws).cpu().numpy()
    assert _rel_close(ew, O.weight_quant_error(wf, r["s"], r["wq"], r["w_scale"]), 1e-12)
    y = torch.from_numpy(r["y"].view(np.int16)).view(torch.bfloat16).cuda()
    rows = np.arange(0, c.tokens, max(1, c.tokens // 7))[:64]
    el = sq.layer_error(x_t, w_t, y, torch.from_numpy(rows.astype(np.int32))).cpu().numpy()
    ref = O.layer_error(xf, wf, r["y"], rows)
    assert _rel_close(el, ref, 1e-4, floor=1e-12)
    ax = torch.from_numpy(r["amax_x"]).cuda()
    for scale in (None, si):
        got = sq.channel_stats(ax, scale).cpu().numpy()
        want = O.channel_stats(r["amax_x"], None if scale is None else r["s_inv"])
        assert _rel_close(got, want, 1e-12)


def test_alpha_sweep_matches_oracle(sq):
    from w8a8_post_quantization_02_b300 import pipeline
    c = synth.workload("single_linear_64x512x512")
    rows = np.arange(0, 64, 3)
    res = pipeline.alpha_sweep(dev(c.x, c.dtype), dev(c.w, c.dtype), [0.3, 0.5, 0.7, 0.9], codes="bf16",
                               rows=torch.from_numpy(rows.astype(np.int32)))
    xf, wf = c.x_f32(), c.w_f32()
    for got in res:
        r = O.run_path(xf, wf, got["alpha"])
        assert _rel_close(got["act_error"], O.act_quant_error(xf, r["s_inv"], r["xq"], r["x_scale"]).sum(), 1e-12)
        assert _rel_close(got["weight_error"], O.weight_quant_error(wf, r["s"], r["wq"], r["w_scale"]).sum(), 1e-12)
        assert _rel_close(got["layer_error"], O.layer_error(xf, wf, r["y"], rows).sum(), 1e-4)
        assert _rel_close(got["x_difficulty_smoothed"], O.channel_stats(r["amax_x"], r["s_inv"])[1], 1e-12)
        assert _rel_close(got["w_difficulty_smoothed"], O.channel_stats(r["amax_w"], r["s"])[1], 1e-12)
    # smoothing moves the spread from X to W as alpha grows (pages: migrate
    # quantization difficulty from activations into weights)
    xd = [g["x_difficulty_smoothed"] for g in res]
    wd = [g["w_difficulty_smoothed"] for g in res]
    assert xd == sorted(xd, reverse=True) and wd == sorted(wd)


def test_full_workload_diagnostics(sq):
    from w8a8_post_quantization_02_b300 import pipeline
    c = synth.workload("down_proj_2048x11008x4096")
    layer = pipeline.Layer.for_case(c)
    layer.load(dev(c.x, c.dtype), dev(c.w, c.dtype))
    layer.step()
    rows = sample_rows(c)[:64]
    d = pipeline.diagnose(layer, torch.from_numpy(rows.astype(np.int32)))
    xf, wf = c.x_f32(), c.w_f32()
    ax, aw = O.calibrate_absmax(xf, 0), O.calibrate_absmax(wf, 1)
    s_ref, si_ref, _ = O.smooth_factors(ax, aw, c.alpha)
    wq_ref, ws_ref, _ = O.fold_quantize_weight(wf, s_ref)
    xq_ref, xs_ref, _ = O.quant_act(xf, si_ref)
    assert _rel_close(d["act_error"], O.act_quant_error(xf, si_ref, xq_ref, xs_ref).sum(), 1e-11)
    assert _rel_close(d["weight_error"], O.weight_quant_error(wf, s_ref, wq_ref, ws_ref).sum(), 1e-11)
    # the layer error of the GPU's own output (within 1 bf16 ulp of the oracle's)
    assert _rel_close(d["layer_error"], O.layer_error(xf, wf, y_bits(layer.y), rows).sum(), 1e-4)
    assert _rel_close(d["x_difficulty"], O.channel_stats(ax)[1], 1e-12)


# ------------------------------------------------------------------ RMSNorm fold
NORM_SHAPES = [
    (64, 512, "f32"), (37, 80, "bf16"), (300, 11008, "bf16"), (9, 16384, "f32"), (4099, 64, "bf16"),
    (700, 4112, "bf16"), (40, 32768, "bf16"), (2048, 4096, "bf16"),
]


@pytest.mark.parametrize("codes", ["i8", "bf16"])
@pytest.mark.parametrize("tokens,cin,dtype", NORM_SHAPES)
def test_rmsnorm_fold_bit_exact(sq, tokens, cin, dtype, codes):
    """Hidden states with outlier channels and a few massive tokens, a
    random gain folded with random factors: codes and scales bit-exact."""
    c = synth.make_case("nrm", tokens, cin, 16, dtype=dtype, outlier_frac=0.01, seed=tokens + 5 * cin,
                        massive_tokens=min(3, tokens), massive_channels=2)
    h = c.x.copy()
    h[tokens // 2, :] = 0   # an all-zero token: r = 1/sqrt(eps)
    if tokens > 2:
        # a token whose float64 sum of squares is a binary32 midpoint that the
        # exact sum lies above: 1 + 2^-24 + 2^-80 rounds up to 1 + 2^-23
        crafted = np.zeros(cin, np.float64)
        crafted[:3] = [1.0, 2.0 ** -12, 2.0 ** -40]
        h[1] = synth.f64_to_bf16_bits(crafted) if dtype == "bf16" else crafted.astype(F32)
    hf = synth.bf16_bits_to_f32(h) if dtype == "bf16" else h
    gamma = (0.5 + synth.uniform(cin, 61, cin)).astype(F32)
    si = (0.25 + 4.0 * synth.uniform(cin, 62, cin)).astype(F32)
    eps = 1e-5
    gf_ref = O.fold_norm_gain(gamma, si)
    gf = sq.fold_norm_gain(torch.from_numpy(gamma).cuda(), torch.from_numpy(si).cuda())
    assert np.array_equal(f32bits(gf), npbits(gf_ref))
    q_ref, xs_ref, nf = O.rmsnorm_quant_act(hf, gf_ref, eps)
    flags = flags_tensor()
    xq, xs = sq.rmsnorm_quant_act(dev(h, dtype), gf, eps, codes, flags)
    assert int(flags.item()) == 0 and not nf
    assert np.array_equal(f32bits(xs), npbits(xs_ref))
    assert np.array_equal(codes_np(xq), q_ref)


def _exact_bf16_bits(v) -> np.ndarray:
    """bf16 bit patterns of values that bf16 holds exactly (subnormals too)."""
    b = np.asarray(v, np.float64).astype(F32).view(np.uint32)
    assert not np.any(b & 0xFFFF)
    return (b >> 16).astype(np.uint16)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("cin", [64, 4096, 8192])
def test_rmsnorm_sum_boundaries(sq, cin, dtype):
    """Sums of squares on and next to binary32 midpoints, and rows whose
    threads hold values far apart or at the ends of the exponent range:
    - 1 + 2^-24 exactly (a tie: even, so 1);
    - 1 + 2^-24 + 2^-56 (just above the tie);
    - 1 + 2^-24 + 2^-120 (a square 2^96 times below the others' unit);
    - a 2^62 value in one thread and 2^-60-sized values in another;
    - rows of 2^-56-sized and 2^40-sized values, one with 1.5 * 2^60 and one
      with 1.5 * 2^61 in its first thread;
    - 1.5 with a 2^-100 value and the bf16 subnormal 2^-130 beside it.
    The scale and the codes must equal the exact-sum oracle's."""
    rng = np.random.default_rng(cin + (7 if dtype == "bf16" else 0))
    rows = np.zeros((10, cin), np.float64)
    rows[0, :2] = [1.0, 2.0 ** -12]
    rows[1, :3] = [1.0, 2.0 ** -12, 2.0 ** -28]
    rows[2, :3] = [1.0, 2.0 ** -12, 2.0 ** -60]
    base = np.round(rng.standard_normal((7, cin)) * 16) / 16   # at most 8 significant bits: exact in bf16
    rows[3] = base[0]
    rows[3, 8] = 2.0 ** 62
    rows[3, 16:24] = base[1, :8] * 2.0 ** -60
    rows[4] = base[2] * 2.0 ** -56
    rows[5] = base[3] * 2.0 ** 40
    rows[5, 0] = 1.5 * 2.0 ** 60
    rows[6] = base[4] * 2.0 ** 40
    rows[6, 0] = 1.5 * 2.0 ** 61
    rows[7] = base[5]
    rows[7, :3] = [1.5, 2.0 ** -100, 2.0 ** -130]
    rows[8] = base[6]
    rows[9, :3] = [1.0, 2.0 ** -12, -(2.0 ** -60)]
    if dtype == "bf16":
        h = _exact_bf16_bits(rows)
        hf = synth.bf16_bits_to_f32(h)
    else:
        h = rows.astype(F32)
        assert np.array_equal(h.astype(np.float64), rows)
        hf = h
    gamma = np.ones(cin, F32)
    eps = 1e-5
    q_ref, xs_ref, nf = O.rmsnorm_quant_act(hf, gamma, eps)
    assert not nf
    assert O.sum_squares_f32(hf[0]) == F32(1.0)
    assert O.sum_squares_f32(hf[1]) == O.sum_squares_f32(hf[2]) == F32(1.0 + 2.0 ** -23)
    flags = flags_tensor()
    xq, xs = sq.rmsnorm_quant_act(dev(h, dtype), torch.from_numpy(gamma).cuda(), eps, "i8", flags)
    assert int(flags.item()) == 0
    assert np.array_equal(f32bits(xs), npbits(xs_ref))
    assert np.array_equal(codes_np(xq), q_ref)


def test_rmsnorm_nonfinite_flag(sq):
    h = torch.ones(4, 64, device="cuda")
    h[2, 9] = float("inf")
    flags = flags_tensor()
    sq.rmsnorm_quant_act(h, torch.ones(64, device="cuda"), 1e-6, "i8", flags)
    assert int(flags.item()) & 1


# ------------------------------------------------------------------ Smooth Rotation
ROT_ACT_SHAPES = [(64, 512, "f32"), (37, 256, "bf16"), (5, 512, "bf16"), (300, 4096, "bf16"), (9, 8192, "f32"),
                  (129, 16384, "bf16"), (40, 32768, "bf16"), (77, 11008, "bf16"),
                  # rows of 2^10 .. 2^14 take the three-phase transform: every length, both input types
                  (33, 1024, "bf16"), (17, 2048, "f32"), (50, 8192, "bf16"), (3, 16384, "f32"), (21, 1024, "f32")]


@pytest.mark.parametrize("qmax", [7, 127])
@pytest.mark.parametrize("tokens,cin,dtype", ROT_ACT_SHAPES)
def test_rotate_quant_act_bit_exact(sq, tokens, cin, dtype, qmax):
    c = synth.make_case("ra", tokens, cin, 16, dtype=dtype, x_std=0.5, fixed_channels=2, fixed_factor=60.0,
                        massive_tokens=min(3, tokens), massive_channels=2, seed=tokens + cin)
    xf = c.x_f32()
    si = (0.25 + 4.0 * synth.uniform(cin, 63, cin)).astype(F32)
    pow2 = cin & (cin - 1) == 0
    for smooth in (False, True):
        for rotate in ((False, True) if pow2 else (False,)):
            for codes in ("i8", "bf16"):
                q_ref, xs_ref, nf = O.rotate_quant_act(xf, si if smooth else None, rotate, qmax)
                flags = flags_tensor()
                xq, xs = sq.rotate_quant_act(dev(c.x, dtype), torch.from_numpy(si).cuda() if smooth else None,
                                             rotate, qmax, codes, flags)
                assert int(flags.item()) == 0 and not nf
                assert np.array_equal(f32bits(xs), npbits(xs_ref)), (smooth, rotate, codes)
                assert np.array_equal(codes_np(xq), q_ref), (smooth, rotate, codes)


ROT_W_SHAPES = [(256, 40, "bf16"), (4096, 264, "bf16"), (8192, 72, "bf16"), (512, 33, "f32"),
                (11008, 24, "bf16"), (1024, 40, "bf16"), (2048, 24, "f32"), (16384, 8, "bf16")]


@pytest.mark.parametrize("qmax", [7, 127])
@pytest.mark.parametrize("cin,cout,dtype", ROT_W_SHAPES)
def test_rotate_fold_quantize_weight_bit_exact(sq, cin, cout, dtype, qmax):
    c = synth.make_case("rw", 1, cin, cout, dtype=dtype, w_std=0.02, seed=cin + cout)
    s = (0.25 + 4.0 * synth.uniform(cin, 64, cin)).astype(F32)
    pow2 = cin & (cin - 1) == 0
    for smooth in (False, True):
        for rotate in ((False, True) if pow2 else (False,)):
            wq_ref, ws_ref, nf = O.rotate_fold_quantize_weight(c.w_f32(), s if smooth else None, rotate, qmax)
            flags = flags_tensor()
            wq, ws = sq.rotate_fold_quantize_weight(dev(c.w, dtype), torch.from_numpy(s).cuda() if smooth else None,
                                                    rotate, qmax, "bf16", flags)
            assert int(flags.item()) == 0 and not nf
            assert np.array_equal(f32bits(ws), npbits(ws_ref)), (smooth, rotate)
            assert np.array_equal(codes_np(wq), wq_ref), (smooth, rotate)


def test_smooth_rotation_w4a4_layer_and_study(sq):
    """W4A4 Smooth Rotation on a down_proj-like layer with massive outliers
    (Cin = 8192, a power of two): the GEMM's accumulators are exact and Y is
    within 1 ulp of the oracle; the four-way study's errors match the
    oracle's."""
    from w8a8_post_quantization_02_b300 import pipeline
    c = synth.make_case("sr", 256, 8192, 512, dtype="bf16", x_std=0.5, w_std=0.02, alpha=0.5,
                        fixed_channels=2, fixed_factor=60.0, massive_tokens=4, massive_channels=2, seed=21)
    xf, wf = c.x_f32(), c.w_f32()
    s_ref, si_ref, _ = O.smooth_factors(O.calibrate_absmax(xf, 0), O.calibrate_absmax(wf, 1), 0.5)
    xq_ref, xs_ref, _ = O.rotate_quant_act(xf, si_ref, True, 7)
    wq_ref, ws_ref, _ = O.rotate_fold_quantize_weight(wf, s_ref, True, 7)
    acc_ref, y_ref = O.w8a8_gemm(xq_ref, xs_ref, wq_ref, ws_ref)
    x_t, w_t = dev(c.x, "bf16"), dev(c.w, "bf16")
    s_t, si_t = sq.smooth_factors(sq.calibrate_absmax(x_t, 0), sq.calibrate_absmax(w_t, 1), 0.5)
    xq, xs = sq.rotate_quant_act(x_t, si_t, True, 7, "bf16")
    wq, ws = sq.rotate_fold_quantize_weight(w_t, s_t, True, 7, "bf16")
    y, acc = sq.w8a8_gemm(xq, xs, wq, ws, want_acc=True)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), acc_ref)
    assert O.bf16_ulp_distance(y_bits(y), y_ref).max() <= 1
    rows = np.arange(0, 256, 5)
    study = pipeline.smooth_rotation_study(x_t, w_t, 0.5, 7, rows=torch.from_numpy(rows.astype(np.int32)))
    for name, smooth, rotate in (("original", False, False), ("smooth", True, False),
                                 ("rotate", False, True), ("smooth_rotate", True, True)):
        xq_r, xs_r, _ = O.rotate_quant_act(xf, si_ref if smooth else None, rotate, 7)
        wq_r, ws_r, _ = O.rotate_fold_quantize_weight(wf, s_ref if smooth else None, rotate, 7)
        _, y_r = O.w8a8_gemm(xq_r, xs_r, wq_r, ws_r)
        want = O.layer_error(xf, wf, y_r, rows).sum()
        assert _rel_close(study[name]["layer_error"], want, 1e-3), name

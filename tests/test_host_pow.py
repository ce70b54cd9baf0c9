"""The smoothing kernel's power routine, compiled for the host, agrees bit
for bit with the oracle's correctly rounded power over the statistics the
five workloads produce and a wide sweep."""
import os
import subprocess

import numpy as np
import pytest

from oracle import sq_oracle as O
from tests._lib_util import ROOT
from w8a8_post_quantization_02_b300 import build_lib, synth

F32 = np.float32


@pytest.fixture(scope="module")
def harness():
    out = os.path.join(ROOT, "_build", "host_pow_harness")
    os.makedirs(os.path.dirname(out), exist_ok=True)
    src = os.path.join(ROOT, "tests", "host_pow_harness.cu")
    deps = [src, os.path.join(build_lib.CSRC, "smooth.cu"), os.path.join(build_lib.CSRC, "sq_common.cuh")]
    if not os.path.exists(out) or any(os.path.getmtime(d) > os.path.getmtime(out) for d in deps):
        subprocess.run([build_lib.nvcc(), src, "-o", out, "-std=c++17", "-O2", "-I", build_lib.INCLUDE,
                        "-I", build_lib.CSRC, "-Xcompiler", "-ffp-contract=off", "-fmad=false"],
                       check=True)
    return out


def run_harness(exe, xs, ys):
    xs = np.asarray(xs, F32)
    ys = np.asarray(ys, F32)
    inp = "\n".join(f"{int(a):08x} {int(b):08x}" for a, b in zip(xs.view(np.uint32), ys.view(np.uint32)))
    out = subprocess.run([exe], input=inp, capture_output=True, text=True, check=True).stdout.split()
    return np.array([int(v, 16) for v in out], dtype=np.uint32).view(F32)


def test_pow_sweep_matches_oracle(harness):
    xs = np.concatenate([
        np.abs(synth.normal(21, 1, 600, 3.0)), np.abs(synth.normal(21, 2, 300, 0.02)),
        np.abs(synth.normal(21, 3, 200, 200.0)), [1e-5, 1.0, 2.0, 0.5, 1000.0, 3.0e38, 1.17549435e-38 * 8],
    ]).astype(F32)
    xs = np.maximum(xs, F32(1e-5))
    for y in (0.5, 0.85, 0.15, 0.8, 0.2, 0.3, 0.7, 0.0, 1.0, 1e-3, 0.999):
        yf = F32(y)
        got = run_harness(harness, xs, np.full(xs.shape, yf))
        want = np.array([O.rn32_pow(x, yf) for x in xs], F32)
        assert np.array_equal(got.view(np.uint32), want.view(np.uint32)), y


def test_pow_on_workload_statistics(harness):
    """The exact (x, y) pairs the smoothing step sees on the down_proj and
    shared-QKV workloads (alpha 0.85 and 0.8), on a row/column sample."""
    for name in ("down_proj_2048x11008x4096", "single_linear_64x512x512"):
        p = dict(synth.WORKLOADS[name])
        p["tokens"] = min(p["tokens"], 64)
        c = synth.make_case(name, **p)
        ax = np.maximum(O.calibrate_absmax(c.x_f32(), 0), F32(1e-5))
        aw = np.maximum(O.calibrate_absmax(c.w_f32()[:, :256], 1), F32(1e-5))
        a = F32(c.alpha)
        b = F32(F32(1) - a)
        idx = np.arange(0, ax.shape[0], max(1, ax.shape[0] // 700))
        got_p = run_harness(harness, ax[idx], np.full(idx.shape, a))
        got_q = run_harness(harness, aw[idx], np.full(idx.shape, b))
        assert np.array_equal(got_p, np.array([O.rn32_pow(v, a) for v in ax[idx]], F32))
        assert np.array_equal(got_q, np.array([O.rn32_pow(v, b) for v in aw[idx]], F32))

"""bench.py's JSON contract on a machine without a GPU: the reference arm
(the CPU oracle) prints one complete line; our arm fails loudly instead of
falling back to the CPU."""
import json
import os
import subprocess
import sys

import pytest
import torch

from tests._lib_util import ROOT

KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
        "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"}


def run_bench(*args, timeout=600):
    env = dict(os.environ, OMP_NUM_THREADS="1")
    return subprocess.run([sys.executable, "bench.py", *args], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=timeout)


def test_reference_arm_line_has_every_key():
    out = run_bench("--impl", "reference", "--steps", "1", "--warmup", "1", "--workload",
                    "single_linear_64x512x512")
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [ln for ln in out.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert KEYS <= set(d), KEYS - set(d)
    assert d["impl"] == "reference" and d["n_gpus"] == 1 and d["value"] > 0 and d["unit"] == "TOPS"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"] == "single_linear_64x512x512"


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the behaviour without a GPU")
def test_our_arm_fails_loudly_without_a_gpu():
    out = run_bench("--steps", "1", "--warmup", "3", "--workload", "single_linear_64x512x512", timeout=300)
    assert out.returncode != 0
    assert not [ln for ln in out.stdout.splitlines() if ln.startswith("{")]

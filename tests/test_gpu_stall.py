"""The kernels' bounded waits, made to run out on a GPU without faulting it.

Each case launches a kernel through its test hook (include/sq.h), whose copy
producer issues nothing, so the first wait for a copy (or for work that
depends on one) runs out after a few milliseconds.  The kernel must raise
SQ_FLAG_TIMEOUT, release what it holds (tensor memory, barriers) and return;
sq_read_device_flags must report SQ_ERR_TIMEOUT; and the same call made
normally right after must be bit-exact against the oracle, which shows that
the device, the kernel's tensor memory and the library are still usable.
"""
import ctypes
import time

import numpy as np
import pytest
import torch

from oracle import sq_oracle as O
from w8a8_post_quantization_02_b300 import synth

pytestmark = pytest.mark.gpu
F32 = np.float32
WAIT_NS = 2_000_000  # 2 ms


@pytest.fixture(scope="module")
def sq():
    from tests._lib_util import ensure_built
    ensure_built()
    from w8a8_post_quantization_02_b300 import sq as sqmod
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sqmod.check_device(torch.cuda.current_device())
    return sqmod


def _codes(m, n, k, seed):
    u = synth.uniform(seed, 5, (m + n) * k)
    c = np.clip(np.floor(u * 255.0) - 127.0, -127, 127).astype(np.int8)
    return c[: m * k].reshape(m, k), c[m * k:].reshape(n, k)


# (m, n, k, codes): the kernel each one reaches
GEMM_CASES = [
    (100, 264, 1024, "bf16"),   # tcgen05, one CTA per tile
    (300, 512, 2048, "bf16"),   # tcgen05, CTA pairs
    (100, 264, 1024, "i8"),     # int8-operand tcgen05, one CTA per tile
    (300, 512, 2048, "i8"),     # int8-operand tcgen05, CTA pairs (odd CTA forwards)
    (8, 4096, 4096, "i8"),      # weight-streaming decode kernel
]


@pytest.mark.parametrize("m,n,k,codes", GEMM_CASES)
def test_gemm_wait_runs_out_then_recovers(sq, m, n, k, codes):
    xq_np, wq_np = _codes(m, n, k, seed=m + n + k)
    xs_np = (0.001 + synth.uniform(1, 6, m)).astype(F32)
    ws_np = (0.0001 + synth.uniform(1, 7, n) * 0.01).astype(F32)
    tdt = torch.bfloat16 if codes == "bf16" else torch.int8
    xq = torch.from_numpy(xq_np.astype(F32) if codes == "bf16" else xq_np).to(tdt).cuda()
    wq = torch.from_numpy(wq_np.astype(F32) if codes == "bf16" else wq_np).to(tdt).cuda()
    xs, ws = torch.from_numpy(xs_np).cuda(), torch.from_numpy(ws_np).cuda()
    y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib = sq.load_library()
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    t0 = time.perf_counter()
    st = lib.sq_test_w8a8_gemm_stalled(P(xq), P(xs), P(wq), P(ws), sq._codes_fmt(codes), m, n, k, P(y),
                                       P(flags), WAIT_NS, sq._stream())
    assert st == sq.SQ_OK
    status, word = sq.read_device_flags(flags, clear=True)
    assert time.perf_counter() - t0 < 10.0
    assert status == sq.SQ_ERR_TIMEOUT and word & sq.SQ_FLAG_TIMEOUT
    assert int(flags.item()) == 0  # cleared by the reader
    # the same product call right after: exact
    y2, acc = sq.w8a8_gemm(xq, xs, wq, ws, want_acc=True, flags=flags)
    ref_acc, ref_y = O.w8a8_gemm(xq_np, xs_np, wq_np, ws_np)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), ref_acc)
    assert O.bf16_ulp_distance(y2.cpu().view(torch.int16).numpy().view(np.uint16), ref_y).max() <= 1
    assert sq.read_device_flags(flags) == (sq.SQ_OK, 0)


@pytest.mark.parametrize("m,n,k", [(100, 264, 1024), (300, 512, 2048)])
def test_widened_gemm_wait_runs_out_then_recovers(sq, m, n, k):
    """1-byte codes with the GEMM's workspace: the widening pass and the fp16
    GEMM after it both run stalled, both waits run out, and the product
    call right after is exact."""
    xq_np, wq_np = _codes(m, n, k, seed=m + 2 * n + k)
    xs_np = (0.001 + synth.uniform(1, 8, m)).astype(F32)
    ws_np = (0.0001 + synth.uniform(1, 9, n) * 0.01).astype(F32)
    xq, wq = torch.from_numpy(xq_np).cuda(), torch.from_numpy(wq_np).cuda()
    xs, ws = torch.from_numpy(xs_np).cuda(), torch.from_numpy(ws_np).cuda()
    y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    nbytes = sq.workspace_bytes(sq.SQ_OP_GEMM, m, n, k, "i8")
    assert nbytes > 0
    work = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    lib = sq.load_library()
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    t0 = time.perf_counter()
    st = lib.sq_test_w8a8_gemm_stalled_ws(P(xq), P(xs), P(wq), P(ws), sq.SQ_CODES_I8, m, n, k, P(y), P(flags),
                                          P(work), nbytes, WAIT_NS, sq._stream())
    assert st == sq.SQ_OK
    status, word = sq.read_device_flags(flags, clear=True)
    assert time.perf_counter() - t0 < 10.0
    assert status == sq.SQ_ERR_TIMEOUT and word & sq.SQ_FLAG_TIMEOUT
    y2, acc = sq.w8a8_gemm(xq, xs, wq, ws, want_acc=True, flags=flags, workspace=work)
    ref_acc, ref_y = O.w8a8_gemm(xq_np, xs_np, wq_np, ws_np)
    assert np.array_equal(acc.cpu().numpy().astype(np.int64), ref_acc)
    assert O.bf16_ulp_distance(y2.cpu().view(torch.int16).numpy().view(np.uint16), ref_y).max() <= 1
    assert sq.read_device_flags(flags) == (sq.SQ_OK, 0)


def test_quant_act_wait_runs_out_then_recovers(sq):
    c = synth.make_case("stall", 300, 4096, 8, dtype="bf16", outlier_frac=0.01, seed=9)
    si = (0.5 + synth.uniform(3, 4, 4096)).astype(F32)
    x = torch.from_numpy(np.ascontiguousarray(c.x).view(np.int16)).view(torch.bfloat16).cuda()
    s_inv = torch.from_numpy(si).cuda()
    xq = torch.empty(300, 4096, dtype=torch.int8, device="cuda")
    x_scale = torch.empty(300, dtype=torch.float32, device="cuda")
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    lib = sq.load_library()
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = lib.sq_test_quant_act_stalled(P(x), sq.SQ_BF16, 300, 4096, 4096, P(s_inv), P(xq), sq.SQ_CODES_I8,
                                       P(x_scale), P(flags), WAIT_NS, sq._stream())
    assert st == sq.SQ_OK
    status, word = sq.read_device_flags(flags, clear=True)
    assert status == sq.SQ_ERR_TIMEOUT and word == sq.SQ_FLAG_TIMEOUT
    xq2, xs2 = sq.quant_act(x, s_inv, "i8", flags)
    q_ref, d_ref, _ = O.quant_act(c.x_f32(), si)
    assert np.array_equal(xq2.cpu().numpy(), q_ref)
    assert np.array_equal(xs2.cpu().numpy().view(np.uint32), d_ref.view(np.uint32))
    assert sq.read_device_flags(flags) == (sq.SQ_OK, 0)


def test_nonfinite_statistic_reported_by_the_reader(sq):
    """A NaN statistic raises SQ_FLAG_NONFINITE, read back as SQ_ERR_NONFINITE."""
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    ax = torch.tensor([1.0, float("nan")] + [1.0] * 14, device="cuda")
    sq.smooth_factors(ax, torch.ones(16, device="cuda"), 0.5, flags)
    assert sq.read_device_flags(flags) == (sq.SQ_ERR_NONFINITE, sq.SQ_FLAG_NONFINITE)

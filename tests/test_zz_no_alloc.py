"""The allocation-free weight fold + quantization entry point.

Callers that cannot give the library device scratch memory (an engine
callback that only receives a stream and its tensors, or a host whose
device memory is fully reserved up front) use
sq_fold_quantize_weight_noalloc, whose scratch is a fixed array inside the
library.  Through the C ABI, two calls in a row must give exactly what the
workspace-taking sq_fold_quantize_weight gives; the second call uses
smaller weights than the first, so stale scratch contents from the first
call would show up as wrong scales.  Both weights have rows whose length in
bytes is not a multiple of 16, which sends them down the two-pass fold, the
path that keeps its per-channel maxima in the scratch array.  Collected
last so that a stop at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from w8a8_post_quantization_02_b300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    from tests._lib_util import ensure_built
    ensure_built()
    from w8a8_post_quantization_02_b300 import sq
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    sq.check_device(torch.cuda.current_device())
    return sq


def _weights(seed, cin, cout, scale):
    c = synth.make_case("w", 1, cin, cout, dtype="bf16", w_std=0.02 * scale, seed=seed)
    w = torch.from_numpy(c.w.view(np.int16)).view(torch.bfloat16).cuda()
    s = (0.5 + torch.from_numpy(synth.uniform(seed, 40, cin)).float()).cuda()
    return w, s


def _with_workspace(sq, w, s, codes):
    return sq.fold_quantize_weight(w, s, codes)


def _no_alloc(sq, w, s, codes):
    L, P = sq.load_library(), ctypes.c_void_p
    cin, cout = w.shape
    wq = torch.empty(cout, cin, device="cuda", dtype=sq._codes_dtype(codes))
    ws = torch.empty(cout, device="cuda", dtype=torch.float32)
    flags = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = L.sq_fold_quantize_weight_noalloc(P(w.data_ptr()), sq.SQ_BF16, cin, cout, w.stride(0),
                                           P(s.data_ptr()), P(wq.data_ptr()), sq._codes_fmt(codes),
                                           P(ws.data_ptr()), P(flags.data_ptr()),
                                           sq._stream())
    assert st == sq.SQ_OK, L.sq_status_string(st)
    torch.cuda.synchronize()
    assert int(flags.item()) == 0
    return wq, ws


@pytest.mark.parametrize("codes", ["i8", "bf16"])
def test_two_calls_match_the_workspace_entry_point(lib, codes):
    sq = lib
    big_w, big_s = _weights(1, 512, 1004, 50.0)
    small_w, small_s = _weights(2, 256, 700, 1.0)
    for w, s in ((big_w, big_s), (small_w, small_s)):
        wq_ref, ws_ref = _with_workspace(sq, w, s, codes)
        wq, ws = _no_alloc(sq, w, s, codes)
        assert torch.equal(wq, wq_ref)
        assert torch.equal(ws.view(torch.int32), ws_ref.view(torch.int32))


def test_rejects_output_widths_beyond_the_scratch(lib):
    sq = lib
    L, P = sq.load_library(), ctypes.c_void_p
    limit = 65536
    t = torch.zeros(64, dtype=torch.float32, device="cuda")
    st = L.sq_fold_quantize_weight_noalloc(P(t.data_ptr()), sq.SQ_F32, 16, limit + 1, limit + 1,
                                           P(t.data_ptr()), P(t.data_ptr()), sq.SQ_CODES_I8,
                                           P(t.data_ptr()), None, sq._stream())
    assert st == sq.SQ_ERR_WORKSPACE

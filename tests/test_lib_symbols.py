"""The C-ABI library loads without a GPU and exports every declared entry
point; host-side argument validation answers without touching a device."""
import ctypes
import subprocess

import pytest

from tests._lib_util import declared_symbols, ensure_built


@pytest.fixture(scope="module")
def lib():
    path = ensure_built()
    from w8a8_post_quantization_02_b300 import sq
    return path, sq.load_library()


def test_header_declares_the_five_steps():
    syms = declared_symbols()
    for name in ("sq_calibrate_absmax", "sq_smooth_factors", "sq_fold_quantize_weight",
                 "sq_quant_act", "sq_w8a8_gemm"):
        assert name in syms


def test_every_declared_symbol_is_exported(lib):
    path, handle = lib
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_symbols():
        assert name in exported, name
        assert getattr(handle, name) is not None


def test_binding_signatures_cover_the_header():
    from w8a8_post_quantization_02_b300 import sq
    assert set(sq.SIGNATURES) == set(declared_symbols())


def test_status_strings(lib):
    _, h = lib
    assert h.sq_status_string(0) == b"ok"
    assert h.sq_status_string(1) == b"invalid argument"
    assert h.sq_status_string(99) == b"unknown status"
    assert h.sq_status_string(6) == b"a bounded device wait ran out"


def test_workspace_sizes(lib):
    _, h = lib
    from w8a8_post_quantization_02_b300 import sq
    assert h.sq_workspace_bytes(sq.SQ_OP_FOLD_QUANTIZE, 0, 11008, 4096, 0) >= 11008 * 4
    assert h.sq_workspace_bytes(sq.SQ_OP_QUANT_ACT, 2048, 0, 4096, 0) == 0
    # GEMM: the widened fp16 operands of 1-byte codes above 64 tokens
    assert h.sq_workspace_bytes(sq.SQ_OP_GEMM, 2048, 11008, 4096, sq.SQ_CODES_I8) == (2048 + 11008) * 4096 * 2
    assert h.sq_workspace_bytes(sq.SQ_OP_GEMM, 2048, 11008, 4096, sq.SQ_CODES_BF16) == 0
    assert h.sq_workspace_bytes(sq.SQ_OP_GEMM, 64, 11008, 4096, sq.SQ_CODES_I8) == 0


def test_argument_validation_needs_no_device(lib):
    _, h = lib
    from w8a8_post_quantization_02_b300 import sq
    P = ctypes.c_void_p
    aligned, odd = P(4096), P(4097)
    # null input
    assert h.sq_calibrate_absmax(None, sq.SQ_BF16, 4, 8, 8, 0, 0, aligned, None) == sq.SQ_ERR_INVALID_ARG
    # ld < cols, bad axis, misaligned base
    assert h.sq_calibrate_absmax(aligned, sq.SQ_BF16, 4, 8, 4, 0, 0, aligned, None) == sq.SQ_ERR_INVALID_ARG
    assert h.sq_calibrate_absmax(aligned, sq.SQ_BF16, 4, 8, 8, 2, 0, aligned, None) == sq.SQ_ERR_INVALID_ARG
    assert h.sq_calibrate_absmax(odd, sq.SQ_BF16, 4, 8, 8, 0, 0, aligned, None) == sq.SQ_ERR_INVALID_ARG
    # alpha outside [0, 1] or NaN
    for alpha in (-0.1, 1.5, float("nan"), float("inf")):
        assert h.sq_smooth_factors(aligned, aligned, 8, alpha, aligned, aligned, None, None) == sq.SQ_ERR_INVALID_ARG
    # cin not a multiple of 16; missing workspace
    assert h.sq_fold_quantize_weight(aligned, sq.SQ_BF16, 24, 8, 8, aligned, aligned, 0, aligned,
                                     None, aligned, 4096, None) == sq.SQ_ERR_INVALID_ARG
    assert h.sq_fold_quantize_weight(aligned, sq.SQ_BF16, 32, 8, 8, aligned, aligned, 0, aligned,
                                     None, None, 0, None) == sq.SQ_ERR_WORKSPACE
    # activation quantization: bad code format, too-wide rows
    assert h.sq_quant_act(aligned, sq.SQ_BF16, 4, 32, 32, aligned, aligned, 7, aligned, None, None) == sq.SQ_ERR_INVALID_ARG
    assert h.sq_quant_act(aligned, sq.SQ_F32, 4, 1 << 20, 1 << 20, aligned, aligned, 0, aligned, None, None) == sq.SQ_ERR_UNSUPPORTED
    # GEMM: k % 16 != 0, zero m, misaligned operand
    assert h.sq_w8a8_gemm(aligned, aligned, aligned, aligned, 0, 4, 4, 24, aligned, None, None, None, 0, None) == sq.SQ_ERR_INVALID_ARG
    assert h.sq_w8a8_gemm(aligned, aligned, aligned, aligned, 0, 0, 4, 32, aligned, None, None, None, 0, None) == sq.SQ_ERR_INVALID_ARG
    assert h.sq_w8a8_gemm(odd, aligned, aligned, aligned, 0, 4, 4, 32, aligned, None, None, None, 0, None) == sq.SQ_ERR_INVALID_ARG
    # GEMM: k beyond the int32 accumulator bound (k * 127^2 >= 2^31)
    assert sq.SQ_GEMM_MAX_K * 127 * 127 < 2 ** 31 <= (sq.SQ_GEMM_MAX_K + 16) * 127 * 127
    assert sq.SQ_GEMM_MAX_K % 16 == 0
    for fmt in (0, 1):
        assert h.sq_w8a8_gemm(aligned, aligned, aligned, aligned, fmt, 4, 4, sq.SQ_GEMM_MAX_K + 16, aligned,
                              None, None, None, 0, None) == sq.SQ_ERR_UNSUPPORTED
    # flag reader: null or misaligned word, bad clear argument
    out = ctypes.c_int32(0)
    assert h.sq_read_device_flags(None, 0, ctypes.byref(out), None) == sq.SQ_ERR_INVALID_ARG
    assert h.sq_read_device_flags(P(4098), 0, ctypes.byref(out), None) == sq.SQ_ERR_INVALID_ARG
    assert h.sq_read_device_flags(aligned, 2, ctypes.byref(out), None) == sq.SQ_ERR_INVALID_ARG
    # layer error: too many sampled rows, zero tokens
    assert h.sq_layer_error(aligned, aligned, sq.SQ_BF16, 4, 32, 8, 32, 8, aligned, aligned, 65, aligned,
                            None) == sq.SQ_ERR_INVALID_ARG
    assert h.sq_layer_error(aligned, aligned, sq.SQ_BF16, 0, 32, 8, 32, 8, aligned, aligned, 4, aligned,
                            None) == sq.SQ_ERR_INVALID_ARG
    # whole path from host memory: null host buffer, cin % 16, missing device buffer, workspace
    full = {n: type("T", (), {"data_ptr": lambda self: 4096})() for n in
            ("x", "w", "amax_x", "amax_w", "s", "s_inv", "wq", "w_scale", "xq", "x_scale", "y")}
    ws = type("W", (), {"data_ptr": lambda self: 8192, "numel": lambda self: 1 << 20,
                        "element_size": lambda self: 1})()
    b = sq.linear_buffers(full, ws)
    L = h.sq_linear_host
    assert L(None, aligned, sq.SQ_BF16, 4, 32, 8, 0.5, 0, aligned, ctypes.byref(b), None, None) == sq.SQ_ERR_INVALID_ARG
    assert L(aligned, aligned, sq.SQ_BF16, 4, 24, 8, 0.5, 0, aligned, ctypes.byref(b), None, None) == sq.SQ_ERR_INVALID_ARG
    assert L(aligned, aligned, sq.SQ_BF16, 4, 32, 8, 1.5, 0, aligned, ctypes.byref(b), None, None) == sq.SQ_ERR_INVALID_ARG
    b.xq = 4097
    assert L(aligned, aligned, sq.SQ_BF16, 4, 32, 8, 0.5, 0, aligned, ctypes.byref(b), None, None) == sq.SQ_ERR_INVALID_ARG
    b.xq = 4096
    b.s = None
    assert L(aligned, aligned, sq.SQ_BF16, 4, 32, 8, 0.5, 0, aligned, ctypes.byref(b), None, None) == sq.SQ_ERR_INVALID_ARG
    b.s = 4096
    b.ws_bytes = 0
    assert L(aligned, aligned, sq.SQ_BF16, 4, 32, 8, 0.5, 0, aligned, ctypes.byref(b), None, None) == sq.SQ_ERR_WORKSPACE


def test_kernel_counts_need_no_device(lib):
    _, h = lib
    from w8a8_post_quantization_02_b300 import sq
    # fold: one kernel when rows are 16-byte aligned and Cin fits 8 CTAs of
    # 1536 rows; else the two-pass path (fill, column maxima, quantize)
    assert h.sq_kernel_count(sq.SQ_OP_FOLD_QUANTIZE, sq.SQ_BF16, 0, 11008, 4096, 11008, 0, 0) == 1
    assert h.sq_kernel_count(sq.SQ_OP_FOLD_QUANTIZE, sq.SQ_BF16, 0, 4096, 11008, 4096, 0, 0) == 1
    assert h.sq_kernel_count(sq.SQ_OP_FOLD_QUANTIZE, sq.SQ_BF16, 0, 300, 80, 300, 0, 0) == 3
    assert h.sq_kernel_count(sq.SQ_OP_FOLD_QUANTIZE, sq.SQ_BF16, 0, 64, 12304, 64, 0, 0) == 3
    for op in (sq.SQ_OP_SMOOTH, sq.SQ_OP_QUANT_ACT):
        assert h.sq_kernel_count(op, sq.SQ_BF16, 2048, 11008, 4096, 4096, 0, 0) == 1
    # GEMM (axis: the code format): one kernel, except 1-byte codes above 64
    # tokens, which are widened in the workspace first
    assert h.sq_kernel_count(sq.SQ_OP_GEMM, sq.SQ_BF16, 2048, 11008, 4096, 0, sq.SQ_CODES_BF16, 0) == 1
    assert h.sq_kernel_count(sq.SQ_OP_GEMM, sq.SQ_BF16, 2048, 11008, 4096, 0, sq.SQ_CODES_I8, 0) == 2
    assert h.sq_kernel_count(sq.SQ_OP_GEMM, sq.SQ_BF16, 64, 11008, 4096, 0, sq.SQ_CODES_I8, 0) == 1
    assert h.sq_kernel_count(99, sq.SQ_BF16, 1, 1, 16, 16, 0, 0) == -1


def test_host_binding_checks_shapes_and_dtypes(lib):
    import torch
    from w8a8_post_quantization_02_b300 import sq
    b = sq.LinearBuffers()
    x = torch.zeros(4, 32, dtype=torch.bfloat16)
    y = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):  # W's dtype differs from X's
        sq.linear_host(x, torch.zeros(32, 8, dtype=torch.float32), 0.5, "i8", y, b)
    with pytest.raises(ValueError):  # X's columns and W's rows do not chain
        sq.linear_host(x, torch.zeros(16, 8, dtype=torch.bfloat16), 0.5, "i8", y, b)
    with pytest.raises(ValueError):  # Y is not tokens x cout
        sq.linear_host(x, torch.zeros(32, 8, dtype=torch.bfloat16), 0.5, "i8", torch.zeros(4, 9, dtype=torch.bfloat16), b)


def test_layer_error_binding_rejects_rows_outside_the_tokens(lib, monkeypatch):
    """A sampled token index outside [0, tokens), or an output of the wrong
    shape, is refused on the host before anything reaches the device."""
    import torch
    from w8a8_post_quantization_02_b300 import sq
    monkeypatch.setattr(sq, "_check_cuda_2d", lambda t, name: None)
    x = torch.zeros(4, 32, dtype=torch.bfloat16)
    w = torch.zeros(32, 8, dtype=torch.bfloat16)
    y = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        sq.layer_error(x, w, y, torch.tensor([0, 4]))
    with pytest.raises(ValueError):
        sq.layer_error(x, w, y, torch.tensor([-1]))
    with pytest.raises(ValueError):
        sq.layer_error(x, w, torch.zeros(3, 8, dtype=torch.bfloat16), torch.tensor([0]))

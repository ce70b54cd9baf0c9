// C ABI entry points: argument validation, workspace sizing and dispatch.
#include "sq_common.cuh"

namespace sq {
sq_status calibrate_absmax(const void*, sq_dtype, int64_t, int64_t, int64_t, int, int, float*,
                           cudaStream_t);
sq_status smooth_factors(const float*, const float*, int64_t, float, float*, float*, int32_t*,
                         cudaStream_t);
sq_status fold_quantize_weight(const void*, sq_dtype, int64_t, int64_t, int64_t, const float*,
                               void*, sq_codes, float*, int32_t*, void*, cudaStream_t);
sq_status quant_act(const void*, sq_dtype, int64_t, int64_t, int64_t, const float*, void*,
                    sq_codes, float*, int32_t*, cudaStream_t);
int64_t quant_act_max_cin(sq_dtype);
sq_status static_act_scale(const float*, const float*, int64_t, float*, int32_t*, cudaStream_t);
sq_status fold_norm_gain(const float*, const float*, int64_t, float*, cudaStream_t);
bool rotate_len_ok(int64_t, sq_dtype, bool);
sq_status rotate_quant_rows(const void*, sq_dtype, int64_t, int64_t, int64_t, const float*, bool, int,
                            int, void*, sq_codes, float*, int32_t*, cudaStream_t);
sq_status fold_transpose(const void*, sq_dtype, int64_t, int64_t, int64_t, const float*, float*,
                         cudaStream_t);
sq_status rmsnorm_quant_act(const void*, sq_dtype, int64_t, int64_t, int64_t, const float*, float,
                            void*, sq_codes, float*, int32_t*, cudaStream_t);
sq_status quant_act_static(const void*, sq_dtype, int64_t, int64_t, int64_t, const float*,
                           const float*, void*, sq_codes, float*, uint32_t*, int32_t*, cudaStream_t);
int fold_kernel_count(sq_dtype, int64_t, int64_t, int64_t);
sq_status act_quant_error(const void*, sq_dtype, int64_t, int64_t, int64_t, const float*, const void*,
                          sq_codes, const float*, double*, cudaStream_t);
sq_status weight_quant_error(const void*, sq_dtype, int64_t, int64_t, int64_t, const float*,
                             const void*, sq_codes, const float*, double*, cudaStream_t);
int layer_error_max_rows();
sq_status layer_error(const void*, const void*, sq_dtype, int64_t, int64_t, int64_t, int64_t, int64_t,
                      const void*, const int32_t*, int, double*, cudaStream_t);
sq_status channel_stats(const float*, const float*, int64_t, double*, cudaStream_t);
int calibrate_kernel_count(sq_dtype, int64_t, int64_t, int64_t, int, int);
sq_status gemm_i8_mma(const int8_t*, const float*, const int8_t*, const float*, int64_t, int64_t,
                      int64_t, void*, int32_t*, cudaStream_t);
sq_status gemm_bf16c_tc(const void*, const float*, const void*, const float*, int64_t, int64_t,
                        int64_t, void*, int32_t*, int32_t*, uint64_t, int, cudaStream_t, bool);
sq_status gemm_i8_widened_tc(const void*, const float*, const void*, const float*, int64_t, int64_t,
                             int64_t, void*, int32_t*, int32_t*, void*, uint64_t, int, cudaStream_t);
size_t gemm_widen_bytes(int64_t, int64_t, int64_t);
sq_status gemm_i8c_tc(const void*, const float*, const void*, const float*, int64_t, int64_t,
                      int64_t, void*, int32_t*, int32_t*, uint64_t, int, cudaStream_t);
sq_status quant_act_stalled(const void*, sq_dtype, int64_t, int64_t, int64_t, const float*, void*,
                            sq_codes, float*, int32_t*, uint64_t, cudaStream_t);
// Bound on each pipeline wait of the GEMM kernels in a product call.
constexpr uint64_t kGemmWaitNs = 2000000000ull;
sq_status gemm_dec(const int8_t*, const float*, const int8_t*, const float*, int64_t, int64_t, int64_t,
                   void*, int32_t*, int32_t*, uint64_t, int, cudaStream_t);
int64_t gemm_dec_max_m();
// Token count above which 1-byte codes run on the tensor cores (below it
// the weight-streaming kernels, whose grids cover the SMs at small M).
constexpr int64_t kI8TensorCoreMinM = 64;

namespace {
bool valid_dtype(sq_dtype d) { return d == SQ_F32 || d == SQ_BF16; }
bool valid_codes(sq_codes c) { return c == SQ_CODES_I8 || c == SQ_CODES_BF16; }
size_t round256(size_t b) { return (b + 255) & ~size_t(255); }
}  // namespace
}  // namespace sq

using namespace sq;

extern "C" {

const char* sq_status_string(sq_status s) {
  switch (s) {
    case SQ_OK: return "ok";
    case SQ_ERR_INVALID_ARG: return "invalid argument";
    case SQ_ERR_NONFINITE: return "non-finite value";
    case SQ_ERR_CUDA: return "CUDA error";
    case SQ_ERR_UNSUPPORTED: return "unsupported request";
    case SQ_ERR_WORKSPACE: return "workspace missing or too small";
    case SQ_ERR_TIMEOUT: return "a bounded device wait ran out";
  }
  return "unknown status";
}

sq_status sq_read_device_flags(int32_t* dev_flags, int clear, int32_t* flags_out,
                               cudaStream_t stream) {
  if (!dev_flags || (clear != 0 && clear != 1) || (reinterpret_cast<uintptr_t>(dev_flags) & 3))
    return SQ_ERR_INVALID_ARG;
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, dev_flags, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return SQ_ERR_CUDA;
  if (clear && cudaMemsetAsync(dev_flags, 0, sizeof(v), stream) != cudaSuccess) return SQ_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SQ_ERR_CUDA;
  if (flags_out) *flags_out = v;
  if (v & SQ_FLAG_TIMEOUT) return SQ_ERR_TIMEOUT;
  if (v & SQ_FLAG_NONFINITE) return SQ_ERR_NONFINITE;
  return SQ_OK;
}

sq_status sq_check_device(int device) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess)
    return SQ_ERR_CUDA;
  return (major == 10 && minor == 3) ? SQ_OK : SQ_ERR_UNSUPPORTED;
}

size_t sq_workspace_bytes(sq_op op, int64_t m, int64_t n, int64_t k, sq_codes fmt) {
  switch (op) {
    case SQ_OP_FOLD_QUANTIZE: return n > 0 ? round256((size_t)n * 4) : 0;
    case SQ_OP_ROTATE_WEIGHT: return (n > 0 && k > 0) ? round256((size_t)n * (size_t)k * 4) : 0;
    case SQ_OP_GEMM:  // 1-byte codes on the tensor cores: both operands widened to fp16
      return (fmt == SQ_CODES_I8 && m > kI8TensorCoreMinM && n > 0 && k > 0) ? round256(gemm_widen_bytes(m, n, k))
                                                                              : 0;
    default: return 0;
  }
}

int sq_kernel_count(sq_op op, sq_dtype dt, int64_t m, int64_t n, int64_t k, int64_t ld, int axis,
                    int accumulate) {
  switch (op) {
    case SQ_OP_CALIBRATE: return calibrate_kernel_count(dt, m, n, ld, axis, accumulate);
    case SQ_OP_SMOOTH: return 1;
    case SQ_OP_FOLD_QUANTIZE: return fold_kernel_count(dt, k, n, ld);
    case SQ_OP_QUANT_ACT: return 1;
    case SQ_OP_STATIC_SCALE: return 1;
    case SQ_OP_QUANT_ACT_STATIC: return 1;
    case SQ_OP_FOLD_NORM_GAIN: return 1;
    case SQ_OP_RMSNORM_QUANT_ACT: return 1;
    case SQ_OP_ROTATE_ACT: return 1;
    case SQ_OP_ROTATE_WEIGHT: return 2;
    case SQ_OP_GEMM:  // axis: the code format (sq_codes)
      return (axis == SQ_CODES_I8 && m > kI8TensorCoreMinM) ? 2 : 1;
  }
  return -1;
}

sq_status sq_calibrate_absmax(const void* a, sq_dtype dt, int64_t rows, int64_t cols, int64_t ld,
                              int axis, int accumulate, float* amax, cudaStream_t stream) {
  if (!a || !amax || !valid_dtype(dt) || rows < 1 || cols < 1 || ld < cols ||
      (axis != 0 && axis != 1) || (accumulate != 0 && accumulate != 1))
    return SQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(a) % elem_bytes(dt)) != 0 || (reinterpret_cast<uintptr_t>(amax) & 3))
    return SQ_ERR_INVALID_ARG;
  return calibrate_absmax(a, dt, rows, cols, ld, axis, accumulate, amax, stream);
}

sq_status sq_smooth_factors(const float* amax_x, const float* amax_w, int64_t cin, float alpha,
                            float* s, float* s_inv, int32_t* dev_flags, cudaStream_t stream) {
  if (!amax_x || !amax_w || !s || !s_inv || cin < 1) return SQ_ERR_INVALID_ARG;
  if (!(alpha >= 0.0f && alpha <= 1.0f)) return SQ_ERR_INVALID_ARG;  // also rejects NaN
  return smooth_factors(amax_x, amax_w, cin, alpha, s, s_inv, dev_flags, stream);
}

sq_status sq_fold_quantize_weight(const void* w, sq_dtype dt, int64_t cin, int64_t cout,
                                  int64_t ldw, const float* s, void* wq, sq_codes fmt,
                                  float* w_scale, int32_t* dev_flags, void* workspace,
                                  size_t ws_bytes, cudaStream_t stream) {
  if (!w || !s || !wq || !w_scale || !valid_dtype(dt) || !valid_codes(fmt) || cin < 1 ||
      cout < 1 || ldw < cout || cin % 16 != 0)
    return SQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(w) % elem_bytes(dt)) != 0 || !aligned16(wq) || (reinterpret_cast<uintptr_t>(s) & 3) ||
      (reinterpret_cast<uintptr_t>(w_scale) & 3))
    return SQ_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < sq_workspace_bytes(SQ_OP_FOLD_QUANTIZE, 0, cout, cin, fmt) ||
      (reinterpret_cast<uintptr_t>(workspace) & 3))
    return SQ_ERR_WORKSPACE;
  return fold_quantize_weight(w, dt, cin, cout, ldw, s, wq, fmt, w_scale, dev_flags, workspace,
                              stream);
}

sq_status sq_quant_act(const void* x, sq_dtype dt, int64_t tokens, int64_t cin, int64_t ldx,
                       const float* s_inv, void* xq, sq_codes fmt, float* x_scale,
                       int32_t* dev_flags, cudaStream_t stream) {
  if (!x || !s_inv || !xq || !x_scale || !valid_dtype(dt) || !valid_codes(fmt) || tokens < 1 ||
      cin < 1 || ldx < cin || cin % 16 != 0)
    return SQ_ERR_INVALID_ARG;
  if (!aligned16(x) || (ldx * elem_bytes(dt)) % 16 != 0 || !aligned16(xq) || !aligned16(s_inv))
    return SQ_ERR_INVALID_ARG;
  if (cin > quant_act_max_cin(dt)) return SQ_ERR_UNSUPPORTED;
  return quant_act(x, dt, tokens, cin, ldx, s_inv, xq, fmt, x_scale, dev_flags, stream);
}

sq_status sq_static_act_scale(const float* amax_x, const float* s_inv, int64_t cin, float* d,
                              int32_t* dev_flags, cudaStream_t stream) {
  if (!amax_x || !s_inv || !d || cin < 1) return SQ_ERR_INVALID_ARG;
  return static_act_scale(amax_x, s_inv, cin, d, dev_flags, stream);
}

sq_status sq_quant_act_static(const void* x, sq_dtype dt, int64_t tokens, int64_t cin, int64_t ldx,
                              const float* s_inv, const float* d, void* xq, sq_codes fmt,
                              float* x_scale, uint32_t* clipped, int32_t* dev_flags,
                              cudaStream_t stream) {
  if (!x || !s_inv || !d || !xq || !x_scale || !valid_dtype(dt) || !valid_codes(fmt) ||
      tokens < 1 || cin < 1 || ldx < cin || cin % 16 != 0)
    return SQ_ERR_INVALID_ARG;
  if (!aligned16(x) || (ldx * elem_bytes(dt)) % 16 != 0 || !aligned16(xq) || !aligned16(s_inv) ||
      (reinterpret_cast<uintptr_t>(clipped) & 3))
    return SQ_ERR_INVALID_ARG;
  if (cin > ((int64_t)1 << 30)) return SQ_ERR_UNSUPPORTED;
  return quant_act_static(x, dt, tokens, cin, ldx, s_inv, d, xq, fmt, x_scale, clipped, dev_flags,
                          stream);
}

sq_status sq_fold_norm_gain(const float* gamma, const float* s_inv, int64_t cin,
                            float* gamma_folded, cudaStream_t stream) {
  if (!gamma || !s_inv || !gamma_folded || cin < 1) return SQ_ERR_INVALID_ARG;
  return fold_norm_gain(gamma, s_inv, cin, gamma_folded, stream);
}

sq_status sq_rmsnorm_quant_act(const void* h, sq_dtype dt, int64_t tokens, int64_t cin,
                               int64_t ldh, const float* gamma_folded, float eps, void* xq,
                               sq_codes fmt, float* x_scale, int32_t* dev_flags,
                               cudaStream_t stream) {
  if (!h || !gamma_folded || !xq || !x_scale || !valid_dtype(dt) || !valid_codes(fmt) || tokens < 1 ||
      cin < 1 || ldh < cin || cin % 16 != 0 || !(eps >= 0.0f) || !(eps < 3.4e38f))
    return SQ_ERR_INVALID_ARG;
  if (!aligned16(h) || (ldh * elem_bytes(dt)) % 16 != 0 || !aligned16(xq) || !aligned16(gamma_folded))
    return SQ_ERR_INVALID_ARG;
  if (cin > quant_act_max_cin(dt)) return SQ_ERR_UNSUPPORTED;
  return rmsnorm_quant_act(h, dt, tokens, cin, ldh, gamma_folded, eps, xq, fmt, x_scale, dev_flags,
                           stream);
}

sq_status sq_rotate_quant_act(const void* x, sq_dtype dt, int64_t tokens, int64_t cin, int64_t ldx,
                              const float* s_inv, int rotate, int qmax, void* xq, sq_codes fmt,
                              float* x_scale, int32_t* dev_flags, cudaStream_t stream) {
  if (!x || !xq || !x_scale || !valid_dtype(dt) || !valid_codes(fmt) || tokens < 1 || cin < 1 ||
      ldx < cin || cin % 16 != 0 || qmax < 1 || qmax > 127 || (rotate != 0 && rotate != 1))
    return SQ_ERR_INVALID_ARG;
  if (!aligned16(x) || (ldx * elem_bytes(dt)) % 16 != 0 || !aligned16(xq) || (s_inv && !aligned16(s_inv)))
    return SQ_ERR_INVALID_ARG;
  if (!rotate_len_ok(cin, dt, rotate != 0)) return SQ_ERR_UNSUPPORTED;
  int l2 = 0;
  while ((1LL << l2) < cin) ++l2;
  return rotate_quant_rows(x, dt, tokens, cin, ldx, s_inv, rotate != 0, qmax, rotate ? l2 : 0, xq, fmt,
                           x_scale, dev_flags, stream);
}

sq_status sq_rotate_fold_quantize_weight(const void* w, sq_dtype dt, int64_t cin, int64_t cout,
                                         int64_t ldw, const float* s, int rotate, int qmax,
                                         void* wq, sq_codes fmt, float* w_scale,
                                         int32_t* dev_flags, void* workspace, size_t ws_bytes,
                                         cudaStream_t stream) {
  if (!w || !wq || !w_scale || !valid_dtype(dt) || !valid_codes(fmt) || cin < 1 || cout < 1 ||
      ldw < cout || cin % 16 != 0 || qmax < 1 || qmax > 127 || (rotate != 0 && rotate != 1))
    return SQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(w) % elem_bytes(dt)) != 0 || !aligned16(wq)) return SQ_ERR_INVALID_ARG;
  if (!workspace || ws_bytes < sq_workspace_bytes(SQ_OP_ROTATE_WEIGHT, 0, cout, cin, fmt) ||
      !aligned16(workspace))
    return SQ_ERR_WORKSPACE;
  if (!rotate_len_ok(cin, SQ_F32, rotate != 0)) return SQ_ERR_UNSUPPORTED;
  float* wt = static_cast<float*>(workspace);
  const sq_status st = fold_transpose(w, dt, cin, cout, ldw, s, wt, stream);
  if (st != SQ_OK) return st;
  return rotate_quant_rows(wt, SQ_F32, cout, cin, cin, nullptr, rotate != 0, qmax, 0, wq, fmt, w_scale,
                           dev_flags, stream);
}

sq_status sq_act_quant_error(const void* x, sq_dtype dt, int64_t tokens, int64_t cin, int64_t ldx,
                             const float* s_inv, const void* xq, sq_codes fmt, const float* x_scale,
                             double* err, cudaStream_t stream) {
  if (!x || !s_inv || !xq || !x_scale || !err || !valid_dtype(dt) || !valid_codes(fmt) || tokens < 1 ||
      cin < 1 || ldx < cin || cin % 16 != 0)
    return SQ_ERR_INVALID_ARG;
  if (!aligned16(x) || (ldx * elem_bytes(dt)) % 16 != 0 || !aligned16(xq) ||
      (reinterpret_cast<uintptr_t>(err) & 7))
    return SQ_ERR_INVALID_ARG;
  return act_quant_error(x, dt, tokens, cin, ldx, s_inv, xq, fmt, x_scale, err, stream);
}

sq_status sq_weight_quant_error(const void* w, sq_dtype dt, int64_t cin, int64_t cout, int64_t ldw,
                                const float* s, const void* wq, sq_codes fmt, const float* w_scale,
                                double* err, cudaStream_t stream) {
  if (!w || !s || !wq || !w_scale || !err || !valid_dtype(dt) || !valid_codes(fmt) || cin < 1 ||
      cout < 1 || ldw < cout)
    return SQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(w) % elem_bytes(dt)) != 0 || (reinterpret_cast<uintptr_t>(err) & 7))
    return SQ_ERR_INVALID_ARG;
  return weight_quant_error(w, dt, cin, cout, ldw, s, wq, fmt, w_scale, err, stream);
}

sq_status sq_layer_error(const void* x, const void* w, sq_dtype dt, int64_t tokens, int64_t cin,
                         int64_t cout, int64_t ldx, int64_t ldw, const void* y,
                         const int32_t* rows, int nrows, double* err, cudaStream_t stream) {
  if (!x || !w || !y || !rows || !err || !valid_dtype(dt) || tokens < 1 || cin < 1 || cout < 1 ||
      ldx < cin || ldw < cout || nrows < 1 || nrows > layer_error_max_rows())
    return SQ_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) % elem_bytes(dt)) != 0 ||
      (reinterpret_cast<uintptr_t>(w) % elem_bytes(dt)) != 0 || (reinterpret_cast<uintptr_t>(y) & 1) ||
      (reinterpret_cast<uintptr_t>(rows) & 3) || (reinterpret_cast<uintptr_t>(err) & 7))
    return SQ_ERR_INVALID_ARG;
  return layer_error(x, w, dt, tokens, cin, cout, ldx, ldw, y, rows, nrows, err, stream);
}

sq_status sq_channel_stats(const float* amax, const float* scale, int64_t n, double* out,
                           cudaStream_t stream) {
  if (!amax || !out || n < 1 || (reinterpret_cast<uintptr_t>(out) & 7)) return SQ_ERR_INVALID_ARG;
  return channel_stats(amax, scale, n, out, stream);
}

namespace {
// The GEMM dispatch shared by sq_w8a8_gemm and its stalled test form.
sq_status w8a8_gemm_dispatch(const void* xq, const float* x_scale, const void* wq,
                             const float* w_scale, sq_codes fmt, int64_t m, int64_t n, int64_t k,
                             void* y, int32_t* acc_out, int32_t* dev_flags, uint64_t wait_ns,
                             int stall, cudaStream_t stream, void* workspace = nullptr,
                             size_t ws_bytes = 0) {
  if (!xq || !x_scale || !wq || !w_scale || !y || !valid_codes(fmt) || m < 1 || n < 1 || k < 16 ||
      k % 16 != 0)
    return SQ_ERR_INVALID_ARG;
  if (!aligned16(xq) || !aligned16(wq) || (reinterpret_cast<uintptr_t>(y) & 3) ||
      (reinterpret_cast<uintptr_t>(acc_out) & 3))
    return SQ_ERR_INVALID_ARG;
  if (k > SQ_GEMM_MAX_K) return SQ_ERR_UNSUPPORTED;  // int32 accumulators could wrap
  if (fmt == SQ_CODES_I8 && m <= gemm_dec_max_m())
    return gemm_dec(static_cast<const int8_t*>(xq), x_scale, static_cast<const int8_t*>(wq), w_scale,
                    m, n, k, y, acc_out, dev_flags, wait_ns, stall, stream);
  if (fmt == SQ_CODES_I8 && m <= kI8TensorCoreMinM) {
    if (stall) return SQ_ERR_UNSUPPORTED;  // the mma.sync kernel has no pipeline waits
    return gemm_i8_mma(static_cast<const int8_t*>(xq), x_scale, static_cast<const int8_t*>(wq),
                       w_scale, m, n, k, y, acc_out, stream);
  }
  if (fmt == SQ_CODES_I8) {
    // with room for the widened operands: one pass widens both to fp16 and
    // the 16-bit-carrier kernel runs; otherwise the kernel that widens in
    // shared memory as it goes
    if (workspace && aligned16(workspace) && ws_bytes >= gemm_widen_bytes(m, n, k))
      return gemm_i8_widened_tc(xq, x_scale, wq, w_scale, m, n, k, y, acc_out, dev_flags, workspace,
                                wait_ns, stall, stream);
    return gemm_i8c_tc(xq, x_scale, wq, w_scale, m, n, k, y, acc_out, dev_flags, wait_ns, stall, stream);
  }
  return gemm_bf16c_tc(xq, x_scale, wq, w_scale, m, n, k, y, acc_out, dev_flags, wait_ns, stall, stream,
                       false);
}
}  // namespace

sq_status sq_w8a8_gemm(const void* xq, const float* x_scale, const void* wq, const float* w_scale,
                       sq_codes fmt, int64_t m, int64_t n, int64_t k, void* y, int32_t* acc_out,
                       int32_t* dev_flags, void* workspace, size_t ws_bytes,
                       cudaStream_t stream) {
  return w8a8_gemm_dispatch(xq, x_scale, wq, w_scale, fmt, m, n, k, y, acc_out, dev_flags, kGemmWaitNs,
                            0, stream, workspace, ws_bytes);
}

sq_status sq_test_w8a8_gemm_stalled(const void* xq, const float* x_scale, const void* wq,
                                    const float* w_scale, sq_codes fmt, int64_t m, int64_t n,
                                    int64_t k, void* y, int32_t* dev_flags, uint64_t wait_ns,
                                    cudaStream_t stream) {
  if (!dev_flags || wait_ns < 100000ull || wait_ns > 1000000000ull) return SQ_ERR_INVALID_ARG;
  return w8a8_gemm_dispatch(xq, x_scale, wq, w_scale, fmt, m, n, k, y, nullptr, dev_flags, wait_ns, 1,
                            stream);
}

sq_status sq_test_w8a8_gemm_stalled_ws(const void* xq, const float* x_scale, const void* wq,
                                       const float* w_scale, sq_codes fmt, int64_t m, int64_t n,
                                       int64_t k, void* y, int32_t* dev_flags, void* workspace,
                                       size_t ws_bytes, uint64_t wait_ns, cudaStream_t stream) {
  if (!dev_flags || wait_ns < 100000ull || wait_ns > 1000000000ull) return SQ_ERR_INVALID_ARG;
  return w8a8_gemm_dispatch(xq, x_scale, wq, w_scale, fmt, m, n, k, y, nullptr, dev_flags, wait_ns, 1,
                            stream, workspace, ws_bytes);
}

sq_status sq_test_quant_act_stalled(const void* x, sq_dtype dt, int64_t tokens, int64_t cin,
                                    int64_t ldx, const float* s_inv, void* xq, sq_codes fmt,
                                    float* x_scale, int32_t* dev_flags, uint64_t wait_ns,
                                    cudaStream_t stream) {
  if (!dev_flags || wait_ns < 100000ull || wait_ns > 1000000000ull) return SQ_ERR_INVALID_ARG;
  if (!x || !s_inv || !xq || !x_scale || !valid_dtype(dt) || !valid_codes(fmt) || tokens < 1 ||
      cin < 1 || ldx < cin || cin % 16 != 0)
    return SQ_ERR_INVALID_ARG;
  if (!aligned16(x) || (ldx * elem_bytes(dt)) % 16 != 0 || !aligned16(xq) || !aligned16(s_inv))
    return SQ_ERR_INVALID_ARG;
  if (cin > quant_act_max_cin(dt)) return SQ_ERR_UNSUPPORTED;
  return quant_act_stalled(x, dt, tokens, cin, ldx, s_inv, xq, fmt, x_scale, dev_flags, wait_ns, stream);
}

sq_status sq_linear_host(const void* x_host, const void* w_host, sq_dtype dt, int64_t tokens,
                         int64_t cin, int64_t cout, float alpha, sq_codes fmt, void* y_host,
                         const sq_linear_buffers* dev, int32_t* dev_flags, cudaStream_t stream) {
  // every condition the steps check, before anything is enqueued
  if (!x_host || !w_host || !y_host || !dev || !valid_dtype(dt) || !valid_codes(fmt) ||
      tokens < 1 || cin < 1 || cout < 1 || cin % 16 != 0 || !(alpha >= 0.0f && alpha <= 1.0f))
    return SQ_ERR_INVALID_ARG;
  const sq_linear_buffers& b = *dev;
  const void* const any[] = {b.x, b.w, b.amax_x, b.amax_w, b.s, b.s_inv, b.wq, b.w_scale, b.xq,
                             b.x_scale, b.y};
  for (const void* p : any)
    if (!p) return SQ_ERR_INVALID_ARG;
  const void* const words[] = {b.amax_x, b.amax_w, b.w_scale, b.x_scale, b.y};
  for (const void* p : words)
    if (reinterpret_cast<uintptr_t>(p) & 3) return SQ_ERR_INVALID_ARG;
  if (!aligned16(b.x) || !aligned16(b.xq) || !aligned16(b.wq) || !aligned16(b.s_inv) ||
      (reinterpret_cast<uintptr_t>(b.s) & 3) || (reinterpret_cast<uintptr_t>(b.w) % elem_bytes(dt)))
    return SQ_ERR_INVALID_ARG;
  if (cin > quant_act_max_cin(dt)) return SQ_ERR_UNSUPPORTED;
  if (!b.workspace || b.ws_bytes < sq_workspace_bytes(SQ_OP_FOLD_QUANTIZE, 0, cout, cin, fmt) ||
      (reinterpret_cast<uintptr_t>(b.workspace) & 3))
    return SQ_ERR_WORKSPACE;

  const size_t eb = (size_t)elem_bytes(dt);
  if (cudaMemcpyAsync(b.x, x_host, (size_t)tokens * cin * eb, cudaMemcpyHostToDevice, stream) !=
          cudaSuccess ||
      cudaMemcpyAsync(b.w, w_host, (size_t)cin * cout * eb, cudaMemcpyHostToDevice, stream) !=
          cudaSuccess)
    return SQ_ERR_CUDA;
  sq_status r;
  if ((r = sq_calibrate_absmax(b.x, dt, tokens, cin, cin, 0, 0, b.amax_x, stream)) != SQ_OK) return r;
  if ((r = sq_calibrate_absmax(b.w, dt, cin, cout, cout, 1, 0, b.amax_w, stream)) != SQ_OK) return r;
  if ((r = sq_smooth_factors(b.amax_x, b.amax_w, cin, alpha, b.s, b.s_inv, dev_flags, stream)) != SQ_OK)
    return r;
  if ((r = sq_fold_quantize_weight(b.w, dt, cin, cout, cout, b.s, b.wq, fmt, b.w_scale, dev_flags,
                                   b.workspace, b.ws_bytes, stream)) != SQ_OK)
    return r;
  if ((r = sq_quant_act(b.x, dt, tokens, cin, cin, b.s_inv, b.xq, fmt, b.x_scale, dev_flags,
                        stream)) != SQ_OK)
    return r;
  // the fold is done with the workspace (same stream): the GEMM may reuse it
  if ((r = sq_w8a8_gemm(b.xq, b.x_scale, b.wq, b.w_scale, fmt, tokens, cout, cin, b.y, nullptr,
                        dev_flags, b.workspace, b.ws_bytes, stream)) != SQ_OK)
    return r;
  if (cudaMemcpyAsync(y_host, b.y, (size_t)tokens * cout * 2, cudaMemcpyDeviceToHost, stream) !=
      cudaSuccess)
    return SQ_ERR_CUDA;
  return SQ_OK;
}

}  // extern "C"

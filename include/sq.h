/*
 * sq.h - C ABI of the B300 (sm_103a) SmoothQuant W8A8 linear-layer path.
 *
 * The path has five steps; each has one entry point below:
 *
 *   1. sq_calibrate_absmax      per-channel max|.| of X and of W
 *   2. sq_smooth_factors        s_j = max|X_j|^a / max|W_j|^(1-a), and 1/s_j
 *   3. sq_fold_quantize_weight  W' = diag(s) W, per-output-channel INT8 codes
 *   4. sq_quant_act             X' = X diag(s)^-1, per-token INT8 codes
 *   5. sq_w8a8_gemm             exact INT8 x INT8 accumulation, bf16 epilogue
 *
 * sq_linear_host runs all five on inputs in host memory (copies included).
 *
 * Orientation (first source page, "Move activation scale without changing
 * the real linear map", paragraph 1): X is [tokens x Cin] and W is
 * [Cin x Cout], so Y = X W; diag(s) multiplies W on its rows (input
 * channels) and diag(s)^-1 multiplies X on its columns.
 *
 * Conventions for every entry point
 *   - Pointers named dev_* or documented as "device" are CUDA device
 *     pointers; all others are host values.  The caller allocates and owns
 *     every buffer (inputs, outputs, workspace).  The library allocates no
 *     memory and keeps no state between calls.
 *   - All work is enqueued on `stream` and returns before it finishes.
 *     Two calls on different streams may run concurrently if their
 *     buffers do not overlap.
 *   - Argument errors are reported synchronously by the return value and
 *     nothing is enqueued.  A failed launch returns SQ_ERR_CUDA.
 *   - Data-dependent conditions found on the device are OR-ed into the
 *     optional device word `dev_flags` (SQ_FLAG_*), which the caller zeroes
 *     and reads back when it wants them; sq_read_device_flags turns the
 *     word into a status (SQ_ERR_TIMEOUT, SQ_ERR_NONFINITE).  The word is
 *     the caller's, one per stream or per layer as it likes, rather than
 *     an error word inside the library: the library keeps no mutable state,
 *     so concurrent streams and captured graphs never share a status.
 *     Kernels never trap.
 *   - Row-major matrices take a leading dimension `ld` in elements.  The
 *     kernels move 16-byte vectors: code buffers, and X in step 4, must be
 *     16-byte aligned with rows a multiple of 16 bytes.  The inputs of steps
 *     1 and 3 need only element alignment (rows that are not 16-byte
 *     aligned take a slower element-wise path).
 *   - The library targets sm_103a only; on any other device the launches
 *     fail with SQ_ERR_CUDA.
 */
#ifndef SQ_B300_H
#define SQ_B300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SQ_OK = 0,
  SQ_ERR_INVALID_ARG = 1,  /* null pointer, bad size, alignment or enum */
  SQ_ERR_NONFINITE = 2,    /* the device word reports a NaN/Inf statistic or scale */
  SQ_ERR_CUDA = 3,         /* a CUDA runtime/driver call or launch failed */
  SQ_ERR_UNSUPPORTED = 4,  /* valid request the library does not implement */
  SQ_ERR_WORKSPACE = 5,    /* workspace pointer missing or too small */
  SQ_ERR_TIMEOUT = 6       /* the device word reports a bounded wait that ran out */
} sq_status;

/* Bits OR-ed into *dev_flags by the kernels. */
#define SQ_FLAG_NONFINITE 0x1 /* a NaN/Inf statistic or scale was seen */
#define SQ_FLAG_TIMEOUT 0x2   /* a bounded pipeline wait ran out */

/* Element type of the floating-point inputs X and W. */
typedef enum { SQ_F32 = 0, SQ_BF16 = 1 } sq_dtype;

/* Storage of INT8 codes.  SQ_CODES_I8 stores each code as int8_t.
 * SQ_CODES_BF16 stores the same integer (-127..127) as an exact bfloat16
 * value; it is the operand format of the sm_103a tensor-core GEMM, since
 * sm_103a's tcgen05.mma has no integer kind.  Both hold identical codes. */
typedef enum { SQ_CODES_I8 = 0, SQ_CODES_BF16 = 1 } sq_codes;

/* Operation ids for sq_workspace_bytes. */
typedef enum {
  SQ_OP_CALIBRATE = 0,
  SQ_OP_SMOOTH = 1,
  SQ_OP_FOLD_QUANTIZE = 2,
  SQ_OP_QUANT_ACT = 3,
  SQ_OP_GEMM = 4,
  SQ_OP_STATIC_SCALE = 5,
  SQ_OP_QUANT_ACT_STATIC = 6,
  SQ_OP_FOLD_NORM_GAIN = 7,
  SQ_OP_RMSNORM_QUANT_ACT = 8,
  SQ_OP_ROTATE_ACT = 9,
  SQ_OP_ROTATE_WEIGHT = 10
} sq_op;

/*
 * Step 1 - calibration statistics.
 * Source: pith.science review of arXiv 2506.01967 (Smooth Rotation),
 * key_machinery (s_j built from max|X_j| and max|W_j|); SmoothQuant glossary
 * (dataterminology.com), "What calibration data does SmoothQuant need?"
 * (statistics from a small calibration set).
 *
 *   a      device, [rows x cols] row-major, element type dt, leading dim ld
 *   axis   0: amax[c] = max_r |a[r,c]|  (X [tokens x Cin] -> amax[Cin])
 *          1: amax[r] = max_c |a[r,c]|  (W [Cin x Cout] -> amax[Cin])
 *   accumulate  0: overwrite amax; 1: amax = max(amax, new) (running max
 *          over calibration batches, or over several weights that share one
 *          activation, e.g. Q/K/V)
 *   amax   device fp32, cols (axis 0) or rows (axis 1) entries
 * NaN inputs propagate: a NaN anywhere makes that channel's statistic NaN
 * (step 2 then flags it).  The column reduction's waits for its copies are
 * bounded; a wait that runs out also leaves NaN statistics behind, so it
 * too surfaces as SQ_FLAG_NONFINITE in step 2.  rows, cols >= 1.
 */
sq_status sq_calibrate_absmax(const void* a, sq_dtype dt, int64_t rows, int64_t cols,
                              int64_t ld, int axis, int accumulate, float* amax,
                              cudaStream_t stream);

/*
 * Step 2 - smoothing factors and their inverses.
 * Source: Smooth Rotation review, key_machinery (a = 0.5 case,
 * s_j = sqrt(max|X_j| / max|W_j|)); first page, paragraph 1 (factors finite
 * and nonzero).  For strength alpha in [0, 1]:
 *   ax = max(amax_x[j], 1e-5f), aw = max(amax_w[j], 1e-5f)
 *   s[j] = clamp(RN(ax^alpha) / RN(aw^(1-alpha)), 1e-5f, 1e5f)
 *   s_inv[j] = 1 / s[j]
 * Each power is the correctly rounded fp32 value, 1-alpha an fp32
 * subtraction, each quotient one IEEE fp32 division.  A non-finite
 * statistic gives s = s_inv = 1 and sets SQ_FLAG_NONFINITE.
 *   amax_x, amax_w  device fp32 [cin];  s, s_inv  device fp32 [cin]
 *   dev_flags       device int32 or NULL
 * alpha outside [0, 1] or not finite -> SQ_ERR_INVALID_ARG.
 */
sq_status sq_smooth_factors(const float* amax_x, const float* amax_w, int64_t cin,
                            float alpha, float* s, float* s_inv, int32_t* dev_flags,
                            cudaStream_t stream);

/*
 * Step 3 - offline fold of diag(s) into W's rows, then symmetric INT8
 * quantization per output channel.
 * Source: first page, paragraph 1 (S multiplies W); learn-kernels.com
 * "Quantization", paragraph 2 (transform applied offline, both operands
 * INT8).  For output channel n:
 *   W'[j,n] = s[j] * W[j,n]               (fp32 multiply)
 *   w_scale[n] = max_j |W'[j,n]| / 127    (fp32 division; 1 if the max is 0)
 *   wq[n,j] = clamp(rne(W'[j,n] / w_scale[n]), -127, 127)
 * where W'/w_scale is the IEEE fp32 quotient (Smooth Rotation review,
 * core_discovery: symmetric round-to-nearest, i.e. round(v / step)).
 *   w      device [cin x cout] row-major, type dt, leading dim ldw
 *   s      device fp32 [cin]
 *   wq     device [cout x cin] codes, row n contiguous (K-major), format fmt
 *   w_scale device fp32 [cout]
 *   workspace  device, >= sq_workspace_bytes(SQ_OP_FOLD_QUANTIZE, 0, cout, cin, fmt)
 * A non-finite column maximum sets SQ_FLAG_NONFINITE.
 */
sq_status sq_fold_quantize_weight(const void* w, sq_dtype dt, int64_t cin, int64_t cout,
                                  int64_t ldw, const float* s, void* wq, sq_codes fmt,
                                  float* w_scale, int32_t* dev_flags, void* workspace,
                                  size_t ws_bytes, cudaStream_t stream);

/*
 * Step 3 without a caller-provided workspace.  The source pages have no
 * counterpart; this is a deployment convenience.  Some callers cannot hand
 * the library device scratch memory: code running inside another engine's
 * execution callback that receives only a stream and its tensors, or a host
 * that reserved its whole device-memory budget up front, must not call
 * cudaMalloc (it can fail for lack of memory or stall every stream on the
 * device).  This entry point computes exactly what sq_fold_quantize_weight
 * computes, with the same arguments minus the workspace, and allocates
 * nothing: its scratch (one 32-bit maximum per output channel) is a fixed
 * array of SQ_NOALLOC_MAX_COUT entries (256 KiB) in the library's device
 * memory, which every GPU that loads the library holds until exit.
 *   - cout > SQ_NOALLOC_MAX_COUT -> SQ_ERR_WORKSPACE (nothing enqueued).
 *   - Each call looks up the array's device address on the current device
 *     (so a device reset, which moves the array, is harmless); a call made
 *     during stream capture reuses the address the last call on that
 *     device found, so make the first call on each device before any
 *     stream capture.
 *   - All calls share the one array: calls whose work overlaps on the GPU
 *     (e.g. on two streams) race and give wrong results.  Each call clears
 *     the entries it uses before using them.
 */
#define SQ_NOALLOC_MAX_COUT 65536
sq_status sq_fold_quantize_weight_noalloc(const void* w, sq_dtype dt, int64_t cin, int64_t cout,
                                          int64_t ldw, const float* s, void* wq, sq_codes fmt,
                                          float* w_scale, int32_t* dev_flags,
                                          cudaStream_t stream);

/*
 * Step 4 - runtime X diag(s)^-1 fused with dynamic per-token INT8
 * quantization (one read of X, one write of the codes).
 * Source: first page, paragraph 3 (the explicit runtime scaling step);
 * learn-kernels.com "Quantization", paragraph 2 (activations to INT8).
 * For token t:
 *   X'[t,j] = X[t,j] * s_inv[j]           (fp32 multiply)
 *   x_scale[t] = max_j |X'[t,j]| / 127    (fp32 division; 1 if the max is 0)
 *   xq[t,j] = clamp(rne(X'[t,j] / x_scale[t]), -127, 127)   (fp32 quotient)
 *   x      device [tokens x cin] row-major, type dt, leading dim ldx
 *   s_inv  device fp32 [cin] (from step 2)
 *   xq     device [tokens x cin] codes, row-major, format fmt
 *   x_scale device fp32 [tokens]
 * A non-finite token maximum sets SQ_FLAG_NONFINITE (its codes are then
 * unspecified).
 */
sq_status sq_quant_act(const void* x, sq_dtype dt, int64_t tokens, int64_t cin, int64_t ldx,
                       const float* s_inv, void* xq, sq_codes fmt, float* x_scale,
                       int32_t* dev_flags, cudaStream_t stream);

/*
 * Step 4, static variant - one calibrated activation scale per tensor.
 * Source: SmoothQuant glossary (dataterminology.com): calibration-based,
 * statistics from a small calibration set; first page, paragraph 3 (the
 * runtime multiply by S^-1).  Two calls:
 *
 * sq_static_act_scale: from the calibration statistics of step 1 (amax_x,
 * a running maximum over the calibration batches) and s_inv of step 2,
 *   d = RN(max_j RN(amax_x[j] * s_inv[j]) / 127)   (1 if the maximum is 0)
 * which is max|X'| / 127 over the calibration data (a binary32 multiply by
 * a fixed positive factor is monotone in |x|).
 *   amax_x, s_inv  device fp32 [cin];  d  device fp32 [1]
 *   dev_flags      device int32 or NULL (SQ_FLAG_NONFINITE)
 *
 * sq_quant_act_static: X' = X * s_inv, codes with the one scale d:
 *   xq[t,j] = clamp(rne(X'[t,j] / d), -127, 127);  x_scale[t] = d
 * (x_scale is filled so that sq_w8a8_gemm's epilogue is unchanged).  Values
 * beyond the calibration maximum saturate; `clipped` (device uint32 or
 * NULL) has the number of elements the clamp changed ADDED to it.  A NaN in
 * X' gives code 0 and +-inf saturates; both raise SQ_FLAG_NONFINITE.  A
 * single streaming pass with no per-token reduction.  Layout and
 * alignment as sq_quant_act; d is read on the device.
 */
sq_status sq_static_act_scale(const float* amax_x, const float* s_inv, int64_t cin, float* d,
                              int32_t* dev_flags, cudaStream_t stream);
sq_status sq_quant_act_static(const void* x, sq_dtype dt, int64_t tokens, int64_t cin, int64_t ldx,
                              const float* s_inv, const float* d, void* xq, sq_codes fmt,
                              float* x_scale, uint32_t* clipped, int32_t* dev_flags,
                              cudaStream_t stream);

/*
 * Step 4 folded into the preceding RMS normalization.
 * Source: first page, paragraph 3: to avoid an extra runtime scaling kernel
 * the inverse factors may be folded into the preceding operation when every
 * consumer keeps its compensation (one s for all consumers of the
 * normalized activation, e.g. Q/K/V).  Reading: the preceding operation is
 * an RMS normalization with a per-channel gain gamma (LLaMA-style layers).
 *
 * sq_fold_norm_gain (offline): gamma_folded[j] = RN(gamma[j] * s_inv[j]).
 *   gamma, s_inv, gamma_folded  device fp32 [cin]
 *
 * sq_rmsnorm_quant_act (runtime, one kernel): for token t of the
 * normalization's input h [tokens x cin],
 *   S_t = the exact sum_j h[t,j]^2, rounded once to binary32 (parts of
 *         squares below 2^-108 of the largest square among the (at most
 *         32) values one thread sums enter only as a sticky bit, so only a
 *         row built to lie within 2^-98 of a binary32 midpoint through
 *         several such parts can round the other way)
 *   r_t = RN(1 / RN(sqrt(RN(RN(S_t / cin) + eps))))   (IEEE binary32 steps)
 *   X'[t,j] = RN(RN(h[t,j] * r_t) * gamma_folded[j])
 * followed by the dynamic per-token quantizer of sq_quant_act (same codes,
 * x_scale, layouts, alignment and limits; h takes the place of x).  A
 * non-finite row gives a non-finite scale and SQ_FLAG_NONFINITE.
 */
sq_status sq_fold_norm_gain(const float* gamma, const float* s_inv, int64_t cin,
                            float* gamma_folded, cudaStream_t stream);
sq_status sq_rmsnorm_quant_act(const void* h, sq_dtype dt, int64_t tokens, int64_t cin,
                               int64_t ldh, const float* gamma_folded, float eps, void* xq,
                               sq_codes fmt, float* x_scale, int32_t* dev_flags,
                               cudaStream_t stream);

/*
 * Smooth Rotation (smoothing, then a Hadamard rotation, low-bit codes).
 * Source: pith.science review of arXiv 2506.01967 ("Smooth Rotation"),
 * key_machinery: X S^-1 R and R^T S W with the same Hadamard matrix R
 * (entries +-1/sqrt(d)), which leaves Y = X W unchanged; core_discovery:
 * symmetric round-to-nearest 4-bit codes on both operands (W4A4).
 *
 * R = H / sqrt(d) with H the Sylvester Hadamard matrix of order d = cin (a
 * power of two).  Z = (X S^-1) H is formed by the fast Walsh-Hadamard
 * transform, stages h = 1, 2, 4, ... in that order, each butterfly
 * (a, b) -> (a + b, a - b) one binary32 addition and subtraction.  Codes
 * clamp(rne(Z / dz), -qmax, qmax) with dz = RN(max|Z| / qmax) per row
 * (1 if the maximum is 0); qmax = 7 gives 4-bit codes, 127 the 8-bit ones.
 * The 1/d of R R^T = H H^T / d is carried by the activation scale as the
 * exact factor 2^-log2(d): x_scale = dz * 2^-log2(d), w_scale = dz, so
 * sq_w8a8_gemm reproduces the layer with its usual epilogue.
 *
 * sq_rotate_quant_act: x [tokens x cin] (ldx), s_inv device fp32 [cin] or
 *   NULL (no smoothing), rotate 0/1 (0: plain per-token codes with qmax);
 *   xq [tokens x cin] codes, x_scale device fp32 [tokens].
 * sq_rotate_fold_quantize_weight: w [cin x cout] (ldw), s device fp32 [cin]
 *   or NULL; wq [cout x cin] codes (K-major), w_scale device fp32 [cout];
 *   workspace >= sq_workspace_bytes(SQ_OP_ROTATE_WEIGHT, 0, cout, cin, fmt)
 *   (the folded weight, transposed, in fp32).
 * Both: 1 <= qmax <= 127; with rotate = 1, cin a power of two with
 * 256 <= cin <= 32768 (bf16) or 128 <= cin <= 16384 (fp32), else
 * SQ_ERR_UNSUPPORTED; alignment as sq_quant_act.  A non-finite row maximum
 * sets SQ_FLAG_NONFINITE.
 */
sq_status sq_rotate_quant_act(const void* x, sq_dtype dt, int64_t tokens, int64_t cin, int64_t ldx,
                              const float* s_inv, int rotate, int qmax, void* xq, sq_codes fmt,
                              float* x_scale, int32_t* dev_flags, cudaStream_t stream);
sq_status sq_rotate_fold_quantize_weight(const void* w, sq_dtype dt, int64_t cin, int64_t cout,
                                         int64_t ldw, const float* s, int rotate, int qmax,
                                         void* wq, sq_codes fmt, float* w_scale,
                                         int32_t* dev_flags, void* workspace, size_t ws_bytes,
                                         cudaStream_t stream);

/*
 * Step 5 - INT8 x INT8 GEMM with exact integer accumulation and a bf16
 * dequantizing epilogue.
 * Source: learn-kernels.com "Quantization", paragraph 2 (the matmul runs on
 * INT8 weights and activations on low-precision hardware paths).
 *   acc[t,n] = sum_j xq[t,j] * wq[n,j]    (exact, |acc| < 2^31)
 *   y[t,n]   = bf16(acc[t,n] * x_scale[t] * w_scale[n])  (fp32 epilogue;
 *              within 1 bf16 ulp of the exactly rounded value)
 *   xq     device [m x k] codes, format fmt (row-major, K contiguous)
 *   wq     device [n x k] codes, format fmt (K contiguous)
 *   y      device bf16 [m x n] row-major
 *   acc_out  device int32 [m x n] or NULL: the exact accumulators
 *   workspace  device, 16-byte aligned; sq_workspace_bytes(SQ_OP_GEMM, m, n,
 *              k, fmt) bytes (0 for SQ_CODES_BF16 and for m <= 64;
 *              (m + n) * k * 2 rounded up to 256 for SQ_CODES_I8 with
 *              m > 64).  A smaller or NULL workspace is not an error: the
 *              call then takes the path that needs none (below).
 * k must be a multiple of 16 and at most SQ_GEMM_MAX_K (beyond it a sum of
 * k products of 127 * 127 could leave int32: SQ_ERR_UNSUPPORTED).
 * SQ_CODES_BF16 runs on the tcgen05 tensor
 * cores (fp32 accumulation in TMEM, converted to int32 every <= 1024
 * products so every partial sum stays an exact integer).  SQ_CODES_I8 reads
 * one byte per code: m <= 16 runs the weight-streaming decode kernel
 * (codes widened to fp16 on chip, mma.sync), 16 < m <= 64 the integer
 * mma.sync kernel, m > 64 the tcgen05 tensor cores: with the workspace, one
 * pass widens both operands' codes to exact fp16 values in it and the
 * 16-bit-carrier kernel multiplies them (two kernels); without it, one
 * kernel widens the codes in shared memory as it goes (slower: the
 * shared-memory banks carry the widening).  Every path accumulates exactly.
 * A pipeline wait that runs out sets SQ_FLAG_TIMEOUT.
 */
#define SQ_GEMM_MAX_K 133136 /* largest multiple of 16 with k * 127^2 < 2^31 */
sq_status sq_w8a8_gemm(const void* xq, const float* x_scale, const void* wq,
                       const float* w_scale, sq_codes fmt, int64_t m, int64_t n, int64_t k,
                       void* y, int32_t* acc_out, int32_t* dev_flags, void* workspace,
                       size_t ws_bytes, cudaStream_t stream);

/*
 * Diagnostics - the second half of the validation order.
 * Source: first page, paragraph 4 (after the unquantized rewrite, quantize
 * and measure activation clipping and weight reconstruction separately);
 * Smooth Rotation review, referee report (layer-wise squared Frobenius
 * quantization error; "quantization difficulty" = standard deviation of
 * channel magnitudes).  Differences x - code * scale are exact in float64;
 * squares and sums are rounded in float64 (order-dependent in the last
 * bits).  None of these is on the timed path.
 *
 * sq_act_quant_error: err[t] = sum_j (RN(X[t,j] * s_inv[j]) - xq[t,j] * x_scale[t])^2
 *   x, s_inv, xq, x_scale as sq_quant_act (same layouts and alignment);
 *   err device double [tokens].
 * sq_weight_quant_error: err[n] = sum_j (RN(s[j] * W[j,n]) - wq[n,j] * w_scale[n])^2
 *   w, s, wq, w_scale as sq_fold_quantize_weight (any row alignment);
 *   err device double [cout].
 * sq_layer_error: for the sampled tokens rows[0..nrows),
 *   err[r] = sum_n ((X W)[rows[r], n] - y[rows[r], n])^2
 *   with X W formed from the unquantized inputs (fp32 chunks of 32 products
 *   summed in float64; relative error ~1e-6 of |X W|).  x [tokens x cin]
 *   (ldx), w [cin x cout] (ldw), both of type dt; y bf16 [tokens x cout]
 *   contiguous; rows device int32 [nrows], 1 <= nrows <= 64; err device
 *   double [nrows] (overwritten).  A sampled index outside [0, tokens) is
 *   never dereferenced: its err entry is NaN.
 * sq_channel_stats: out[0] = mean, out[1] = population standard deviation
 *   of v_j = RN(amax[j] * scale[j]) (scale NULL: v_j = amax[j]); with
 *   amax = max|X_j| and scale = s_inv, the channel magnitudes after
 *   smoothing.  out device double [2].
 */
sq_status sq_act_quant_error(const void* x, sq_dtype dt, int64_t tokens, int64_t cin, int64_t ldx,
                             const float* s_inv, const void* xq, sq_codes fmt, const float* x_scale,
                             double* err, cudaStream_t stream);
sq_status sq_weight_quant_error(const void* w, sq_dtype dt, int64_t cin, int64_t cout, int64_t ldw,
                                const float* s, const void* wq, sq_codes fmt, const float* w_scale,
                                double* err, cudaStream_t stream);
sq_status sq_layer_error(const void* x, const void* w, sq_dtype dt, int64_t tokens, int64_t cin,
                         int64_t cout, int64_t ldx, int64_t ldw, const void* y,
                         const int32_t* rows, int nrows, double* err, cudaStream_t stream);
sq_status sq_channel_stats(const float* amax, const float* scale, int64_t n, double* out,
                           cudaStream_t stream);

/*
 * The whole path on host-resident inputs, one call per layer.  No source
 * page defines this call; it is the end-to-end form of steps 1-5 above for
 * callers whose X and W live in host memory.  Enqueued on `stream`, in this
 * order: copy X and W from host to the caller's device buffers; step 1 on X
 * (axis 0) and on W (axis 1); step 2 with strength alpha; step 3; step 4
 * (dynamic per-token scale); step 5 without the accumulators; copy Y back
 * to host memory.  Every intermediate stays in `dev` for the caller.
 *   x_host  host [tokens x cin], type dt, contiguous
 *   w_host  host [cin x cout], type dt, contiguous
 *   y_host  host bf16 [tokens x cout], contiguous
 *   dev     host pointer to the caller's device buffers (layouts and formats
 *           as in steps 1-5, all contiguous): x, w as above; amax_x,
 *           amax_w, s, s_inv fp32 [cin]; wq [cout x cin] and xq
 *           [tokens x cin] codes in format fmt; w_scale fp32 [cout];
 *           x_scale fp32 [tokens]; y bf16 [tokens x cout]; workspace of at
 *           least sq_workspace_bytes(SQ_OP_FOLD_QUANTIZE, 0, cout, cin, fmt)
 *           (steps 3 and 5 use it in turn: with sq_workspace_bytes(SQ_OP_GEMM,
 *           tokens, cout, cin, fmt) bytes as well, step 5 takes its widening
 *           path for 1-byte codes)
 *   dev_flags  device int32 or NULL, as in the steps
 * The copies are asynchronous only from page-locked host memory
 * (cudaHostAlloc or cudaHostRegister); from pageable memory CUDA stages them
 * and the call may block.  The host buffers must stay valid, and y_host
 * unread, until `stream` has finished the call's work.  All arguments are
 * checked before anything is enqueued (cin a multiple of 16, x, xq and wq
 * 16-byte aligned, every other buffer 4-byte aligned, cin within step 4's
 * limit); a failing copy or launch returns SQ_ERR_CUDA with the earlier
 * work of the call already enqueued.
 */
typedef struct {
  void* x;
  void* w;
  float* amax_x;
  float* amax_w;
  float* s;
  float* s_inv;
  void* wq;
  float* w_scale;
  void* xq;
  float* x_scale;
  void* y;
  void* workspace;
  size_t ws_bytes;
} sq_linear_buffers;

sq_status sq_linear_host(const void* x_host, const void* w_host, sq_dtype dt, int64_t tokens,
                         int64_t cin, int64_t cout, float alpha, sq_codes fmt, void* y_host,
                         const sq_linear_buffers* dev, int32_t* dev_flags, cudaStream_t stream);

/* Workspace bytes an operation needs for these sizes (0 if none). */
size_t sq_workspace_bytes(sq_op op, int64_t m, int64_t n, int64_t k, sq_codes fmt);

/*
 * Number of kernels one call of `op` enqueues for these sizes, assuming
 * every pointer is 16-byte aligned and every workspace has the size
 * sq_workspace_bytes asks for: `ld` is the leading dimension (in elements,
 * type dt) of the call's input matrix; `axis` and `accumulate` are
 * SQ_OP_CALIBRATE's, except that for SQ_OP_GEMM `axis` carries the code
 * format (sq_codes).  Sizes follow each entry point's own
 * names: calibrate (m = rows, n = cols), smooth (k = cin), fold
 * (k = cin, n = cout), quant_act (m = tokens, k = cin), GEMM (m, n, k).
 * For budgeting launches (e.g. in a CUDA graph) and reading a profiler's
 * launch list.  -1 for an unknown op.
 */
int sq_kernel_count(sq_op op, sq_dtype dt, int64_t m, int64_t n, int64_t k, int64_t ld, int axis,
                    int accumulate);

/*
 * Read (and optionally clear) a device flag word and turn it into a status.
 * Source: none on the pages; it is the boundary's status convention for the
 * data-dependent conditions above.  Enqueues a 4-byte device-to-host copy of
 * *dev_flags on `stream` (after the work already there), then, with clear =
 * 1, zeroes the word, and waits for the stream: a synchronizing call, not
 * for use inside stream capture.  Returns SQ_ERR_TIMEOUT if
 * SQ_FLAG_TIMEOUT is set, else SQ_ERR_NONFINITE if SQ_FLAG_NONFINITE is
 * set, else SQ_OK; flags_out (host, or NULL) receives the raw word.
 *   dev_flags  device int32, 4-byte aligned;  clear  0 or 1
 */
sq_status sq_read_device_flags(int32_t* dev_flags, int clear, int32_t* flags_out,
                               cudaStream_t stream);

/*
 * Test hooks for the bounded waits.  No source page has a counterpart: they
 * let a test drive the abort path of the kernels' pipelines on a GPU without
 * faulting it.  Each call enqueues the same kernel as its product entry
 * point, with its copy producer stalled (it issues no copies), so the first
 * wait for a copy (or for work that depends on one) runs out after wait_ns
 * nanoseconds; the kernel then sets SQ_FLAG_TIMEOUT in *dev_flags, stops,
 * releases what it holds (tensor memory, barriers) and returns, leaving the
 * device usable for the next call.  Outputs are unspecified.
 *   sq_test_w8a8_gemm_stalled: the kernel sq_w8a8_gemm would run for these
 *     arguments (SQ_ERR_UNSUPPORTED for the one GEMM kernel without pipeline
 *     waits: 1-byte codes with 17 to 64 tokens).
 *   sq_test_w8a8_gemm_stalled_ws: the same with a workspace, so 1-byte codes
 *     above 64 tokens take the widening path; its widening pass and its
 *     GEMM both run stalled.
 *   sq_test_quant_act_stalled: the kernel of sq_quant_act.
 * dev_flags is required; 1e5 <= wait_ns <= 1e9 (else SQ_ERR_INVALID_ARG).
 * Other arguments as the product entry points.
 */
sq_status sq_test_w8a8_gemm_stalled(const void* xq, const float* x_scale, const void* wq,
                                    const float* w_scale, sq_codes fmt, int64_t m, int64_t n,
                                    int64_t k, void* y, int32_t* dev_flags, uint64_t wait_ns,
                                    cudaStream_t stream);
sq_status sq_test_w8a8_gemm_stalled_ws(const void* xq, const float* x_scale, const void* wq,
                                       const float* w_scale, sq_codes fmt, int64_t m, int64_t n,
                                       int64_t k, void* y, int32_t* dev_flags, void* workspace,
                                       size_t ws_bytes, uint64_t wait_ns, cudaStream_t stream);
sq_status sq_test_quant_act_stalled(const void* x, sq_dtype dt, int64_t tokens, int64_t cin,
                                    int64_t ldx, const float* s_inv, void* xq, sq_codes fmt,
                                    float* x_scale, int32_t* dev_flags, uint64_t wait_ns,
                                    cudaStream_t stream);

/* Static text for a status code. */
const char* sq_status_string(sq_status status);

/* SQ_OK if `device` is an sm_103 GPU this library can run on, else
 * SQ_ERR_UNSUPPORTED (or SQ_ERR_CUDA if the query fails). */
sq_status sq_check_device(int device);

#ifdef __cplusplus
}
#endif

#endif /* SQ_B300_H */

// Step 4, static variant: one calibrated activation scale per tensor.
//
// Source: SmoothQuant glossary (dataterminology.com): the method is
// calibration-based, with statistics from a small calibration set; first
// page ("Move activation scale without changing the real linear map"),
// paragraph 3: the runtime step multiplies activations by S^-1.
//
// k_static_scale reduces d = max_j RN(amax_x[j] * s_inv[j]) / 127 on one
// block (a binary32 multiply by a fixed positive factor is monotone in |x|,
// so this is the largest |X'| the calibration data produced).  The
// quantization with that one scale runs in the activation kernel (act.cu)
// in its static mode.
#include "sq_async.cuh"

namespace sq {
namespace {
using namespace async;

__global__ void __launch_bounds__(1024) k_static_scale(const float* __restrict__ amax_x,
                                                       const float* __restrict__ s_inv,
                                                       int64_t cin, float* __restrict__ d_out,
                                                       int32_t* flags) {
  __shared__ uint32_t red[32];
  uint32_t m = 0u;
  for (int64_t j = threadIdx.x; j < cin; j += blockDim.x) {
    const float v = __fmul_rn(amax_x[j], s_inv[j]);
    m = max(m, __float_as_uint(v) & 0x7FFFFFFFu);  // NaN sorts above +inf
  }
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    uint32_t v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0u;
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    if (threadIdx.x == 0) {
      float d, inv;
      scale_and_inverse(__uint_as_float(v), d, inv);
      *d_out = d;
      if (!finite_bits(v)) raise_flag(flags, SQ_FLAG_NONFINITE);
    }
  }
}

}  // namespace

sq_status static_act_scale(const float* amax_x, const float* s_inv, int64_t cin, float* d,
                           int32_t* flags, cudaStream_t st) {
  k_static_scale<<<1, 1024, 0, st>>>(amax_x, s_inv, cin, d, flags);
  return launch_status();
}

}  // namespace sq

// Quantization diagnostics: the second half of the pages' validation order.
//
// Sources: first page ("Move activation scale without changing the real
// linear map"), paragraph 4: once the unquantized rewrite checks out,
// quantize and measure activation clipping and weight reconstruction
// separately; pith.science review of arXiv 2506.01967 (Smooth Rotation),
// referee report: the layer-wise squared Frobenius quantization error and
// the "quantization difficulty" (standard deviation of channel magnitudes).
//
// Each difference x - code * scale is exact in float64 (a 24-bit value
// minus a 7-bit code times a 24-bit scale, within half a step of each
// other); squares and sums are rounded in float64.  The layer error forms
// X W from the unquantized inputs in fp32 chunks of 32 products (exact
// products for bf16 inputs) summed in float64.
#include <cuda_bf16.h>

#include "sq_common.cuh"

namespace sq {
namespace {

template <bool BF16>
SQ_DEVINL void unpack16(uint4 v, float* f) {
  if constexpr (BF16) {
    f[0] = bf16lo_to_f32(v.x);
    f[1] = bf16hi_to_f32(v.x);
    f[2] = bf16lo_to_f32(v.y);
    f[3] = bf16hi_to_f32(v.y);
    f[4] = bf16lo_to_f32(v.z);
    f[5] = bf16hi_to_f32(v.z);
    f[6] = bf16lo_to_f32(v.w);
    f[7] = bf16hi_to_f32(v.w);
  } else {
    f[0] = __uint_as_float(v.x);
    f[1] = __uint_as_float(v.y);
    f[2] = __uint_as_float(v.z);
    f[3] = __uint_as_float(v.w);
  }
}

// Code number e of a group starting at byte p (int8 or bf16 storage).
template <int CODES>
SQ_DEVINL double code_at(const uint8_t* p, int e) {
  if constexpr (CODES == SQ_CODES_BF16)
    return (double)__uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(p)[e] << 16);
  else
    return (double)reinterpret_cast<const int8_t*>(p)[e];
}

SQ_DEVINL double warp_sum(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// err[t] = sum_j (RN(X[t,j] * s_inv[j]) - xq[t,j] * x_scale[t])^2; one warp per token.
template <bool BF16, int CODES>
__global__ void __launch_bounds__(256) k_act_error(const uint8_t* __restrict__ x, int64_t tokens,
                                                   int64_t cin, int64_t ldx_bytes,
                                                   const float* __restrict__ s_inv,
                                                   const uint8_t* __restrict__ xq,
                                                   const float* __restrict__ x_scale,
                                                   double* __restrict__ err) {
  constexpr int E = BF16 ? 8 : 4;
  constexpr int CB = CODES == SQ_CODES_BF16 ? 2 : 1;
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= tokens) return;
  const double d = (double)x_scale[t];
  const uint8_t* row = x + t * ldx_bytes;
  const uint8_t* qrow = xq + t * cin * CB;
  double acc = 0.0;
  for (int64_t v = lane; v * E < cin; v += 32) {
    float f[E];
    unpack16<BF16>(ld_stream16(row + v * 16), f);
#pragma unroll
    for (int e = 0; e < E; ++e) {
      const float xs = __fmul_rn(f[e], s_inv[v * E + e]);
      const double diff = fma(-code_at<CODES>(qrow + v * E * CB, e), d, (double)xs);  // exact
      acc = fma(diff, diff, acc);
    }
  }
  acc = warp_sum(acc);
  if (lane == 0) err[t] = acc;
}

// err[n] = sum_j (RN(s_j * W[j,n]) - wq[n,j] * w_scale[n])^2.  A block owns
// 64 output channels and walks Cin in 64-row tiles of W (row-major) and of
// the codes (output-channel-major), both staged in shared memory.
constexpr int kT = 64;

template <bool BF16, int CODES>
__global__ void __launch_bounds__(256) k_weight_error(const uint8_t* __restrict__ w, int64_t cin,
                                                      int64_t cout, int64_t ldw_bytes,
                                                      const float* __restrict__ s,
                                                      const uint8_t* __restrict__ wq,
                                                      const float* __restrict__ w_scale,
                                                      double* __restrict__ err) {
  constexpr int EB = BF16 ? 2 : 4;
  constexpr int CB = CODES == SQ_CODES_BF16 ? 2 : 1;
  __shared__ float ws[kT][kT + 1];     // W'[j][n] of the tile (fp32, after the fold)
  __shared__ float codes[kT][kT + 1];  // code[n][j] (an exact integer)
  __shared__ double part[4][kT];
  const int tid = threadIdx.x;
  const int64_t n0 = (int64_t)blockIdx.x * kT;
  const int nl = tid & (kT - 1), jg = tid >> 6;  // channel, group of 16 rows
  const double dn = n0 + nl < cout ? (double)w_scale[n0 + nl] : 0.0;
  double acc = 0.0;
  for (int64_t j0 = 0; j0 < cin; j0 += kT) {
    // W tile: 64 rows x 64 channels, element loads (rows of any alignment)
    for (int i = tid; i < kT * kT; i += 256) {
      const int jl = i / kT, c = i % kT;
      const int64_t j = j0 + jl, n = n0 + c;
      float v = 0.0f;
      if (j < cin && n < cout) {
        const uint8_t* p = w + j * ldw_bytes + n * EB;
        const float raw = BF16 ? __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t*>(p) << 16)
                               : *reinterpret_cast<const float*>(p);
        v = __fmul_rn(s[j], raw);
      }
      ws[jl][c] = v;
    }
    // code tile: 64 channels x 64 rows
    for (int i = tid; i < kT * kT; i += 256) {
      const int c = i / kT, jl = i % kT;
      const int64_t j = j0 + jl, n = n0 + c;
      codes[c][jl] = (j < cin && n < cout) ? (float)code_at<CODES>(wq + (n * cin + j) * CB, 0) : 0.0f;
    }
    __syncthreads();
#pragma unroll 4
    for (int k = 0; k < 16; ++k) {
      const int jl = jg * 16 + k;
      const double diff = fma(-(double)codes[nl][jl], dn, (double)ws[jl][nl]);  // exact
      acc = fma(diff, diff, acc);
    }
    __syncthreads();
  }
  part[jg][nl] = acc;
  __syncthreads();
  if (tid < kT && n0 + tid < cout)
    err[n0 + tid] = ((part[0][tid] + part[1][tid]) + part[2][tid]) + part[3][tid];
}

// err[r] += sum over this block's 64 channels of ((X W)[rows[r], n] - Y[rows[r], n])^2.
constexpr int kMaxRows = 64;
constexpr int kJ = 32;

template <bool BF16>
__global__ void __launch_bounds__(256) k_layer_error(const uint8_t* __restrict__ x,
                                                     const uint8_t* __restrict__ w, int64_t cin,
                                                     int64_t cout, int64_t ldx_bytes,
                                                     int64_t ldw_bytes,
                                                     const __nv_bfloat16* __restrict__ y,
                                                     const int32_t* __restrict__ rows, int nrows,
                                                     int64_t tokens, double* __restrict__ err) {
  constexpr int EB = BF16 ? 2 : 4;
  __shared__ float xs[kMaxRows][kJ + 1];
  __shared__ float wsm[kJ][kT + 1];
  __shared__ double red[kMaxRows][kT / 32];
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t n0 = (int64_t)blockIdx.x * kT;
  const int nl = tid & (kT - 1), rg = tid >> 6;  // channel, group of 16 sampled rows
  double acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.0;
  auto load = [](const uint8_t* p) {
    return BF16 ? __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t*>(p) << 16)
                : *reinterpret_cast<const float*>(p);
  };
  for (int64_t j0 = 0; j0 < cin; j0 += kJ) {
    for (int i = tid; i < kMaxRows * kJ; i += 256) {
      const int r = i / kJ, jl = i % kJ;
      const int64_t j = j0 + jl;
      // a sampled index outside [0, tokens) is never dereferenced
      const bool ok = r < nrows && j < cin && rows[r] >= 0 && rows[r] < tokens;
      xs[r][jl] = ok ? load(x + (int64_t)rows[r] * ldx_bytes + j * EB) : 0.0f;
    }
    for (int i = tid; i < kJ * kT; i += 256) {
      const int jl = i / kT, c = i % kT;
      const int64_t j = j0 + jl, n = n0 + c;
      wsm[jl][c] = (j < cin && n < cout) ? load(w + j * ldw_bytes + n * EB) : 0.0f;
    }
    __syncthreads();
    float part[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) part[i] = 0.0f;
#pragma unroll 8
    for (int jl = 0; jl < kJ; ++jl) {
      const float wv = wsm[jl][nl];
#pragma unroll
      for (int i = 0; i < 16; ++i) part[i] = fmaf(xs[rg * 16 + i][jl], wv, part[i]);
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] += (double)part[i];
    __syncthreads();
  }
  const int64_t n = n0 + nl;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const int r = rg * 16 + i;
    double sq = 0.0;
    if (r < nrows && n < cout && rows[r] >= 0 && rows[r] < tokens) {
      const double diff = acc[i] - (double)__bfloat162float(y[(int64_t)rows[r] * cout + n]);
      sq = diff * diff;
    }
    sq = warp_sum(sq);
    if (lane == 0) red[r][(tid >> 5) & 1] = sq;
  }
  __syncthreads();
  if (tid < nrows) {
    if (rows[tid] >= 0 && rows[tid] < tokens)
      atomicAdd(&err[tid], red[tid][0] + red[tid][1]);
    else
      err[tid] = __longlong_as_double(0x7FF8000000000000ll);  // NaN: no such token
  }
}

// out = (mean, population std) of v_j = RN(amax[j] * scale[j]) (scale may be null).
__global__ void __launch_bounds__(1024) k_channel_stats(const float* __restrict__ amax,
                                                        const float* __restrict__ scale, int64_t n,
                                                        double* __restrict__ out) {
  __shared__ double red[32];
  __shared__ double mean_sh;
  auto value = [&](int64_t j) {
    return (double)(scale ? __fmul_rn(amax[j], scale[j]) : amax[j]);
  };
  auto block_sum = [&](double v) {
    v = warp_sum(v);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    double t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0;
    if (threadIdx.x < 32) t = warp_sum(t);
    __syncthreads();
    return t;  // valid in thread 0
  };
  double s = 0.0;
  for (int64_t j = threadIdx.x; j < n; j += blockDim.x) s += value(j);
  s = block_sum(s);
  if (threadIdx.x == 0) mean_sh = s / (double)n;
  __syncthreads();
  const double mean = mean_sh;
  double q = 0.0;
  for (int64_t j = threadIdx.x; j < n; j += blockDim.x) {
    const double dv = value(j) - mean;
    q = fma(dv, dv, q);
  }
  q = block_sum(q);
  if (threadIdx.x == 0) {
    out[0] = mean;
    out[1] = sqrt(q / (double)n);
  }
}

}  // namespace

sq_status act_quant_error(const void* x, sq_dtype dt, int64_t tokens, int64_t cin, int64_t ldx,
                          const float* s_inv, const void* xq, sq_codes fmt, const float* x_scale,
                          double* err, cudaStream_t st) {
  const uint8_t* xb = static_cast<const uint8_t*>(x);
  const uint8_t* qb = static_cast<const uint8_t*>(xq);
  const int64_t ldb = ldx * elem_bytes(dt);
  const unsigned grid = (unsigned)((tokens + 7) / 8);
#define SQ_AE(B, C) k_act_error<B, C><<<grid, 256, 0, st>>>(xb, tokens, cin, ldb, s_inv, qb, x_scale, err)
  if (dt == SQ_BF16) {
    if (fmt == SQ_CODES_BF16) SQ_AE(true, SQ_CODES_BF16); else SQ_AE(true, SQ_CODES_I8);
  } else {
    if (fmt == SQ_CODES_BF16) SQ_AE(false, SQ_CODES_BF16); else SQ_AE(false, SQ_CODES_I8);
  }
#undef SQ_AE
  return launch_status();
}

sq_status weight_quant_error(const void* w, sq_dtype dt, int64_t cin, int64_t cout, int64_t ldw,
                             const float* s, const void* wq, sq_codes fmt, const float* w_scale,
                             double* err, cudaStream_t st) {
  const uint8_t* wb = static_cast<const uint8_t*>(w);
  const uint8_t* qb = static_cast<const uint8_t*>(wq);
  const int64_t ldb = ldw * elem_bytes(dt);
  const unsigned grid = (unsigned)((cout + kT - 1) / kT);
#define SQ_WE(B, C) k_weight_error<B, C><<<grid, 256, 0, st>>>(wb, cin, cout, ldb, s, qb, w_scale, err)
  if (dt == SQ_BF16) {
    if (fmt == SQ_CODES_BF16) SQ_WE(true, SQ_CODES_BF16); else SQ_WE(true, SQ_CODES_I8);
  } else {
    if (fmt == SQ_CODES_BF16) SQ_WE(false, SQ_CODES_BF16); else SQ_WE(false, SQ_CODES_I8);
  }
#undef SQ_WE
  return launch_status();
}

int layer_error_max_rows() { return kMaxRows; }

sq_status layer_error(const void* x, const void* w, sq_dtype dt, int64_t tokens, int64_t cin,
                      int64_t cout, int64_t ldx, int64_t ldw, const void* y, const int32_t* rows,
                      int nrows, double* err, cudaStream_t st) {
  if (cudaMemsetAsync(err, 0, sizeof(double) * nrows, st) != cudaSuccess) return SQ_ERR_CUDA;
  const unsigned grid = (unsigned)((cout + kT - 1) / kT);
  const int eb = elem_bytes(dt);
  const uint8_t* xb = static_cast<const uint8_t*>(x);
  const uint8_t* wb = static_cast<const uint8_t*>(w);
  const __nv_bfloat16* yb = static_cast<const __nv_bfloat16*>(y);
  if (dt == SQ_BF16)
    k_layer_error<true><<<grid, 256, 0, st>>>(xb, wb, cin, cout, ldx * eb, ldw * eb, yb, rows, nrows, tokens, err);
  else
    k_layer_error<false><<<grid, 256, 0, st>>>(xb, wb, cin, cout, ldx * eb, ldw * eb, yb, rows, nrows, tokens, err);
  return launch_status();
}

sq_status channel_stats(const float* amax, const float* scale, int64_t n, double* out,
                        cudaStream_t st) {
  k_channel_stats<<<1, 1024, 0, st>>>(amax, scale, n, out);
  return launch_status();
}

}  // namespace sq

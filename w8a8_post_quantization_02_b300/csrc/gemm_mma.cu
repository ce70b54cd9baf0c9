// Step 5, integer path: INT8 x INT8 -> INT32 GEMM on the legacy integer
// tensor-core instruction (mma.sync m16n8k32 s8), exact by construction,
// with the bf16 dequantizing epilogue.
//
// Source: learn-kernels.com "Quantization", paragraph 2 (both matmul
// operands INT8); paragraph 1 (a decode step is bound by streaming the
// weights).  This path reads the int8 weight codes directly, one byte per
// weight, so it is the weight-streaming (decode, small m) path.
//
// A block owns 16*MT tokens x 16 output channels and its 8 warps split K
// in runs of 8/MT consecutive 64-wide steps whose loads are all issued
// before their MMAs.  Each lane loads 16 contiguous codes per row per step;
// the same permutation of k inside the step is used for A and B, so every
// product pairs matching k and the sum is unchanged.
#include <cuda_bf16.h>

#include "sq_common.cuh"

namespace sq {
namespace {

SQ_DEVINL void mma_s8(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                      uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

constexpr int kWarps = 8;
constexpr int kBN = 16;  // output channels per block (two n8 tiles)

template <int MT>
__global__ void __launch_bounds__(kWarps * 32) k_gemm_i8_mma(
    const int8_t* __restrict__ xq, const float* __restrict__ x_scale, const int8_t* __restrict__ wq,
    const float* __restrict__ w_scale, int64_t M, int64_t N, int64_t K,
    __nv_bfloat16* __restrict__ y, int32_t* __restrict__ acc_out) {
  constexpr int BM = 16 * MT;
  __shared__ int32_t tile[BM][kBN];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, tq = lane & 3;
  const int64_t m0 = (int64_t)blockIdx.y * BM, n0 = (int64_t)blockIdx.x * kBN;

  for (int i = threadIdx.x; i < BM * kBN; i += blockDim.x) (&tile[0][0])[i] = 0;

  int acc[MT][2][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int r = 0; r < 4; ++r) acc[mt][nt][r] = 0;

  const int64_t nsteps = (K + 63) / 64;
  const int8_t* brow[2];
  bool bval[2];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const int64_t n = n0 + nt * 8 + g;
    bval[nt] = n < N;
    brow[nt] = wq + (bval[nt] ? n : 0) * K;
  }
  const int8_t* arow[MT][2];
  bool aval[MT][2];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int64_t m = m0 + mt * 16 + g + h * 8;
      aval[mt][h] = m < M;
      arow[mt][h] = xq + (aval[mt][h] ? m : 0) * K;
    }

  // each warp takes U consecutive 64-wide k steps at a time and issues all
  // of their loads before the MMAs, so U x 2 weight loads per lane are in
  // flight (a decode step is bound by streaming the weights)
  constexpr int U = 8 / MT;
  for (int64_t s0 = (int64_t)warp * U; s0 < nsteps; s0 += (int64_t)kWarps * U) {
    uint4 b[U][2];
    uint4 a[U][MT][2];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int64_t k = (s0 + u) * 64 + tq * 16;
      const bool kin = k < K;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
        b[u][nt] = (kin && bval[nt]) ? ld_stream16(brow[nt] + k) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int h = 0; h < 2; ++h)
          a[u][mt][h] = (kin && aval[mt][h]) ? ld_ro16(arow[mt][h] + k) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int mt = 0; mt < MT; ++mt)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          mma_s8(acc[mt][nt], a[u][mt][0].x, a[u][mt][1].x, a[u][mt][0].y, a[u][mt][1].y, b[u][nt].x,
                 b[u][nt].y);
          mma_s8(acc[mt][nt], a[u][mt][0].z, a[u][mt][1].z, a[u][mt][0].w, a[u][mt][1].w, b[u][nt].z,
                 b[u][nt].w);
        }
  }
  __syncthreads();  // tile zeroed
#pragma unroll
  for (int mt = 0; mt < MT; ++mt)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      atomicAdd(&tile[mt * 16 + g][nt * 8 + tq * 2 + 0], acc[mt][nt][0]);
      atomicAdd(&tile[mt * 16 + g][nt * 8 + tq * 2 + 1], acc[mt][nt][1]);
      atomicAdd(&tile[mt * 16 + g + 8][nt * 8 + tq * 2 + 0], acc[mt][nt][2]);
      atomicAdd(&tile[mt * 16 + g + 8][nt * 8 + tq * 2 + 1], acc[mt][nt][3]);
    }
  __syncthreads();
  for (int i = threadIdx.x; i < BM * kBN; i += blockDim.x) {
    const int r = i / kBN, c = i % kBN;
    const int64_t m = m0 + r, n = n0 + c;
    if (m >= M || n >= N) continue;
    const int32_t v = tile[r][c];
    if (acc_out) acc_out[m * N + n] = v;
    const float f = __fmul_rn(__fmul_rn(__int2float_rn(v), x_scale[m]), w_scale[n]);
    y[m * N + n] = __float2bfloat16_rn(f);
  }
}

}  // namespace

sq_status gemm_i8_mma(const int8_t* xq, const float* x_scale, const int8_t* wq,
                      const float* w_scale, int64_t m, int64_t n, int64_t k, void* y,
                      int32_t* acc_out, cudaStream_t st) {
  __nv_bfloat16* yb = static_cast<__nv_bfloat16*>(y);
  const unsigned gx = (unsigned)((n + kBN - 1) / kBN);
  if (m <= 16) {
    k_gemm_i8_mma<1><<<dim3(gx, 1), kWarps * 32, 0, st>>>(xq, x_scale, wq, w_scale, m, n, k, yb, acc_out);
  } else if (m <= 32) {
    k_gemm_i8_mma<2><<<dim3(gx, 1), kWarps * 32, 0, st>>>(xq, x_scale, wq, w_scale, m, n, k, yb, acc_out);
  } else {
    const unsigned gy = (unsigned)((m + 63) / 64);
    k_gemm_i8_mma<4><<<dim3(gx, gy), kWarps * 32, 0, st>>>(xq, x_scale, wq, w_scale, m, n, k, yb, acc_out);
  }
  return launch_status();
}

}  // namespace sq

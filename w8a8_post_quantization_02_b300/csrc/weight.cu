// Step 3: offline fold of diag(s) into W's rows and per-output-channel
// symmetric INT8 quantization, written K-major ([Cout x Cin]) for the GEMM.
//
// Sources: first page ("Move activation scale without changing the real
// linear map"), paragraph 1: S multiplies W on the input-channel side;
// learn-kernels.com "Quantization", paragraph 2: the transform is applied
// offline and the weights are quantized to INT8.
//
// Pass 1 streams W once and reduces max_j |s_j * W[j,n]| per output
// channel n (8 warps per block over rows, one atomicMax per column per
// block, into a caller-provided workspace).  Pass 2 streams W again in
// 64 x 64 tiles, recomputes W' = s_j * W[j,n], quantizes with the channel's
// 1/d, transposes through shared memory and writes each output channel's
// codes contiguously.
#include "sq_common.cuh"

namespace sq {

__global__ void k_fill_u32(uint32_t* p, int64_t n, uint32_t v);  // calib.cu

namespace {

template <bool BF16>
SQ_DEVINL void load_row_vec(const uint8_t* row, int64_t c, float (&f)[8]) {
  // 8 consecutive elements starting at column c (c % 8 == 0, in bounds)
  if constexpr (BF16) {
    uint4 v = ld_stream16(row + c * 2);
    f[0] = bf16lo_to_f32(v.x);
    f[1] = bf16hi_to_f32(v.x);
    f[2] = bf16lo_to_f32(v.y);
    f[3] = bf16hi_to_f32(v.y);
    f[4] = bf16lo_to_f32(v.z);
    f[5] = bf16hi_to_f32(v.z);
    f[6] = bf16lo_to_f32(v.w);
    f[7] = bf16hi_to_f32(v.w);
  } else {
    uint4 a = ld_stream16(row + c * 4), b = ld_stream16(row + c * 4 + 16);
    f[0] = __uint_as_float(a.x);
    f[1] = __uint_as_float(a.y);
    f[2] = __uint_as_float(a.z);
    f[3] = __uint_as_float(a.w);
    f[4] = __uint_as_float(b.x);
    f[5] = __uint_as_float(b.y);
    f[6] = __uint_as_float(b.z);
    f[7] = __uint_as_float(b.w);
  }
}

// ALIGNED: row starts are 16-byte aligned, so in-bounds groups of 8 use
// vector loads; otherwise elements are loaded one by one.
template <bool BF16, bool ALIGNED>
SQ_DEVINL void load_row_vec_masked(const uint8_t* row, int64_t c, int64_t cols, float (&f)[8]) {
  if (ALIGNED && c + 8 <= cols) {
    load_row_vec<BF16>(row, c, f);
    return;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float v = 0.0f;
    if (c + e < cols)
      v = BF16 ? __uint_as_float((uint32_t)reinterpret_cast<const uint16_t*>(row)[c + e] << 16)
               : reinterpret_cast<const float*>(row)[c + e];
    f[e] = v;
  }
}

// Pass 1: amax_bits[n] = max(amax_bits[n], max_j |s_j * W[j, n]|).  A block
// covers 256 columns (8 per thread) and a range of rows.
template <bool BF16, bool ALIGNED>
__global__ void __launch_bounds__(kThreads) k_fold_colmax(const uint8_t* __restrict__ w,
                                                          int64_t cin, int64_t cout,
                                                          int64_t ldw_bytes,
                                                          const float* __restrict__ s,
                                                          int64_t rows_per_block,
                                                          uint32_t* __restrict__ amax_bits) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t c = (int64_t)blockIdx.x * 256 + (int64_t)lane * 8;
  const int64_t r0 = (int64_t)blockIdx.y * rows_per_block;
  const int64_t r1 = min(cin, r0 + rows_per_block);
  uint32_t m[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
  if (c < cout) {
    int64_t r = r0 + warp;
    for (; r + 8 < r1; r += 16) {
      float f0[8], f1[8];
      load_row_vec_masked<BF16, ALIGNED>(w + r * ldw_bytes, c, cout, f0);
      load_row_vec_masked<BF16, ALIGNED>(w + (r + 8) * ldw_bytes, c, cout, f1);
      const float s0 = s[r], s1 = s[r + 8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        m[e] = max(m[e], abs_bits(__fmul_rn(s0, f0[e])));
        m[e] = max(m[e], abs_bits(__fmul_rn(s1, f1[e])));
      }
    }
    for (; r < r1; r += 8) {
      float f0[8];
      load_row_vec_masked<BF16, ALIGNED>(w + r * ldw_bytes, c, cout, f0);
      const float s0 = s[r];
#pragma unroll
      for (int e = 0; e < 8; ++e) m[e] = max(m[e], abs_bits(__fmul_rn(s0, f0[e])));
    }
  }
  __shared__ uint32_t red[kThreads / 32][32][8];
#pragma unroll
  for (int e = 0; e < 8; ++e) red[warp][lane][e] = m[e];
  __syncthreads();
  if (warp == 0 && c < cout) {
    for (int w2 = 1; w2 < kThreads / 32; ++w2)
#pragma unroll
      for (int e = 0; e < 8; ++e) m[e] = max(m[e], red[w2][lane][e]);
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (c + e < cout) atomicMax(amax_bits + c + e, m[e]);
  }
}

// Pass 2: a block quantizes a tile of 64 input channels (j) x 64 output
// channels (n) and writes wq[n, j0 .. j0+63].
constexpr int TJ = 64, TN = 64;

template <bool BF16, bool ALIGNED, int CODES>
__global__ void __launch_bounds__(kThreads) k_fold_quant(const uint8_t* __restrict__ w, int64_t cin,
                                                         int64_t cout, int64_t ldw_bytes,
                                                         const float* __restrict__ s,
                                                         const uint32_t* __restrict__ amax_bits,
                                                         uint8_t* __restrict__ wq,
                                                         float* __restrict__ w_scale,
                                                         int32_t* flags) {
  constexpr int CB = CODES == SQ_CODES_BF16 ? 2 : 1;
  constexpr int ROWB = TJ * CB + 16;  // padded bytes per output-channel row of the tile
  __shared__ float inv_s[TN];
  __shared__ __align__(16) uint8_t tile[TN * ROWB];
  const int64_t j0 = (int64_t)blockIdx.y * TJ, n0 = (int64_t)blockIdx.x * TN;
  if (threadIdx.x < TN) {
    const int64_t n = n0 + threadIdx.x;
    float d = 1.0f, inv = 1.0f;
    if (n < cout) {
      const uint32_t ab = amax_bits[n];
      scale_and_inverse(__uint_as_float(ab), d, inv);
      if (blockIdx.y == 0) {
        w_scale[n] = d;
        if (!finite_bits(ab)) raise_flag(flags, SQ_FLAG_NONFINITE);
      }
    }
    inv_s[threadIdx.x] = inv;
  }
  __syncthreads();
  // each thread: 2 (row j, 8-column group) items of the 64 x 64 tile
#pragma unroll
  for (int it = 0; it < 2; ++it) {
    const int item = threadIdx.x + it * kThreads;  // 0..511
    const int jl = item >> 3, g = item & 7;
    const int64_t j = j0 + jl, c = n0 + g * 8;
    float f[8];
    float sj = 0.0f;
    if (j < cin) {
      load_row_vec_masked<BF16, ALIGNED>(w + j * ldw_bytes, c, cout, f);
      sj = s[j];
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = 0.0f;
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float m = code_magic(__fmul_rn(sj, f[e]), inv_s[g * 8 + e]);
      uint8_t* dst = tile + (g * 8 + e) * ROWB + jl * CB;
      if constexpr (CODES == SQ_CODES_BF16)
        *reinterpret_cast<uint16_t*>(dst) = (uint16_t)magic_to_bf16bits(m);
      else
        *dst = (uint8_t)(__float_as_uint(m) & 0xFFu);
    }
  }
  __syncthreads();
  // write: each output-channel row segment is TJ*CB bytes = 4 (i8) or 8
  // (bf16) 16-byte vectors
  constexpr int VPR = TJ * CB / 16;
  for (int item = threadIdx.x; item < TN * VPR; item += kThreads) {
    const int nl = item / VPR, q = item % VPR;
    const int64_t n = n0 + nl, j = j0 + q * (16 / CB);
    if (n >= cout || j >= cin) continue;  // cin % 16 == 0, so a vector is all-in or all-out
    const uint4 v = *reinterpret_cast<const uint4*>(tile + nl * ROWB + q * 16);
    st16(wq + (n * cin + j) * CB, v);
  }
}

}  // namespace

sq_status fold_quantize_weight(const void* w, sq_dtype dt, int64_t cin, int64_t cout, int64_t ldw,
                               const float* s, void* wq, sq_codes fmt, float* w_scale,
                               int32_t* flags, void* workspace, cudaStream_t st) {
  const bool bf16 = dt == SQ_BF16;
  const uint8_t* wb = static_cast<const uint8_t*>(w);
  const int64_t ldb = ldw * elem_bytes(dt);
  uint32_t* amax = static_cast<uint32_t*>(workspace);
  {
    int g = (int)std::min<int64_t>((cout + 255) / 256, 1024);
    k_fill_u32<<<g, 256, 0, st>>>(amax, cout, 0u);
  }
  const bool aligned = aligned16(w) && ldb % 16 == 0;
  {
    const int64_t gx = (cout + 255) / 256;
    int64_t gy = std::max<int64_t>(1, (int64_t)sm_count() * 4 / gx);
    gy = std::min<int64_t>(gy, (cin + 127) / 128);
    gy = std::max<int64_t>(gy, 1);
    const int64_t rpb = (cin + gy - 1) / gy;
    gy = (cin + rpb - 1) / rpb;
    dim3 grid((unsigned)gx, (unsigned)gy);
    if (bf16)
      aligned ? k_fold_colmax<true, true><<<grid, kThreads, 0, st>>>(wb, cin, cout, ldb, s, rpb, amax)
              : k_fold_colmax<true, false><<<grid, kThreads, 0, st>>>(wb, cin, cout, ldb, s, rpb, amax);
    else
      aligned ? k_fold_colmax<false, true><<<grid, kThreads, 0, st>>>(wb, cin, cout, ldb, s, rpb, amax)
              : k_fold_colmax<false, false><<<grid, kThreads, 0, st>>>(wb, cin, cout, ldb, s, rpb, amax);
  }
  {
    dim3 grid((unsigned)((cout + TN - 1) / TN), (unsigned)((cin + TJ - 1) / TJ));
    uint8_t* q = static_cast<uint8_t*>(wq);
#define SQ_FQ(B, A, C) k_fold_quant<B, A, C><<<grid, kThreads, 0, st>>>(wb, cin, cout, ldb, s, amax, q, w_scale, flags)
    if (bf16) {
      if (fmt == SQ_CODES_BF16) aligned ? SQ_FQ(true, true, SQ_CODES_BF16) : SQ_FQ(true, false, SQ_CODES_BF16);
      else aligned ? SQ_FQ(true, true, SQ_CODES_I8) : SQ_FQ(true, false, SQ_CODES_I8);
    } else {
      if (fmt == SQ_CODES_BF16) aligned ? SQ_FQ(false, true, SQ_CODES_BF16) : SQ_FQ(false, false, SQ_CODES_BF16);
      else aligned ? SQ_FQ(false, true, SQ_CODES_I8) : SQ_FQ(false, false, SQ_CODES_I8);
    }
#undef SQ_FQ
  }
  return launch_status();
}

}  // namespace sq

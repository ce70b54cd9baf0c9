// Step 1: per-channel absolute-maximum statistics (calibration).
//
// Source: pith.science review of arXiv 2506.01967 (Smooth Rotation),
// key_machinery: the smoothing factor is built from max|X_j| over tokens and
// max|W_j| over output channels.  Both reductions are HBM-bound streams:
// 16-byte vector loads, integer max on |x| bit patterns (NaN sorts above
// +inf, so NaN propagates), warp shuffles / shared memory, and one
// atomicMax per column per block for the column reduction.
#include "sq_common.cuh"

namespace sq {

__global__ void k_fill_u32(uint32_t* p, int64_t n, uint32_t v) {
  int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  for (; i < n; i += (int64_t)gridDim.x * blockDim.x) p[i] = v;
}

// Per 16-byte vector: fold |elements| into 4 running words.
//  bf16: each word holds two 16-bit maxima (SIMD unsigned max);
//  f32 : each word holds one 32-bit maximum.
template <bool BF16>
SQ_DEVINL void fold_vec(uint4 v, uint32_t (&m)[4]) {
  if (BF16) {
    m[0] = __vmaxu2(m[0], v.x & 0x7FFF7FFFu);
    m[1] = __vmaxu2(m[1], v.y & 0x7FFF7FFFu);
    m[2] = __vmaxu2(m[2], v.z & 0x7FFF7FFFu);
    m[3] = __vmaxu2(m[3], v.w & 0x7FFF7FFFu);
  } else {
    m[0] = max(m[0], v.x & 0x7FFFFFFFu);
    m[1] = max(m[1], v.y & 0x7FFFFFFFu);
    m[2] = max(m[2], v.z & 0x7FFFFFFFu);
    m[3] = max(m[3], v.w & 0x7FFFFFFFu);
  }
}

// Load one 16-byte vector's worth of row elements starting at column c;
// elements at or past `cols` read as zero.  ALIGNED: every row start is
// 16-byte aligned, so in-bounds vectors use one 16-byte load; otherwise the
// elements are loaded one by one.
template <bool BF16, bool ALIGNED>
SQ_DEVINL uint4 load_vec_masked(const uint8_t* row, int64_t c, int64_t cols) {
  constexpr int VEC = BF16 ? 8 : 4;
  if (ALIGNED && c + VEC <= cols) return ld_stream16(row + c * (BF16 ? 2 : 4));
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  if (BF16) {
    const uint16_t* p = reinterpret_cast<const uint16_t*>(row);
    for (int e = 0; e < VEC; ++e)
      if (c + e < cols) w[e >> 1] |= (uint32_t)p[c + e] << (16 * (e & 1));
  } else {
    const uint32_t* p = reinterpret_cast<const uint32_t*>(row);
    for (int e = 0; e < VEC; ++e)
      if (c + e < cols) w[e] = p[c + e];
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// axis 0: out_bits[c] = max(out_bits[c], max_r |a[r, c]|).  A block covers a
// strip of 32*VEC columns and a range of rows; its 8 warps stride the rows.
template <bool BF16, bool ALIGNED>
__global__ void __launch_bounds__(kThreads) k_colmax(const uint8_t* __restrict__ a, int64_t rows,
                                                     int64_t cols, int64_t ld_bytes,
                                                     int64_t rows_per_block,
                                                     uint32_t* __restrict__ out_bits) {
  constexpr int VEC = BF16 ? 8 : 4;
  constexpr int UNROLL = 4;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t c = (int64_t)blockIdx.x * 32 * VEC + (int64_t)lane * VEC;
  const int64_t r0 = (int64_t)blockIdx.y * rows_per_block;
  const int64_t r1 = min(rows, r0 + rows_per_block);
  uint32_t m[4] = {0u, 0u, 0u, 0u};
  if (c < cols) {
    int64_t r = r0 + warp;
    for (; r + (UNROLL - 1) * 8 < r1; r += UNROLL * 8) {
      uint4 v[UNROLL];
#pragma unroll
      for (int u = 0; u < UNROLL; ++u)
        v[u] = load_vec_masked<BF16, ALIGNED>(a + (r + u * 8) * ld_bytes, c, cols);
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) fold_vec<BF16>(v[u], m);
    }
    for (; r < r1; r += 8) fold_vec<BF16>(load_vec_masked<BF16, ALIGNED>(a + r * ld_bytes, c, cols), m);
  }
  __shared__ uint32_t red[kThreads / 32][32][4];
#pragma unroll
  for (int i = 0; i < 4; ++i) red[warp][lane][i] = m[i];
  __syncthreads();
  if (warp == 0 && c < cols) {
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        m[i] = BF16 ? __vmaxu2(m[i], red[w][lane][i]) : max(m[i], red[w][lane][i]);
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      if (c + e >= cols) break;
      uint32_t b = BF16 ? ((m[e >> 1] >> (16 * (e & 1))) & 0xFFFFu) << 16 : m[e];
      atomicMax(out_bits + c + e, b);
    }
  }
}

// axis 1: out[r] = max_c |a[r, c]| (optionally max with the old out[r]).
// One warp per row.
template <bool BF16, bool ALIGNED>
__global__ void __launch_bounds__(kThreads) k_rowmax(const uint8_t* __restrict__ a, int64_t rows,
                                                     int64_t cols, int64_t ld_bytes,
                                                     uint32_t* __restrict__ out_bits,
                                                     int accumulate) {
  constexpr int VEC = BF16 ? 8 : 4;
  constexpr int UNROLL = 4;
  const int lane = threadIdx.x & 31;
  const int64_t r = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  if (r >= rows) return;
  const uint8_t* row = a + r * ld_bytes;
  const int64_t nvec = (cols + VEC - 1) / VEC;
  uint32_t m[4] = {0u, 0u, 0u, 0u};
  int64_t v = lane;
  for (; v + (UNROLL - 1) * 32 < nvec; v += UNROLL * 32) {
    uint4 x[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) x[u] = load_vec_masked<BF16, ALIGNED>(row, (v + u * 32) * VEC, cols);
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) fold_vec<BF16>(x[u], m);
  }
  for (; v < nvec; v += 32) fold_vec<BF16>(load_vec_masked<BF16, ALIGNED>(row, v * VEC, cols), m);
  uint32_t b;
  if (BF16) {
    b = __vmaxu2(__vmaxu2(m[0], m[1]), __vmaxu2(m[2], m[3]));  // per-half maxima
    b = max(b & 0xFFFFu, b >> 16) << 16;
  } else {
    b = max(max(m[0], m[1]), max(m[2], m[3]));
  }
  b = __reduce_max_sync(0xFFFFFFFFu, b);
  if (lane == 0) out_bits[r] = accumulate ? max(out_bits[r], b) : b;
}

sq_status calibrate_absmax(const void* a, sq_dtype dt, int64_t rows, int64_t cols, int64_t ld,
                           int axis, int accumulate, float* amax, cudaStream_t st) {
  const bool bf16 = dt == SQ_BF16;
  const int64_t ld_bytes = ld * elem_bytes(dt);
  const uint8_t* base = static_cast<const uint8_t*>(a);
  uint32_t* out = reinterpret_cast<uint32_t*>(amax);
  const bool aligned = aligned16(a) && ld_bytes % 16 == 0;
  if (axis == 0) {
    const int vec = bf16 ? 8 : 4;
    if (!accumulate) {
      int g = (int)std::min<int64_t>((cols + 255) / 256, 1024);
      k_fill_u32<<<g, 256, 0, st>>>(out, cols, 0u);
    }
    const int64_t gx = (cols + 32 * vec - 1) / (32 * vec);
    // >= 128 rows per block (16 per warp, 4-deep unrolled 16-byte loads),
    // but enough blocks to cover every SM about 4 times when rows allow
    int64_t gy = std::max<int64_t>(1, (int64_t)sm_count() * 4 / gx);
    gy = std::min<int64_t>(gy, (rows + 127) / 128);
    gy = std::max<int64_t>(gy, 1);
    const int64_t rpb = (rows + gy - 1) / gy;
    gy = (rows + rpb - 1) / rpb;
    dim3 grid((unsigned)gx, (unsigned)gy);
    if (bf16)
      aligned ? k_colmax<true, true><<<grid, kThreads, 0, st>>>(base, rows, cols, ld_bytes, rpb, out)
              : k_colmax<true, false><<<grid, kThreads, 0, st>>>(base, rows, cols, ld_bytes, rpb, out);
    else
      aligned ? k_colmax<false, true><<<grid, kThreads, 0, st>>>(base, rows, cols, ld_bytes, rpb, out)
              : k_colmax<false, false><<<grid, kThreads, 0, st>>>(base, rows, cols, ld_bytes, rpb, out);
  } else {
    const int64_t g = (rows + kThreads / 32 - 1) / (kThreads / 32);
    if (bf16)
      aligned ? k_rowmax<true, true><<<(unsigned)g, kThreads, 0, st>>>(base, rows, cols, ld_bytes, out, accumulate)
              : k_rowmax<true, false><<<(unsigned)g, kThreads, 0, st>>>(base, rows, cols, ld_bytes, out, accumulate);
    else
      aligned ? k_rowmax<false, true><<<(unsigned)g, kThreads, 0, st>>>(base, rows, cols, ld_bytes, out, accumulate)
              : k_rowmax<false, false><<<(unsigned)g, kThreads, 0, st>>>(base, rows, cols, ld_bytes, out, accumulate);
  }
  return launch_status();
}

}  // namespace sq

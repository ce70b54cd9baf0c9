// Step 1: per-channel absolute-maximum statistics (calibration).
//
// Source: pith.science review of arXiv 2506.01967 (Smooth Rotation),
// key_machinery: the smoothing factor is built from max|X_j| over tokens and
// max|W_j| over output channels.  Both reductions are HBM-bound streams;
// maxima of magnitudes are exact in any order, and NaN propagates.
//
// Column maxima (axis 0, rows 16-byte aligned): the matrix is cut into
// strips of 128 bytes of columns; a cluster of 1-8 CTAs owns a strip and
// splits its rows; each CTA streams its rows through a 4-stage ring of
// 128-row TMA boxes (128-byte swizzle, conflict-free reads), and the
// cluster combines its partial maxima through distributed shared memory,
// so one kernel writes every column once, with no atomics and no zeroing.
// Other alignments: each block reduces a strip of rows and merges with one
// atomicMax per column into a zeroed output.
//
// Row maxima (axis 1): one warp per row, eight 16-byte loads in flight per
// lane.
#include "sq_async.cuh"

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
    m[0] = async::absmax_nan_bf16x2(m[0], v.x);
    m[1] = async::absmax_nan_bf16x2(m[1], v.y);
    m[2] = async::absmax_nan_bf16x2(m[2], v.z);
    m[3] = async::absmax_nan_bf16x2(m[3], v.w);
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
  for (int i = 0; i < 4; ++i) red[warp][lane][i] = m[i] & (BF16 ? 0x7FFF7FFFu : 0xFFFFFFFFu);
  __syncthreads();
  if (warp == 0 && c < cols) {
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (BF16) m[i] &= 0x7FFF7FFFu;
        m[i] = BF16 ? __vmaxu2(m[i], red[w][lane][i]) : max(m[i], red[w][lane][i]);
      }
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
  constexpr int UNROLL = 8;
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
#pragma unroll
    for (int i = 0; i < 4; ++i) m[i] &= 0x7FFF7FFFu;  // drop the meaningless signs
    b = __vmaxu2(__vmaxu2(m[0], m[1]), __vmaxu2(m[2], m[3]));  // per-half maxima
    b = max(b & 0xFFFFu, b >> 16) << 16;
  } else {
    b = max(max(m[0], m[1]), max(m[2], m[3]));
  }
  b = __reduce_max_sync(0xFFFFFFFFu, b);
  if (lane == 0) out_bits[r] = accumulate ? max(out_bits[r], b) : b;
}

// ---------------------------------------------------------------- column maxima, TMA strips
namespace colstrip {
using namespace async;

constexpr int kThreads = 256;
constexpr int kBoxRows = 128;
constexpr int kRowBytes = 128;           // strip width: 128 bytes (128-byte swizzle)
constexpr int kStages = 4;
constexpr int kBoxBytes = kBoxRows * kRowBytes;
constexpr uint64_t kWaitNs = 1000000000ull;

struct Smem {
  uint8_t box[kStages][kBoxBytes];
  uint32_t red[4][8][4];  // [row group][chunk][word]
  uint32_t part[32];      // this CTA's maxima as |.| bit patterns (read by the cluster)
  uint64_t full[kStages];
};

// One CTA of a CL-CTA cluster: rows [rank*R, rank*R + R) of the strip of
// columns [c0, c0 + 128 bytes).  Every wait is bounded; one that runs out
// (a copy that never lands) turns the strip's maxima into NaN.  Words of `part`: chunk c (16 bytes) word q
// holds columns c*EPC + q (fp32) or c*EPC + 2q, +1 (two bf16 halves).
template <bool BF16, int CL>
__global__ void __launch_bounds__(kThreads) k_colmax_strip(const __grid_constant__ CUtensorMap map,
                                                           int64_t rows, int64_t cols,
                                                           int rows_per_cta, int accumulate,
                                                           uint32_t* __restrict__ out_bits,
                                                           int32_t* flags) {
  constexpr int EPC = BF16 ? 8 : 4;
  constexpr int SW = 8 * EPC;
  extern __shared__ uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, lane = tid & 31;
  const uint32_t rank = CL > 1 ? cluster_ctarank() : 0u;
  const int64_t c0 = (int64_t)(blockIdx.x / CL) * SW;
  const int64_t r0 = (int64_t)rank * rows_per_cta;
  const int64_t left = rows - r0;
  const int nrows = left <= 0 ? 0 : (int)(left < rows_per_cta ? left : rows_per_cta);
  const int nbox = (nrows + kBoxRows - 1) / kBoxRows;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) mbar_init(&sm.full[s], 1);
    fence_mbar_init();
    prefetch_tensormap(&map);
    for (int b = 0; b < kStages && b < nbox; ++b) {
      mbar_expect_tx(&sm.full[b], kBoxBytes);
      tma_load_2d(sm.box[b], &map, &sm.full[b], (int)c0, (int)(r0 + b * kBoxRows));
    }
  }
  __syncthreads();

  // 8 consecutive lanes read 8 consecutive rows of one chunk: with the
  // 128-byte swizzle (chunk index XOR row bits 0-2) they hit 8 different
  // bank groups.
  const int c = (tid >> 3) & 7;
  const int rsub = (tid & 7) + 8 * (tid >> 6);  // 0..31
  uint32_t m[4] = {0u, 0u, 0u, 0u};
  bool aborted = false;
  int b = 0;
  for (; b < nbox; ++b) {
    const int stage = b % kStages;
    const bool ok = mbar_wait_bounded(&sm.full[stage], (uint32_t)(b / kStages) & 1u, kWaitNs);
    if (ok) {
#pragma unroll
      for (int k = 0; k < kBoxRows / 32; ++k) {
        const int r = rsub + 32 * k;
        const uint4 v = *reinterpret_cast<const uint4*>(sm.box[stage] + r * kRowBytes +
                                                        ((c ^ (r & 7)) << 4));
        if constexpr (BF16) {
          m[0] = absmax_nan_bf16x2(m[0], v.x);
          m[1] = absmax_nan_bf16x2(m[1], v.y);
          m[2] = absmax_nan_bf16x2(m[2], v.z);
          m[3] = absmax_nan_bf16x2(m[3], v.w);
        } else {
          m[0] = __float_as_uint(absmax_nan(__uint_as_float(m[0]), __uint_as_float(v.x)));
          m[1] = __float_as_uint(absmax_nan(__uint_as_float(m[1]), __uint_as_float(v.y)));
          m[2] = __float_as_uint(absmax_nan(__uint_as_float(m[2]), __uint_as_float(v.z)));
          m[3] = __float_as_uint(absmax_nan(__uint_as_float(m[3]), __uint_as_float(v.w)));
        }
      }
    }
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    if (tid == 0 && b + kStages < nbox) {  // the stage is free: refill it
      mbar_expect_tx(&sm.full[stage], kBoxBytes);
      tma_load_2d(sm.box[stage], &map, &sm.full[stage], (int)c0,
                  (int)(r0 + (int64_t)(b + kStages) * kBoxRows));
    }
  }
  // magnitudes as bit patterns (the packed max leaves meaningless signs)
  const uint32_t mask = BF16 ? 0x7FFF7FFFu : 0x7FFFFFFFu;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t v = m[i] & mask;
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) {
      const uint32_t u = __shfl_xor_sync(0xFFFFFFFFu, v, o);
      v = BF16 ? __vmaxu2(v, u) : max(v, u);
    }
    m[i] = v;
  }
  if ((lane & 7) == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) sm.red[tid >> 6][c][i] = m[i];
  }
  __syncthreads();
  if (tid < 32) {
    uint32_t v = 0u;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const uint32_t u = sm.red[g][tid >> 2][tid & 3];
      v = BF16 ? __vmaxu2(v, u) : max(v, u);
    }
    // a wait that ran out makes this strip's statistics NaN, which the
    // smoothing step reports as SQ_FLAG_NONFINITE
    sm.part[tid] = aborted ? mask : v;
  }
  if constexpr (CL > 1) {
    cluster_arrive();
    cluster_wait();
  } else {
    __syncthreads();
  }
  if (rank == 0 && tid < 32) {
    uint32_t v = sm.part[tid];
    if constexpr (CL > 1) {
      const uint32_t a = su32(&sm.part[tid]);
#pragma unroll
      for (int q = 1; q < CL; ++q) {
        const uint32_t u = ld_cluster_u32(mapa(a, (uint32_t)q));
        v = BF16 ? __vmaxu2(v, u) : max(v, u);
      }
    }
    const int cc = tid >> 2, q = tid & 3;
    if constexpr (BF16) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int64_t col = c0 + cc * EPC + 2 * q + h;
        if (col < cols) {
          uint32_t bits = ((v >> (16 * h)) & 0xFFFFu) << 16;
          if (accumulate) bits = max(bits, out_bits[col]);
          out_bits[col] = bits;
        }
      }
    } else {
      const int64_t col = c0 + cc * EPC + q;
      if (col < cols) out_bits[col] = accumulate ? max(v, out_bits[col]) : v;
    }
  }
  if (aborted && tid == 0) {
    raise_flag(flags, SQ_FLAG_TIMEOUT);
    for (int k = 0; k < kStages && b + k < nbox; ++k)
      mbar_wait_bounded(&sm.full[(b + k) % kStages], (uint32_t)((b + k) / kStages) & 1u, 10000000ull);
  }
  if constexpr (CL > 1) {
    cluster_arrive();  // rank 0 has read every peer's `part`
    cluster_wait();
  }
}

int64_t rows_per_cta(int64_t rows, int cl) {
  const int64_t r = (rows + cl - 1) / cl;
  return (r + kBoxRows - 1) / kBoxRows * kBoxRows;
}

// Cluster size: the largest that keeps the grid within one wave of three
// CTAs per SM (the shared memory of a CTA allows three), no more CTAs per
// strip than 128-row boxes.  A second, partial wave measured slower on B300
// than fewer, longer CTAs (8192 x 8192 bf16: 25.4 us instead of 29.0 us).
int cluster_size(int64_t rows, int64_t cols, sq_dtype dt) {
  const int64_t strips = (cols * elem_bytes(dt) + kRowBytes - 1) / kRowBytes;
  const int64_t boxes = (rows + kBoxRows - 1) / kBoxRows;
  int cl = 1;
  while (cl < 8 && strips * cl * 2 <= 3 * (int64_t)sm_count() && cl * 2 <= boxes) cl *= 2;
  return cl;
}

bool applies(sq_dtype dt, int64_t rows, int64_t cols, int64_t ld) {
  return (ld * elem_bytes(dt)) % 16 == 0 && rows < ((int64_t)1 << 31) && cols < ((int64_t)1 << 31);
}

template <bool BF16, int CL>
sq_status launch(const CUtensorMap& map, int64_t rows, int64_t cols, int rpc, int accumulate,
                 uint32_t* out, cudaStream_t st) {
  auto kern = k_colmax_strip<BF16, CL>;
  const size_t smem = sizeof(Smem) + 1024;
  static std::atomic<uint64_t> attr_done{0};
  if (!once_per_device(attr_done, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      }))
    return SQ_ERR_CUDA;
  const int64_t strips = (cols * (BF16 ? 2 : 4) + kRowBytes - 1) / kRowBytes;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(strips * CL), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CL;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, map, rows, cols, rpc, accumulate, out, (int32_t*)nullptr) !=
      cudaSuccess)
    return SQ_ERR_CUDA;
  return launch_status();
}

template <bool BF16>
sq_status launch_cl(int cl, const CUtensorMap& map, int64_t rows, int64_t cols, int rpc,
                    int accumulate, uint32_t* out, cudaStream_t st) {
  switch (cl) {
    case 1: return launch<BF16, 1>(map, rows, cols, rpc, accumulate, out, st);
    case 2: return launch<BF16, 2>(map, rows, cols, rpc, accumulate, out, st);
    case 4: return launch<BF16, 4>(map, rows, cols, rpc, accumulate, out, st);
    default: return launch<BF16, 8>(map, rows, cols, rpc, accumulate, out, st);
  }
}

sq_status colmax(const void* a, sq_dtype dt, int64_t rows, int64_t cols, int64_t ld, int accumulate,
                 uint32_t* out, cudaStream_t st) {
  const int eb = elem_bytes(dt);
  auto fn = tensor_map_encoder();
  if (!fn) return SQ_ERR_CUDA;
  const int cl = cluster_size(rows, cols, dt);
  const int rpc = (int)rows_per_cta(rows, cl);
  CUtensorMap map;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)(ld * eb)};
  cuuint32_t box[2] = {(cuuint32_t)(kRowBytes / eb), (cuuint32_t)kBoxRows};
  cuuint32_t estr[2] = {1, 1};
  if (fn(&map, dt == SQ_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
         const_cast<void*>(a), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return SQ_ERR_CUDA;
  return dt == SQ_BF16 ? launch_cl<true>(cl, map, rows, cols, rpc, accumulate, out, st)
                       : launch_cl<false>(cl, map, rows, cols, rpc, accumulate, out, st);
}

}  // namespace colstrip

int calibrate_kernel_count(sq_dtype dt, int64_t rows, int64_t cols, int64_t ld, int axis,
                           int accumulate) {
  if (axis == 1) return 1;
  if (colstrip::applies(dt, rows, cols, ld)) return 1;
  return accumulate ? 1 : 2;
}

sq_status calibrate_absmax(const void* a, sq_dtype dt, int64_t rows, int64_t cols, int64_t ld,
                           int axis, int accumulate, float* amax, cudaStream_t st) {
  const bool bf16 = dt == SQ_BF16;
  const int64_t ld_bytes = ld * elem_bytes(dt);
  const uint8_t* base = static_cast<const uint8_t*>(a);
  uint32_t* out = reinterpret_cast<uint32_t*>(amax);
  const bool aligned = aligned16(a) && ld_bytes % 16 == 0;
  if (axis == 0 && aligned && colstrip::applies(dt, rows, cols, ld))
    return colstrip::colmax(a, dt, rows, cols, ld, accumulate, out, st);
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

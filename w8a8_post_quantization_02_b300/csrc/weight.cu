// Step 3: offline fold of diag(s) into W's rows and per-output-channel
// symmetric INT8 quantization, written K-major ([Cout x Cin]) for the GEMM.
//
// Sources: first page ("Move activation scale without changing the real
// linear map"), paragraph 1: S multiplies W on the input-channel side;
// learn-kernels.com "Quantization", paragraph 2: the transform is applied
// offline and the weights are quantized to INT8.
//
// Single-pass path (rows of W 16-byte aligned, Cin <= 12288): W is cut into
// strips of 64 bytes of columns (32 bf16 / 16 fp32 output channels).  A
// cluster of 1-8 CTAs owns one strip and splits its rows; each CTA loads its
// part of the strip into shared memory with 2-D TMA copies (64-byte
// swizzle, so both passes over it are free of bank conflicts), reduces
// max_j |s_j * W[j,n]| over its rows, and the cluster combines the partial
// maxima through distributed shared memory.  Each CTA then quantizes its
// rows from shared memory and writes each output channel's codes as
// contiguous runs.  W is read from HBM once and the codes written once.
//
// Two-pass path (any alignment or width): pass 1 streams W and reduces
// the column maxima (one atomicMax per column per block, into the caller's
// workspace); pass 2 streams W again in 64 x 64 tiles, quantizes, transposes
// through shared memory and writes the codes.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "sq_async.cuh"

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
  __shared__ float d_s[TN], inv_s[TN];
  __shared__ bool fast_s[TN];
  __shared__ __align__(16) uint8_t tile[TN * ROWB];
  const int64_t j0 = (int64_t)blockIdx.y * TJ, n0 = (int64_t)blockIdx.x * TN;
  if (threadIdx.x < TN) {
    const int64_t n = n0 + threadIdx.x;
    float d = 1.0f, inv = 1.0f;
    bool fast = true;
    if (n < cout) {
      const uint32_t ab = amax_bits[n];
      scale_and_inverse(__uint_as_float(ab), d, inv);
      fast = fast_quotient_ok(ab);
      if (blockIdx.y == 0) {
        w_scale[n] = d;
        if (!finite_bits(ab)) raise_flag(flags, SQ_FLAG_NONFINITE);
      }
    }
    d_s[threadIdx.x] = d;
    inv_s[threadIdx.x] = inv;
    fast_s[threadIdx.x] = fast;
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
      const int ch = g * 8 + e;
      const float v = __fmul_rn(sj, f[e]);
      const float m = fast_s[ch] ? magic_of(quot_rn(v, d_s[ch], inv_s[ch])) : code_div_magic(v, d_s[ch], 127.0f);
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


// ---------------------------------------------------------------- single pass
namespace strip {
using namespace async;

constexpr int kThreads = 256;
constexpr int kBoxRows = 128;                       // rows per TMA box
constexpr int kRowBytes = 64;                       // strip row = 64 bytes (64-byte swizzle)
constexpr int kMaxRows = 1536;                      // rows per CTA: 96 KiB of strip
constexpr int kMaxBoxes = kMaxRows / kBoxRows;
constexpr uint64_t kWaitNs = 1000000000ull;         // bound on every mbarrier wait (1 s)

// Byte offset of 16-byte chunk c of strip row r in the TMA 64-byte swizzle:
// the chunk index is XOR-ed with bits 1-2 of the row.
SQ_DEVINL uint32_t chunk_off(int r, int c) {
  return (uint32_t)r * kRowBytes + ((uint32_t)(c ^ ((r >> 1) & 3)) << 4);
}

template <bool BF16>
SQ_DEVINL void unpack_chunk(uint4 v, float* f) {
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

template <int EPC>
struct Layout {
  static constexpr int SW = 4 * EPC;  // output channels per strip
  size_t strip, s, red, part, inv, dsc, flag, bars, total;
  explicit __host__ __device__ Layout(int rows_per_cta) {
    strip = 0;                                     // 1024-aligned base
    s = strip + (size_t)rows_per_cta * kRowBytes;  // fp32 [R]
    red = s + (size_t)rows_per_cta * 4;            // u32 [8 warps][4 chunks][EPC]
    part = red + 8 * 4 * EPC * 4;                  // u32 [SW], read by the whole cluster
    inv = part + SW * 4;                           // fp32 [SW]: RN(1/d)
    dsc = inv + SW * 4;                            // fp32 [SW]: d
    flag = dsc + SW * 4;                           // int: some channel needs the division
    bars = (flag + 4 + 7) & ~size_t(7);            // mbarriers [kMaxBoxes]
    total = bars + kMaxBoxes * 8;
  }
};

// One CTA of a CL-CTA cluster: rows [rank*R, rank*R + R) of the strip of
// output channels [n0, n0 + SW).
// MINB: 3 builds the kernel for three CTAs per SM (at most 80 registers,
// a few bytes spilled), 0 leaves the compiler's choice (83-88 registers, so
// two CTAs per SM).  See launch_cl for which runs.
template <bool BF16, int CODES, int CL, int MINB>
__global__ void __launch_bounds__(kThreads, MINB) k_fold_strip(const __grid_constant__ CUtensorMap map_w,
                                                         const float* __restrict__ s, int64_t cin,
                                                         int64_t cout, int rows_per_cta,
                                                         uint8_t* __restrict__ wq,
                                                         float* __restrict__ w_scale,
                                                         int32_t* flags) {
  constexpr int EPC = BF16 ? 8 : 4;  // elements per 16-byte chunk
  constexpr int SW = 4 * EPC;
  constexpr int CB = CODES == SQ_CODES_BF16 ? 2 : 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const Layout<EPC> L(rows_per_cta);
  uint8_t* strip = base + L.strip;
  float* s_sm = reinterpret_cast<float*>(base + L.s);
  uint32_t* red = reinterpret_cast<uint32_t*>(base + L.red);
  uint32_t* part = reinterpret_cast<uint32_t*>(base + L.part);
  float* inv_sm = reinterpret_cast<float*>(base + L.inv);
  float* d_sm = reinterpret_cast<float*>(base + L.dsc);
  int* clamp_flag = reinterpret_cast<int*>(base + L.flag);
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + L.bars);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = CL > 1 ? cluster_ctarank() : 0u;
  const int64_t n0 = (int64_t)(blockIdx.x / CL) * SW;
  const int64_t j0 = (int64_t)rank * rows_per_cta;
  const int64_t left = cin - j0;
  const int rows = left <= 0 ? 0 : (int)(left < rows_per_cta ? left : rows_per_cta);  // multiple of 16
  const int nbox = (rows + kBoxRows - 1) / kBoxRows;

  if (tid == 0) {
    for (int b = 0; b < nbox; ++b) mbar_init(&bars[b], 1);
    *clamp_flag = 0;
    fence_mbar_init();
    prefetch_tensormap(&map_w);
    for (int b = 0; b < nbox; ++b) {
      mbar_expect_tx(&bars[b], kBoxRows * kRowBytes);
      tma_load_2d(strip + (size_t)b * kBoxRows * kRowBytes, &map_w, &bars[b], (int)n0,
                  (int)(j0 + b * kBoxRows));
    }
  }
  for (int i = tid; i < rows; i += kThreads) s_sm[i] = s[j0 + i];
  __syncthreads();

  // ---- pass 1: max over this CTA's rows of |s_j * W[j, n]| per channel.
  // 8 consecutive lanes read 8 consecutive rows of one chunk: conflict-free.
  bool ok = true;
  {
    const int c = (tid >> 3) & 3;
    const int rsub = (tid & 7) + 8 * warp;  // 0..63
    float m[EPC];
#pragma unroll
    for (int e = 0; e < EPC; ++e) m[e] = 0.0f;
    for (int b = 0; b < nbox; ++b) {
      ok = mbar_wait_bounded(&bars[b], 0, kWaitNs) && ok;
      const int r1 = min(rows, (b + 1) * kBoxRows);
      for (int r = b * kBoxRows + rsub; r < r1; r += 64) {
        float f[EPC];
        unpack_chunk<BF16>(*reinterpret_cast<const uint4*>(strip + chunk_off(r, c)), f);
        const float sj = s_sm[r];
#pragma unroll
        for (int e = 0; e < EPC; e += 2) mul2_rn(f[e], f[e + 1], sj, sj);
#pragma unroll
        for (int e = 0; e < EPC; ++e) m[e] = absmax_nan(m[e], f[e]);
      }
    }
    uint32_t mb[EPC];
#pragma unroll
    for (int e = 0; e < EPC; ++e) {
      mb[e] = __float_as_uint(m[e]) & 0x7FFFFFFFu;
      mb[e] = max(mb[e], __shfl_xor_sync(0xFFFFFFFFu, mb[e], 1));
      mb[e] = max(mb[e], __shfl_xor_sync(0xFFFFFFFFu, mb[e], 2));
      mb[e] = max(mb[e], __shfl_xor_sync(0xFFFFFFFFu, mb[e], 4));
    }
    if ((lane & 7) == 0) {
#pragma unroll
      for (int e = 0; e < EPC; ++e) red[(warp * 4 + c) * EPC + e] = mb[e];
    }
  }
  __syncthreads();
  if (tid < SW) {
    uint32_t v = 0u;
#pragma unroll
    for (int w = 0; w < 8; ++w) v = max(v, red[w * SW + tid]);
    part[tid] = v;
  }
  // ---- combine the cluster's partial maxima (distributed shared memory)
  if constexpr (CL > 1) {
    cluster_arrive();
    cluster_wait();
  } else {
    __syncthreads();
  }
  if (tid < SW) {
    uint32_t v = 0u;
    if constexpr (CL > 1) {
      const uint32_t a = su32(&part[tid]);
#pragma unroll
      for (int q = 0; q < CL; ++q) v = max(v, ld_cluster_u32(mapa(a, (uint32_t)q)));
    } else {
      v = part[tid];
    }
    float d, inv;
    scale_and_inverse(__uint_as_float(v), d, inv);
    inv_sm[tid] = inv;
    d_sm[tid] = d;
    const int64_t n = n0 + tid;
    if (n < cout) {
      // a finite maximum >= 2^-93: the quotient W'/d comes from quot_rn and
      // no code leaves [-127, 127]; otherwise the CTA divides and clamps
      if (!fast_quotient_ok(v)) *clamp_flag = 1;
      if (rank == 0) {
        w_scale[n] = d;
        if (!finite_bits(v)) raise_flag(flags, SQ_FLAG_NONFINITE);
      }
    }
  }
  if constexpr (CL > 1) cluster_arrive();  // done reading the peers' shared memory
  __syncthreads();

  // ---- pass 2: codes of 8 consecutive rows x one chunk per thread, in
  // two halves of 4 rows packed as they are produced (few live registers)
  {
    const int c = tid & 3;
    const bool clamp = *clamp_flag != 0;
    float inv[EPC], dch[EPC];
#pragma unroll
    for (int e = 0; e < EPC; ++e) {
      inv[e] = inv_sm[c * EPC + e];
      dch[e] = d_sm[c * EPC + e];
    }
    for (int g = tid >> 2; g * 8 < rows; g += kThreads / 4) {
      constexpr int WPC = CODES == SQ_CODES_BF16 ? 4 : 2;  // 32-bit words per channel
      uint32_t out[EPC][WPC];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float q[4][EPC];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int r = g * 8 + h * 4 + k;
          unpack_chunk<BF16>(*reinterpret_cast<const uint4*>(strip + chunk_off(r, c)), q[k]);
          const float sj = s_sm[r];
#pragma unroll
          for (int e = 0; e < EPC; e += 2) mul2_rn(q[k][e], q[k][e + 1], sj, sj);
          if (!clamp) {
#pragma unroll
            for (int e = 0; e < EPC; e += 2) {
              quot2_rn(q[k][e], q[k][e + 1], dch[e], dch[e + 1], inv[e], inv[e + 1]);
              add2_rn(q[k][e], q[k][e + 1], kMagic, kMagic);
            }
          } else {
#pragma unroll
            for (int e = 0; e < EPC; ++e) q[k][e] = code_div_magic(q[k][e], dch[e], 127.0f);
          }
        }
#pragma unroll
        for (int e = 0; e < EPC; ++e) {
          if constexpr (CODES == SQ_CODES_BF16) {
#pragma unroll
            for (int k = 0; k < 4; k += 2) {
              float c0 = q[k][e], c1 = q[k + 1][e];
              add2_rn(c0, c1, -kMagic, -kMagic);  // exact integers
              out[e][h * 2 + k / 2] = __byte_perm(__float_as_uint(c0), __float_as_uint(c1), 0x7632);
            }
          } else {
            out[e][h] = pack4_codes(q[0][e], q[1][e], q[2][e], q[3][e]);
          }
        }
      }
      const int64_t jrow = j0 + (int64_t)g * 8;
#pragma unroll
      for (int e = 0; e < EPC; ++e) {
        const int64_t n = n0 + c * EPC + e;
        if (n >= cout) continue;
        uint8_t* dst = wq + (n * cin + jrow) * CB;
        if constexpr (CODES == SQ_CODES_BF16)
          st16(dst, make_uint4(out[e][0], out[e][1], out[e][2], out[e][3]));
        else
          st8(dst, make_uint2(out[e][0], out[e][1]));
      }
    }
  }

  if (!ok && tid == 0) {
    raise_flag(flags, SQ_FLAG_TIMEOUT);
    for (int b = 0; b < nbox; ++b) mbar_wait_bounded(&bars[b], 0, 10000000ull);
  }
  if constexpr (CL > 1) cluster_wait();  // peers may still read `part` until here
}

// Rows per CTA for cluster size cl (a multiple of the TMA box height).
int64_t rows_per_cta(int64_t cin, int cl) {
  const int64_t r = (cin + cl - 1) / cl;
  return (r + kBoxRows - 1) / kBoxRows * kBoxRows;
}

template <bool BF16, int CODES, int CL, int MINB>
sq_status launch(const CUtensorMap& map, const float* s, int64_t cin, int64_t cout, int rpc,
                 uint8_t* wq, float* w_scale, int32_t* flags, cudaStream_t st) {
  constexpr int EPC = BF16 ? 8 : 4;
  auto kern = k_fold_strip<BF16, CODES, CL, MINB>;
  const size_t smem = Layout<EPC>(rpc).total + 1024;
  static std::atomic<uint64_t> attr_done{0};
  if (!once_per_device(attr_done, [&] {
        const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)Layout<EPC>(kMaxRows).total + 1024);
        return e != cudaSuccess ? e
                                : cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
      }))
    return SQ_ERR_CUDA;
  const int64_t strips = (cout + 4 * EPC - 1) / (4 * EPC);
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
  if (cudaLaunchKernelEx(&cfg, kern, map, s, cin, cout, rpc, wq, w_scale, flags) != cudaSuccess)
    return SQ_ERR_CUDA;
  return launch_status();
}

template <bool BF16, int CODES, int MINB>
sq_status launch_cl_b(int cl, const CUtensorMap& map, const float* s, int64_t cin, int64_t cout,
                      int rpc, uint8_t* wq, float* w_scale, int32_t* flags, cudaStream_t st) {
  switch (cl) {
    case 1: return launch<BF16, CODES, 1, MINB>(map, s, cin, cout, rpc, wq, w_scale, flags, st);
    case 2: return launch<BF16, CODES, 2, MINB>(map, s, cin, cout, rpc, wq, w_scale, flags, st);
    case 4: return launch<BF16, CODES, 4, MINB>(map, s, cin, cout, rpc, wq, w_scale, flags, st);
    default: return launch<BF16, CODES, 8, MINB>(map, s, cin, cout, rpc, wq, w_scale, flags, st);
  }
}

// The three-CTA build where shared memory lets three CTAs share an SM (at
// most 1024 rows per CTA) and the grid holds at least two such waves.
// Measured on B300 (bf16 W, 1-byte codes): 4096 x 11008 54.5 -> 51.1 us,
// 8192 x 10240 98.7 -> 87.5 us (bf16 codes 60.7 -> 53.8, 110 -> 96); the
// 4096 x 4096 decode weight (512 CTAs) and CTAs of 1408 rows (two per SM by
// shared memory) were slower with it (25.2 -> 28.4, 60.1 -> 62.6 us).
template <bool BF16, int CODES>
sq_status launch_cl(int cl, const CUtensorMap& map, const float* s, int64_t cin, int64_t cout,
                    int rpc, uint8_t* wq, float* w_scale, int32_t* flags, cudaStream_t st) {
  constexpr int EPC = BF16 ? 8 : 4;
  const int64_t ctas = (cout + 4 * EPC - 1) / (4 * EPC) * cl;
  if (rpc <= 1024 && ctas >= 2 * 3 * (int64_t)sm_count())
    return launch_cl_b<BF16, CODES, 3>(cl, map, s, cin, cout, rpc, wq, w_scale, flags, st);
  return launch_cl_b<BF16, CODES, 0>(cl, map, s, cin, cout, rpc, wq, w_scale, flags, st);
}

int cluster_size(int64_t cin) {
  for (int c : {1, 2, 4, 8})
    if (rows_per_cta(cin, c) <= kMaxRows) return c;
  return 0;
}

bool applies(sq_dtype dt, int64_t cin, int64_t cout, int64_t ldw) {
  return (ldw * elem_bytes(dt)) % 16 == 0 && cin <= ((int64_t)1 << 30) &&
         cout <= ((int64_t)1 << 30) && cluster_size(cin) != 0;
}

// SQ_ERR_UNSUPPORTED when the single-pass path does not apply (the caller
// then takes the two-pass path); otherwise the launch status.
sq_status fold_single_pass(const void* w, sq_dtype dt, int64_t cin, int64_t cout, int64_t ldw,
                           const float* s, void* wq, sq_codes fmt, float* w_scale, int32_t* flags,
                           cudaStream_t st) {
  const int eb = elem_bytes(dt);
  if (!aligned16(w) || !applies(dt, cin, cout, ldw)) return SQ_ERR_UNSUPPORTED;
  const int cl = cluster_size(cin);
  const int rpc = (int)rows_per_cta(cin, cl);
  auto fn = tensor_map_encoder();
  if (!fn) return SQ_ERR_CUDA;
  CUtensorMap map;
  cuuint64_t dims[2] = {(cuuint64_t)cout, (cuuint64_t)cin};
  cuuint64_t strides[1] = {(cuuint64_t)(ldw * eb)};
  cuuint32_t box[2] = {(cuuint32_t)(kRowBytes / eb), (cuuint32_t)kBoxRows};
  cuuint32_t estr[2] = {1, 1};
  if (fn(&map, dt == SQ_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
         const_cast<void*>(w), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return SQ_ERR_CUDA;
  uint8_t* q = static_cast<uint8_t*>(wq);
  if (dt == SQ_BF16)
    return fmt == SQ_CODES_BF16
               ? launch_cl<true, SQ_CODES_BF16>(cl, map, s, cin, cout, rpc, q, w_scale, flags, st)
               : launch_cl<true, SQ_CODES_I8>(cl, map, s, cin, cout, rpc, q, w_scale, flags, st);
  return fmt == SQ_CODES_BF16
             ? launch_cl<false, SQ_CODES_BF16>(cl, map, s, cin, cout, rpc, q, w_scale, flags, st)
             : launch_cl<false, SQ_CODES_I8>(cl, map, s, cin, cout, rpc, q, w_scale, flags, st);
}

}  // namespace strip

}  // namespace

int fold_kernel_count(sq_dtype dt, int64_t cin, int64_t cout, int64_t ldw) {
  return strip::applies(dt, cin, cout, ldw) ? 1 : 3;
}

sq_status fold_quantize_weight(const void* w, sq_dtype dt, int64_t cin, int64_t cout, int64_t ldw,
                               const float* s, void* wq, sq_codes fmt, float* w_scale,
                               int32_t* flags, void* workspace, cudaStream_t st) {
  {
    const sq_status r = strip::fold_single_pass(w, dt, cin, cout, ldw, s, wq, fmt, w_scale, flags, st);
    if (r != SQ_ERR_UNSUPPORTED) return r;
  }
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

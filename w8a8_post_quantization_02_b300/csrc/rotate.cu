// Smooth Rotation: smoothing, then a Hadamard rotation, then low-bit codes.
//
// Source: pith.science review of arXiv 2506.01967 ("Smooth Rotation"),
// key_machinery: scale activations by S^-1 and weights by S, then multiply
// both by the same Hadamard matrix R with entries +-1/sqrt(d), so the
// linear map is unchanged; core_discovery: 4-bit symmetric round-to-nearest
// codes on both operands (W4A4).
//
// k_rotate_rows quantizes rows: each CTA takes rows r = blockIdx.x,
// + gridDim.x, ...; a row (d = 2^L elements) is held in registers, thread
// t owning the 16-byte vectors v = t + i * blockDim.x.  The unnormalized
// fast Walsh-Hadamard transform runs its stages in ascending order
// h = 1, 2, 4, ... exactly as the definition (butterfly (a, b) ->
// (a + b, a - b) in binary32): stages inside a vector in registers, across
// lanes by warp shuffles, across warps through shared memory, across a
// thread's vectors in registers.  The row's max|Z| gives the scale
// d = RN(max|Z| / qmax) and codes clamp(rne(RN(Z / d)), -qmax, qmax).
// The 1/d_len of R R^T = H H^T / d_len rides on the activation scale as the
// exact power of two 2^-L.  The same kernel quantizes the rows of the
// transposed, folded weight (k_fold_transpose), one row per output channel.
#include "sq_async.cuh"

namespace sq {
namespace {
using namespace async;

template <bool BF16>
SQ_DEVINL void unpack_vec(uint4 v, float* f) {
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

// The butterfly for the element whose index has bit h clear (lo = true):
// a + b; for its partner: a - b, with a the element whose bit is clear.
SQ_DEVINL float butterfly(float mine, float partner, bool lo) {
  return lo ? __fadd_rn(mine, partner) : __fsub_rn(partner, mine);
}

// One row per CTA iteration; blockDim.x threads (a multiple of 32, at most
// 1024), VPT vectors of E elements each per thread.  ROTATE requires
// nvec == blockDim.x * VPT (the whole power-of-two row in registers).
template <bool BF16, int CODES, int VPT, bool ROTATE>
__global__ void __launch_bounds__(1024) k_rotate_rows(const uint8_t* __restrict__ x, int64_t rows,
                                                      int nvec, int64_t ld_bytes,
                                                      const float* __restrict__ col_scale,
                                                      float qmax, int log2_len,
                                                      uint8_t* __restrict__ q,
                                                      float* __restrict__ row_scale,
                                                      int32_t* flags) {
  constexpr int E = BF16 ? 8 : 4;
  constexpr int CB = CODES == SQ_CODES_BF16 ? 2 : 1;
  extern __shared__ __align__(16) float row_sm[];  // [nvec * E] (cross-warp stages), then [32] maxima
  uint32_t* red = reinterpret_cast<uint32_t*>(row_sm + (ROTATE ? nvec * E : 0));
  const int nt = blockDim.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nw = nt >> 5;
  const int64_t rowlen = (int64_t)nvec * E;

  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint8_t* src = x + r * ld_bytes;
    float f[VPT][E];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = tid + i * nt;
      if (v < nvec) {
        unpack_vec<BF16>(ld_stream16(src + (int64_t)v * 16), f[i]);
        if (col_scale) {
#pragma unroll
          for (int e = 0; e < E; e += 4) {
            const uint4 s4 = ld_ro16(col_scale + (int64_t)v * E + e);
            mul2_rn(f[i][e], f[i][e + 1], __uint_as_float(s4.x), __uint_as_float(s4.y));
            mul2_rn(f[i][e + 2], f[i][e + 3], __uint_as_float(s4.z), __uint_as_float(s4.w));
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) f[i][e] = 0.0f;
      }
    }
    if constexpr (ROTATE) {
      // stages inside a vector: h = 1, 2 (, 4)
#pragma unroll
      for (int h = 1; h < E; h <<= 1)
#pragma unroll
        for (int i = 0; i < VPT; ++i)
#pragma unroll
          for (int e = 0; e < E; ++e)
            if ((e & h) == 0) {
              const float a = f[i][e], b = f[i][e + h];
              f[i][e] = __fadd_rn(a, b);
              f[i][e + h] = __fsub_rn(a, b);
            }
      // across lanes: h = E * m, m = 1 .. 16
#pragma unroll
      for (int m = 1; m < 32; m <<= 1) {
        const bool lo = (lane & m) == 0;
#pragma unroll
        for (int i = 0; i < VPT; ++i)
#pragma unroll
          for (int e = 0; e < E; ++e) f[i][e] = butterfly(f[i][e], __shfl_xor_sync(0xFFFFFFFFu, f[i][e], m), lo);
      }
      // across warps: h = 32 E * m, through shared memory
      for (int m = 1; m < nw; m <<= 1) {
#pragma unroll
        for (int i = 0; i < VPT; ++i)
#pragma unroll
          for (int e = 0; e < E; ++e) row_sm[(int64_t)(tid + i * nt) * E + e] = f[i][e];
        __syncthreads();
        const bool lo = (warp & m) == 0;
        const int ptid = tid ^ (m << 5);
#pragma unroll
        for (int i = 0; i < VPT; ++i)
#pragma unroll
          for (int e = 0; e < E; ++e)
            f[i][e] = butterfly(f[i][e], row_sm[(int64_t)(ptid + i * nt) * E + e], lo);
        __syncthreads();
      }
      // across a thread's vectors: h = nt * E * m
#pragma unroll
      for (int m = 1; m < VPT; m <<= 1)
#pragma unroll
        for (int i = 0; i < VPT; ++i)
          if ((i & m) == 0)
#pragma unroll
            for (int e = 0; e < E; ++e) {
              const float a = f[i][e], b = f[i + m][e];
              f[i][e] = __fadd_rn(a, b);
              f[i + m][e] = __fsub_rn(a, b);
            }
    }
    // row maximum (NaN sorts above +inf as bits)
    uint32_t mb = 0u;
#pragma unroll
    for (int i = 0; i < VPT; ++i)
#pragma unroll
      for (int e = 0; e < E; ++e) mb = max(mb, __float_as_uint(f[i][e]) & 0x7FFFFFFFu);
    mb = __reduce_max_sync(0xFFFFFFFFu, mb);
    if (lane == 0) red[warp] = mb;
    __syncthreads();
    uint32_t amax = 0u;
    for (int w = 0; w < nw; ++w) amax = max(amax, red[w]);
    __syncthreads();  // red is rewritten by the next row
    const float am = __uint_as_float(amax);
    const float d = (amax == 0u) ? 1.0f : __fdiv_rn(am, qmax);
    const float inv = __fdiv_rn(1.0f, d);
    const bool fast = fast_quotient_ok(amax);  // then no code leaves [-qmax, qmax]
    if (tid == 0) {
      row_scale[r] = log2_len ? ldexpf(d, -log2_len) : d;
      if (!finite_bits(amax)) raise_flag(flags, SQ_FLAG_NONFINITE);
    }
    uint8_t* qrow = q + r * rowlen * CB;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = tid + i * nt;
      if (v >= nvec) continue;
      float c[E];
      if (fast) {
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          float a = f[i][e], b = f[i][e + 1];
          quot2_rn(a, b, d, d, inv, inv);
          add2_rn(a, b, kMagic, kMagic);
          c[e] = a;
          c[e + 1] = b;
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) c[e] = code_div_magic(f[i][e], d, qmax);
      }
      if constexpr (CODES == SQ_CODES_BF16) {
        uint32_t w[E / 2];
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          float c0 = c[e], c1 = c[e + 1];
          add2_rn(c0, c1, -kMagic, -kMagic);  // exact integers
          w[e / 2] = __byte_perm(__float_as_uint(c0), __float_as_uint(c1), 0x7632);
        }
        if constexpr (E == 8)
          st16(qrow + (size_t)v * 16, make_uint4(w[0], w[1], w[2], w[3]));
        else
          st8(qrow + (size_t)v * 8, make_uint2(w[0], w[1]));
      } else {
        if constexpr (E == 8)
          st8(qrow + (size_t)v * 8,
              make_uint2(pack4_codes(c[0], c[1], c[2], c[3]), pack4_codes(c[4], c[5], c[6], c[7])));
        else
          *reinterpret_cast<uint32_t*>(qrow + (size_t)v * 4) = pack4_codes(c[0], c[1], c[2], c[3]);
      }
    }
  }
}

// Rows of d = 2^L elements, L in [10, 14], on T = d / 32 threads that each
// hold 32 elements; the transform's stages run in registers in three phases
// of at most five index bits, with the row transposed through shared memory
// between phases (two copies of the row per row, instead of a shuffle for
// every element at each lane stage and a copy at each warp stage):
//   phase 1: bits 0-4 in the thread, thread t holds elements 32 t .. +31;
//   phase 2: bits 5-9, thread u = (bits 10.. , bits 0-4) holds
//            (u >> 5) << 10 | v << 5 | (u & 31), v = 0 .. 31;
//   phase 3 (L > 10): bits 10 .. L-1 (n3 = L - 10 of them) and bits
//            0 .. J-1 (J = 5 - n3), thread w = bits J .. 9 holds
//            h << 10 | w << J | j, so each group of 2^J codes it writes is
//            contiguous.
// Every stage is the same butterfly in the same ascending order h = 1, 2,
// 4, ... as the row-per-vector kernel above, so the results are the same
// bit for bit.  Shared-memory rows are padded by 4 floats every 32
// (index i at i + 4 (i / 32)): both transposes are conflict-free and the
// phase-1 writes and phase-3 reads stay 16-byte vectors.
SQ_DEVINL int pad_idx(int i) { return i + ((i >> 5) << 2); }

template <int N>
SQ_DEVINL void stages_in_regs(float (&f)[N], int first_h, int last_h) {
#pragma unroll
  for (int h = 1; h < N; h <<= 1) {
    if (h < first_h || h > last_h) continue;
#pragma unroll
    for (int k = 0; k < N; ++k)
      if ((k & h) == 0) {
        const float a = f[k], b = f[k + h];
        f[k] = __fadd_rn(a, b);
        f[k + h] = __fsub_rn(a, b);
      }
  }
}

// CTAs per SM the kernel is built for (the shared-memory rows allow this
// many; more registers per thread would leave fewer resident)
constexpr int rows_t_min_blocks(int L) { return L >= 14 ? 1 : L == 13 ? 3 : L == 12 ? 6 : 8; }

template <bool BF16, int CODES, int L>
__global__ void __launch_bounds__(1 << (L - 5), rows_t_min_blocks(L)) k_rotate_rows_t(const uint8_t* __restrict__ x, int64_t rows,
                                                                int64_t ld_bytes,
                                                                const float* __restrict__ col_scale,
                                                                float qmax, int log2_len,
                                                                uint8_t* __restrict__ q,
                                                                float* __restrict__ row_scale,
                                                                int32_t* flags) {
  constexpr int D = 1 << L, T = D >> 5, NW = T / 32;
  constexpr int P = D + (D >> 3);            // padded floats per row copy
  constexpr int N3 = L > 10 ? L - 10 : 0;    // phase-3 bits above 9
  constexpr int J = 5 - N3;                  // phase-3 low bits (a contiguous group of 2^J)
  constexpr int CB = CODES == SQ_CODES_BF16 ? 2 : 1;
  extern __shared__ __align__(16) float sm_rt[];
  float* buf0 = sm_rt;
  float* buf1 = sm_rt + P;
  uint32_t* red = reinterpret_cast<uint32_t*>(sm_rt + 2 * P);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // this thread's 64 (bf16) or 128 (fp32) bytes of a row; the next row's
  // are loaded while the current one is transformed.  Each load instruction
  // covers 16 of every thread's 64 or 128 bytes, so a warp's four or eight
  // loads share their 32-byte sectors: rows of 2^13 and more keep them in L1
  // (measured on B300, 8192 x 8192: 134 us against 153 us streaming past L1),
  // shorter rows stream past it (2048 x 4096: 25 us against 45 us, their
  // six or more CTAs per SM leaving L1 too little room beside shared memory)
  constexpr int NV = BF16 ? 4 : 8;
  auto ld_row = [](const uint8_t* p) {
    if constexpr (L >= 13) return ld_ro16(p);
    else return ld_stream16(p);
  };
  uint4 raw[NV];
  const int64_t tid_off = (int64_t)tid * 32 * (BF16 ? 2 : 4);
  if (blockIdx.x < rows) {
#pragma unroll
    for (int q4 = 0; q4 < NV; ++q4) raw[q4] = ld_row(x + (int64_t)blockIdx.x * ld_bytes + tid_off + 16 * q4);
  }
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    // phase 1: elements 32 tid .. 32 tid + 31, scaled by the column factors
    float f[32];
#pragma unroll
    for (int q4 = 0; q4 < NV; ++q4) unpack_vec<BF16>(raw[q4], f + q4 * (BF16 ? 8 : 4));
    if (r + gridDim.x < rows) {
#pragma unroll
      for (int q4 = 0; q4 < NV; ++q4) raw[q4] = ld_row(x + (r + gridDim.x) * ld_bytes + tid_off + 16 * q4);
    }
    if (col_scale) {
#pragma unroll
      for (int k = 0; k < 32; k += 4) {
        const uint4 s4 = ld_ro16(col_scale + (int64_t)tid * 32 + k);
        mul2_rn(f[k], f[k + 1], __uint_as_float(s4.x), __uint_as_float(s4.y));
        mul2_rn(f[k + 2], f[k + 3], __uint_as_float(s4.z), __uint_as_float(s4.w));
      }
    }
    stages_in_regs<32>(f, 1, 16);
    {
      float* dst = buf0 + pad_idx(tid * 32);
#pragma unroll
      for (int k = 0; k < 32; k += 4) *reinterpret_cast<float4*>(dst + k) = make_float4(f[k], f[k + 1], f[k + 2], f[k + 3]);
    }
    __syncthreads();
    // phase 2
    const int lo5 = tid & 31, hi = tid >> 5;
#pragma unroll
    for (int v = 0; v < 32; ++v) f[v] = buf0[pad_idx((hi << 10) | (v << 5) | lo5)];
    stages_in_regs<32>(f, 1, 16);
    if constexpr (L > 10) {
#pragma unroll
      for (int v = 0; v < 32; ++v) buf1[pad_idx((hi << 10) | (v << 5) | lo5)] = f[v];
      __syncthreads();
      // phase 3: f[h * 2^J + j] is element h << 10 | tid << J | j
#pragma unroll
      for (int h = 0; h < (1 << N3); ++h) {
        const float* s3 = buf1 + pad_idx((h << 10) | (tid << J));
        if constexpr (J >= 2) {
#pragma unroll
          for (int j = 0; j < (1 << J); j += 4) {
            const float4 t4 = *reinterpret_cast<const float4*>(s3 + j);
            f[h * (1 << J) + j] = t4.x;
            f[h * (1 << J) + j + 1] = t4.y;
            f[h * (1 << J) + j + 2] = t4.z;
            f[h * (1 << J) + j + 3] = t4.w;
          }
        } else {
          const float2 t2 = *reinterpret_cast<const float2*>(s3);
          f[h * 2] = t2.x;
          f[h * 2 + 1] = t2.y;
        }
      }
      stages_in_regs<32>(f, 1 << J, 16);
    }
    // row maximum (NaN sorts above +inf as bits)
    uint32_t mb = 0u;
#pragma unroll
    for (int k = 0; k < 32; ++k) mb = max(mb, __float_as_uint(f[k]) & 0x7FFFFFFFu);
    mb = __reduce_max_sync(0xFFFFFFFFu, mb);
    if (lane == 0) red[warp] = mb;
    __syncthreads();
    uint32_t amax = 0u;
#pragma unroll
    for (int w = 0; w < NW; ++w) amax = max(amax, red[w]);
    const float am = __uint_as_float(amax);
    const float d = (amax == 0u) ? 1.0f : __fdiv_rn(am, qmax);
    const float inv = __fdiv_rn(1.0f, d);
    const bool fast = fast_quotient_ok(amax);  // then no code leaves [-qmax, qmax]
    if (tid == 0) {
      row_scale[r] = log2_len ? ldexpf(d, -log2_len) : d;
      if (!finite_bits(amax)) raise_flag(flags, SQ_FLAG_NONFINITE);
    }
    float (&c)[32] = f;  // the codes (as magic-number floats) replace the values
    if (fast) {
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        float a = f[k], b = f[k + 1];
        quot2_rn(a, b, d, d, inv, inv);
        add2_rn(a, b, kMagic, kMagic);
        c[k] = a;
        c[k + 1] = b;
      }
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k) c[k] = code_div_magic(f[k], d, qmax);
    }
    // codes: groups of G contiguous elements starting at element e0(g)
    constexpr int G = L > 10 ? (1 << J) : 1;
    uint8_t* qrow = q + r * (int64_t)D * CB;
#pragma unroll
    for (int g = 0; g < 32 / G; ++g) {
      const int e0 = L > 10 ? ((g << 10) | (tid << J)) : ((g << 5) | lo5);
      uint8_t* dst = qrow + (int64_t)e0 * CB;
      if constexpr (CODES == SQ_CODES_BF16) {
        if constexpr (G == 1) {
          float c0 = c[g], c1 = 0.0f;
          add2_rn(c0, c1, -kMagic, -kMagic);
          *reinterpret_cast<uint16_t*>(dst) = (uint16_t)(__float_as_uint(c0) >> 16);
        } else {
          uint32_t w[G / 2];
#pragma unroll
          for (int e = 0; e < G; e += 2) {
            float c0 = c[g * G + e], c1 = c[g * G + e + 1];
            add2_rn(c0, c1, -kMagic, -kMagic);  // exact integers
            w[e / 2] = __byte_perm(__float_as_uint(c0), __float_as_uint(c1), 0x7632);
          }
          if constexpr (G == 2) *reinterpret_cast<uint32_t*>(dst) = w[0];
          else if constexpr (G == 4) st8(dst, make_uint2(w[0], w[1]));
#pragma unroll
          for (int e = 0; G >= 8 && e < G / 2; e += 4) st16(dst + 4 * e, make_uint4(w[e], w[e + 1], w[e + 2], w[e + 3]));
        }
      } else {
        if constexpr (G < 4) {
#pragma unroll
          for (int e = 0; e < G; ++e) dst[e] = (uint8_t)(__float_as_uint(c[g * G + e]) & 0xFFu);
        } else {
          uint32_t w[G / 4];
#pragma unroll
          for (int e = 0; e < G; e += 4)
            w[e / 4] = pack4_codes(c[g * G + e], c[g * G + e + 1], c[g * G + e + 2], c[g * G + e + 3]);
          if constexpr (G == 4) *reinterpret_cast<uint32_t*>(dst) = w[0];
          else if constexpr (G == 8) st8(dst, make_uint2(w[0], w[1]));
          else st16(dst, make_uint4(w[0], w[1], w[2], w[3]));
        }
      }
    }
  }
}

template <bool BF16, int CODES, int L>
sq_status launch_rows_t(const uint8_t* x, int64_t rows, int64_t ld_bytes, const float* col_scale, int qmax,
                        int log2_len, uint8_t* q, float* row_scale, int32_t* flags, cudaStream_t st) {
  auto kern = k_rotate_rows_t<BF16, CODES, L>;
  constexpr int D = 1 << L;
  const size_t smem = (size_t)2 * (D + D / 8) * 4 + 32 * 4;
  static std::atomic<uint64_t> attr_done{0};
  if (!once_per_device(attr_done, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      }))
    return SQ_ERR_CUDA;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, D / 32, smem) != cudaSuccess) return SQ_ERR_CUDA;
  occ = std::max(1, std::min(occ, 8));
  const int64_t grid = std::min<int64_t>(rows, (int64_t)sm_count() * occ);
  kern<<<(unsigned)grid, D / 32, smem, st>>>(x, rows, ld_bytes, col_scale, (float)qmax, log2_len, q, row_scale,
                                            flags);
  return launch_status();
}

// wt[n, j] = RN(s[j] * W[j, n]) (s may be null: W[j, n]), fp32, 32 x 32 tiles.
template <bool BF16>
__global__ void __launch_bounds__(256) k_fold_transpose(const uint8_t* __restrict__ w, int64_t cin,
                                                        int64_t cout, int64_t ldw_bytes,
                                                        const float* __restrict__ s,
                                                        float* __restrict__ wt) {
  __shared__ float tile[32][33];
  const int64_t j0 = (int64_t)blockIdx.y * 32, n0 = (int64_t)blockIdx.x * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 8 rows of 32
  for (int k = ty; k < 32; k += 8) {
    const int64_t j = j0 + k, n = n0 + tx;
    float v = 0.0f;
    if (j < cin && n < cout) {
      const uint8_t* p = w + j * ldw_bytes + n * (BF16 ? 2 : 4);
      v = BF16 ? __uint_as_float((uint32_t)*reinterpret_cast<const uint16_t*>(p) << 16)
               : *reinterpret_cast<const float*>(p);
      if (s) v = __fmul_rn(s[j], v);
    }
    tile[k][tx] = v;
  }
  __syncthreads();
  for (int k = ty; k < 32; k += 8) {
    const int64_t n = n0 + k, j = j0 + tx;
    if (n < cout && j < cin) wt[n * cin + j] = tile[tx][k];
  }
}

template <bool BF16, int CODES, int VPT, bool ROTATE>
sq_status launch_rows(const uint8_t* x, int64_t rows, int nvec, int64_t ld_bytes,
                      const float* col_scale, int qmax, int log2_len, int nt, uint8_t* q,
                      float* row_scale, int32_t* flags, cudaStream_t st) {
  auto kern = k_rotate_rows<BF16, CODES, VPT, ROTATE>;
  const size_t smem = (ROTATE ? (size_t)nvec * (BF16 ? 8 : 4) * 4 : 0) + 32 * 4;
  static std::atomic<uint64_t> attr_done{0};
  if (!once_per_device(attr_done, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
      }))
    return SQ_ERR_CUDA;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, nt, smem) != cudaSuccess) return SQ_ERR_CUDA;
  occ = std::max(1, std::min(occ, 8));
  const int64_t grid = std::min<int64_t>(rows, (int64_t)sm_count() * occ);
  kern<<<(unsigned)grid, nt, smem, st>>>(x, rows, nvec, ld_bytes, col_scale, (float)qmax, log2_len, q,
                                         row_scale, flags);
  return launch_status();
}

// pow2_shift: the row scales are multiplied by 2^-pow2_shift (exactly).
template <bool BF16, int CODES>
sq_status rows_dispatch(const uint8_t* x, int64_t rows, int64_t len, int64_t ld_bytes,
                        const float* col_scale, bool rotate, int qmax, int pow2_shift, uint8_t* q,
                        float* row_scale, int32_t* flags, cudaStream_t st) {
  constexpr int E = BF16 ? 8 : 4;
  const int nvec = (int)(len / E);
  const int log2_len = pow2_shift;
  // without the rotation: the fewest threads (>= 32) holding the row in 1,
  // 2 or 4 vectors each
  int vpt = 1;
  while (vpt < 4 && (nvec + vpt - 1) / vpt > 1024) vpt *= 2;
  int nt = (nvec + vpt - 1) / vpt;
  if (nt > 1024) return SQ_ERR_UNSUPPORTED;
  nt = (nt + 31) / 32 * 32;
  if (rotate) {
    // a power-of-two row, whole warps of whole vectors, as many vectors per
    // thread as allowed (4): every factor of 2 in the vectors per thread
    // moves one transform stage from shared memory (two block barriers)
    // into registers, and smaller blocks let more rows share an SM
    vpt = 4;
    while (vpt > 1 && nvec / vpt < 32) vpt /= 2;
    nt = nvec / vpt;
    if (nt < 32 || nt > 1024 || nt * vpt != nvec) return SQ_ERR_UNSUPPORTED;
  }
  if (rotate) {
    // rows of 2^10 .. 2^14 elements: the three-phase kernel (transposes
    // through shared memory instead of shuffle and shared-memory stages)
    int lg = 0;
    while ((int64_t)1 << lg < len) ++lg;
    switch (lg) {
      case 10: return launch_rows_t<BF16, CODES, 10>(x, rows, ld_bytes, col_scale, qmax, log2_len, q, row_scale, flags, st);
      case 11: return launch_rows_t<BF16, CODES, 11>(x, rows, ld_bytes, col_scale, qmax, log2_len, q, row_scale, flags, st);
      case 12: return launch_rows_t<BF16, CODES, 12>(x, rows, ld_bytes, col_scale, qmax, log2_len, q, row_scale, flags, st);
      case 13: return launch_rows_t<BF16, CODES, 13>(x, rows, ld_bytes, col_scale, qmax, log2_len, q, row_scale, flags, st);
      case 14: return launch_rows_t<BF16, CODES, 14>(x, rows, ld_bytes, col_scale, qmax, log2_len, q, row_scale, flags, st);
      default: break;
    }
    switch (vpt) {
      case 1: return launch_rows<BF16, CODES, 1, true>(x, rows, nvec, ld_bytes, col_scale, qmax, log2_len, nt, q, row_scale, flags, st);
      case 2: return launch_rows<BF16, CODES, 2, true>(x, rows, nvec, ld_bytes, col_scale, qmax, log2_len, nt, q, row_scale, flags, st);
      default: return launch_rows<BF16, CODES, 4, true>(x, rows, nvec, ld_bytes, col_scale, qmax, log2_len, nt, q, row_scale, flags, st);
    }
  }
  switch (vpt) {
    case 1: return launch_rows<BF16, CODES, 1, false>(x, rows, nvec, ld_bytes, col_scale, qmax, log2_len, nt, q, row_scale, flags, st);
    case 2: return launch_rows<BF16, CODES, 2, false>(x, rows, nvec, ld_bytes, col_scale, qmax, log2_len, nt, q, row_scale, flags, st);
    default: return launch_rows<BF16, CODES, 4, false>(x, rows, nvec, ld_bytes, col_scale, qmax, log2_len, nt, q, row_scale, flags, st);
  }
}

}  // namespace

bool rotate_len_ok(int64_t len, sq_dtype dt, bool rotate) {
  const int E = dt == SQ_BF16 ? 8 : 4;
  if (len % E != 0 || len / E > 4096) return false;
  if (!rotate) return true;
  return (len & (len - 1)) == 0 && len >= 32 * E;
}

sq_status rotate_quant_rows(const void* x, sq_dtype dt, int64_t rows, int64_t len, int64_t ld,
                            const float* col_scale, bool rotate, int qmax, int pow2_shift, void* q,
                            sq_codes fmt, float* row_scale, int32_t* flags, cudaStream_t st) {
  const uint8_t* xb = static_cast<const uint8_t*>(x);
  uint8_t* qb = static_cast<uint8_t*>(q);
  const int64_t ldb = ld * elem_bytes(dt);
  if (dt == SQ_BF16)
    return fmt == SQ_CODES_BF16
               ? rows_dispatch<true, SQ_CODES_BF16>(xb, rows, len, ldb, col_scale, rotate, qmax, pow2_shift, qb, row_scale, flags, st)
               : rows_dispatch<true, SQ_CODES_I8>(xb, rows, len, ldb, col_scale, rotate, qmax, pow2_shift, qb, row_scale, flags, st);
  return fmt == SQ_CODES_BF16
             ? rows_dispatch<false, SQ_CODES_BF16>(xb, rows, len, ldb, col_scale, rotate, qmax, pow2_shift, qb, row_scale, flags, st)
             : rows_dispatch<false, SQ_CODES_I8>(xb, rows, len, ldb, col_scale, rotate, qmax, pow2_shift, qb, row_scale, flags, st);
}

sq_status fold_transpose(const void* w, sq_dtype dt, int64_t cin, int64_t cout, int64_t ldw,
                         const float* s, float* wt, cudaStream_t st) {
  const dim3 grid((unsigned)((cout + 31) / 32), (unsigned)((cin + 31) / 32));
  const uint8_t* wb = static_cast<const uint8_t*>(w);
  const int64_t ldb = ldw * elem_bytes(dt);
  if (dt == SQ_BF16)
    k_fold_transpose<true><<<grid, 256, 0, st>>>(wb, cin, cout, ldb, s, wt);
  else
    k_fold_transpose<false><<<grid, 256, 0, st>>>(wb, cin, cout, ldb, s, wt);
  return launch_status();
}

}  // namespace sq

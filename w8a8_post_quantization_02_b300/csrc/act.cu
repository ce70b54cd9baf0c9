// Step 4: runtime X * diag(s)^-1 fused with dynamic per-token INT8
// quantization.
//
// Sources: first page ("Move activation scale without changing the real
// linear map"), paragraph 3: the explicit runtime scaling step that
// multiplies activations by S^-1; learn-kernels.com "Quantization",
// paragraph 2: activations are quantized to INT8.
//
// A group of 32-256 threads owns one token row at a time.  The row is read
// once from HBM with 16-byte streaming loads and kept in registers (up to
// 16 vectors per thread), scaled by s_inv (L1-resident), reduced to the
// row's max|X'| (integer max on |x| bits, so NaN/Inf are caught), and
// quantized from the registers.  HBM traffic per element: one read of X plus one write of the
// code, and 4 bytes per token for the scale.
#include "sq_common.cuh"

namespace sq {
namespace {

template <bool BF16>
struct ActVec;
template <>
struct ActVec<true> {
  static constexpr int kElems = 8;
};
template <>
struct ActVec<false> {
  static constexpr int kElems = 4;
};

template <bool BF16>
SQ_DEVINL void unpack(uint4 v, float (&f)[ActVec<BF16>::kElems]) {
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

// Max of a u32 over the TPR threads of the block (all get the result).
template <int TPR>
SQ_DEVINL uint32_t row_max_u32(uint32_t v, uint32_t* red) {
  v = __reduce_max_sync(0xFFFFFFFFu, v);
  if constexpr (TPR == 32) {
    return v;
  } else {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    uint32_t r = red[lane < (TPR / 32) ? lane : 0];
    r = __reduce_max_sync(0xFFFFFFFFu, r);
    __syncthreads();  // red is reused by the next row
    return r;
  }
}

template <bool BF16>
SQ_DEVINL void scale_vec(uint4 raw, const float* si_ptr, float (&f)[ActVec<BF16>::kElems]) {
  constexpr int E = ActVec<BF16>::kElems;
  unpack<BF16>(raw, f);
#pragma unroll
  for (int q = 0; q < E; q += 4) {
    const uint4 si = ld_ro16(si_ptr + q);
    f[q + 0] = __fmul_rn(f[q + 0], __uint_as_float(si.x));
    f[q + 1] = __fmul_rn(f[q + 1], __uint_as_float(si.y));
    f[q + 2] = __fmul_rn(f[q + 2], __uint_as_float(si.z));
    f[q + 3] = __fmul_rn(f[q + 3], __uint_as_float(si.w));
  }
}

// A block of TPR threads owns one token row at a time (grid-stride over
// rows).  Each thread keeps VPT raw 16-byte vectors of X in registers:
// pass 1 forms X' = X * s_inv and the row's max|X'|, pass 2 recomputes X'
// from the registers and writes the codes, so X is read from HBM once.
template <bool BF16, int VPT, int CODES, int TPR>
__global__ void __launch_bounds__(TPR) k_quant_act(const uint8_t* __restrict__ x, int64_t tokens,
                                                   int64_t cin, int64_t ldx_bytes,
                                                   const float* __restrict__ s_inv,
                                                   uint8_t* __restrict__ xq,
                                                   float* __restrict__ x_scale, int32_t* flags) {
  constexpr int E = ActVec<BF16>::kElems;
  constexpr int CB = CODES == SQ_CODES_BF16 ? 2 : 1;  // bytes per code
  __shared__ uint32_t red[TPR / 32];
  const int64_t nvec = cin / E;
  for (int64_t t = blockIdx.x; t < tokens; t += gridDim.x) {
    const uint8_t* row = x + t * ldx_bytes;
    uint4 raw[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int64_t v = threadIdx.x + (int64_t)i * TPR;
      raw[i] = v < nvec ? ld_stream16(row + v * 16) : make_uint4(0u, 0u, 0u, 0u);
    }
    uint32_t amax = 0u;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int64_t v = threadIdx.x + (int64_t)i * TPR;
      if (v < nvec) {
        float f[E];
        scale_vec<BF16>(raw[i], s_inv + v * E, f);
#pragma unroll
        for (int e = 0; e < E; ++e) amax = max(amax, abs_bits(f[e]));
      }
    }
    amax = row_max_u32<TPR>(amax, red);
    float d, inv;
    scale_and_inverse(__uint_as_float(amax), d, inv);
    if (threadIdx.x == 0) {
      x_scale[t] = d;
      if (!finite_bits(amax)) raise_flag(flags, SQ_FLAG_NONFINITE);
    }
    uint8_t* qrow = xq + t * cin * CB;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int64_t v = threadIdx.x + (int64_t)i * TPR;
      if (v >= nvec) continue;
      float f[E], m[E];
      scale_vec<BF16>(raw[i], s_inv + v * E, f);
#pragma unroll
      for (int e = 0; e < E; ++e) m[e] = code_magic(f[e], inv);
      if constexpr (CODES == SQ_CODES_BF16) {
        if constexpr (E == 8) {
          st16(qrow + v * 16, make_uint4(pack2_bf16codes(m[0], m[1]), pack2_bf16codes(m[2], m[3]),
                                         pack2_bf16codes(m[4], m[5]), pack2_bf16codes(m[6], m[7])));
        } else {
          st8(qrow + v * 8, make_uint2(pack2_bf16codes(m[0], m[1]), pack2_bf16codes(m[2], m[3])));
        }
      } else {
        if constexpr (E == 8) {
          st8(qrow + v * 8, make_uint2(pack4_codes(m[0], m[1], m[2], m[3]),
                                       pack4_codes(m[4], m[5], m[6], m[7])));
        } else {
          *reinterpret_cast<uint32_t*>(qrow + v * 4) = pack4_codes(m[0], m[1], m[2], m[3]);
        }
      }
    }
  }
}

template <bool BF16, int CODES, int TPR>
sq_status launch_act_tpr(int vpt, const uint8_t* x, int64_t tokens, int64_t cin, int64_t ldx_bytes,
                         const float* s_inv, uint8_t* xq, float* x_scale, int32_t* flags,
                         cudaStream_t st) {
  // up to 2048 resident threads and 32 resident blocks per SM
  const int per_sm = std::min(32, 2048 / TPR);
  const int64_t grid = std::min<int64_t>(tokens, (int64_t)sm_count() * per_sm);
#define SQ_ACT_CASE(V)                                                                             \
  case V:                                                                                          \
    k_quant_act<BF16, V, CODES, TPR><<<(unsigned)grid, TPR, 0, st>>>(x, tokens, cin, ldx_bytes,     \
                                                                     s_inv, xq, x_scale, flags);   \
    break;
  switch (vpt) {
    SQ_ACT_CASE(1)
    SQ_ACT_CASE(2)
    SQ_ACT_CASE(4)
    SQ_ACT_CASE(8)
    SQ_ACT_CASE(12)
    SQ_ACT_CASE(16)
    default:
      return SQ_ERR_UNSUPPORTED;
  }
#undef SQ_ACT_CASE
  return launch_status();
}

int round_vpt(int64_t v) {
  for (int c : {1, 2, 4, 8, 12, 16})
    if (v <= c) return c;
  return 0;
}

template <bool BF16, int CODES>
sq_status launch_act_codes(int64_t nvec, const uint8_t* x, int64_t tokens, int64_t cin,
                           int64_t ldx_bytes, const float* s_inv, uint8_t* xq, float* x_scale,
                           int32_t* flags, cudaStream_t st) {
  // the narrowest row group (one warp when it fits) whose threads hold the
  // row in at most 16 vectors each
  if (nvec <= 32 * 16)
    return launch_act_tpr<BF16, CODES, 32>(round_vpt((nvec + 31) / 32), x, tokens, cin, ldx_bytes,
                                           s_inv, xq, x_scale, flags, st);
  if (nvec <= 64 * 16)
    return launch_act_tpr<BF16, CODES, 64>(round_vpt((nvec + 63) / 64), x, tokens, cin, ldx_bytes,
                                           s_inv, xq, x_scale, flags, st);
  if (nvec <= 128 * 16)
    return launch_act_tpr<BF16, CODES, 128>(round_vpt((nvec + 127) / 128), x, tokens, cin,
                                            ldx_bytes, s_inv, xq, x_scale, flags, st);
  return launch_act_tpr<BF16, CODES, 256>(round_vpt((nvec + 255) / 256), x, tokens, cin, ldx_bytes,
                                          s_inv, xq, x_scale, flags, st);
}

}  // namespace

// Largest Cin held in registers: 16 vectors x 256 threads x (8 bf16 | 4 f32).
int64_t quant_act_max_cin(sq_dtype dt) { return (int64_t)16 * 256 * (dt == SQ_BF16 ? 8 : 4); }

sq_status quant_act(const void* x, sq_dtype dt, int64_t tokens, int64_t cin, int64_t ldx,
                    const float* s_inv, void* xq, sq_codes fmt, float* x_scale, int32_t* flags,
                    cudaStream_t st) {
  const bool bf16 = dt == SQ_BF16;
  const int64_t nvec = cin / (bf16 ? 8 : 4);
  const uint8_t* xb = static_cast<const uint8_t*>(x);
  uint8_t* qb = static_cast<uint8_t*>(xq);
  const int64_t ldb = ldx * elem_bytes(dt);
  if (bf16) {
    return fmt == SQ_CODES_BF16
               ? launch_act_codes<true, SQ_CODES_BF16>(nvec, xb, tokens, cin, ldb, s_inv, qb, x_scale, flags, st)
               : launch_act_codes<true, SQ_CODES_I8>(nvec, xb, tokens, cin, ldb, s_inv, qb, x_scale, flags, st);
  }
  return fmt == SQ_CODES_BF16
             ? launch_act_codes<false, SQ_CODES_BF16>(nvec, xb, tokens, cin, ldb, s_inv, qb, x_scale, flags, st)
             : launch_act_codes<false, SQ_CODES_I8>(nvec, xb, tokens, cin, ldb, s_inv, qb, x_scale, flags, st);
}

}  // namespace sq

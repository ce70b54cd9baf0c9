// Step 4: runtime X * diag(s)^-1 fused with dynamic per-token INT8
// quantization.
//
// Sources: first page ("Move activation scale without changing the real
// linear map"), paragraph 3: the explicit runtime scaling step that
// multiplies activations by S^-1; learn-kernels.com "Quantization",
// paragraph 2: activations are quantized to INT8.
//
// Persistent kernel: each CTA owns every gridDim.x-th token row.  Rows
// stream from HBM into a ring of shared-memory stages with one-dimensional
// bulk copies (TMA), several rows ahead of the threads, so the reads of
// later rows overlap the arithmetic and the code stores of earlier ones.
// Every thread owns the same column vectors of every row and keeps their
// s^-1 in registers.  Pass 1 forms X' = X * s^-1 (kept in registers) and
// the row's max|X'|; one block barrier combines the warps' maxima (and
// frees the stage for the next copy); pass 2 writes the codes
// rne(RN(X' / d)), the binary32 quotient formed by quot_rn.  HBM
// traffic per element: one read of X and one write of the code, plus 4
// bytes per token for the scale.  The same kernel serves the static
// variant (one calibrated scale for every token, SmoothQuant glossary:
// calibration-based): no row maximum, the clamp can act and is counted.
#include "sq_async.cuh"

namespace sq {
namespace {
using namespace async;

constexpr uint64_t kWaitNs = 1000000000ull;  // bound on every mbarrier wait of a product call (1 s)
constexpr int kMaxStages = 8;

template <bool BF16>
SQ_DEVINL void unpack(uint4 v, float* f) {
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

// E consecutive s^-1 values starting at element e0 (16-byte aligned).
template <int E>
SQ_DEVINL void load_sinv(const float* s_inv, int64_t e0, float* f) {
#pragma unroll
  for (int q = 0; q < E; q += 4) {
    const uint4 v = ld_ro16(s_inv + e0 + q);
    f[q + 0] = __uint_as_float(v.x);
    f[q + 1] = __uint_as_float(v.y);
    f[q + 2] = __uint_as_float(v.z);
    f[q + 3] = __uint_as_float(v.w);
  }
}

constexpr int kDynamic = 0;  // per-token scale from the row's max|X'|
constexpr int kStatic = 1;   // one calibrated scale for every token
constexpr int kNorm = 2;     // RMS normalization with the folded gain, then per-token scale

// Flag bits beside a warp's exponent in the kNorm exchange: bits were
// dropped below the unit; a thread of the warp used the fast sum.
constexpr uint32_t kStickyBit = 1u << 16, kFastBit = 1u << 17;

// 128-bit unsigned integer as (hi, lo).
struct U128 {
  uint64_t hi, lo;
};
SQ_DEVINL U128 add128(U128 a, U128 b) {
  U128 r;
  r.lo = a.lo + b.lo;
  r.hi = a.hi + b.hi + (r.lo < a.lo ? 1ull : 0ull);
  return r;
}
SQ_DEVINL U128 sub128(U128 a, U128 b) {  // a - b, a >= b
  U128 r;
  r.lo = a.lo - b.lo;
  r.hi = a.hi - b.hi - (a.lo < b.lo ? 1ull : 0ull);
  return r;
}

// Exact sums of squares as 128-bit fixed-point integers.  For h with
// binary32 exponent field e (>= 1 after subnormals) and 24-bit significand
// m, h^2 = m^2 * 2^(2e - 300).  A partial sum relative to exponent E holds
// I = sum m^2 * 2^(62 - 2 (E - e)), i.e. sum h^2 = I * 2^(2E - 362); every
// term is below 2^110, so a row of 32768 terms stays below 2^125.  Bits of
// a term more than 2^62 below the largest fall below the unit: they are
// dropped, and `sticky` records that a nonzero part was dropped, so that a
// sum that would otherwise sit exactly on a binary32 midpoint is known to
// lie above it.
SQ_DEVINL U128 shl128(uint64_t v, int sh, bool& sticky) {  // v * 2^sh, v < 2^48, sh <= 62
  U128 r;
  if (sh >= 0) {
    r.lo = v << sh;
    r.hi = sh ? (v >> (64 - sh)) : 0ull;
  } else {
    const int k = -sh;
    sticky |= (k < 64 ? (v & ((1ull << k) - 1ull)) : v) != 0ull;
    r.lo = k < 64 ? (v >> k) : 0ull;
    r.hi = 0ull;
  }
  return r;
}

SQ_DEVINL U128 shr128(U128 x, int sh) {  // x / 2^sh truncated, sh >= 0
  if (sh == 0) return x;
  U128 r;
  if (sh >= 128) {
    r.hi = r.lo = 0ull;
  } else if (sh >= 64) {
    r.lo = x.hi >> (sh - 64);
    r.hi = 0ull;
  } else {
    r.lo = (x.lo >> sh) | (x.hi << (64 - sh));
    r.hi = x.hi >> sh;
  }
  return r;
}

// The same, recording in `sticky` whether nonzero bits were shifted out.
SQ_DEVINL U128 shr128(U128 x, int sh, bool& sticky) {
  if (sh == 0) return x;
  bool lost;
  if (sh >= 128)
    lost = (x.hi | x.lo) != 0ull;
  else if (sh >= 64)
    lost = x.lo != 0ull || (sh > 64 && (x.hi & ((1ull << (sh - 64)) - 1ull)) != 0ull);
  else
    lost = (x.lo & ((1ull << sh) - 1ull)) != 0ull;
  sticky |= lost;
  return shr128(x, sh);
}

// Add h^2 for the element with |h| bits b to the sum I relative to exponent
// E.  bf16-origin values (low 16 significand bits zero) within 2^15 of the
// largest take a single 32 x 32 -> 64-bit multiply-add into the high word.
template <bool BF16>
SQ_DEVINL void add_square(U128& acc, uint32_t b, int E, bool& sticky) {
  const int e = (int)(b >> 23);
  const int d2 = 2 * (E - (e ? e : 1));
  if constexpr (BF16) {
    const uint32_t m8 = ((b >> 16) & 0x7Fu) | (e ? 0x80u : 0u);
    const uint32_t sq = m8 * m8;                 // < 2^16
    if (d2 <= 30) {                              // sq * 2^(94 - d2): bits 64.. of the sum
      const uint64_t add = (uint64_t)sq * (uint64_t)(1u << (30 - d2));
      acc.hi += add;
      return;
    }
    acc = add128(acc, shl128((uint64_t)sq << 32, 62 - d2, sticky));
  } else {
    const uint64_t m = (uint64_t)((b & 0x7FFFFFu) | (e ? 0x800000u : 0u));
    acc = add128(acc, shl128(m * m, 62 - d2, sticky));
  }
}

// I * 2^u rounded once to binary32 (nearest, ties to even; subnormal
// results rounded at their own position, overflow to +inf).  `sticky`: the
// true value lies strictly above I * 2^u by less than one unit.
SQ_DEVINL float u128_scaled_to_f32(U128 x, int u, bool sticky) {
  if (x.hi == 0 && x.lo == 0) return 0.0f;
  const int t = x.hi ? 127 - __clzll((long long)x.hi) : 63 - __clzll((long long)x.lo);  // top bit
  const int shift = max(t - 23, -149 - u);     // bits below `shift` are rounded off
  // at most 24 significant bits: exact, and a sticky part below the unit is
  // under half a unit of the result
  if (shift <= 0) return ldexpf((float)x.lo, u);
  // the sums held here stay below 2^125, so a shift of 128 or more means a
  // value below 2^-152: under half the smallest subnormal
  if (shift >= 128) return 0.0f;
  const U128 q128 = shr128(x, shift);
  uint32_t q = (uint32_t)q128.lo;              // < 2^24
  // remainder against half a unit at `shift`
  U128 rem;
  if (shift >= 64) {
    rem.hi = (shift == 64) ? 0ull : (x.hi & ((1ull << (shift - 64)) - 1ull));
    rem.lo = x.lo;
  } else {
    rem.hi = 0ull;
    rem.lo = x.lo & ((1ull << shift) - 1ull);
  }
  U128 half;
  if (shift - 1 >= 64) {
    half.hi = 1ull << (shift - 1 - 64);
    half.lo = 0ull;
  } else {
    half.hi = 0ull;
    half.lo = 1ull << (shift - 1);
  }
  const bool gt = rem.hi > half.hi || (rem.hi == half.hi && rem.lo > half.lo);
  const bool eq = rem.hi == half.hi && rem.lo == half.lo;
  if (gt || (eq && (sticky || (q & 1u)))) ++q;
  return ldexpf((float)q, shift + u);          // q <= 2^24: exact scaling
}

// Fast sum of squares of one thread's bf16-origin values, used when the
// thread's largest exponent field et lies in [kFastLo, kFastHi].  With
// U = 2^(2 (et - 127)) every square is below 4U.  Each square is split on
// the grid 2^-16 U by an add of sigma = 192 U (hi = RN(h^2 + sigma) - sigma,
// exact by Sterbenz's lemma) and lo = h^2 - hi (one fused multiply-add,
// exact: a bf16 square has 16 significant bits).  The hi parts sum exactly
// (multiples of 2^-16 U below 2^7 U); the lo parts, each at most 2^-17 U,
// sum with rounding error below 2^-33 U for 32 values (two running sums of
// 16, each add off by at most 2^-38 U, the last by 2^-37 U), and squares
// below the normal range add at most 32 * 2^-150 <= 2^-35 U (U >= 2^-110).
// So the result, returned in the fixed-point form relative to et (rounded
// there at 2^-68 U), is within 2^-32.6 U of the thread's exact sum, and U is
// at most its largest square.
constexpr int kFastLo = 72, kFastHi = 187;
template <int N>
SQ_DEVINL U128 fast_sum_squares_bf16(const float* h, int et) {
  static_assert(N % 2 == 0 && N <= 32, "at most 32 values, in pairs");
  const float sigma = __uint_as_float(((uint32_t)(2 * et - 120) << 23) | 0x400000u);  // 192 U
  float sh0 = 0.0f, sh1 = 0.0f, sl0 = 0.0f, sl1 = 0.0f;
#pragma unroll
  for (int k = 0; k < N; k += 2) {
    float t0 = h[k], t1 = h[k + 1];
    fma2_rn(t0, t1, h[k], h[k + 1], sigma, sigma);      // RN(h^2 + sigma)
    add2_rn(t0, t1, -sigma, -sigma);                    // hi, exact
    float l0 = h[k], l1 = h[k + 1];
    fma2_rn(l0, l1, h[k], h[k + 1], -t0, -t1);          // lo = h^2 - hi, exact
    add2_rn(sh0, sh1, t0, t1);
    add2_rn(sl0, sl1, l0, l1);
  }
  const float s_hi = __fadd_rn(sh0, sh1);  // exact
  const float s_lo = __fadd_rn(sl0, sl1);
  // s_hi = H * 2^-16 U: H << 92 in units of 2^(2 et - 362)
  const uint32_t H = __float2uint_rn(__fmul_rn(s_hi, __uint_as_float((uint32_t)(397 - 2 * et) << 23)));
  // s_lo / U, then at the unit 2^-68 U (2^40 units): |L| <= 2^56
  const long long L =
      __float2ll_rn(__fmul_rn(__fmul_rn(s_lo, __uint_as_float((uint32_t)(381 - 2 * et) << 23)), 0x1p68f));
  const U128 a = {(uint64_t)H << 28, 0ull};
  const U128 b = {(uint64_t)(L >> 24), (uint64_t)L << 40};  // L * 2^40, two's complement
  return add128(a, b);                                         // the sum is positive
}

// Exact sum of squares of one thread's values relative to exponent et.
template <bool BF16, int N>
SQ_DEVINL U128 exact_sum_squares(const float* h, int et, bool& sticky) {
  U128 acc = {0ull, 0ull};
#pragma unroll
  for (int k = 0; k < N; ++k) add_square<BF16>(acc, __float_as_uint(h[k]) & 0x7FFFFFFFu, et, sticky);
  return acc;
}

// Sum of a warp's 128-bit partial sums, each relative to its lane's exponent
// et, aligned to the warp's largest exponent (returned in ew).
SQ_DEVINL U128 warp_sum128(U128 acc, int et, int& ew, bool& sticky) {
  ew = (int)__reduce_max_sync(0xFFFFFFFFu, (uint32_t)et);
  acc = shr128(acc, 2 * (ew - et), sticky);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    U128 other;
    other.hi = __shfl_xor_sync(0xFFFFFFFFu, acc.hi, o);
    other.lo = __shfl_xor_sync(0xFFFFFFFFu, acc.lo, o);
    acc = add128(acc, other);
  }
  return acc;
}

// Sum of the NW warps' partial sums (red_s, with exponents and flag bits in
// red_e) in every warp: lane w aligns warp w's sum to the row's largest
// exponent eb and a butterfly over the first NW lanes adds them (integer
// sums: the order does not matter).  Returns the OR of the flag bits.
template <int NW>
SQ_DEVINL U128 block_sum128(const U128* red_s, const uint32_t* red_e, int lane, int& eb,
                            uint32_t& bits) {
  static_assert((NW & (NW - 1)) == 0 && NW <= 32, "power-of-two warp count");
  const uint32_t re = lane < NW ? red_e[lane] : 1u;
  const int ew_l = (int)(re & 0xFFFFu);
  eb = (int)__reduce_max_sync(0xFFFFFFFFu, (uint32_t)ew_l);
  bool sticky = false;
  U128 tot = {0ull, 0ull};
  if (lane < NW) tot = shr128(red_s[lane], 2 * (eb - ew_l), sticky);
#pragma unroll
  for (int o = NW / 2; o > 0; o >>= 1) {
    U128 other;
    other.hi = __shfl_xor_sync(0xFFFFFFFFu, tot.hi, o);
    other.lo = __shfl_xor_sync(0xFFFFFFFFu, tot.lo, o);
    tot = add128(tot, other);
  }
  bits = __reduce_or_sync(0xFFFFFFFFu, (re & ~0xFFFFu) | (sticky ? kStickyBit : 0u));
  return tot;
}

// r = RN(1 / RN(sqrt(RN(RN(s / K) + eps)))), every step one IEEE binary32
// operation.
// For K = 2^k, RN(s / K) is RN(s * 2^-k): both round the same real number
// once.
SQ_DEVINL float rms_factor(float s, int K, float eps) {
  const float q = (K & (K - 1)) == 0 ? __fmul_rn(s, __uint_as_float((uint32_t)(127 - (31 - __clz(K))) << 23))
                                     : __fdiv_rn(s, (float)K);
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(q, eps)));
}

// NT threads per CTA, each owning VPT 16-byte vectors of every row (vector
// v = tid + i*NT).  With NT <= 512 the thread's s^-1 values stay in
// registers; with 1024 threads (rows longer than 32 KiB) the register
// budget is 64 per thread, so they are re-read through L1 for each row, and
// so are the RMS-normalizing mode's gains in its 256- and 512-thread blocks:
// that leaves 62 registers, four 256-thread or two 512-thread blocks per SM
// instead of two or one (B300: 8192 x 8192 104 -> 94 us, 2048 x 11008
// 55 -> 47 us, 4096 x 16384 113 -> 100 us; the 128-thread block, already
// at its four blocks per SM, kept its registers).
// MODE kStatic: one calibrated scale *d_static for every token instead of
// the row maximum (no reduction; the clamp can act and `clipped` counts it).
// MODE kNorm: `s_inv` holds the folded gain gamma' and the row is first
// RMS-normalized: S, the exact sum of squares rounded once to binary32
// (128-bit fixed point, order-independent; bf16 rows take a split sum on the
// floating-point pipe whose error bound decides the rounding, and redo the
// exact sum in the rare rows where it cannot), then
// r = RN(1 / RN(sqrt(RN(RN(S / K) + eps)))) in IEEE binary32 and
// X' = RN(RN(h * r) * gamma').  Three block barriers per row (five when the
// exact sum is redone).
// From 512 threads up the kernel is built for one block per SM, which leaves
// the compiler its full register budget (0 below: no minimum; the
// RMS-normalizing mode's 512-thread block for two, see above).  Measured on
// B300: 2048 x 11008 bf16 24.7 -> 22.4 us (RMS-normalizing mode 70.2 ->
// 62.0), 4096 x 16384 55.4 -> 45.1 us (175 -> 146); with the same bound on
// the 256-thread block of 8192-element rows the RMS-normalizing mode lost
// 4 %, so it applies to the larger blocks only.
template <bool BF16, int CODES, int NT, int VPT, int MODE>
__global__ void __launch_bounds__(NT, (MODE == kNorm && NT == 512) ? 2 : (NT >= 512 ? 1 : 0)) k_quant_act(const uint8_t* __restrict__ x, int64_t tokens,
                                                  int nvec, int64_t ldx_bytes,
                                                  const float* __restrict__ s_inv,
                                                  uint8_t* __restrict__ xq,
                                                  float* __restrict__ x_scale, int32_t* flags,
                                                  int stages, const float* __restrict__ d_static,
                                                  uint32_t* clipped, float eps, uint64_t wait_ns,
                                                  int stall) {
  constexpr bool STATIC = MODE == kStatic;
  constexpr bool NORM = MODE == kNorm;
  constexpr int E = BF16 ? 8 : 4;
  constexpr int NW = NT / 32;
  constexpr int CB = CODES == SQ_CODES_BF16 ? 2 : 1;
  constexpr bool kSiReg = NT <= 512 && !(NORM && NT >= 256);
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t row_bytes = (uint32_t)nvec * 16u;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)stages * row_bytes);
  uint32_t* red = reinterpret_cast<uint32_t*>(full + kMaxStages);  // [2][NW]
  uint32_t* red_e = red + 2 * NW;                                    // [2][NW] (kNorm)
  U128* red_s = reinterpret_cast<U128*>(full + kMaxStages + 2 * NW); // [2][NW] (kNorm)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int cin = nvec * E;

  float si[kSiReg ? VPT : 1][E];
  if constexpr (kSiReg) {
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = tid + i * NT;
      if (v < nvec) {
        load_sinv<E>(s_inv, (int64_t)v * E, si[i]);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) si[i][e] = 0.0f;
      }
    }
  }

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) mbar_init(&full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  const uint64_t pol = policy_evict_first();  // X is read once here
  if (tid == 0 && !stall) {  // stall: no copies (the bounded waits' test; 0 on every product call)
    for (int i = 0; i < stages; ++i) {
      const int64_t r = blockIdx.x + (int64_t)i * gridDim.x;
      if (r >= tokens) break;
      mbar_expect_tx(&full[i], row_bytes);
      bulk_g2s_hint(smem + (size_t)i * row_bytes, x + r * ldx_bytes, row_bytes, &full[i], pol);
    }
  }

  float d_fix = 1.0f, inv_fix = 1.0f;
  bool fast_fix = false;
  if constexpr (STATIC) {
    d_fix = *d_static;
    inv_fix = __fdiv_rn(1.0f, d_fix);
    fast_fix = fast_scale_ok(d_fix);
  }
  uint32_t nclip = 0u;
  bool nonfinite = false;
  int it = 0;
  bool aborted = false;
  for (int64_t r = blockIdx.x; r < tokens; r += gridDim.x, ++it) {
    const int stage = it % stages;
    const uint32_t parity = (uint32_t)(it / stages) & 1u;
    const bool ok = mbar_wait_bounded(&full[stage], parity, wait_ns);
    const uint8_t* buf = smem + (size_t)stage * row_bytes;

    // pass 1: X' = X * s^-1 into registers, and the thread's max|X'|
    float p[VPT][E];
    float m = 0.0f;
    if constexpr (NORM) {
      // the row into registers and the thread's largest binary32 exponent
      uint32_t tb = 0u;
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = tid + i * NT;
        if (ok && v < nvec) {
          const uint4 raw = *reinterpret_cast<const uint4*>(buf + (size_t)v * 16);
          unpack<BF16>(raw, p[i]);
          if constexpr (BF16) {  // packed magnitudes, NaN kept (exponent 255)
            tb = absmax_nan_bf16x2(tb, absmax_nan_bf16x2(absmax_nan_bf16x2(raw.x, raw.y),
                                                         absmax_nan_bf16x2(raw.z, raw.w)));
          } else {
#pragma unroll
            for (int e = 0; e < E; ++e) tb = max(tb, __float_as_uint(p[i][e]) & 0x7FFFFFFFu);
          }
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) p[i][e] = 0.0f;
        }
      }
      if constexpr (BF16) tb = max(tb & 0x7FFFu, (tb >> 16) & 0x7FFFu) << 16;
      const int et = max(1, (int)(tb >> 23));  // 255: a non-finite value
      // the thread's sum of squares relative to et: the fast split sum for
      // bf16 values in its exponent range (within 2^-31 U), else exact
      bool fast = false;
      if constexpr (BF16) fast = et >= kFastLo && et <= kFastHi;
      bool sticky = false;
      U128 acc = {0ull, 0ull};
      if (fast) {
        if constexpr (BF16) acc = fast_sum_squares_bf16<VPT * E>(&p[0][0], et);
      } else if (et < 255) {
        acc = exact_sum_squares<BF16, VPT * E>(&p[0][0], et, sticky);
      }
      int ew;
      acc = warp_sum128(acc, et, ew, sticky);
      const uint32_t wbits = (__any_sync(0xFFFFFFFFu, sticky) ? kStickyBit : 0u) |
                             (__any_sync(0xFFFFFFFFu, fast) ? kFastBit : 0u);
      if (lane == 0) {
        red_s[(it & 1) * NW + warp] = acc;
        red_e[(it & 1) * NW + warp] = (uint32_t)ew | wbits;
      }
      if (__syncthreads_or(!ok)) {
        aborted = true;
        break;
      }
      if (tid == 0) {  // the row is in registers: refill the stage
        const int64_t rn = r + (int64_t)stages * gridDim.x;
        if (rn < tokens) {
          mbar_expect_tx(&full[stage], row_bytes);
          bulk_g2s_hint(const_cast<uint8_t*>(buf), x + rn * ldx_bytes, row_bytes, &full[stage], pol);
        }
      }
      // Warp 0 alone forms the row's factor r (the block's total, the bound
      // check and the scalar chain); the other warps wait for it at a
      // barrier instead of repeating that work.
      //
      // S32 = RN(S), S the exact sum.  With fast sums in the total T, S lies
      // within 2^-32.6 S of T (every thread's error is below 2^-32.6 U and
      // its U is at most its largest square, so those bounds add up to at
      // most 2^-32.6 S; dropped bits below the unit are under 2^-90 S), so
      // if T - B and T + B round alike for B = 2^-32 T + 1 that is RN(S).
      // Otherwise (a midpoint within B of T: about 2^-8 of random rows)
      // every thread forms its exact sum and the block adds them again.
      // r = RN(1 / RN(sqrt(RN(RN(S32 / K) + eps)))), every step one IEEE
      // binary32 operation.
      float* rn_s = reinterpret_cast<float*>(red_s + 2 * NW);  // [2]
      uint32_t* st_s = reinterpret_cast<uint32_t*>(rn_s + 2);   // [2]: 1 redo, 2 finite
      if (warp == 0) {
        int eb;
        uint32_t bbits;
        const U128 tot = block_sum128<NW>(red_s + (it & 1) * NW, red_e + (it & 1) * NW, lane, eb, bbits);
        // lanes 0 and 1 round T - B and T + B side by side (T alone, with
        // the sticky bit, when every thread summed exactly)
        const bool finite = eb < 255;
        const bool fast_row = (bbits & kFastBit) != 0u;
        float f = 0.0f;
        if (finite && lane < 2) {
          const U128 bnd = add128(shr128(tot, 32), U128{0ull, 1ull});
          f = !fast_row ? u128_scaled_to_f32(tot, 2 * eb - 362, (bbits & kStickyBit) != 0u)
                        : u128_scaled_to_f32(lane == 0 ? sub128(tot, bnd) : add128(tot, bnd), 2 * eb - 362, false);
        }
        const float f1 = __shfl_sync(0xFFFFFFFFu, f, 1);
        if (lane == 0) {
          const bool redo = finite && fast_row && __float_as_uint(f) != __float_as_uint(f1);
          if (finite && !redo) rn_s[it & 1] = rms_factor(f, cin, eps);
          st_s[it & 1] = (redo ? 1u : 0u) | (finite ? 2u : 0u);
        }
      }
      __syncthreads();
      const uint32_t st = st_s[it & 1];
      const bool row_finite = (st & 2u) != 0u;
      if (st & 1u) {
        // the other exchange slot: its last readers (the previous row's warp
        // 0) are past this row's first barrier, and the next row writes it
        // only after this row's last barrier
        sticky = false;
        acc = {0ull, 0ull};
        if (et < 255) acc = exact_sum_squares<BF16, VPT * E>(&p[0][0], et, sticky);
        acc = warp_sum128(acc, et, ew, sticky);
        const bool wst = __any_sync(0xFFFFFFFFu, sticky);
        const int slot = ((it + 1) & 1) * NW;
        if (lane == 0) {
          red_s[slot + warp] = acc;
          red_e[slot + warp] = (uint32_t)ew | (wst ? kStickyBit : 0u);
        }
        __syncthreads();
        if (warp == 0) {
          int eb;
          uint32_t bbits;
          const U128 tot = block_sum128<NW>(red_s + slot, red_e + slot, lane, eb, bbits);
          if (lane == 0)
            rn_s[it & 1] = rms_factor(u128_scaled_to_f32(tot, 2 * eb - 362, (bbits & kStickyBit) != 0u), cin, eps);
        }
        __syncthreads();
      }
      const float rn32 = row_finite ? rn_s[it & 1] : 0.0f;
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = tid + i * NT;
        if (!(v < nvec)) continue;
        float sv[E];
        if constexpr (kSiReg) {
#pragma unroll
          for (int e = 0; e < E; ++e) sv[e] = si[i][e];
        } else {
          load_sinv<E>(s_inv, (int64_t)v * E, sv);
        }
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          mul2_rn(p[i][e], p[i][e + 1], rn32, rn32);
          mul2_rn(p[i][e], p[i][e + 1], sv[e], sv[e + 1]);
        }
#pragma unroll
        for (int e = 0; e < E; ++e) m = absmax_nan(m, p[i][e]);
      }
      if (!row_finite) m = __int_as_float(0x7FFFFFFF);  // the row's scale is NaN
      const uint32_t mbx = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m) & 0x7FFFFFFFu);
      if (lane == 0) red[(it & 1) * NW + warp] = mbx;
      __syncthreads();
    } else {
#pragma unroll
      for (int i = 0; i < VPT; ++i) {
        const int v = tid + i * NT;
        if (ok && v < nvec) {
          unpack<BF16>(*reinterpret_cast<const uint4*>(buf + (size_t)v * 16), p[i]);
          float sv[E];
          if constexpr (kSiReg) {
#pragma unroll
            for (int e = 0; e < E; ++e) sv[e] = si[i][e];
          } else {
            load_sinv<E>(s_inv, (int64_t)v * E, sv);
          }
#pragma unroll
          for (int e = 0; e < E; e += 2) mul2_rn(p[i][e], p[i][e + 1], sv[e], sv[e + 1]);
          if constexpr (!STATIC) {
#pragma unroll
            for (int e = 0; e < E; ++e) m = absmax_nan(m, p[i][e]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) p[i][e] = 0.0f;
        }
      }
      if constexpr (!STATIC) {
        const uint32_t mb = __reduce_max_sync(0xFFFFFFFFu, __float_as_uint(m) & 0x7FFFFFFFu);
        if (lane == 0) red[(it & 1) * NW + warp] = mb;
      }
      if (__syncthreads_or(!ok)) {
        aborted = true;
        break;
      }
      // every thread has read this stage: refill it with the row `stages`
      // iterations ahead
      if (tid == 0) {
        const int64_t rn = r + (int64_t)stages * gridDim.x;
        if (rn < tokens) {
          mbar_expect_tx(&full[stage], row_bytes);
          bulk_g2s_hint(const_cast<uint8_t*>(buf), x + rn * ldx_bytes, row_bytes, &full[stage], pol);
        }
      }
    }
    float d, inv;
    bool no_clamp;
    if constexpr (STATIC) {
      d = d_fix;
      inv = inv_fix;
      no_clamp = false;
      if (tid == 0) x_scale[r] = d;
    } else {
      uint32_t amax = 0u;
#pragma unroll
      for (int w = 0; w < NW; ++w) amax = max(amax, red[(it & 1) * NW + w]);
      scale_and_inverse(__uint_as_float(amax), d, inv);
      if (tid == 0) {
        x_scale[r] = d;
        if (!finite_bits(amax)) raise_flag(flags, SQ_FLAG_NONFINITE);
      }
      // With a finite max >= 2^-93 the quotient X'/d comes from quot_rn and
      // no code can leave [-127, 127], so the clamp is skipped; any other
      // row (tiny, zero or non-finite maximum) divides element by element.
      no_clamp = fast_quotient_ok(amax);
    }

    // pass 2: codes = rne(RN(X' / d)), via the magic-number add
    uint8_t* qrow = xq + r * (int64_t)nvec * E * CB;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
      const int v = tid + i * NT;
      if (v >= nvec) continue;
      float q[E];
      if (no_clamp) {
        // two quotients per instruction, then the rounding add
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          float a = p[i][e], b = p[i][e + 1];
          quot2_rn(a, b, d, d, inv, inv);
          add2_rn(a, b, kMagic, kMagic);
          q[e] = a;
          q[e + 1] = b;
        }
      } else if constexpr (STATIC) {
        // the quotient (quot_rn inside its range, else an IEEE division),
        // clamp, then the rounding add.  A NaN gives code 0 and +-inf
        // saturates; neither counts as clipped, both are flagged.
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const float q0 = __fmul_rn(p[i][e], inv);
          const float t = (fast_fix && fabsf(q0) < 256.0f) ? quot_refine(p[i][e], d, inv, q0)
                                                           : __fdiv_rn(p[i][e], d);
          const float a = fabsf(t);
          const bool finite = a <= 3.4028234663852886e38f;
          nonfinite |= !finite;
          nclip += (finite && a >= 127.5f) ? 1u : 0u;
          q[e] = __fadd_rn((t == t) ? fminf(fmaxf(t, -127.0f), 127.0f) : 0.0f, kMagic);
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) q[e] = code_div_magic(p[i][e], d, 127.0f);
      }
      if constexpr (CODES == SQ_CODES_BF16) {
        uint32_t w[E / 2];
#pragma unroll
        for (int e = 0; e < E; e += 2) {
          float c0 = q[e], c1 = q[e + 1];
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
              make_uint2(pack4_codes(q[0], q[1], q[2], q[3]), pack4_codes(q[4], q[5], q[6], q[7])));
        else
          *reinterpret_cast<uint32_t*>(qrow + (size_t)v * 4) = pack4_codes(q[0], q[1], q[2], q[3]);
      }
    }
  }

  if constexpr (STATIC) {
    if (clipped) {
      nclip = __reduce_add_sync(0xFFFFFFFFu, nclip);
      if (lane == 0 && nclip) atomicAdd(clipped, nclip);
    }
    if (__any_sync(0xFFFFFFFFu, nonfinite) && lane == 0) raise_flag(flags, SQ_FLAG_NONFINITE);
  }
  if (aborted && tid == 0) {
    raise_flag(flags, SQ_FLAG_TIMEOUT);
    // let every copy this CTA issued land before its shared memory is freed
    for (int k = 0; k < stages && !stall; ++k) {
      const int j = it + k;
      if (blockIdx.x + (int64_t)j * gridDim.x >= tokens) break;
      mbar_wait_bounded(&full[j % stages], (uint32_t)(j / stages) & 1u, 10000000ull);
    }
  }
}

struct ActLaunch {
  int stages;
  size_t smem;
  int grid;
};

struct Static {
  int mode;            // kDynamic, kStatic or kNorm
  const float* d;      // kStatic: the calibrated scale
  uint32_t* clipped;   // kStatic: clip counter or null
  float eps;           // kNorm
  uint64_t wait_ns = kWaitNs;  // bound on each wait for a row's copy
  int stall = 0;               // 1: no copies are issued (the bounded waits' test)
};

template <bool BF16, int CODES, int NT, int VPT, int MODE>
sq_status launch_act(int nvec, const uint8_t* x, int64_t tokens, int64_t ldx_bytes,
                     const float* s_inv, uint8_t* xq, float* x_scale, int32_t* flags, Static sc,
                     cudaStream_t st) {
  auto kern = k_quant_act<BF16, CODES, NT, VPT, MODE>;
  static std::atomic<uint64_t> attr_done{0};
  if (!once_per_device(attr_done, [&] {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
      }))
    return SQ_ERR_CUDA;
  const size_t row_bytes = (size_t)nvec * 16;
  // about 32 KiB of rows in flight per CTA, at least two stages, so several
  // CTAs share an SM.  Measured on B300 against 64 KiB: 2048 x 4096 bf16
  // 11.2 instead of 13.0 us, 8192 x 8192 41.2 instead of 43.0 us, and in
  // the RMS-normalizing mode 24.8 instead of 27.7 us (2048 x 4096).
  const size_t in_flight = 32768;
  const int stages = (int)std::max<size_t>(2, std::min<size_t>(kMaxStages, in_flight / row_bytes));
  const size_t smem = stages * row_bytes + kMaxStages * 8 + 2 * (NT / 32) * (4 + 4 + 16) + 16 + 16;
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, NT, smem) != cudaSuccess)
    return SQ_ERR_CUDA;
  occ = std::max(1, std::min(occ, 4));
  const int64_t grid = std::min<int64_t>(tokens, (int64_t)sm_count() * occ);
  kern<<<(unsigned)grid, NT, smem, st>>>(x, tokens, nvec, ldx_bytes, s_inv, xq, x_scale, flags,
                                         stages, sc.d, sc.clipped, sc.eps, sc.wait_ns, sc.stall);
  return launch_status();
}

template <bool BF16, int CODES, int NT, int MODE>
sq_status launch_act_vpt(int nvec, const uint8_t* x, int64_t tokens, int64_t ldx_bytes,
                         const float* s_inv, uint8_t* xq, float* x_scale, int32_t* flags,
                         Static sc, cudaStream_t st) {
  switch ((nvec + NT - 1) / NT) {
    case 1: return launch_act<BF16, CODES, NT, 1, MODE>(nvec, x, tokens, ldx_bytes, s_inv, xq, x_scale, flags, sc, st);
    case 2: return launch_act<BF16, CODES, NT, 2, MODE>(nvec, x, tokens, ldx_bytes, s_inv, xq, x_scale, flags, sc, st);
    case 3: return launch_act<BF16, CODES, NT, 3, MODE>(nvec, x, tokens, ldx_bytes, s_inv, xq, x_scale, flags, sc, st);
    case 4: return launch_act<BF16, CODES, NT, 4, MODE>(nvec, x, tokens, ldx_bytes, s_inv, xq, x_scale, flags, sc, st);
    default: return SQ_ERR_UNSUPPORTED;
  }
}

template <bool BF16, int CODES, int NT>
sq_status launch_act_nt(int nvec, const uint8_t* x, int64_t tokens, int64_t ldx_bytes,
                        const float* s_inv, uint8_t* xq, float* x_scale, int32_t* flags,
                        Static sc, cudaStream_t st) {
  switch (sc.mode) {
    case kStatic: return launch_act_vpt<BF16, CODES, NT, kStatic>(nvec, x, tokens, ldx_bytes, s_inv, xq, x_scale, flags, sc, st);
    case kNorm: return launch_act_vpt<BF16, CODES, NT, kNorm>(nvec, x, tokens, ldx_bytes, s_inv, xq, x_scale, flags, sc, st);
    default: return launch_act_vpt<BF16, CODES, NT, kDynamic>(nvec, x, tokens, ldx_bytes, s_inv, xq, x_scale, flags, sc, st);
  }
}

template <bool BF16, int CODES>
sq_status launch_act_codes(int nvec, const uint8_t* x, int64_t tokens, int64_t ldx_bytes,
                           const float* s_inv, uint8_t* xq, float* x_scale, int32_t* flags,
                           Static sc, cudaStream_t st) {
  // the smallest block whose threads hold the row in at most 4 vectors each
  if (nvec <= 128 * 4)
    return launch_act_nt<BF16, CODES, 128>(nvec, x, tokens, ldx_bytes, s_inv, xq, x_scale, flags, sc, st);
  if (nvec <= 256 * 4)
    return launch_act_nt<BF16, CODES, 256>(nvec, x, tokens, ldx_bytes, s_inv, xq, x_scale, flags, sc, st);
  if (nvec <= 512 * 4)
    return launch_act_nt<BF16, CODES, 512>(nvec, x, tokens, ldx_bytes, s_inv, xq, x_scale, flags, sc, st);
  return launch_act_nt<BF16, CODES, 1024>(nvec, x, tokens, ldx_bytes, s_inv, xq, x_scale, flags, sc, st);
}

sq_status quant_act_any(const void* x, sq_dtype dt, int64_t tokens, int64_t cin, int64_t ldx,
                        const float* s_inv, void* xq, sq_codes fmt, float* x_scale,
                        int32_t* flags, Static sc, cudaStream_t st) {
  const bool bf16 = dt == SQ_BF16;
  const int nvec = (int)(cin / (bf16 ? 8 : 4));
  const uint8_t* xb = static_cast<const uint8_t*>(x);
  uint8_t* qb = static_cast<uint8_t*>(xq);
  const int64_t ldb = ldx * elem_bytes(dt);
  if (bf16) {
    return fmt == SQ_CODES_BF16
               ? launch_act_codes<true, SQ_CODES_BF16>(nvec, xb, tokens, ldb, s_inv, qb, x_scale, flags, sc, st)
               : launch_act_codes<true, SQ_CODES_I8>(nvec, xb, tokens, ldb, s_inv, qb, x_scale, flags, sc, st);
  }
  return fmt == SQ_CODES_BF16
             ? launch_act_codes<false, SQ_CODES_BF16>(nvec, xb, tokens, ldb, s_inv, qb, x_scale, flags, sc, st)
             : launch_act_codes<false, SQ_CODES_I8>(nvec, xb, tokens, ldb, s_inv, qb, x_scale, flags, sc, st);
}

}  // namespace

// Largest Cin: a 64 KiB row (two stages fit one CTA's shared memory), i.e.
// 4096 vectors of 16 bytes held by 1024 threads x 4.
int64_t quant_act_max_cin(sq_dtype dt) { return (int64_t)4096 * (dt == SQ_BF16 ? 8 : 4); }

sq_status quant_act(const void* x, sq_dtype dt, int64_t tokens, int64_t cin, int64_t ldx,
                    const float* s_inv, void* xq, sq_codes fmt, float* x_scale, int32_t* flags,
                    cudaStream_t st) {
  return quant_act_any(x, dt, tokens, cin, ldx, s_inv, xq, fmt, x_scale, flags, Static{kDynamic, nullptr, nullptr, 0.0f}, st);
}

sq_status quant_act_stalled(const void* x, sq_dtype dt, int64_t tokens, int64_t cin, int64_t ldx,
                            const float* s_inv, void* xq, sq_codes fmt, float* x_scale, int32_t* flags,
                            uint64_t wait_ns, cudaStream_t st) {
  return quant_act_any(x, dt, tokens, cin, ldx, s_inv, xq, fmt, x_scale, flags,
                       Static{kDynamic, nullptr, nullptr, 0.0f, wait_ns, 1}, st);
}

sq_status quant_act_static(const void* x, sq_dtype dt, int64_t tokens, int64_t cin, int64_t ldx,
                           const float* s_inv, const float* d, void* xq, sq_codes fmt,
                           float* x_scale, uint32_t* clipped, int32_t* flags, cudaStream_t st) {
  return quant_act_any(x, dt, tokens, cin, ldx, s_inv, xq, fmt, x_scale, flags, Static{kStatic, d, clipped, 0.0f}, st);
}

sq_status rmsnorm_quant_act(const void* h, sq_dtype dt, int64_t tokens, int64_t cin, int64_t ldh,
                            const float* gamma_folded, float eps, void* xq, sq_codes fmt,
                            float* x_scale, int32_t* flags, cudaStream_t st) {
  return quant_act_any(h, dt, tokens, cin, ldh, gamma_folded, xq, fmt, x_scale, flags, Static{kNorm, nullptr, nullptr, eps}, st);
}

namespace {
__global__ void k_fold_norm_gain(const float* __restrict__ gamma, const float* __restrict__ s_inv,
                                 int64_t n, float* __restrict__ out) {
  for (int64_t j = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; j < n; j += (int64_t)gridDim.x * blockDim.x)
    out[j] = __fmul_rn(gamma[j], s_inv[j]);
}
}  // namespace

sq_status fold_norm_gain(const float* gamma, const float* s_inv, int64_t cin, float* out,
                         cudaStream_t st) {
  const int g = (int)std::min<int64_t>((cin + 255) / 256, 1024);
  k_fold_norm_gain<<<g, 256, 0, st>>>(gamma, s_inv, cin, out);
  return launch_status();
}

}  // namespace sq

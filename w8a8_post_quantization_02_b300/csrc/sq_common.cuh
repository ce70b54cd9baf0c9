// Shared device/host helpers of the sm_103a SmoothQuant W8A8 library.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>

#include "sq.h"

#define SQ_DEVINL __device__ __forceinline__

namespace sq {

constexpr int kThreads = 256;  // block size of the streaming kernels

// ---------------------------------------------------------------- host side
inline sq_status launch_status() {
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? SQ_OK : SQ_ERR_CUDA;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Kernel attributes (shared-memory limits) are per device: `set` runs once
// for each device the calling thread has current (device ids below 64 are
// remembered in `done`; others run it every time).  Safe to call from
// several host threads: `set` is idempotent.  False if `set` failed.
template <typename F>
inline bool once_per_device(std::atomic<uint64_t>& done, F set) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  const uint64_t bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return true;
  if (set() != cudaSuccess) return false;
  done.fetch_or(bit, std::memory_order_release);
  return true;
}

inline int elem_bytes(sq_dtype dt) { return dt == SQ_F32 ? 4 : 2; }

inline int code_bytes(sq_codes f) { return f == SQ_CODES_BF16 ? 2 : 1; }

// SM count of the current device, queried once per device (ids below 64).
inline int sm_count() {
  static std::atomic<int> cache[64];  // zero-initialized: static storage
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  if (dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// ---------------------------------------------------------------- device side
// 16-byte streaming load that bypasses L1 allocation (read-once data).
SQ_DEVINL uint4 ld_stream16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// 8-byte streaming load that bypasses L1 allocation (read-once data).
SQ_DEVINL uint2 ld_stream8(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}

// 16-byte load through the read-only path (reused data such as s_inv).
SQ_DEVINL uint4 ld_ro16(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

SQ_DEVINL void st16(void* p, uint4 v) {
  asm volatile("st.global.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

SQ_DEVINL void st8(void* p, uint2 v) {
  asm volatile("st.global.v2.u32 [%0], {%1,%2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

SQ_DEVINL float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
SQ_DEVINL float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// |x| as ordered bits: for non-negative floats (and NaN, which sorts above
// +inf) unsigned comparison of the bit patterns orders like the values.
SQ_DEVINL uint32_t abs_bits(float x) { return __float_as_uint(x) & 0x7FFFFFFFu; }

SQ_DEVINL void raise_flag(int32_t* flags, int32_t bit) {
  if (flags) atomicOr(flags, bit);
}

SQ_DEVINL bool finite_bits(uint32_t absb) { return absb < 0x7F800000u; }

// Symmetric INT8 scale for a maximum magnitude: d = amax / 127 (IEEE fp32
// division), 1 when amax == 0, and its reciprocal RN(1/d) (IEEE division),
// which the quotient below refines.
SQ_DEVINL void scale_and_inverse(float amax, float& d, float& inv) {
  d = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 127.0f);
  inv = __fdiv_rn(1.0f, d);
}

// The quantizer's code is rne(RN(v / d)): the IEEE binary32 quotient,
// rounded to the nearest integer.  quot_rn forms that quotient with one
// multiply and four fused multiply-adds instead of a division:
//   q0 = RN(v * y)                     y = RN(1/d), so |q0 - v/d| < 1.5 ulp
//   q1 = RN(q0 + RN(v - d q0) * y)     |q1 - v/d| < 1 ulp (faithful)
//   q2 = RN(q1 + (v - d q1) * y)       the remainder v - d q1 is exact
// and q2 = RN(v / d) by Markstein's theorem (P. Markstein, IBM J. Res. Dev.
// 34(1), 1990; also Cornea, Harrison and Tang, "Scientific Computing on
// Itanium-based Systems", 2002): with y correctly rounded and q1 faithful,
// one residual correction gives the correctly rounded quotient.  Its
// premises hold when d lies in [2^-100, 2^120] and |v / d| <= 256: then
// no product, remainder or correction leaves the normal range (a remainder
// is a multiple of 2^(e_d + e_q - 46) >= 2^-148 whenever |v / d| >= 2^-2,
// and below that every candidate rounds to code 0).  Every caller checks
// those bounds and otherwise takes __fdiv_rn.
SQ_DEVINL float quot_refine(float v, float d, float y, float q0) {
  const float r0 = __fmaf_rn(-d, q0, v);
  const float q1 = __fmaf_rn(r0, y, q0);
  const float r1 = __fmaf_rn(-d, q1, v);
  return __fmaf_rn(r1, y, q1);
}
SQ_DEVINL float quot_rn(float v, float d, float y) { return quot_refine(v, d, y, __fmul_rn(v, y)); }

// A row or channel maximum at or above 2^-93 (and finite) gives
// d = RN(amax / qmax) >= 2^-100 for any qmax <= 127, inside quot_rn's range;
// and since every |v| <= amax, |v / d| <= qmax * (1 + 2^-23), whose
// rounding to an integer never exceeds qmax: no clamp is needed.
constexpr uint32_t kFastAmaxBits = 0x11000000u;  // 2^-93
SQ_DEVINL bool fast_quotient_ok(uint32_t amax_bits) {
  return amax_bits >= kFastAmaxBits && amax_bits < 0x7F800000u;
}
// d within quot_rn's range, for a scale not derived from the values it
// divides (the static activation scale): [2^-100, 2^120].
SQ_DEVINL bool fast_scale_ok(float d) {
  const uint32_t b = __float_as_uint(d);
  return b >= 0x0D800000u && b <= 0x7B800000u;
}

// rne(q) returned as the float q' = code + 1.5*2^23, whose low byte is the
// two's-complement code and whose value minus 1.5*2^23 is the code
// exactly.  The add rounds to nearest-even on the integer grid because
// 1.5*2^23 + [-127.5, 127.5] lies in [2^23, 2^24).
constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
SQ_DEVINL float magic_of(float q) { return __fadd_rn(q, kMagic); }

// clamp(rne(RN(v / d)), -qmax, qmax) as a magic float, for any v and d:
// one IEEE division; a NaN quotient gives code 0, +-inf saturates.
SQ_DEVINL float code_div_magic(float v, float d, float qmax) {
  const float t = __fdiv_rn(v, d);
  return __fadd_rn((t == t) ? fminf(fmaxf(t, -qmax), qmax) : 0.0f, kMagic);
}

SQ_DEVINL uint32_t magic_to_bf16bits(float m) {
  // exact integer value as fp32, then its upper half is the exact bf16
  return __float_as_uint(__fsub_rn(m, kMagic)) >> 16;
}

// Pack the low bytes of four magic floats into one word (code0 in byte 0).
SQ_DEVINL uint32_t pack4_codes(float m0, float m1, float m2, float m3) {
  uint32_t lo = __byte_perm(__float_as_uint(m0), __float_as_uint(m1), 0x0040);
  uint32_t hi = __byte_perm(__float_as_uint(m2), __float_as_uint(m3), 0x0040);
  return __byte_perm(lo, hi, 0x5410);
}

// Four int8 codes (code k in byte k of w) -> the same four integers as
// exact fp16 values: codes 0 and 1 in lo (code 0 in the low half), 2 and 3
// in hi.  Flipping a byte's top bit gives u = code + 128 in [1, 255]; the
// fp16 bit pattern 0x6400 | u is exactly 1024 + u; subtracting 1152
// (0x6480) is exact (both operands within a factor of two) and leaves the
// code.
SQ_DEVINL void codes4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(lo) : "r"(__byte_perm(u, 0x64646464u, 0x4140)), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(hi) : "r"(__byte_perm(u, 0x64646464u, 0x4342)), "r"(0x64806480u));
}

SQ_DEVINL uint32_t pack2_bf16codes(float m0, float m1) {
  return magic_to_bf16bits(m0) | (magic_to_bf16bits(m1) << 16);
}

}  // namespace sq

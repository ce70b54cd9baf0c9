// Step 2: smoothing factors s_j = max|X_j|^a / max|W_j|^(1-a) and 1/s_j.
//
// Source: pith.science review of arXiv 2506.01967 (Smooth Rotation),
// key_machinery: at a = 0.5, s_j = sqrt(max|X_j| / max|W_j|); first page
// ("Move activation scale without changing the real linear map"),
// paragraph 1: the factors must be finite and nonzero.
//
// Each power is returned correctly rounded to fp32, so the result does not
// depend on any library's pow.  The power is evaluated as exp(y * ln x) in
// double-double arithmetic (error-free two-sum / two-product
// transformations, Dekker 1971 and Knuth TAOCP vol. 2), with
//   ln m   = 2 atanh((m-1)/(m+1)) for m in [sqrt(1/2), sqrt(2))   (series)
//   exp r  = (Taylor series of exp(r / 2^10))^(2^10)
// which is accurate to about 2^-95 relative; the double-double value is then
// rounded once to fp32.  That path is slow (fp64 division-heavy), so the
// kernel first tries IEEE sqrt (alpha = 1/2) or a double-precision pow whose
// rounding to fp32 is provably decided (pow_rn32 below).  This file is
// compiled with -fmad=false.
#include <math.h>
#include <string.h>

#include "sq_common.cuh"

namespace sq {
namespace {

// The arithmetic below is also compiled for the host by a self-check, so
// it avoids device-only intrinsics.
#define SQ_HD __host__ __device__ __forceinline__

SQ_HD uint32_t f2u(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}
SQ_HD float u2f(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

struct dd {
  double hi, lo;
};

SQ_HD dd two_sum(double a, double b) {
  double s = a + b;
  double bb = s - a;
  double e = (a - (s - bb)) + (b - bb);
  return {s, e};
}
SQ_HD dd fast_two_sum(double a, double b) {  // requires |a| >= |b|
  double s = a + b;
  return {s, b - (s - a)};
}
SQ_HD dd two_prod(double a, double b) {
  double p = a * b;
  return {p, fma(a, b, -p)};
}
SQ_HD dd dd_add(dd a, dd b) {
  dd s = two_sum(a.hi, b.hi);
  dd t = two_sum(a.lo, b.lo);
  s.lo += t.hi;
  s = fast_two_sum(s.hi, s.lo);
  s.lo += t.lo;
  return fast_two_sum(s.hi, s.lo);
}
SQ_HD dd dd_neg(dd a) { return {-a.hi, -a.lo}; }
SQ_HD dd dd_sub(dd a, dd b) { return dd_add(a, dd_neg(b)); }
SQ_HD dd dd_mul(dd a, dd b) {
  dd p = two_prod(a.hi, b.hi);
  p.lo += a.hi * b.lo;
  p.lo += a.lo * b.hi;
  return fast_two_sum(p.hi, p.lo);
}
SQ_HD dd dd_mul_d(dd a, double b) {
  dd p = two_prod(a.hi, b);
  p.lo += a.lo * b;
  return fast_two_sum(p.hi, p.lo);
}
// a / b by long division with three double quotient digits.
SQ_HD dd dd_div(dd a, dd b) {
  double q1 = a.hi / b.hi;
  dd r = dd_sub(a, dd_mul_d(b, q1));
  double q2 = r.hi / b.hi;
  r = dd_sub(r, dd_mul_d(b, q2));
  double q3 = r.hi / b.hi;
  dd q = fast_two_sum(q1, q2);
  return dd_add(q, dd{q3, 0.0});
}
SQ_HD dd dd_scale2(dd a, int e) { return {ldexp(a.hi, e), ldexp(a.lo, e)}; }

// ln 2 split into two doubles (hi = RN(ln 2), lo = RN(ln 2 - hi)).
constexpr double kLn2Hi = 0x1.62e42fefa39efp-1;
constexpr double kLn2Lo = 0x1.abc9e3b39803fp-56;

// Natural log of a positive normal float, in double-double.
SQ_HD dd ln_dd(float x) {
  uint32_t b = f2u(x);
  int e = (int)((b >> 23) & 0xFF) - 127;
  double m = (double)u2f((b & 0x007FFFFFu) | 0x3F800000u);  // [1, 2)
  if (m > 1.4142135623730951) {
    m *= 0.5;
    e += 1;
  }
  // t = (m - 1) / (m + 1); both operands are exact doubles.
  dd t = dd_div(dd{m - 1.0, 0.0}, dd{m + 1.0, 0.0});
  dd t2 = dd_mul(t, t);
  // sum_{k=0}^{N} t^(2k) / (2k+1) by Horner in t^2; |t| <= 0.1716, so 23
  // terms leave a remainder below 2^-110.
  constexpr int N = 22;
  dd S = dd_div(dd{1.0, 0.0}, dd{2.0 * N + 1.0, 0.0});
  for (int k = N - 1; k >= 0; --k)
    S = dd_add(dd_mul(S, t2), dd_div(dd{1.0, 0.0}, dd{2.0 * k + 1.0, 0.0}));
  dd lnm = dd_mul_d(dd_mul(t, S), 2.0);
  dd eln2 = dd_add(two_prod(kLn2Hi, (double)e), dd{kLn2Lo * (double)e, 0.0});
  return dd_add(eln2, lnm);
}

// exp of a double-double argument with |z| < 700.
SQ_HD dd exp_dd(dd z) {
  double k = rint(z.hi / kLn2Hi);
  dd kln2 = dd_add(two_prod(kLn2Hi, k), dd{kLn2Lo * k, 0.0});
  dd r = dd_scale2(dd_sub(z, kln2), -10);  // |r| <= 0.35 / 1024
  // Taylor series 1 + r (1 + r/2 (1 + r/3 (... (1 + r/9)))) ; the omitted
  // terms are below 2^-110 relative.
  dd acc = {1.0, 0.0};
  for (int i = 9; i >= 1; --i) acc = dd_add(dd{1.0, 0.0}, dd_mul(dd_div(r, dd{(double)i, 0.0}), acc));
  for (int i = 0; i < 10; ++i) acc = dd_mul(acc, acc);
  return dd_scale2(acc, (int)k);
}

// Round a double-double (hi + lo, |lo| <= ulp(hi)/2) to the nearest float,
// ties to even.  Only when hi is itself a float midpoint can lo move the
// result; then the sign of lo decides.
SQ_HD float dd_to_float_rn(dd v) {
  float f = (float)v.hi;  // round-to-nearest-even conversion
  double fd = (double)f;
  if (fd == v.hi || v.lo == 0.0) return f;
  float g = (v.hi > fd) ? nextafterf(f, INFINITY) : nextafterf(f, -INFINITY);
  double mid = 0.5 * (fd + (double)g);  // exact in double
  if (v.hi != mid) return f;
  // hi sits exactly on the midpoint between f and g: lo decides
  bool above = v.lo > 0.0;
  float lo_c = fd < (double)g ? f : g, hi_c = fd < (double)g ? g : f;
  return above ? hi_c : lo_c;
}

// Correctly rounded x^y for finite normal x > 0 and 0 <= y <= 1.
SQ_HD float pow_cr(float x, float y) {
  if (y == 0.0f || x == 1.0f) return 1.0f;
  if (y == 1.0f) return x;
  dd z = dd_mul_d(ln_dd(x), (double)y);
  return dd_to_float_rn(exp_dd(z));
}

// x^y correctly rounded to fp32, cheaply when possible: IEEE sqrt for
// y = 1/2; otherwise CUDA's double-precision pow (documented error <= 2 ulp
// of double, i.e. relative 2^-51) decides the fp32 rounding whenever its
// result lies farther than 2^-48 (relative) from both fp32 rounding
// boundaries around it; only near a boundary is the double-double path run.
SQ_DEVINL float pow_rn32(float x, float y) {
  if (y == 0.0f || x == 1.0f) return 1.0f;
  if (y == 1.0f) return x;
  if (y == 0.5f) return __fsqrt_rn(x);
  const double r = pow((double)x, (double)y);
  const float f = __double2float_rn(r);
  const double fd = (double)f;
  const double m_hi = 0.5 * (fd + (double)nextafterf(f, INFINITY));
  const double m_lo = 0.5 * (fd + (double)nextafterf(f, 0.0f));
  const double tol = r * 0x1p-48;
  if (r - m_lo > tol && m_hi - r > tol) return f;
  return pow_cr(x, y);
}

constexpr int kSmoothThreads = 64;

// Two threads per channel: the even lane of each pair raises max|X_j| to
// alpha, the odd lane max|W_j| to 1 - alpha, so the (double-precision)
// powers of a block run on twice as many warps.
__global__ void __launch_bounds__(kSmoothThreads) k_smooth(const float* __restrict__ amax_x,
                                                     const float* __restrict__ amax_w, int64_t cin,
                                                     float alpha, float* __restrict__ s,
                                                     float* __restrict__ s_inv, int32_t* flags) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t j = t >> 1;
  const bool odd = (t & 1) != 0;
  const bool in = j < cin;
  float ax = in ? amax_x[j] : 1.0f, aw = in ? amax_w[j] : 1.0f;
  const bool finite = isfinite(ax) && isfinite(aw);
  ax = fmaxf(ax, 1e-5f);
  aw = fmaxf(aw, 1e-5f);
  const float beta = __fsub_rn(1.0f, alpha);
  // one call with per-lane operands (not two branches), so the pair does
  // not diverge
  const float mine = finite ? pow_rn32(odd ? aw : ax, odd ? beta : alpha) : 1.0f;
  const float other = __shfl_xor_sync(0xFFFFFFFFu, mine, 1);  // every lane reaches this
  if (!in || odd) return;
  if (!finite) {
    s[j] = 1.0f;
    s_inv[j] = 1.0f;
    raise_flag(flags, SQ_FLAG_NONFINITE);
    return;
  }
  float sj = __fdiv_rn(mine, other);
  sj = fminf(fmaxf(sj, 1e-5f), 1e5f);
  s[j] = sj;
  s_inv[j] = __fdiv_rn(1.0f, sj);
}

}  // namespace

sq_status smooth_factors(const float* amax_x, const float* amax_w, int64_t cin, float alpha,
                         float* s, float* s_inv, int32_t* flags, cudaStream_t st) {
  const int64_t g = (2 * cin + kSmoothThreads - 1) / kSmoothThreads;
  k_smooth<<<(unsigned)g, kSmoothThreads, 0, st>>>(amax_x, amax_w, cin, alpha, s, s_inv, flags);
  return launch_status();
}

}  // namespace sq

// sin and cos of the rotary angles pos * inv_freq, accurate to ~1e-14 plus
// the float64 rounding of the angle itself, with few float64 operations
// (float64 is a narrow pipe on GB300: about 2 fused multiply-adds per SM and
// clock, against 128 in float32).
//
// Method:
//  1. float64: the angle a = pos * inv_freq and one reduction by quarter
//     turns, q = rint(a * 2/pi), x = a - q * pi/2 with pi/2 split in two
//     doubles (Cody-Waite), |x| <= pi/4 (+ rounding); x is passed on as a
//     float-float pair (x_hi + x_lo, x_lo the float of the float64 remainder).
//  2. float32, float-float arithmetic (error-free sums and products via
//     fused multiply-add): with k = round(64 |x|) and d = |x| - k/64
//     (|d| <= 1/128), the addition theorems
//        sin|x| = sin(k/64) cos d + cos(k/64) sin d
//        cos|x| = cos(k/64) cos d - sin(k/64) sin d
//     with sin(k/64), cos(k/64) from a 51-entry float-float table built on
//     the host in long double, and the short series
//        sin d = d - d^3/6 + d^5/120,  cos d = 1 - d^2/2 + d^4/24
//     (truncation below 1e-18 for |d| <= 1/128).
//  3. signs and the quadrant q mod 4 put the result back.
// Host and device share the code so the CPU tests can check it against the
// C library's long-double sin/cos.
#pragma once

#include <cuda_runtime.h>

#include <cmath>

namespace pkvqk {

constexpr int kSinCosKnots = 51;   // k/64 for k = 0 .. 50 covers [0, pi/4 + 1/128]

// sin(k/64) and cos(k/64) as float-float pairs: {sin_hi, sin_lo, cos_hi, cos_lo}.
inline void build_sincos_table(float tab[kSinCosKnots][4]) {
  for (int k = 0; k < kSinCosKnots; ++k) {
    const long double x = static_cast<long double>(k) / 64.0L;
    const long double s = sinl(x), c = cosl(x);
    const float sh = static_cast<float>(s), ch = static_cast<float>(c);
    tab[k][0] = sh;
    tab[k][1] = static_cast<float>(s - static_cast<long double>(sh));
    tab[k][2] = ch;
    tab[k][3] = static_cast<float>(c - static_cast<long double>(ch));
  }
}

// ------------------------------------------------ float-float arithmetic

// Separately rounded float32 add/multiply: on the device never fused into a
// multiply-add by the compiler (the error-free transforms depend on it); the
// host build of the CPU check disables contraction.
#ifdef __CUDA_ARCH__
#define PKVQK_ADD(a, b) __fadd_rn((a), (b))
#define PKVQK_SUB(a, b) __fsub_rn((a), (b))
#define PKVQK_MUL(a, b) __fmul_rn((a), (b))
#else
#define PKVQK_ADD(a, b) ((a) + (b))
#define PKVQK_SUB(a, b) ((a) - (b))
#define PKVQK_MUL(a, b) ((a) * (b))
#endif

struct FF {
  float hi, lo;
};

// s + e = a + b exactly (any magnitudes).
__host__ __device__ __forceinline__ FF two_sum(float a, float b) {
  const float s = PKVQK_ADD(a, b);
  const float bb = PKVQK_SUB(s, a);
  const float e = PKVQK_ADD(PKVQK_SUB(a, PKVQK_SUB(s, bb)), PKVQK_SUB(b, bb));
  return {s, e};
}

// s + e = a + b exactly, for |a| >= |b| (or a == 0).
__host__ __device__ __forceinline__ FF fast_two_sum(float a, float b) {
  const float s = PKVQK_ADD(a, b);
  return {s, PKVQK_SUB(b, PKVQK_SUB(s, a))};
}

__host__ __device__ __forceinline__ FF ff_mul(FF a, FF b) {
  const float p = PKVQK_MUL(a.hi, b.hi);
  float e = fmaf(a.hi, b.hi, -p);                 // a.hi * b.hi = p + e exactly
  e = fmaf(a.hi, b.lo, fmaf(a.lo, b.hi, e));
  return fast_two_sum(p, e);
}

__host__ __device__ __forceinline__ FF ff_add(FF a, FF b) {
  FF s = two_sum(a.hi, b.hi);
  return fast_two_sum(s.hi, PKVQK_ADD(s.lo, PKVQK_ADD(a.lo, b.lo)));
}

// ------------------------------------------------------------ the angles

// Step 1: the angle pos * inv_freq reduced by quarter turns; returns q mod 4
// and |x| <= pi/4 (+ rounding) as a float-float pair.
__host__ __device__ __forceinline__ int reduce_angle(double pos, double inv_freq, FF* x) {
  const double kPiO2Hi = 1.5707963267948966;          // pi/2 rounded to double
  const double kPiO2Lo = 6.123233995736766e-17;       // pi/2 - kPiO2Hi
  const double kTwoOverPi = 0.63661977236758134;
  const double a = pos * inv_freq;
  const double q = rint(a * kTwoOverPi);
  double r = fma(-q, kPiO2Hi, a);
  r = fma(-q, kPiO2Lo, r);
  const float hi = static_cast<float>(r);
  x->hi = hi;
  x->lo = static_cast<float>(r - static_cast<double>(hi));
  return static_cast<int>(static_cast<long long>(q) & 3);
}

// Steps 2 and 3: sin and cos of x + quadrant * pi/2 as float-float pairs.
// tab: build_sincos_table's values (any memory the caller can index).
__host__ __device__ __forceinline__ void sincos_ff(FF x, int quadrant,
                                                   const float (*tab)[4], FF* s_out,
                                                   FF* c_out) {
  const bool neg = x.hi < 0.f;
  if (neg) {
    x.hi = -x.hi;
    x.lo = -x.lo;
  }
  int k = static_cast<int>(x.hi * 64.f + 0.5f);
  k = k < 0 ? 0 : (k > kSinCosKnots - 1 ? kSinCosKnots - 1 : k);
  // d = x - k/64: x.hi - k/64 is exact (the two are within a factor of 2,
  // or k == 0)
  const FF d = fast_two_sum(PKVQK_SUB(x.hi, static_cast<float>(k) * (1.f / 64.f)), x.lo);
  // sin d = d + d^3 (-1/6 + d^2/120); the correction is below 7e-8, so the
  // float32 evaluation from d.hi is accurate to ~1e-15
  const float d2 = PKVQK_MUL(d.hi, d.hi);
  const float sc = d.hi * d2 * fmaf(d2, 1.f / 120.f, -1.f / 6.f);
  const FF sd = fast_two_sum(d.hi, PKVQK_ADD(d.lo, sc));
  // cos d = 1 - d^2/2 + d^4/24 with d^2 as an exact product plus tail
  float e2 = fmaf(d.hi, d.hi, -d2);
  e2 = fmaf(2.f * d.hi, d.lo, e2);
  FF cd = two_sum(1.f, -0.5f * d2);
  cd = fast_two_sum(cd.hi, PKVQK_ADD(cd.lo, fmaf(d2 * d2, 1.f / 24.f, -0.5f * e2)));
  const FF sk = {tab[k][0], tab[k][1]}, ck = {tab[k][2], tab[k][3]};
  FF sn = ff_add(ff_mul(sk, cd), ff_mul(ck, sd));
  const FF m = ff_mul(sk, sd);
  FF cs = ff_add(ff_mul(ck, cd), FF{-m.hi, -m.lo});
  if (neg) {
    sn.hi = -sn.hi;
    sn.lo = -sn.lo;
  }
  // (sin, cos)(x + quadrant * pi/2)
  const FF sv = (quadrant & 1) ? cs : sn;
  const FF cv = (quadrant & 1) ? sn : cs;
  *s_out = (quadrant & 2) ? FF{-sv.hi, -sv.lo} : sv;
  *c_out = ((quadrant + 1) & 2) ? FF{-cv.hi, -cv.lo} : cv;
}

}  // namespace pkvqk

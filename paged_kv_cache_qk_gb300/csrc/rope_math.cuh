// sin and cos of a reduced rotary angle, to ~1e-15 absolute, with few
// float64 operations (float64 is a narrow pipe on GB300).
//
// Method: Taylor series of sin and cos about 0 (the Maclaurin series), after
// reducing the angle to |x| <= pi/4 by quarter turns.  The leading terms run
// in float64; each series' tail, a few 1e-7 of the result at most, runs in
// float32, whose relative error there is below 1e-14 of the result.
//   sin x = x + x^3 (-1/3! + x^2 (1/5! + x^2 (-1/7! + x^2 Qs(x^2))))
//   cos x = 1 + x^2 (-1/2! + x^2 (1/4! + x^2 (-1/6! + x^2 (1/8! + x^2 Qc(x^2)))))
//   Qs(y) = 1/9! - y/11! + y^2/13! - y^3/15!   (float32; truncation < 1e-15)
//   Qc(y) = -1/10! + y/12! - y^2/14!        (float32; truncation < 2e-15)
// Host and device share the code so the CPU tests can check it against the C
// library's long-double sin/cos.
#pragma once

#include <cuda_runtime.h>

#include <cmath>

namespace pkvqk {

// Input: |red| <= pi (+ rounding), e.g. an angle reduced by whole turns.
__host__ __device__ inline void sincos_reduced(double red, double* s_out, double* c_out) {
  const double kPiO2Hi = 1.5707963267948966;          // pi/2 rounded to double
  const double kPiO2Lo = 6.123233995736766e-17;       // pi/2 - kPiO2Hi
  const double kTwoOverPi = 0.63661977236758134;
  const double q = rint(red * kTwoOverPi);            // quarter turns, in {-2, ..., 2}
  double x = fma(-q, kPiO2Hi, red);
  x = fma(-q, kPiO2Lo, x);                            // |x| <= pi/4 (+ rounding)
  const double y = x * x;
  const float yf = static_cast<float>(y);
  // float32 tails
  const float qs = fmaf(fmaf(fmaf(yf, -7.6471637318198164e-13f, 1.6059043836821613e-10f), yf,
                             -2.5052108385441720e-08f),
                        yf, 2.7557319223985893e-06f);
  const float qc = fmaf(fmaf(yf, -1.1470745597729725e-11f, 2.0876756987868099e-09f), yf,
                        -2.7557319223985888e-07f);
  // float64 leading terms
  double ps = fma(y, static_cast<double>(qs), -1.9841269841269841e-04);
  ps = fma(y, ps, 8.3333333333333333e-03);
  ps = fma(y, ps, -1.6666666666666667e-01);
  const double sx = fma(x * y, ps, x);
  double pc = fma(y, static_cast<double>(qc), 2.4801587301587302e-05);
  pc = fma(y, pc, -1.3888888888888889e-03);
  pc = fma(y, pc, 4.1666666666666667e-02);
  pc = fma(y, pc, -0.5);
  const double cx = fma(y, pc, 1.0);
  // undo the quarter turns: (sin, cos)(x + q pi/2)
  const int k = static_cast<int>(q) & 3;
  const double sv = (k & 1) ? cx : sx;
  const double cv = (k & 1) ? sx : cx;
  *s_out = (k & 2) ? -sv : sv;
  *c_out = ((k + 1) & 2) ? -cv : cv;
}

}  // namespace pkvqk

// Host-side check of the rotary sin/cos of rope_math.cuh against the C
// library's long-double sin/cos.  Prints
//   (1) the largest absolute errors of sincos_ff over reduced angles in
//       [-pi/4, pi/4] (every quadrant, knot edges included),
//   (2) the largest absolute errors of the whole path reduce_angle +
//       sincos_ff for the RoPE angles pos * theta^(-2i/128), theta = 1e6,
//       pos in [0, 65535], against sinl/cosl of the exact product.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include "../../paged_kv_cache_qk_gb300/csrc/rope_math.cuh"

int main(int argc, char** argv) {
  const long n = argc > 1 ? atol(argv[1]) : 2000000;
  float tab[pkvqk::kSinCosKnots][4];
  pkvqk::build_sincos_table(tab);
  const double pi = 3.14159265358979323846;
  uint64_t st = 88172645463325252ull;
  auto rnd = [&]() {
    st ^= st << 13; st ^= st >> 7; st ^= st << 17;
    return (st >> 11) * (1.0 / 9007199254740992.0);   // [0, 1)
  };
  // (1) reduced angles, given as float-float pairs
  double es = 0, ec = 0;
  auto check_reduced = [&](double r, int quad) {
    pkvqk::FF x{static_cast<float>(r), 0.f};
    x.lo = static_cast<float>(r - static_cast<double>(x.hi));
    pkvqk::FF s, c;
    pkvqk::sincos_ff(x, quad, tab, &s, &c);
    const long double a = static_cast<long double>(r) + quad * (static_cast<long double>(pi) / 2);
    const long double aa = static_cast<long double>(r) + quad * 1.5707963267948966192313216916397514L;
    (void)a;
    const double ds = std::fabs(static_cast<double>((static_cast<long double>(s.hi) + s.lo) - sinl(aa)));
    const double dc = std::fabs(static_cast<double>((static_cast<long double>(c.hi) + c.lo) - cosl(aa)));
    if (ds > es) es = ds;
    if (dc > ec) ec = dc;
  };
  for (long i = 0; i < n; ++i) check_reduced((2 * rnd() - 1) * pi / 4, static_cast<int>(i & 3));
  for (int k = -51; k <= 51; ++k)
    for (double e : {0.0, 0.5 / 64, -0.5 / 64, 0.49999 / 64, -0.49999 / 64, 1e-12, -1e-12}) {
      const double r = k / 64.0 + e;
      if (std::fabs(r) <= pi / 4 + 1e-9)
        for (int q = 0; q < 4; ++q) check_reduced(r, q);
    }
  // (2) the whole path on RoPE angles
  double fs = 0, fc = 0;
  for (long j = 0; j < n / 8; ++j) {
    const int i = static_cast<int>(rnd() * 64);
    const double pos = std::floor(rnd() * 65536.0);
    const double inv_freq = std::pow(1.0e6, -2.0 * i / 128.0);
    pkvqk::FF x, s, c;
    const int q = pkvqk::reduce_angle(pos, inv_freq, &x);
    pkvqk::sincos_ff(x, q, tab, &s, &c);
    const long double a = static_cast<long double>(pos) * static_cast<long double>(inv_freq);
    const double ds = std::fabs(static_cast<double>((static_cast<long double>(s.hi) + s.lo) - sinl(a)));
    const double dc = std::fabs(static_cast<double>((static_cast<long double>(c.hi) + c.lo) - cosl(a)));
    if (ds > fs) fs = ds;
    if (dc > fc) fc = dc;
  }
  std::printf("%.3e %.3e %.3e %.3e\n", es, ec, fs, fc);
  return 0;
}

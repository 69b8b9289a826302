// Host-side check of pkvqk::sincos_reduced against the C library's
// long-double sin/cos: prints the largest absolute errors over a sweep of
// reduced angles in [-pi, pi] and some edge values.
#include <cmath>
#include <cstdio>
#include <cstdint>
#include "../../paged_kv_cache_qk_gb300/csrc/rope_math.cuh"

int main(int argc, char** argv) {
  const long n = argc > 1 ? atol(argv[1]) : 2000000;
  const double pi = 3.14159265358979323846;
  double es = 0, ec = 0, worst_s = 0, worst_c = 0;
  uint64_t st = 88172645463325252ull;
  auto check = [&](double r) {
    double s, c;
    pkvqk::sincos_reduced(r, &s, &c);
    const long double rl = r;
    const double ds = std::fabs(static_cast<double>(static_cast<long double>(s) - sinl(rl)));
    const double dc = std::fabs(static_cast<double>(static_cast<long double>(c) - cosl(rl)));
    if (ds > es) { es = ds; worst_s = r; }
    if (dc > ec) { ec = dc; worst_c = r; }
  };
  for (long i = 0; i < n; ++i) {
    st ^= st << 13; st ^= st >> 7; st ^= st << 17;
    const double u = (st >> 11) * (1.0 / 9007199254740992.0);   // [0, 1)
    check((2 * u - 1) * pi);
  }
  const double edges[] = {0.0, -0.0, 1e-300, -1e-20, pi, -pi, pi / 4, -pi / 4, pi / 2, -pi / 2,
                          3 * pi / 4, -3 * pi / 4, 0.7853981633974483, 0.7853981633974484,
                          2.356194490192345, 3.141592653589793};
  for (double e : edges) check(e);
  std::printf("%.3e %.3e %.17g %.17g\n", es, ec, worst_s, worst_c);
  return 0;
}

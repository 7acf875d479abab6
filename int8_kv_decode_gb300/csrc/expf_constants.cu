// Host-side constants of the table-driven exp used by exact mode
// ("Kestrel_VLLM - 18" §3.3: 64-entry table of 2^(j/64), K = 64/ln2,
// C2 = ln2/64, C0 = 1/6, C1 = 1/2, each rounded to nearest double).
//
// They are derived here in double-double arithmetic (about 104 significant
// bits) from first principles, then rounded once to double:
//   ln2      = 2 atanh(1/3) = 2 sum_k (1/3)^(2k+1) / (2k+1)
//   2^(1/64) = six nested square roots of 2 (Newton steps in double-double)
//   T[j]     = (2^(1/64))^j by repeated double-double products
// This file must be built without floating-point contraction so that the
// error-free transformations below stay exact (-ffp-contract=off, --fmad=false).
#include <cmath>

#include "kattn_internal.cuh"

namespace kattn {
namespace {

struct dd {
  double hi, lo;
};

dd two_sum(double a, double b) {
  const double s = a + b;
  const double bb = s - a;
  const double e = (a - (s - bb)) + (b - bb);
  return {s, e};
}

dd quick_two_sum(double a, double b) {
  const double s = a + b;
  return {s, b - (s - a)};
}

dd two_prod(double a, double b) {
  const double p = a * b;
  return {p, std::fma(a, b, -p)};
}

dd add(dd a, dd b) {
  dd s = two_sum(a.hi, b.hi);
  s.lo += a.lo + b.lo;
  return quick_two_sum(s.hi, s.lo);
}

dd mul(dd a, dd b) {
  dd p = two_prod(a.hi, b.hi);
  p.lo += a.hi * b.lo + a.lo * b.hi;
  return quick_two_sum(p.hi, p.lo);
}

dd div(dd a, dd b) {
  const double q1 = a.hi / b.hi;
  dd r = add(a, mul(b, dd{-q1, 0.0}));
  const double q2 = r.hi / b.hi;
  r = add(r, mul(b, dd{-q2, 0.0}));
  const double q3 = r.hi / b.hi;
  return add(quick_two_sum(q1, q2), dd{q3, 0.0});
}

dd sqrt_dd(dd a) {
  dd x{std::sqrt(a.hi), 0.0};
  for (int it = 0; it < 3; ++it) {  // x <- (x + a/x) / 2
    const dd t = add(x, div(a, x));
    x = dd{t.hi * 0.5, t.lo * 0.5};
  }
  return x;
}

dd ln2_dd() {
  // 2 * sum_{k>=0} u^(2k+1)/(2k+1), u = 1/3; terms fall by 9x each.
  const dd u = div(dd{1.0, 0.0}, dd{3.0, 0.0});
  const dd u2 = mul(u, u);
  dd pw = u, sum{0.0, 0.0};
  for (int k = 0; k < 40; ++k) {
    sum = add(sum, div(pw, dd{(double)(2 * k + 1), 0.0}));
    pw = mul(pw, u2);
  }
  return dd{sum.hi * 2.0, sum.lo * 2.0};
}

// Round a normalised double-double to the nearest double.
double to_double(dd a) { return a.hi + a.lo; }

ExpfConsts build() {
  ExpfConsts c{};
  const dd ln2 = ln2_dd();
  c.K = to_double(div(dd{64.0, 0.0}, ln2));
  c.C2 = to_double(ln2) / 64.0;  // exact scaling by a power of two
  c.C0 = 1.0 / 6.0;              // IEEE division is correctly rounded
  c.C1 = 0.5;
  dd root{2.0, 0.0};
  for (int i = 0; i < 6; ++i) root = sqrt_dd(root);
  dd pw{1.0, 0.0};
  for (int j = 0; j < 64; ++j) {
    c.T[j] = to_double(pw);
    pw = mul(pw, root);
  }
  return c;
}

}  // namespace

const ExpfConsts& expf_constants() {
  static const ExpfConsts c = build();
  return c;
}

}  // namespace kattn

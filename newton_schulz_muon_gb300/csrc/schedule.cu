// Per-iteration Newton-Schulz coefficients (host only).
//
// DeepSpeed issue "[RFC] Enable Correct and High-Performance Muon Optimizer under
// ZeRO CPU Offload", follow-up list: Newton-Schulz with per-iteration optimised
// coefficients ("Polar Express", arXiv:2505.16932) as an ns_method option, so
// that fewer iterations reach the same polar-factor accuracy.  The pages print no
// coefficients; the construction here is the greedy minimax one: iteration k
// uses the odd quintic p_k(x) = a x + b x^3 + c x^5 minimising max |1 - p_k(x)|
// on the interval [l_k, s u_k] that holds the singular values (s >= 1 a safety
// widening), and the next interval is its image [1 - E_k, 1 + E_k].  After the
// Frobenius normalisation the singular values lie in (0, 1], so u_0 = 1 and l_0
// is the caller's lower bound.
//
// The minimax quintic is found by the exchange (Remez) iteration on the basis
// x, x^3, x^5: on a reference of four points solve p(t_i) + (-1)^i E = 1; move
// the reference to the interval ends and the critical points of p inside (the
// roots of p'(x) = a + 3 b x^2 + 5 c x^4, a quadratic in x^2); stop when the
// largest error there equals |E|.  On an interval shorter than 1e-4 the basis is
// nearly dependent (fits differ in coefficients, not in their ~1e-13 errors) and
// the fit tends to the quintic flat to third order at 1, (15 x - 10 x^3 + 3 x^5)
// / 8, which is used there.
#include <cmath>
#include <cstdint>

#include "kernels.h"
#include "muon.h"

namespace muon {
namespace {

// 4 x 4 linear solve by Gaussian elimination with partial pivoting; false if singular.
bool solve4(double m[4][5], double out[4]) {
  for (int col = 0; col < 4; ++col) {
    int piv = col;
    for (int r = col + 1; r < 4; ++r)
      if (std::fabs(m[r][col]) > std::fabs(m[piv][col])) piv = r;
    if (std::fabs(m[piv][col]) < 1e-300) return false;
    if (piv != col)
      for (int c = 0; c < 5; ++c) std::swap(m[piv][c], m[col][c]);
    for (int r = 0; r < 4; ++r) {
      if (r == col) continue;
      const double f = m[r][col] / m[col][col];
      for (int c = col; c < 5; ++c) m[r][c] -= f * m[col][c];
    }
  }
  for (int i = 0; i < 4; ++i) out[i] = m[i][4] / m[i][i];
  return true;
}

double err_at(const double co[3], double x) {
  const double x2 = x * x;
  return 1.0 - x * (co[0] + x2 * (co[1] + x2 * co[2]));
}

// Odd quintic closest to 1 in the max norm on [lo, hi]; returns the largest
// |1 - p| reached on the interval (ends and interior critical points).
double minimax_quintic(double lo, double hi, double co[3]) {
  if (hi - lo < 1e-4) {  // nearly dependent basis: the flat quintic, error ~2.5 ((hi - lo) / 2)^3
    co[0] = 15.0 / 8.0;
    co[1] = -10.0 / 8.0;
    co[2] = 3.0 / 8.0;
    return std::fmax(std::fabs(err_at(co, lo)), std::fabs(err_at(co, hi)));
  }
  double t[4];
  for (int i = 0; i < 4; ++i) t[i] = lo + (hi - lo) * (1.0 - std::cos(3.14159265358979323846 * i / 3.0)) / 2.0;
  double E = 0.0, worst = 0.0;
  for (int iter = 0; iter < 100; ++iter) {
    double m[4][5], sol[4];
    for (int i = 0; i < 4; ++i) {
      m[i][0] = t[i];
      m[i][1] = t[i] * t[i] * t[i];
      m[i][2] = m[i][1] * t[i] * t[i];
      m[i][3] = (i & 1) ? -1.0 : 1.0;
      m[i][4] = 1.0;
    }
    if (!solve4(m, sol)) break;
    co[0] = sol[0];
    co[1] = sol[1];
    co[2] = sol[2];
    E = sol[3];
    // critical points: 5 c y^2 + 3 b y + a = 0, y = x^2
    double crit[2];
    int nc = 0;
    const double qa = 5.0 * co[2], qb = 3.0 * co[1], qc = co[0];
    const double disc = qb * qb - 4.0 * qa * qc;
    if (qa != 0.0 && disc >= 0.0) {
      const double sq = std::sqrt(disc);
      // the numerically stable pair of roots
      const double q = -0.5 * (qb + std::copysign(sq, qb));
      const double ys[2] = {q / qa, q != 0.0 ? qc / q : 0.0};
      for (double y : ys) {
        if (y <= 0.0) continue;
        const double x = std::sqrt(y);
        if (x > lo && x < hi) crit[nc++] = x;
      }
    }
    if (nc == 2 && crit[0] > crit[1]) std::swap(crit[0], crit[1]);
    worst = std::fmax(std::fabs(err_at(co, lo)), std::fabs(err_at(co, hi)));
    for (int i = 0; i < nc; ++i) worst = std::fmax(worst, std::fabs(err_at(co, crit[i])));
    if (nc != 2) break;  // no interior pair to exchange with: keep this fit
    t[0] = lo;
    t[1] = crit[0];
    t[2] = crit[1];
    t[3] = hi;
    if (worst - std::fabs(E) <= 1e-14 * std::fmax(1.0, std::fabs(E))) break;
  }
  return worst;
}

}  // namespace
}  // namespace muon

extern "C" muon_status muon_polar_express_coefficients(int32_t n_iters, double lower, double safety,
                                                       float* coeffs_out, double* err_out) {
  using namespace muon;
  if (!coeffs_out) return set_error(MUON_ERR_INVALID, "NULL coefficient buffer");
  if (n_iters < 1 || n_iters > MUON_MAX_NS_STEPS)
    return set_error(MUON_ERR_INVALID, "n_iters must be in [1, 16]");
  if (!(lower > 0.0 && lower < 1.0)) return set_error(MUON_ERR_INVALID, "lower must be in (0, 1)");
  if (!(safety >= 1.0 && safety <= 2.0)) return set_error(MUON_ERR_INVALID, "safety must be in [1, 2]");
  double lo = lower, hi = 1.0;
  for (int k = 0; k < n_iters; ++k) {
    double co[3];
    const double e = minimax_quintic(lo, hi * safety, co);
    if (!std::isfinite(e) || !std::isfinite(co[0]) || !std::isfinite(co[1]) || !std::isfinite(co[2]))
      return set_error(MUON_ERR_INVALID, "the minimax fit did not converge");
    for (int j = 0; j < 3; ++j) coeffs_out[3 * k + j] = (float)co[j];
    if (err_out) err_out[k] = e;
    lo = 1.0 - e;
    hi = 1.0 + e;
    if (lo <= 0.0) return set_error(MUON_ERR_INVALID, "lower bound too small for a quintic step");
  }
  return MUON_OK;
}

// fp32 momentum with the rounding of one correctly rounded operation, shared by
// the momentum kernel and the small-matrix Newton-Schulz kernel (which computes
// the momentum in its first pass): mu*m and w*g are split exactly into (high,
// low) pairs with fma, then added as double-word numbers (Joldes, Muller,
// Popescu, "Tight and rigorous error bounds for basic building blocks of
// double-word arithmetic", 2017, accurate DW+DW).  The high word of the result is
// within 3u^2 relative of the exact value, so it is the nearest float or its
// neighbour: within 1 ulp.
#pragma once

namespace muon {
namespace {

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bp = __fsub_rn(s, a);
  const float ap = __fsub_rn(s, bp);
  e = __fadd_rn(__fsub_rn(a, ap), __fsub_rn(b, bp));
}

__device__ __forceinline__ void fast_two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  e = __fsub_rn(b, __fsub_rn(s, a));
}

// mu * m + w * g (w = 1 - mu for the EMA form, 1 for the SGD form)
__device__ __forceinline__ float dot2_accurate(float mu, float m, float w, float g) {
  const float ph = __fmul_rn(mu, m), pl = __fmaf_rn(mu, m, -ph);
  const float qh = __fmul_rn(w, g), ql = __fmaf_rn(w, g, -qh);
  float sh, sl, th, tl, vh, vl, zh, zl;
  two_sum(ph, qh, sh, sl);
  two_sum(pl, ql, th, tl);
  fast_two_sum(sh, __fadd_rn(sl, th), vh, vl);
  fast_two_sum(vh, __fadd_rn(tl, vl), zh, zl);
  return zh;
}

// The Newton-Schulz input: Nesterov look-ahead mu * M_new + w * g, or M_new.
__device__ __forceinline__ float nesterov_input(int nesterov, float mu, float m_new, float w, float g) {
  return nesterov ? __fmaf_rn(mu, m_new, __fmul_rn(w, g)) : m_new;
}

}  // namespace
}  // namespace muon

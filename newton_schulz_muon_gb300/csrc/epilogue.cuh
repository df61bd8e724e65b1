// Epilogue pieces shared by the Newton-Schulz kernels: bf16 packing and the
// weight update applied from the last iteration's accumulators.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"

namespace muon {
namespace {

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// Fused weight update for 32 consecutive columns [c0, c0 + valid) of row r of
// U (the last iteration's output, wide orientation) of bucket-local matrix `mat`:
//   apply: W <- W - lr (s U + wd W), s = sqrt(max(1, rows/cols)), in the caller's
//          layout (U transposed back for tall matrices);
//   emit:  U' = s U in fp32, in the same layout.
// Sources: "Muon Optimizer + FSDP", section 背景 (W_t = W_t - lr * U_t).
__device__ __forceinline__ void fused_apply_chunk(const ApplyArgs& A, int mat, int64_t r, int64_t c0, int64_t valid,
                                                  const float (&u)[32]) {
  int lo = 0, hi = A.n_segs - 1;
  while (lo < hi) {  // last run with mat0 <= mat
    const int mid = (lo + hi + 1) >> 1;
    if (A.seg[mid].mat0 <= mat) lo = mid; else hi = mid - 1;
  }
  const ApplySeg& S = A.seg[lo];
  if (!A.emit && A.skip_nonfinite && A.flags[mat]) return;
  const int64_t base = (int64_t)(mat - S.mat0) * S.stride;
  const float sc = S.shape_scale;
  const int n = valid < 32 ? (int)valid : 32;
  // element j of the chunk lives at base + off0 + j * step in the caller's layout:
  // a wide matrix keeps U's row (step 1), a tall one is U transposed (step = cols)
  const int64_t off0 = S.transposed ? c0 * S.cols + r : r * S.cols + c0;
  const int64_t step = S.transposed ? S.cols : 1;
  if (A.emit) {
    float* out = reinterpret_cast<float*>(S.w) + base + off0;
    if (!S.transposed && n == 32 && ((S.cols & 3) == 0) && ((S.stride & 3) == 0)) {
#pragma unroll
      for (int q = 0; q < 8; ++q)
        reinterpret_cast<float4*>(out)[q] =
            make_float4(sc * u[4 * q], sc * u[4 * q + 1], sc * u[4 * q + 2], sc * u[4 * q + 3]);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < n) out[j * step] = sc * u[j];
    }
    return;
  }
  if (A.param_dtype == 0) {
    float* w = reinterpret_cast<float*>(S.w) + base + off0;
    float x[32];
    if (!S.transposed && n == 32 && ((S.cols & 3) == 0) && ((S.stride & 3) == 0)) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 t = reinterpret_cast<const float4*>(w)[q];
        x[4 * q] = t.x; x[4 * q + 1] = t.y; x[4 * q + 2] = t.z; x[4 * q + 3] = t.w;
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] = __fmaf_rn(-A.lr, __fmaf_rn(sc, u[j], __fmul_rn(A.wd, x[j])), x[j]);
#pragma unroll
      for (int q = 0; q < 8; ++q)
        reinterpret_cast<float4*>(w)[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    } else {
      // all loads first, then all stores: the 32 addresses are distinct
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] = j < n ? w[j * step] : 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (j < n) w[j * step] = __fmaf_rn(-A.lr, __fmaf_rn(sc, u[j], __fmul_rn(A.wd, x[j])), x[j]);
    }
  } else {
    __nv_bfloat16* w = reinterpret_cast<__nv_bfloat16*>(S.w) + base + off0;
    if (!S.transposed && n == 32 && ((S.cols & 7) == 0) && ((S.stride & 7) == 0)) {
      // the row's 32 weights are 64 contiguous, 16-byte aligned bytes
      uint4 raw[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) raw[q] = reinterpret_cast<const uint4*>(w)[q];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t h[4] = {raw[q].x, raw[q].y, raw[q].z, raw[q].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162*>(&h[e]);
          const int j = 8 * q + 2 * e;
          const float x0 = __low2float(p), x1 = __high2float(p);
          h[e] = pack_bf16x2(__fmaf_rn(-A.lr, __fmaf_rn(sc, u[j], __fmul_rn(A.wd, x0)), x0),
                             __fmaf_rn(-A.lr, __fmaf_rn(sc, u[j + 1], __fmul_rn(A.wd, x1)), x1));
        }
        raw[q] = make_uint4(h[0], h[1], h[2], h[3]);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) reinterpret_cast<uint4*>(w)[q] = raw[q];
      return;
    }
    // a tall matrix's column of W is contiguous across the lanes of a warp
    float x[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = j < n ? __bfloat162float(w[j * step]) : 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j)
      if (j < n) w[j * step] = __float2bfloat16_rn(__fmaf_rn(-A.lr, __fmaf_rn(sc, u[j], __fmul_rn(A.wd, x[j])), x[j]));
  }
}

}  // namespace
}  // namespace muon

// HBM-bound kernels of the Muon step on sm_103a:
//
//  * momentum_prep: fused fp32 momentum update (EMA or SGD form) with optional
//    Nesterov look-ahead, sum of squares of the Newton-Schulz input V for the
//    Frobenius norm (warp shuffles, fixed-order block reduction, one partial per
//    tile), and the bf16 (or tf32 hi/lo) cast of V into the workspace in wide
//    orientation (transposed through shared memory when rows > cols).
//    Sources: "Muon Optimizer + FSDP", section 背景 (M_t = momentum_update(grad)
//    feeds NewtonSchulz); section 内存控制方案 item 4 (bf16 Newton-Schulz buffers,
//    normalisation scalars kept in fp32).
//  * norm_finalize: per matrix (one block), sums its tile partials in a fixed order (fp64),
//    and stores s = 1 / (||V||_F + eps) and a non-finite flag.  s is folded into
//    the first Newton-Schulz iteration's GEMM epilogues instead of rescaling X0.
//  * apply: W <- W - lr (sqrt(max(1, rows/cols)) U + wd W), un-transposing U
//    through shared memory for tall matrices ("Muon Optimizer + FSDP", 背景:
//    W_t = W_t - lr * U_t); or, for the offload path, U' = sqrt(max(1,rows/cols)) U
//    written in fp32 for the host.
//
// Every kernel works on 64 x 64 tiles of one logical matrix (rows x cols, the
// caller's layout).  Full tiles of aligned matrices use 16-byte accesses.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "device.cuh"
#include "kernels.h"
#include "epilogue.cuh"
#include "momentum.cuh"

namespace muon {
namespace {

constexpr int kT = kPrepTile;       // 64
constexpr int kThreads = 256;       // 16 x 16 threads, 4 x 4 elements each

struct Tile {
  int seg;
  int64_t mat;   // matrix within the run
  int64_t r0, c0;
};

template <typename Seg>
__device__ __forceinline__ Tile decode_tile(const Seg* segs, int n_segs, int64_t t) {
  int lo = 0, hi = n_segs - 1;
  while (lo < hi) {  // last segment with block0 <= t
    const int mid = (lo + hi + 1) >> 1;
    if (segs[mid].block0 <= t) lo = mid; else hi = mid - 1;
  }
  const Seg& s = segs[lo];
  const int64_t local = t - s.block0;
  Tile tile;
  tile.seg = lo;
  tile.mat = local / s.tiles_per_mat;
  const int64_t tt = local % s.tiles_per_mat;
  tile.r0 = (tt / s.tiles_c) * kT;
  tile.c0 = (tt % s.tiles_c) * kT;
  return tile;
}

__device__ __forceinline__ float load_grad(const void* g, int64_t i, int dtype) {
  if (dtype == 1) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(g)[i]);
  return reinterpret_cast<const float*>(g)[i];
}

__device__ __forceinline__ void store_x(void* x_hi, float* x_lo, int64_t i, float v, int tf32) {
  if (tf32) {
    const float h = round_tf32(v);
    reinterpret_cast<float*>(x_hi)[i] = h;
    x_lo[i] = v - h;
  } else {
    reinterpret_cast<__nv_bfloat16*>(x_hi)[i] = __float2bfloat16_rn(v);
  }
}

// Eight consecutive elements of X0 from index i (a multiple of 8 in a row of whole
// 16-byte units): one 16-byte bf16 store, or two for each of the tf32 hi and lo parts.
__device__ __forceinline__ void store_x8(void* x_hi, float* x_lo, int64_t i, const float v[8], int tf32) {
  if (tf32) {
    float h[8], l[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      h[j] = round_tf32(v[j]);
      l[j] = v[j] - h[j];
    }
    float4* hp = reinterpret_cast<float4*>(reinterpret_cast<float*>(x_hi) + i);
    float4* lp = reinterpret_cast<float4*>(x_lo + i);
    hp[0] = make_float4(h[0], h[1], h[2], h[3]);
    hp[1] = make_float4(h[4], h[5], h[6], h[7]);
    lp[0] = make_float4(l[0], l[1], l[2], l[3]);
    lp[1] = make_float4(l[4], l[5], l[6], l[7]);
  } else {
    *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(x_hi) + i) =
        make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                   pack_bf16x2(v[6], v[7]));
  }
}

// Thread (tx, ty) of a 64 x 64 tile: rows ty and ty + 32, columns 8 tx .. 8 tx + 7,
// so that a full tile of a matrix whose rows are whole 16-byte units moves with
// 16-byte accesses (bf16 G and X0: one per row; fp32 M: two per row).
__global__ void __launch_bounds__(kThreads) momentum_prep_kernel(const __grid_constant__ PrepArgs a) {
  __shared__ float vt[kT][kT + 1];
  __shared__ float red[kThreads / 32];
  const int64_t t = blockIdx.x;
  if (t >= a.total_tiles) return;
  const Tile tile = decode_tile(a.seg, a.n_segs, t);
  const PrepSeg& s = a.seg[tile.seg];
  const int64_t rows = s.rows, cols = s.cols;
  const int64_t base = tile.mat * s.stride;
  const int tx = threadIdx.x & 7, ty = threadIdx.x >> 3;
  const float mu = a.mu, omu = a.omu;
  float sumsq = 0.f;
  float v[2][8];

  const bool full = (tile.r0 + kT <= rows) && (tile.c0 + kT <= cols);
  const bool vec = full && ((cols & 7) == 0) && ((s.stride & 7) == 0);
  float* mrow = s.m + base;
  if (vec) {
    // all loads of the thread's 2 x 8 elements first, then arithmetic, then stores
    float4 mv[2][2];
    float gv[2][8];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int64_t off = (tile.r0 + ty + 32 * k) * cols + tile.c0 + 8 * tx;
      mv[k][0] = __ldcs(reinterpret_cast<const float4*>(mrow + off));
      mv[k][1] = __ldcs(reinterpret_cast<const float4*>(mrow + off + 4));
      if (a.grad_dtype == 1) {
        const uint4 raw = __ldcs(reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(s.g) + base + off));
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162*>(&w[h]);
          gv[k][2 * h] = __low2float(p);
          gv[k][2 * h + 1] = __high2float(p);
        }
      } else {
        const float* gp = reinterpret_cast<const float*>(s.g) + base + off;
        const float4 f0 = __ldcs(reinterpret_cast<const float4*>(gp));
        const float4 f1 = __ldcs(reinterpret_cast<const float4*>(gp + 4));
        gv[k][0] = f0.x; gv[k][1] = f0.y; gv[k][2] = f0.z; gv[k][3] = f0.w;
        gv[k][4] = f1.x; gv[k][5] = f1.y; gv[k][6] = f1.z; gv[k][7] = f1.w;
      }
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const float mo[8] = {mv[k][0].x, mv[k][0].y, mv[k][0].z, mv[k][0].w,
                           mv[k][1].x, mv[k][1].y, mv[k][1].z, mv[k][1].w};
      float mn[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        mn[j] = dot2_accurate(mu, mo[j], omu, gv[k][j]);
        v[k][j] = nesterov_input(a.nesterov, mu, mn[j], omu, gv[k][j]);
        sumsq = __fmaf_rn(v[k][j], v[k][j], sumsq);
      }
      mv[k][0] = make_float4(mn[0], mn[1], mn[2], mn[3]);
      mv[k][1] = make_float4(mn[4], mn[5], mn[6], mn[7]);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int64_t off = (tile.r0 + ty + 32 * k) * cols + tile.c0 + 8 * tx;
      __stcs(reinterpret_cast<float4*>(mrow + off), mv[k][0]);
      __stcs(reinterpret_cast<float4*>(mrow + off + 4), mv[k][1]);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int64_t r = tile.r0 + ty + 32 * k;
      const int64_t c = tile.c0 + 8 * tx;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v[k][j] = 0.f;
        if (r < rows && c + j < cols) {
          const int64_t off = r * cols + c + j;
          const float gj = load_grad(s.g, base + off, a.grad_dtype);
          const float mn = dot2_accurate(mu, mrow[off], omu, gj);
          mrow[off] = mn;
          v[k][j] = nesterov_input(a.nesterov, mu, mn, omu, gj);
          sumsq = __fmaf_rn(v[k][j], v[k][j], sumsq);
        }
      }
    }
  }

  // X0 = cast(V) in wide orientation (the 1/(||V||+eps) factor is applied later);
  // in 3xTF32 mode also X0^T, the layout the UPDATE GEMM reads.
  const int64_t xb = tile.mat * s.x_mstride;
  const bool need_vt = s.transposed || a.tf32;
  if (need_vt) {
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
      for (int j = 0; j < 8; ++j) vt[ty + 32 * k][8 * tx + j] = v[k][j];
    __syncthreads();
  }
  // P[r][c] = V[r][c]
  auto store_direct = [&](void* hi, float* lo, int64_t ld, int64_t base) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int64_t r = tile.r0 + ty + 32 * k;
      const int64_t c = tile.c0 + 8 * tx;
      if (full && (ld & 7) == 0) {
        store_x8(hi, lo, base + r * ld + c, v[k], a.tf32);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (r < rows && c + j < cols) store_x(hi, lo, base + r * ld + c + j, v[k][j], a.tf32);
      }
    }
  };
  // P[c][r] = V[r][c]: P row = source column, P column = source row
  auto store_transposed = [&](void* hi, float* lo, int64_t ld, int64_t base) {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int xi = ty + 32 * k;
      const int64_t xr = tile.c0 + xi;
      const int64_t xc = tile.r0 + 8 * tx;
      float w8[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) w8[j] = vt[8 * tx + j][xi];
      if (full && (ld & 7) == 0) {
        store_x8(hi, lo, base + xr * ld + xc, w8, a.tf32);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (xr < cols && xc + j < rows) store_x(hi, lo, base + xr * ld + xc + j, w8[j], a.tf32);
      }
    }
  };
  if (!s.transposed) store_direct(s.x_hi, s.x_lo, s.x_ld, xb);
  else store_transposed(s.x_hi, s.x_lo, s.x_ld, xb);
  if (a.tf32) {
    const int64_t tb = tile.mat * s.xt_mstride;
    if (!s.transposed) store_transposed(s.xt_hi, s.xt_lo, s.xt_ld, tb);
    else store_direct(s.xt_hi, s.xt_lo, s.xt_ld, tb);
  }

  sumsq = warp_sum(sumsq);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sumsq;
  __syncthreads();
  if (threadIdx.x == 0) {
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) tot += red[w];
    a.partials[t] = tot;
  }
}

// One block per matrix: each thread sums a fixed strided subset of the matrix's
// tile partials in fp64, then a fixed-shape tree combines them (deterministic).
__global__ void __launch_bounds__(256) norm_finalize_kernel(const __grid_constant__ PrepArgs a) {
  __shared__ double red[256];
  const int mat = blockIdx.x;
  if (mat >= a.n_mats) return;
  int si = 0;
  for (int i = 1; i < a.n_segs; ++i)
    if (a.seg[i].mat0 <= mat) si = i;
  const PrepSeg& s = a.seg[si];
  const int64_t first = s.block0 + (int64_t)(mat - s.mat0) * s.tiles_per_mat;
  double acc = 0.0;
  for (int64_t i = threadIdx.x; i < s.tiles_per_mat; i += 256) acc += (double)a.partials[first + i];
  red[threadIdx.x] = acc;
  __syncthreads();
#pragma unroll
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double tot = red[0];
    const bool finite = isfinite(tot);
    a.scale[mat] = finite ? (float)(1.0 / (sqrt(tot) + (double)a.eps)) : 0.f;
    a.flags[mat] = finite ? 0 : 1;
    s.norm_out[mat - s.mat0] = (float)sqrt(tot);
    if (!finite) atomicAdd(&a.status->nonfinite, 1u);
  }
}

// ---------------------------------------------------------------------------
// apply / emit
// ---------------------------------------------------------------------------
__device__ __forceinline__ float load_u(const void* hi, const float* lo, int64_t i, int tf32) {
  if (tf32) return reinterpret_cast<const float*>(hi)[i] + lo[i];
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(hi)[i]);
}

__global__ void __launch_bounds__(kThreads) apply_kernel(const __grid_constant__ ApplyArgs a) {
  __shared__ float ut[kT][kT + 1];
  const int64_t t = blockIdx.x;
  if (t >= a.total_tiles) return;
  const Tile tile = decode_tile(a.seg, a.n_segs, t);
  const ApplySeg& s = a.seg[tile.seg];
  const int mat = s.mat0 + (int)tile.mat;
  if (!a.emit && a.skip_nonfinite && a.flags[mat]) return;  // whole tile belongs to one matrix
  const int64_t rows = s.rows, cols = s.cols;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int64_t ub = tile.mat * s.u_mstride;
  const float us = a.unnormalized ? a.scale[mat] : 1.0f;
  const bool full = (tile.r0 + kT <= rows) && (tile.c0 + kT <= cols);
  float u[4][4];

  if (s.transposed) {
    // U_wide is cols x rows; gather the tile's transpose through shared memory.
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int wi = ty + 16 * k;            // wide row = W column
      const int64_t wr = tile.c0 + wi;
      const int64_t wc = tile.r0 + 4 * tx;   // wide column = W row
#pragma unroll
      for (int j = 0; j < 4; ++j)
        ut[wi][4 * tx + j] = (wr < cols && wc + j < rows) ? load_u(s.u_hi, s.u_lo, ub + wr * s.u_ld + wc + j, a.tf32) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < 4; ++k)
#pragma unroll
      for (int j = 0; j < 4; ++j) u[k][j] = ut[4 * tx + j][ty + 16 * k];
  } else {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int64_t r = tile.r0 + ty + 16 * k;
      const int64_t c = tile.c0 + 4 * tx;
      if (full && !a.tf32) {
        const uint2 raw = *reinterpret_cast<const uint2*>(
            reinterpret_cast<const __nv_bfloat16*>(s.u_hi) + ub + r * s.u_ld + c);
        const __nv_bfloat162 p0 = *reinterpret_cast<const __nv_bfloat162*>(&raw.x);
        const __nv_bfloat162 p1 = *reinterpret_cast<const __nv_bfloat162*>(&raw.y);
        u[k][0] = __low2float(p0); u[k][1] = __high2float(p0);
        u[k][2] = __low2float(p1); u[k][3] = __high2float(p1);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          u[k][j] = (r < rows && c + j < cols) ? load_u(s.u_hi, s.u_lo, ub + r * s.u_ld + c + j, a.tf32) : 0.f;
      }
    }
  }

  const int64_t wb = tile.mat * s.stride;
  const float sc = s.shape_scale;
  const bool vec = full && ((cols & 3) == 0) && ((s.stride & 3) == 0);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int64_t r = tile.r0 + ty + 16 * k;
    const int64_t c = tile.c0 + 4 * tx;
    const int64_t off = wb + r * cols + c;
    if (a.emit) {
      float* out = reinterpret_cast<float*>(s.w);
      if (vec) {
        *reinterpret_cast<float4*>(out + off) =
            make_float4(sc * (us * u[k][0]), sc * (us * u[k][1]), sc * (us * u[k][2]), sc * (us * u[k][3]));
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (r < rows && c + j < cols) out[off + j] = sc * (us * u[k][j]);
      }
      continue;
    }
    if (a.param_dtype == 0) {
      float* w = reinterpret_cast<float*>(s.w);
      if (vec) {
        float4 w4 = *reinterpret_cast<const float4*>(w + off);
        float wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j)
          wv[j] = __fmaf_rn(-a.lr, __fmaf_rn(sc, us * u[k][j], __fmul_rn(a.wd, wv[j])), wv[j]);
        *reinterpret_cast<float4*>(w + off) = make_float4(wv[0], wv[1], wv[2], wv[3]);
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (r < rows && c + j < cols) {
            const float wv = w[off + j];
            w[off + j] = __fmaf_rn(-a.lr, __fmaf_rn(sc, us * u[k][j], __fmul_rn(a.wd, wv)), wv);
          }
      }
    } else {
      __nv_bfloat16* w = reinterpret_cast<__nv_bfloat16*>(s.w);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (r < rows && c + j < cols) {
          const float wv = __bfloat162float(w[off + j]);
          w[off + j] = __float2bfloat16_rn(
              __fmaf_rn(-a.lr, __fmaf_rn(sc, us * u[k][j], __fmul_rn(a.wd, wv)), wv));
        }
    }
  }
}

// The failure-path self-test: one thread waits on an mbarrier whose phase nothing
// completes, with the bounded wait every kernel of the library uses, which gives up
// after limit_ns and sets kStatusWaitTimeout in the device status word.
__global__ void wait_selftest_kernel(DeviceStatus* status, unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) (void)mbar_wait(&bar, 0u, &abort_flag, &status->flags, limit_ns);
}

}  // namespace

cudaError_t launch_wait_selftest(DeviceStatus* status, unsigned long long limit_ns, cudaStream_t s) {
  wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s) {
  if (a.total_tiles <= 0) return cudaSuccess;
  momentum_prep_kernel<<<(unsigned)a.total_tiles, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_norm(const PrepArgs& a, cudaStream_t s) {
  if (a.n_mats <= 0) return cudaSuccess;
  norm_finalize_kernel<<<a.n_mats, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_apply(const ApplyArgs& a, cudaStream_t s) {
  if (a.total_tiles <= 0) return cudaSuccess;
  apply_kernel<<<(unsigned)a.total_tiles, kThreads, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace muon

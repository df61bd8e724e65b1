// Newton-Schulz GEMMs on the sm_103a tensor cores (tcgen05 + TMEM, fed by TMA).
//
// One quintic iteration on a wide matrix X (m x n, m <= n) is three GEMMs
// (DeepSpeed issue "[RFC] Enable Correct and High-Performance Muon Optimizer
// under ZeRO CPU Offload", section 2: "5~6 iterations" of Newton-Schulz on the
// full 2-D matrix; "Muon Optimizer + FSDP", section 背景):
//
//   GRAM   A  = X X^T            m x m, symmetric: only tiles touching the upper
//                                triangle are computed; the epilogue writes the
//                                upper part and mirrors it into the lower part.
//   POLY   B  = c (A A) + b A    m x m, symmetric (a polynomial of A); A A is read
//                                as A A^T so both operands are K-major rows; the
//                                b A term is added in the epilogue.
//   UPDATE X' = (B X) + a X      m x n; B rows are K-major, X is read MN-major
//                                (n contiguous); the a X term is added in the
//                                epilogue.
//
// In the first iteration X holds the un-normalised V; the per-matrix factor
// s = 1/(||V||_F + eps) is applied in the epilogues (GRAM: s^2, UPDATE: s).
//
// Kernel structure (one persistent CTA per SM, 192 threads):
//   warp 0  lane 0: TMA producer over a 4-stage shared-memory ring
//                   (A 128 x 64 bf16 + B 256 x 64 bf16 per stage, 128-byte swizzle)
//   warp 1  lane 0: tcgen05.mma issuer, M=128 N=256 K=16, fp32 accumulators in
//                   TMEM, two accumulator buffers (512 columns) so the epilogue of
//                   one tile overlaps the main loop of the next
//   warps 2-5:      epilogue; warp w reads TMEM lanes 32*(w%4)..+31 with
//                   tcgen05.ld, applies alpha/beta, converts to bf16 and stores.
// Tiles of all same-shape groups of a micro-bucket (and of all its matrices) are
// numbered in one space and dealt round-robin to the CTAs.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "device.cuh"
#include "kernels.h"

namespace muon {
namespace {

constexpr int kBK = 64;  // bf16 elements per 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kThreadsG = 192;
constexpr uint32_t kABytes = kBM * kBK * 2;   // 16 KB
constexpr uint32_t kBBytes = kBN * kBK * 2;   // 32 KB
constexpr uint32_t kStageBytes = kABytes + kBBytes;
constexpr uint32_t kTmemCols = 512;
constexpr size_t kSmemBytes = (size_t)kStages * kStageBytes + 1024;

struct TileCoord {
  int g, b, bi, bj;
};

__device__ __forceinline__ TileCoord decode_tile(const GemmArgs& a, int t) {
  int g = 0;
  for (int i = 1; i < a.n_groups; ++i)
    if (a.g[i].tile0 <= t) g = i;
  const GemmGroup& G = a.g[g];
  const int local = t - G.tile0;
  TileCoord tc;
  tc.g = g;
  tc.b = local / G.tiles_per_mat;
  int tt = local % G.tiles_per_mat;
  if (a.mode == kUpdate) {
    tc.bi = tt / G.tiles_n;
    tc.bj = tt % G.tiles_n;
  } else {
    // upper-triangle tiles, column block by column block
    tc.bi = 0;
    tc.bj = 0;
    for (int bj = 0; bj < G.tiles_n; ++bj) {
      const int cnt = min(G.tiles_m, (bj * kBN + kBN - 1) / kBM + 1);
      if (tt < cnt) {
        tc.bi = tt;
        tc.bj = bj;
        break;
      }
      tt -= cnt;
    }
  }
  return tc;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

__global__ void __launch_bounds__(kThreadsG, 1) ns_gemm_bf16_kernel(const __grid_constant__ GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full_bar[kStages];
  __shared__ __align__(8) uint64_t empty_bar[kStages];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  unsigned* status = &a.status->flags;
  volatile int* abort_p = &abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull_bar[i], 1);
      mbar_init(&tempty_bar[i], 128);
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < a.n_groups; ++i) {
      tma_prefetch_desc(&a.g[i].map_a);
      tma_prefetch_desc(&a.g[i].map_b);
    }
  }
  if (warp == 1) {
    tmem_alloc(&tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = tmem_slot;
  const int mode = a.mode;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int stage = 0;
      uint32_t phase = 0;
      for (int t = blockIdx.x; t < a.total_tiles; t += gridDim.x) {
        const TileCoord tc = decode_tile(a, t);
        const GemmGroup& G = a.g[tc.g];
        const int kblocks = (G.K + kBK - 1) / kBK;
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&empty_bar[stage], phase ^ 1u, abort_p, status)) { ok = false; break; }
          uint8_t* sa = smem + (size_t)stage * kStageBytes;
          uint8_t* sb = sa + kABytes;
          mbar_arrive_expect_tx(&full_bar[stage], kStageBytes);
          const int k0 = kb * kBK;
          tma_load_3d(sa, &G.map_a, &full_bar[stage], k0, tc.bi * kBM, tc.b);
          if (mode == kUpdate) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              tma_load_3d(sb + q * 8192, &G.map_b, &full_bar[stage], tc.bj * kBN + q * 64, k0, tc.b);
          } else {
#pragma unroll
            for (int h = 0; h < 2; ++h)
              tma_load_3d(sb + h * 16384, &G.map_b, &full_bar[stage], k0, tc.bj * kBN + h * 128, tc.b);
          }
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
      if (*abort_p) {
        // let loads already issued land before the CTA exits (bounded)
        for (int s = 0; s < kStages; ++s) {
          (void)mbar_wait(&full_bar[s], phase ^ (s < stage ? 0u : 1u), nullptr, nullptr, 100000000ull);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      const uint32_t idesc = make_idesc(1u, kBM, kBN, mode == kUpdate ? 1u : 0u);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int t = blockIdx.x; t < a.total_tiles; t += gridDim.x) {
        const TileCoord tc = decode_tile(a, t);
        const GemmGroup& G = a.g[tc.g];
        const int kblocks = (G.K + kBK - 1) / kBK;
        if (!mbar_wait(&tempty_bar[acc], acc_phase ^ 1u, abort_p, status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!mbar_wait(&full_bar[stage], phase, abort_p, status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + (size_t)stage * kStageBytes);
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t ad = smem_desc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = (mode == kUpdate) ? smem_desc_sw128(sb + kk * 2048, 8192, 1024)
                                                  : smem_desc_sw128(sb + kk * 32, 16, 1024);
            mma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          mma_commit(&empty_bar[stage]);
          if (++stage == kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(&tfull_bar[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // every MMA issued by this thread has completed before TMEM is freed
      mma_commit(&drain_bar);
      (void)mbar_wait(&drain_bar, 0u, nullptr, status);
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int quad = warp & 3;
    const int row_in_tile = quad * 32 + lane;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int t = blockIdx.x; t < a.total_tiles; t += gridDim.x) {
      const TileCoord tc = decode_tile(a, t);
      const GemmGroup& G = a.g[tc.g];
      // warp-uniform decision: tcgen05.ld below needs every lane of the warp
      const bool got = mbar_wait(&tfull_bar[acc], acc_phase, abort_p, status);
      if (!__all_sync(0xffffffffu, got)) break;
      tc_fence_after();
      float alpha = a.alpha, beta = a.beta;
      if (a.use_scale) {
        const float s = a.scale[G.mat_base + tc.b];
        if (mode == kGram) alpha *= s * s;
        if (mode == kUpdate) { alpha *= s; beta *= s; }
      }
      const bool sym = (mode != kUpdate);
      const int64_t r = (int64_t)tc.bi * kBM + row_in_tile;
      __nv_bfloat16* C = reinterpret_cast<__nv_bfloat16*>(G.c_hi) + (int64_t)tc.b * G.c_mstride;
      const __nv_bfloat16* D = reinterpret_cast<const __nv_bfloat16*>(G.d_hi) + (int64_t)tc.b * G.c_mstride;
      const int64_t ld = G.c_ld;
#pragma unroll 1
      for (int cc = 0; cc < kBN / 32; ++cc) {
        float v[32];
        tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * kBN + cc * 32), v);
        const int64_t c0 = (int64_t)tc.bj * kBN + cc * 32;
        if (r >= G.M || c0 >= G.N) continue;
        const bool cols_full = (c0 + 32 <= G.N);
        if (mode != kGram) {
          const __nv_bfloat16* drow = D + r * ld + c0;
          if (cols_full) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 raw = *reinterpret_cast<const uint4*>(drow + 8 * q);
              const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                const __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162*>(&w4[h]);
                v[8 * q + 2 * h] = alpha * v[8 * q + 2 * h] + beta * __low2float(p);
                v[8 * q + 2 * h + 1] = alpha * v[8 * q + 2 * h + 1] + beta * __high2float(p);
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              v[j] = alpha * v[j] + (c0 + j < G.N ? beta * __bfloat162float(drow[j]) : 0.f);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= alpha;
        }
        // direct store of row r (upper part only in the symmetric modes)
        __nv_bfloat16* crow = C + r * ld + c0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int64_t cq = c0 + 8 * q;
          if (cq + 8 <= G.N && (!sym || cq >= r)) {
            uint4 raw;
            raw.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
            raw.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
            raw.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
            raw.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
            *reinterpret_cast<uint4*>(crow + 8 * q) = raw;
          } else {
#pragma unroll
            for (int h = 0; h < 8; ++h) {
              const int64_t c = cq + h;
              if (c < G.N && (!sym || c >= r)) crow[8 * q + h] = __float2bfloat16_rn(v[8 * q + h]);
            }
          }
        }
        // mirror of the strictly upper part: C[c][r] = C[r][c]
        if (sym) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int64_t c = c0 + j;
            if (c > r && c < G.N) C[c * ld + r] = __float2bfloat16_rn(v[j]);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty_bar[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

}  // namespace

size_t gemm_smem_bytes(bool tf32) {
  (void)tf32;
  return kSmemBytes;
}

cudaError_t launch_gemm(const GemmArgs& a, int num_sms, bool tf32, cudaStream_t s) {
  if (tf32) return cudaErrorNotSupported;
  if (a.total_tiles <= 0) return cudaSuccess;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(ns_gemm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int grid = a.total_tiles < num_sms ? a.total_tiles : num_sms;
  ns_gemm_bf16_kernel<<<grid, kThreadsG, kSmemBytes, s>>>(a);
  return cudaGetLastError();
}

}  // namespace muon

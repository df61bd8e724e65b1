// Newton-Schulz GEMMs on the sm_103a tensor cores (tcgen05 + TMEM, fed by TMA).
//
// One quintic iteration on a wide matrix X (m x n, m <= n) is three GEMMs
// (DeepSpeed issue "[RFC] Enable Correct and High-Performance Muon Optimizer
// under ZeRO CPU Offload", section 2: "5~6 iterations" of Newton-Schulz on the
// full 2-D matrix; "Muon Optimizer + FSDP", section 背景):
//
//   GRAM   A  = X X^T            m x m, symmetric: only tiles touching the upper
//                                triangle are computed.
//   POLY   B  = c (A A) + b A    m x m, symmetric (a polynomial of A); A A is read
//                                as A A^T (both operands rows of A); the b A term
//                                is added in the epilogue, and in bf16 also a on
//                                the diagonal: B' = a I + B.
//   UPDATE X' = B' X (bf16)      m x n; B rows are the A operand; bf16 reads X MN-major
//          X' = (B X) + a X      (n contiguous); 3xTF32 reads the rows of X^T
//          (3xTF32)              (K-major, kept beside X in that mode), writes
//                                X'^T as well, and adds the a X term in the
//                                epilogue.
// Folding a I into B changes only where bf16 rounding falls: near convergence B'
// has eigenvalues near 1 where B has them near a - 1, so rounding B' to bf16 loses
// less than rounding B, and the UPDATE epilogue reads no addend.
//
// Symmetric storage.  The GRAM and POLY tiles are the 256 x 256 blocks on and
// above the diagonal.  In bf16 a diagonal block is computed, and written, whole,
// and a block above it also writes its transpose (one more TMA box per chunk from
// the same staging), so A and B' are whole and every operand is read in place
// (K-major rows).  Storing only the computed blocks and reading the blocks left of
// an operand's rows transposed (MN-major) was measured slower: the transposed A
// operand slows the mainloop more than the extra boxes cost the epilogue.  3xTF32
// mirrors the strictly upper part element by element.
//
// In the first iteration X holds the un-normalised V; the per-matrix factor
// s = 1/(||V||_F + eps) is applied in the epilogues (GRAM: s^2, UPDATE: s).  The
// last UPDATE applies the weight update (or writes the offload update U') from
// its epilogue instead of storing X.
//
// Kernel structure (one persistent CTA per SM, 320 threads):
//   warp 0:         TMA producer (converged warp, lane 0 issues) over a shared-memory
//                   ring of 128-byte-swizzled stages, as many as fit beside the
//                   epilogue staging: bf16 -- A 128 x 64 + B (256 / cluster) x 64
//                   per stage; 3xTF32 -- A 128 x 32 and B x 32, each as a
//                   tf32-high and a tf32-low fp32 copy
//   warp 1:         tcgen05.mma issuer (converged warp, lane 0 issues), M=128 x
//                   cluster, N=256 (K=16 bf16 / K=8 tf32), fp32 accumulators in
//                   TMEM, two accumulator buffers (512 columns) so the epilogue of
//                   one tile overlaps the main loop of the next.  3xTF32 issues
//                   hi*hi + hi*lo + lo*hi per k step.
//   warps 2-9:      epilogue; warp w reads TMEM lanes 32*(w%4)..+31 with
//                   tcgen05.ld (two warps per lane quadrant, 128 columns each),
//                   adds the alpha/beta term, converts and stores.  bf16: each
//                   warp owns 8 KB of shared memory through which its 32 x 32
//                   chunks pass as TMA boxes -- the addend is requested one
//                   chunk ahead (across tiles) into two slots with their own
//                   mbarriers, the output leaves as TMA stores, and the last
//                   UPDATE's weights move by cp.async, one chunk ahead.
// Tiles of all same-shape groups of a micro-bucket (and of all its matrices) are
// numbered in one space; a host-computed longest-processing-time schedule gives
// each cluster its list of tiles.
//
// kCL = 2 (the default for m > 128): a cluster of two CTAs on two SMs computes a
// 256 x 256 tile with one tcgen05.mma.cta_group::2 (M=256, N=256) issued by the
// even CTA.  Each CTA holds its own 128 rows of A and one 128-wide half of B, so
// each SM streams half as many B bytes through its shared memory as a single-SM
// 128 x 256 tile (whose operand reads plus TMA fills otherwise saturate shared
// memory bandwidth).  Both CTAs' TMA loads complete on the even CTA's barrier;
// its commits release stages and accumulators in both CTAs; each CTA drains the
// 128 accumulator rows in its own Tensor Memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "device.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace muon {
namespace {

constexpr int kThreadsG = 320;  // producer warp, MMA warp, 8 epilogue warps
constexpr uint32_t kTmemCols = 512;

// Per-precision, per-cluster-size constants.  A "part" is one copy of an operand
// tile: bf16 has one, 3xTF32 a tf32-high and a tf32-low fp32 copy.  Rows are 128
// bytes (one swizzle atom wide).  Each CTA holds 128 rows of A and kBN / kCL rows
// (K-major) or columns (MN-major) of B per part.
template <bool kTF32, int kCL>
struct Cfg {
  static constexpr int kBK = kTF32 ? 32 : 64;            // k elements per 128-byte row
  static constexpr int kParts = kTF32 ? 2 : 1;
  static constexpr uint32_t kA = kBM * 128;               // 16 KB
  static constexpr int kBRows = kBN / kCL;                // B rows (or columns) held by one CTA
  static constexpr uint32_t kB = kBRows * 128;            // 32 KB or 16 KB
  static constexpr uint32_t kStage = kParts * (kA + kB);
  // bf16 epilogue: per epilogue warp 8 KB -- the output chunk (32 x 32 bf16) and
  // two addend chunks (the current one and the next, TMA boxes), or two 32 x 32
  // chunks of the last UPDATE's weights
  static constexpr uint32_t kWarpStaging = 8192u;
  static constexpr uint32_t kStaging = kTF32 ? 0u : 8u * kWarpStaging;
  // as many stages as fit in the 227 KB of dynamic shared memory a CTA may use
  // (1 KB kept for the 1024-byte alignment of the ring, 1 KB for static data)
  static constexpr int kStages = (int)((232448u - 2048u - kStaging) / kStage);
  static constexpr uint32_t kTx = kCL * kStage;           // bytes landing per stage on the leader's barrier
  static constexpr int kInstK = kTF32 ? 8 : 16;           // k per MMA instruction
  static constexpr int kChunks = kBRows / kBK;            // MN-major 128-byte column chunks per CTA
  static constexpr uint32_t kChunkBytes = kBK * 128;      // one chunk: kBK k-rows of 128 B
  static constexpr uint32_t kFormat = kTF32 ? 2u : 1u;    // tf32 / bf16 in the instruction descriptor
  static constexpr size_t kSmem = (size_t)kStages * kStage + kStaging + 1024;
};

struct TileCoord {
  int g, b, bi, bj;
};

// Tile t of the launch -> group, matrix, row block and column block.  Row blocks
// are kBM * kCL rows high (one per cluster); the CTA of rank `rank` takes 128-row
// tile bi = row_block * kCL + rank.
template <int kCL>
__device__ __forceinline__ TileCoord decode_tile(const GemmArgs& a, int t, int rank) {
  int g = 0;
  for (int i = 1; i < a.n_groups; ++i)
    if (a.g[i].tile0 <= t) g = i;
  const GemmGroup& G = a.g[g];
  const int local = t - G.tile0;
  TileCoord tc;
  tc.g = g;
  tc.b = local / G.tiles_per_mat;
  int tt = local % G.tiles_per_mat;
  int pi = 0;
  if (a.mode == kUpdate) {
    pi = tt / G.tiles_n;
    tc.bj = tt % G.tiles_n;
  } else {
    // upper-triangle row blocks, column block by column block
    tc.bj = 0;
    for (int bj = 0; bj < G.tiles_n; ++bj) {
      const int cnt = min(G.tiles_m, (bj * kBN + kBN - 1) / (kBM * kCL) + 1);
      if (tt < cnt) {
        pi = tt;
        tc.bj = bj;
        break;
      }
      tt -= cnt;
    }
  }
  tc.bi = pi * kCL + rank;
  return tc;
}

__device__ __forceinline__ uint4 pack8v(const float* v) {
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}

// ---------------------------------------------------------------------------
// epilogue element access: 32 consecutive columns of one row
// ---------------------------------------------------------------------------
template <bool kTF32>
struct Epi;

template <>
struct Epi<true> {  // 3xTF32: fp32 tf32-high + fp32 low parts (the bf16 epilogue is staged, below)
  static __device__ __forceinline__ void add_d(float (&v)[32], const GemmGroup& G, int64_t off, bool full,
                                               int64_t valid, float alpha, float beta) {
    const float* dh = reinterpret_cast<const float*>(G.d_hi) + off;
    const float* dl = G.d_lo + off;
    if (full) {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float4 h = *reinterpret_cast<const float4*>(dh + 4 * q);
        const float4 l = *reinterpret_cast<const float4*>(dl + 4 * q);
        v[4 * q + 0] = alpha * v[4 * q + 0] + beta * (h.x + l.x);
        v[4 * q + 1] = alpha * v[4 * q + 1] + beta * (h.y + l.y);
        v[4 * q + 2] = alpha * v[4 * q + 2] + beta * (h.z + l.z);
        v[4 * q + 3] = alpha * v[4 * q + 3] + beta * (h.w + l.w);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = alpha * v[j] + (j < valid ? beta * (dh[j] + dl[j]) : 0.f);
    }
  }
  static __device__ __forceinline__ void store8(const GemmGroup& G, int64_t off, const float* v, bool all8,
                                                unsigned mask) {
    float* ch = reinterpret_cast<float*>(G.c_hi) + off;
    float* cl = G.c_lo + off;
    float hi[8], lo[8];
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      hi[h] = round_tf32(v[h]);
      lo[h] = v[h] - hi[h];
    }
    if (all8) {
      *reinterpret_cast<float4*>(ch) = make_float4(hi[0], hi[1], hi[2], hi[3]);
      *reinterpret_cast<float4*>(ch + 4) = make_float4(hi[4], hi[5], hi[6], hi[7]);
      *reinterpret_cast<float4*>(cl) = make_float4(lo[0], lo[1], lo[2], lo[3]);
      *reinterpret_cast<float4*>(cl + 4) = make_float4(lo[4], lo[5], lo[6], lo[7]);
    } else {
#pragma unroll
      for (int h = 0; h < 8; ++h)
        if (mask & (1u << h)) {
          ch[h] = hi[h];
          cl[h] = lo[h];
        }
    }
  }
  static __device__ __forceinline__ void store1(const GemmGroup& G, int64_t off, float v) {
    const float h = round_tf32(v);
    reinterpret_cast<float*>(G.c_hi)[off] = h;
    G.c_lo[off] = v - h;
  }
  // the transposed copy X'^T of the UPDATE output
  static __device__ __forceinline__ void store1t(const GemmGroup& G, int64_t off, float v) {
    const float h = round_tf32(v);
    reinterpret_cast<float*>(G.ct_hi)[off] = h;
    G.ct_lo[off] = v - h;
  }
};

// ---------------------------------------------------------------------------
// bf16 epilogue staging.  A 32 x 32 bf16 chunk is held as 32 rows of four
// 16-byte units, unit u of row i at position i * 4 + (u ^ ((i / 2) % 4)): the
// order in which a TMA box of 64-byte rows lands with the 64-byte swizzle (the
// buffers are 2 KB aligned), so such chunks move as TMA boxes.  The same idea
// with eight units per row, position i * 8 + (u ^ (i % 8)), holds a 32 x 32 fp32
// piece of weights, whose global rows move eight (or four) rows per warp step
// with 16-byte lanes.  A lane reads its own row back (the TMEM row layout).
// ---------------------------------------------------------------------------
__device__ __forceinline__ int unit4(int i, int u) { return i * 4 + (u ^ ((i >> 1) & 3)); }
__device__ __forceinline__ int unit8(int i, int u) { return i * 8 + (u ^ (i & 7)); }

// The weights (or U' output) of one matrix for the staged update: a wide matrix
// whose rows are whole 16-byte units.  ok = false leaves the matrix to
// fused_apply_chunk (tall matrices, unaligned rows, skipped matrices).
struct StagedTarget {
  uint8_t* w;
  int64_t ld;
  float sc;
  bool bf16, ok;
};

__device__ __forceinline__ StagedTarget staged_target(const ApplyArgs& A, int mat) {
  int lo = 0, hi = A.n_segs - 1;
  while (lo < hi) {  // last run with mat0 <= mat
    const int mid = (lo + hi + 1) >> 1;
    if (A.seg[mid].mat0 <= mat) lo = mid; else hi = mid - 1;
  }
  const ApplySeg& S = A.seg[lo];
  StagedTarget t;
  t.bf16 = !A.emit && A.param_dtype != 0;
  const int64_t per = t.bf16 ? 8 : 4;  // elements per 16-byte unit
  t.w = reinterpret_cast<uint8_t*>(S.w) + (int64_t)(mat - S.mat0) * S.stride * (t.bf16 ? 2 : 4);
  t.ld = S.cols;
  t.sc = S.shape_scale;
  t.ok = !S.transposed && (S.cols % per) == 0 && (S.stride % per) == 0 &&
         (reinterpret_cast<uintptr_t>(t.w) & 15u) == 0 && !(!A.emit && A.skip_nonfinite && A.flags[mat]);
  return t;
}

// Starts copying the weights of rows row0 .. +31, columns c0 .. +31 into `buf`
// (nothing when emitting U').
__device__ __forceinline__ void staged_load(const ApplyArgs& A, const StagedTarget& t, int64_t M, int64_t N,
                                            int64_t row0, int64_t c0, int lane, uint4* buf) {
  if (A.emit) return;
  if (t.bf16) {
    const int g = lane & 3;
#pragma unroll 1
    for (int qq = 0; qq < 4; ++qq) {
      const int i = 8 * qq + (lane >> 2);
      const int64_t rr = row0 + i, cg = c0 + 8 * g;
      if (rr < M && cg < N)
        cp_async_16(buf + unit4(i, g), reinterpret_cast<const __nv_bfloat16*>(t.w) + rr * t.ld + cg);
    }
  } else {
    const int g = lane & 7;
#pragma unroll 1
    for (int qq = 0; qq < 8; ++qq) {
      const int i = 4 * qq + (lane >> 3);
      const int64_t rr = row0 + i, cg = c0 + 4 * g;
      if (rr < M && cg < N)
        cp_async_16(buf + unit8(i, g), reinterpret_cast<const float*>(t.w) + rr * t.ld + cg);
    }
  }
}

// Lane = row of the chunk, u = its 32 values of U: W <- W - lr (s U + wd W) in
// the buffer (U' = s U when emitting); then the rows go back to the tensor.
__device__ __forceinline__ void staged_update_store(const ApplyArgs& A, const StagedTarget& t, int64_t M, int64_t N,
                                                    int64_t row0, int64_t c0, int lane, const float (&u)[32],
                                                    uint4* buf) {
  if (t.bf16) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4& cell = buf[unit4(lane, q)];
      uint32_t h[4] = {cell.x, cell.y, cell.z, cell.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162*>(&h[e]);
        const int j = 8 * q + 2 * e;
        const float x0 = __low2float(p), x1 = __high2float(p);
        h[e] = pack_bf16x2(__fmaf_rn(-A.lr, __fmaf_rn(t.sc, u[j], __fmul_rn(A.wd, x0)), x0),
                           __fmaf_rn(-A.lr, __fmaf_rn(t.sc, u[j + 1], __fmul_rn(A.wd, x1)), x1));
      }
      cell = make_uint4(h[0], h[1], h[2], h[3]);
    }
  } else {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float4* cell = reinterpret_cast<float4*>(buf + unit8(lane, q));
      float4 w = A.emit ? make_float4(0.f, 0.f, 0.f, 0.f) : *cell;
      float* wv = reinterpret_cast<float*>(&w);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        wv[e] = A.emit ? t.sc * u[4 * q + e]
                       : __fmaf_rn(-A.lr, __fmaf_rn(t.sc, u[4 * q + e], __fmul_rn(A.wd, wv[e])), wv[e]);
      *cell = w;
    }
  }
  __syncwarp();
  if (t.bf16) {
    const int g = lane & 3;
#pragma unroll
    for (int qq = 0; qq < 4; ++qq) {
      const int i = 8 * qq + (lane >> 2);
      const int64_t rr = row0 + i, cg = c0 + 8 * g;
      if (rr < M && cg < N)
        *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(t.w) + rr * t.ld + cg) = buf[unit4(i, g)];
    }
  } else {
    const int g = lane & 7;
#pragma unroll
    for (int qq = 0; qq < 8; ++qq) {
      const int i = 4 * qq + (lane >> 3);
      const int64_t rr = row0 + i, cg = c0 + 4 * g;
      if (rr < M && cg < N)
        *reinterpret_cast<uint4*>(reinterpret_cast<float*>(t.w) + rr * t.ld + cg) = buf[unit8(i, g)];
    }
  }
}

template <bool kTF32, int kCL>
__global__ void __launch_bounds__(kThreadsG, 1) ns_gemm_kernel(const __grid_constant__ GemmArgs a) {
  using C = Cfg<kTF32, kCL>;
  static_assert(kCL == 1 || kCL == 2, "one CTA, or a pair of CTAs on two SMs");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full_bar[C::kStages];
  __shared__ __align__(8) uint64_t empty_bar[C::kStages];
  __shared__ __align__(8) uint64_t tfull_bar[2];
  __shared__ __align__(8) uint64_t tempty_bar[2];
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ __align__(8) uint64_t addend_bar[16];  // two per epilogue warp
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rank = kCL > 1 ? (int)cluster_ctarank() : 0;
  const bool leader = rank == 0;
  const int cluster_id = blockIdx.x / kCL;
  constexpr uint16_t kPair = (1u << kCL) - 1u;
  unsigned* status = &a.status->flags;
  volatile int* abort_p = &abort_flag;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tfull_bar[i], 1);
      // single CTA: every epilogue thread arrives; pair: one lane per epilogue warp of both CTAs
      mbar_init(&tempty_bar[i], kCL == 1 ? 256 : 8 * kCL);
    }
    mbar_init(&drain_bar, 1);
    for (int i = 0; i < 16; ++i) mbar_init(&addend_bar[i], 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    for (int i = 0; i < a.n_groups; ++i) {
      tma_prefetch_desc(&a.g[i].map_a);
      tma_prefetch_desc(&a.g[i].map_b);
      if (kTF32) {
        tma_prefetch_desc(&a.g[i].map_a_lo);
        tma_prefetch_desc(&a.g[i].map_b_lo);
      }
    }
  }
  if (warp == 1) {
    tmem_alloc<kCL>(&tmem_slot, kTmemCols);
    tmem_relinquish<kCL>();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (kCL > 1) cluster_sync();  // barriers of both CTAs exist before any remote signal
  tc_fence_after();
  // The prologue above overlaps the previous launch's last tiles; its outputs (X,
  // A, B', the norm scales) are read only after it has completed.
  griddep_launch_dependents();
  griddep_wait();
  const uint32_t tmem_base = tmem_slot;
  const int mode = a.mode;
  const bool mn_b = (mode == kUpdate) && !kTF32;  // B operand read MN-major
#ifdef MUON_DEBUG
  // Debug build: the tile schedule lives in the caller's workspace; every thread
  // checks this cluster's range of it (offsets in order and within the tile count,
  // every tile index in range) before any role uses it, and on a bad entry no role
  // runs a tile.  The release build leaves these loops exactly as they are.
  bool sched_ok;
  {
    const int lo = a.sched_off[cluster_id], hi = a.sched_off[cluster_id + 1];
    sched_ok = cluster_id < a.n_clusters && 0 <= lo && lo <= hi && hi <= a.total_tiles;
    for (int si = lo; sched_ok && si < hi; ++si) {
      const int t = a.sched_units[si];
      sched_ok = 0 <= t && t < a.total_tiles;
    }
    if (!sched_ok && threadIdx.x == 0) guard_fail(status, abort_p);
  }
#define MUON_SCHED_OK sched_ok &&
#else
#define MUON_SCHED_OK
#endif

  if (warp == 0) {
    // ---------------- TMA producer (both CTAs) ----------------
    // The whole warp walks the schedule and waits (converged); lane 0 issues.
    // Issuing from a lone lane of a diverged warp is several times slower.
    int stage = 0;
    uint32_t phase = 0;
    for (int si = a.sched_off[cluster_id]; MUON_SCHED_OK si < a.sched_off[cluster_id + 1]; ++si) {
      const int t = a.sched_units[si];
      const TileCoord tc = decode_tile<kCL>(a, t, rank);
      const GemmGroup& G = a.g[tc.g];
      const int kblocks = (G.K + C::kBK - 1) / C::kBK;
      bool ok = true;
      for (int kb = 0; kb < kblocks; ++kb) {
        const bool got = mbar_wait(&empty_bar[stage], phase ^ 1u, abort_p, status);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        if (lane == 0) {
          uint8_t* sa = smem + (size_t)stage * C::kStage;
          uint8_t* sb = sa + C::kParts * C::kA;
          if (leader) mbar_arrive_expect_tx(&full_bar[stage], C::kTx);
          const uint32_t bar = kCL > 1 ? mapa_shared(&full_bar[stage], 0) : smem_u32(&full_bar[stage]);
          const int k0 = kb * C::kBK;
#pragma unroll
          for (int part = 0; part < C::kParts; ++part) {
            const CUtensorMap* ma = part ? &G.map_a_lo : &G.map_a;
            const CUtensorMap* mb = part ? &G.map_b_lo : &G.map_b;
            uint8_t* sbp = sb + part * C::kB;
            if constexpr (kCL == 1) {
              tma_load_3d(sa + part * C::kA, ma, &full_bar[stage], k0, tc.bi * kBM, tc.b);
              if (mn_b) {
#pragma unroll
                for (int q = 0; q < C::kChunks; ++q)
                  tma_load_3d(sbp + q * C::kChunkBytes, mb, &full_bar[stage], tc.bj * kBN + q * C::kBK, k0, tc.b);
              } else {
#pragma unroll
                for (int h = 0; h < 2; ++h)
                  tma_load_3d(sbp + h * (C::kB / 2), mb, &full_bar[stage], k0, tc.bj * kBN + h * 128, tc.b);
              }
            } else {
              // own 128 rows of A and own half of B, completing on the even CTA's barrier
              tma_load_3d_pair(sa + part * C::kA, ma, bar, k0, tc.bi * kBM, tc.b);
              if (mn_b) {
#pragma unroll
                for (int q = 0; q < C::kChunks; ++q)
                  tma_load_3d_pair(sbp + q * C::kChunkBytes, mb, bar, tc.bj * kBN + rank * C::kBRows + q * C::kBK,
                                   k0, tc.b);
              } else {
                tma_load_3d_pair(sbp, mb, bar, k0, tc.bj * kBN + rank * C::kBRows, tc.b);
              }
            }
          }
        }
        __syncwarp();
        if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
    }
    if (*abort_p && (kCL == 1 || leader) && lane == 0) {
      // let loads already issued land before the CTA exits (bounded)
      for (int s = 0; s < C::kStages; ++s)
        (void)mbar_wait(&full_bar[s], phase ^ (s < stage ? 0u : 1u), nullptr, nullptr, 100000000ull);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (leader) {
      // ---------------- MMA issuer (the even CTA) ----------------
      // converged warp; lane 0 issues the MMAs and the commits that track them
      const uint32_t idesc = make_idesc(C::kFormat, kBM * kCL, kBN, mn_b ? 1u : 0u);
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      for (int si = a.sched_off[cluster_id]; MUON_SCHED_OK si < a.sched_off[cluster_id + 1]; ++si) {
      const int t = a.sched_units[si];
        const TileCoord tc = decode_tile<kCL>(a, t, rank);
        const GemmGroup& G = a.g[tc.g];
        const int kblocks = (G.K + C::kBK - 1) / C::kBK;
        const bool free_acc = mbar_wait(&tempty_bar[acc], acc_phase ^ 1u, abort_p, status);
        if (!__all_sync(0xffffffffu, free_acc)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * kBN);
        bool ok = true;
        for (int kb = 0; kb < kblocks; ++kb) {
          // the TMA bytes are visible to the tensor core once the barrier completes
          const bool got = mbar_wait(&full_bar[stage], phase, abort_p, status);
          if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
#ifdef MUON_DEBUG
          // debug build: the stage's operands lie inside the ring, the accumulator in
          // the allocated Tensor Memory columns
          if (!(stage >= 0 && stage < C::kStages && (uint32_t)(acc + 1) * kBN <= kTmemCols)) {
            guard_fail(status, abort_p);
            ok = false;
            break;
          }
#endif
          if (lane == 0) {
            const uint32_t sa = smem_u32(smem + (size_t)stage * C::kStage);
            const uint32_t sb = sa + C::kParts * C::kA;
#pragma unroll
            for (int kk = 0; kk < C::kBK / C::kInstK; ++kk) {
              const uint64_t ad = smem_desc_sw128(sa + kk * 32, 16, 1024);
              const uint64_t bd = mn_b ? smem_desc_sw128(sb + kk * C::kInstK * 128, C::kChunkBytes, 1024)
                                       : smem_desc_sw128(sb + kk * 32, 16, 1024);
              const uint32_t accumulate = (kb | kk) != 0 ? 1u : 0u;
              if constexpr (kTF32) {
                const uint64_t ad_lo = smem_desc_sw128(sa + C::kA + kk * 32, 16, 1024);
                const uint64_t bd_lo = smem_desc_sw128(sb + C::kB + kk * 32, 16, 1024);  // tf32 B is K-major
                mma<true, kCL>(d_tmem, ad_lo, bd, idesc, accumulate);
                mma<true, kCL>(d_tmem, ad, bd_lo, idesc, 1u);
                mma<true, kCL>(d_tmem, ad, bd, idesc, 1u);
              } else {
                mma<false, kCL>(d_tmem, ad, bd, idesc, accumulate);
              }
            }
            if constexpr (kCL > 1) mma_commit_multicast<kCL>(&empty_bar[stage], kPair);
            else mma_commit<kCL>(&empty_bar[stage]);
          }
          __syncwarp();
          if (++stage == C::kStages) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (lane == 0) {
          if constexpr (kCL > 1) mma_commit_multicast<kCL>(&tfull_bar[acc], kPair);
          else mma_commit<kCL>(&tfull_bar[acc]);
        }
        __syncwarp();
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // every MMA issued by lane 0 has completed before TMEM is freed
      if (lane == 0) {
        mma_commit<kCL>(&drain_bar);
        (void)mbar_wait(&drain_bar, 0u, nullptr, status);
      }
      __syncwarp();
    }
  } else {
    // ---------------- epilogue (warps 2..9 of both CTAs) ----------------
    // warp w reads TMEM lanes 32*(w%4)..+31; the two warps of a lane quadrant
    // split the 256 accumulator columns into 32-column chunks
    const int quad = warp & 3;
    const int half = (warp - 2) >> 2;
    const int ew = warp - 2;
    // bf16 staging of this warp (after the ring), in 32 x 32 boxes of the 64-byte
    // swizzle: the output chunk and its transpose (first 4 KB) and two POLY
    // addend slots filled by TMA (last 4 KB); the last UPDATE uses the two halves
    // as weight slots instead
    uint8_t* wst = smem + (size_t)C::kStages * C::kStage + (size_t)ew * C::kWarpStaging;
    uint4* rowbuf = reinterpret_cast<uint4*>(wst);
    __nv_bfloat16* tbuf = reinterpret_cast<__nv_bfloat16*>(wst + 2048u);  // POLY: the chunk transposed
    uint4* dbuf = reinterpret_cast<uint4*>(wst + 4096u);  // addend slot s at dbuf + s * 128
    uint64_t* dbar = &addend_bar[2 * ew];
    const uint32_t tempty_lead[2] = {kCL > 1 ? mapa_shared(&tempty_bar[0], 0) : 0u,
                                     kCL > 1 ? mapa_shared(&tempty_bar[1], 0) : 0u};
    const int s_end = a.sched_off[cluster_id + 1];
    // addend chunks are requested in the order they are used, one ahead, across
    // tiles: request q lands in slot q % 2 and completes phase (q / 2) % 2
    const bool has_d = !kTF32 && mode == kPoly;
    int d_req = 0, d_use = 0;
    auto d_request = [&](const GemmGroup& Gx, int b, int64_t r0, int64_t c) {
      const int s = d_req & 1;
      if (lane == 0) {
        mbar_arrive_expect_tx(&dbar[s], 2048u);
        tma_load_3d(dbuf + s * 128, &Gx.map_d, &dbar[s], (int)c, (int)r0, b);
      }
      ++d_req;
    };
    // last UPDATE: the weights of staged chunk q arrive by cp.async in slot q % 2
    // (the first or the second 4 KB of the staging, free of addends in UPDATE),
    // one cp.async group per chunk, requested one chunk ahead across tiles
    int w_req = 0, w_use = 0;
    auto w_slot = [&](int q) { return reinterpret_cast<uint4*>(wst + (q & 1) * 4096u); };
    int acc = 0;
    uint32_t acc_phase = 0;
    bool failed = false;
    for (int si = a.sched_off[cluster_id]; MUON_SCHED_OK si < s_end && !failed; ++si) {
      const int t = a.sched_units[si];
      const TileCoord tc = decode_tile<kCL>(a, t, rank);
      const GemmGroup& G = a.g[tc.g];
      const int64_t row0 = (int64_t)tc.bi * kBM + quad * 32;  // first row of this warp's 32
      const int64_t r = row0 + lane;
      const int64_t mb = (int64_t)tc.b * G.c_mstride;
      const int64_t ld = G.c_ld;
      const int64_t c_first = (int64_t)tc.bj * kBN + half * (kBN / 2);
      // this warp's chunks that start inside the matrix
      const int nch = c_first < G.N ? (int)min((int64_t)(kBN / 64), (G.N - c_first + 31) / 32) : 0;
      StagedTarget stg{};
      if constexpr (!kTF32) {
        // the first addend chunk loads while the accumulator is awaited, unless
        // the previous tile requested it already
        if (has_d && nch > 0 && d_req == d_use) d_request(G, tc.b, row0, c_first);
        if (a.fuse_apply) {
          stg = staged_target(a.apply, G.mat_base + tc.b);
          if (stg.ok && nch > 0 && w_req == w_use) {  // not requested by the previous tile
            staged_load(a.apply, stg, G.M, G.N, row0, c_first, lane, w_slot(w_req++));
            cp_async_commit();
          }
        }
      }
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
#pragma unroll 1
      for (int k = 0; k < (kTF32 ? kBN / 64 : nch); ++k) {
        const int cc = half * (kBN / 64) + k;
        const int64_t c0 = (int64_t)tc.bj * kBN + cc * 32;
        if constexpr (!kTF32) {
          const bool staged = a.fuse_apply && stg.ok;
          // the next addend chunk: this tile's next, else the next tile's first
          if (has_d && d_req == d_use + 1) {
            if (k + 1 < nch) {
              d_request(G, tc.b, row0, c0 + 32);
            } else if (si + 1 < s_end) {
              const TileCoord tn = decode_tile<kCL>(a, a.sched_units[si + 1], rank);
              const GemmGroup& Gn = a.g[tn.g];
              const int64_t cn = (int64_t)tn.bj * kBN + half * (kBN / 2);
              if (cn < Gn.N) d_request(Gn, tn.b, (int64_t)tn.bi * kBM + quad * 32, cn);
            }
          }
          float v[32];
          tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * kBN + cc * 32), v);
          if (staged && w_req == w_use + 1) {
            // the next chunk's weights (this tile's next chunk, else the next tile's
            // first), requested after the accumulator load, which would otherwise
            // queue behind these copies
            if (k + 1 < nch) {
              staged_load(a.apply, stg, G.M, G.N, row0, c0 + 32, lane, w_slot(w_req++));
              cp_async_commit();
            } else if (si + 1 < s_end) {
              const TileCoord tn = decode_tile<kCL>(a, a.sched_units[si + 1], rank);
              const GemmGroup& Gn = a.g[tn.g];
              const int64_t cn = (int64_t)tn.bj * kBN + half * (kBN / 2);
              const StagedTarget sn = staged_target(a.apply, Gn.mat_base + tn.b);
              if (sn.ok && cn < Gn.N) {
                staged_load(a.apply, sn, Gn.M, Gn.N, (int64_t)tn.bi * kBM + quad * 32, cn, lane, w_slot(w_req++));
                cp_async_commit();
              }
            }
          }
          const bool row_ok = r < G.M;
          const int64_t valid = G.N - c0;
          if (has_d) {
            const int s = d_use & 1;
            const bool landed = mbar_wait(&dbar[s], (uint32_t)(d_use >> 1) & 1u, abort_p, status);
            if (!__all_sync(0xffffffffu, landed)) { failed = true; break; }
            ++d_use;
            const uint4* dcur = dbuf + s * 128;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 raw = dcur[unit4(lane, q)];
              const uint32_t w4[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                const __nv_bfloat162 p2 = *reinterpret_cast<const __nv_bfloat162*>(&w4[h]);
                v[8 * q + 2 * h] = alpha * v[8 * q + 2 * h] + beta * __low2float(p2);
                v[8 * q + 2 * h + 1] = alpha * v[8 * q + 2 * h + 1] + beta * __high2float(p2);
              }
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] *= alpha;
          }
          if (a.fuse_apply) {  // last iteration: update the weights directly, X is not stored
            if (staged) {
              // this chunk's group is the oldest; the next chunk's may stay in flight
              if (w_req - w_use > 1) cp_async_wait<1>(); else cp_async_wait<0>();
              __syncwarp();
              staged_update_store(a.apply, stg, G.M, G.N, row0, c0, lane, v, w_slot(w_use++));
            } else if (row_ok) {
              fused_apply_chunk(a.apply, G.mat_base + tc.b, r, c0, valid, v);
            }
            __syncwarp();  // this weight slot is refilled two chunks later
            continue;
          }
          if (c0 == row0 && a.diag != 0.f) {  // a chunk on the diagonal: element (lane, lane)
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (j == lane) v[j] += a.diag;
          }
          // Every chunk of a tile leaves as one TMA box.  The symmetric products
          // also write the transpose of a chunk above the diagonal blocks (row
          // block left of the column block); the diagonal blocks are computed and
          // written whole, so A and B' are whole for the next GEMM.
          if (row0 >= G.M) {
            __syncwarp();
            continue;
          }
          const bool mirror = mode != kUpdate && (row0 >> 8) < (c0 >> 8);
          if (lane == 0) bulk_wait_group_read<0>();  // the last boxes have left the staging
          __syncwarp();
#pragma unroll
          for (int q = 0; q < 4; ++q) rowbuf[unit4(lane, q)] = pack8v(v + 8 * q);
          if (mirror) {
            // row j of the transpose is column j of the chunk; lane = its element
            const int e = lane & 7, u = lane >> 3;
#pragma unroll
            for (int j = 0; j < 32; ++j) tbuf[j * 32 + ((u ^ ((j >> 1) & 3)) << 3) + e] = __float2bfloat16_rn(v[j]);
          }
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&G.map_c, rowbuf, (int)c0, (int)row0, tc.b);
            if (mirror) tma_store_3d(&G.map_c, tbuf, (int)row0, (int)c0, tc.b);
            bulk_commit_group();
          }
          __syncwarp();
          continue;
        } else {
          float v[32];
          tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * kBN + cc * 32), v);
          if (r >= G.M || c0 >= G.N) continue;
          const int64_t valid = G.N - c0;  // columns of this chunk inside the matrix
          if (mode != kGram) {
            Epi<true>::add_d(v, G, mb + r * ld + c0, valid >= 32, valid, alpha, beta);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] *= alpha;
          }
          if (a.fuse_apply) {  // last iteration: update the weights directly, X is not stored
            fused_apply_chunk(a.apply, G.mat_base + tc.b, r, c0, valid, v);
            continue;
          }
          // direct store of row r (upper part only in the symmetric modes)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int64_t cq = c0 + 8 * q;
            unsigned mask = 0;
#pragma unroll
            for (int h = 0; h < 8; ++h)
              if (cq + h < G.N && (!sym || cq + h >= r)) mask |= 1u << h;
            Epi<true>::store8(G, mb + r * ld + cq, v + 8 * q, mask == 0xFFu, mask);
          }
          if (mode == kUpdate) {  // X'^T[c][r] for the next UPDATE's K-major B operand
            const int64_t mbt = (int64_t)tc.b * G.ct_mstride;
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c0 + j < G.N) Epi<true>::store1t(G, mbt + (c0 + j) * G.ct_ld + r, v[j]);
          }
          // mirror of the strictly upper part: C[c][r] = C[r][c]
          if (sym) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int64_t c = c0 + j;
              if (c > r && c < G.N) Epi<true>::store1(G, mb + c * ld + r, v[j]);
            }
          }
        }
      }
      if (failed) break;
      tc_fence_before();
      if constexpr (kCL == 1) {
        mbar_arrive(&tempty_bar[acc]);
      } else {
        __syncwarp();
        // hand the accumulator back to the MMA issuer: this warp's tcgen05.ld have
        // completed (wait::ld) and are ordered before the arrive by the fence above
        if (lane == 0) mbar_arrive_cluster_relaxed(tempty_lead[acc]);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if constexpr (!kTF32) {
      if (lane == 0) {
        // addend boxes still in flight land before the CTA exits (bounded), and
        // the output boxes are written
        for (int q = d_use; q < d_req; ++q)
          (void)mbar_wait(&dbar[q & 1], (uint32_t)(q >> 1) & 1u, nullptr, nullptr, 100000000ull);
        bulk_wait_group<0>();
      }
      __syncwarp();
    }
  }

  cp_async_wait<0>();  // no copy into shared memory outlives the CTA
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  // neither CTA frees Tensor Memory or exits while the pair's MMAs or signals may still reach it
  if constexpr (kCL > 1) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<kCL>(tmem_base, kTmemCols);
  }
}

template <bool kTF32, int kCL>
int max_clusters_impl(int num_sms) {
  static int cached = 0;
  if (cached) return cached;
  auto kernel = ns_gemm_kernel<kTF32, kCL>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cfg<kTF32, kCL>::kSmem) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  int n = num_sms / kCL;
  if (kCL > 1) {
    cudaLaunchConfig_t q = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = kCL;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    q.gridDim = dim3(num_sms / kCL * kCL);
    q.blockDim = dim3(kThreadsG);
    q.dynamicSmemBytes = Cfg<kTF32, kCL>::kSmem;
    q.attrs = at;
    q.numAttrs = 1;
    int m = 0;
    if (cudaOccupancyMaxActiveClusters(&m, kernel, &q) == cudaSuccess && m > 0) n = m;
    cudaGetLastError();
  }
  cached = n;
  return n;
}

template <bool kTF32, int kCL>
cudaError_t launch_impl(const GemmArgs& a, int num_sms, cudaStream_t s) {
  const int maxc = max_clusters_impl<kTF32, kCL>(num_sms);
  if (maxc <= 0) return cudaErrorInvalidConfiguration;
  if (a.n_clusters <= 0 || a.n_clusters > maxc) return cudaErrorInvalidValue;
  auto kernel = ns_gemm_kernel<kTF32, kCL>;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  cfg.gridDim = dim3(a.n_clusters * kCL);
  cfg.blockDim = dim3(kThreadsG);
  cfg.dynamicSmemBytes = Cfg<kTF32, kCL>::kSmem;
  cfg.stream = s;
  // may start as the previous kernel of the stream drains (the kernel waits for it
  // with griddepcontrol.wait before reading anything it wrote)
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (kCL > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = kCL;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

}  // namespace

size_t gemm_smem_bytes(bool tf32) { return tf32 ? Cfg<true, 1>::kSmem : Cfg<false, 1>::kSmem; }

int gemm_max_clusters(bool tf32, int cluster, int num_sms) {
  if (cluster == 2) return tf32 ? max_clusters_impl<true, 2>(num_sms) : max_clusters_impl<false, 2>(num_sms);
  return tf32 ? max_clusters_impl<true, 1>(num_sms) : max_clusters_impl<false, 1>(num_sms);
}

cudaError_t launch_gemm(const GemmArgs& a, int num_sms, bool tf32, int cluster, cudaStream_t s) {
  if (a.total_tiles <= 0) return cudaSuccess;
  if (cluster == 2) return tf32 ? launch_impl<true, 2>(a, num_sms, s) : launch_impl<false, 2>(a, num_sms, s);
  return tf32 ? launch_impl<true, 1>(a, num_sms, s) : launch_impl<false, 1>(a, num_sms, s);
}

#undef MUON_SCHED_OK

}  // namespace muon

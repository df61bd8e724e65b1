// Newton-Schulz for wide matrices of at most 128 rows (m <= 128, any n): one CTA
// takes one matrix through every quintic iteration in a single launch.
//
// The iteration is the one of the grouped GEMM kernel (DeepSpeed issue "[RFC]
// Enable Correct and High-Performance Muon Optimizer under ZeRO CPU Offload",
// section 2; "Muon Optimizer + FSDP", section 背景):
//   A = X X^T,  B' = a I + b A + c A A,  X' = B' X
// (X' = a X + (b A + c A A) X with the a X term carried by B', as the grouped
// kernel does in bf16: near convergence B' has eigenvalues near 1 where b A + c A A
// has them near a - 1, so rounding B' to bf16 loses less, and the UPDATE
// epilogue reads no X).
// The matrices this kernel exists for are the per-head slices of a fused QKV
// projection (128 rows each; DeepSpeed issue #8463, section 4.D).  At m = 128 the
// three GEMMs of one iteration do ~3 flops per byte of X, so a launch per GEMM
// streams X, A and B through HBM every iteration.  Here A and B never leave the
// SM, and X is read once and written once per iteration:
//
//   * A and B' (128 x 128 bf16, 32 KB) live in shared memory in the tcgen05
//     128-byte-swizzled K-major layout; B' overwrites A in place (each epilogue
//     thread reads its A elements before writing the same B' elements, after the
//     A A product has completed).
//   * X is streamed in 128-column chunks (two 128-row x 64-column boxes) through
//     a TMA ring.  The same boxes serve both uses: K-major operand of the Gram,
//     MN-major B operand of the UPDATE (k = the 128 rows).  Rows >= m and columns
//     >= n are zero-filled by TMA, so padding contributes nothing.  Successive
//     passes over X alternate direction, so a pass begins on the chunks the
//     previous one wrote last (still in L2 more often).  Every MMA has
//     N = 128: on one SM a tcgen05.mma of M = 128 takes at least ~60 cycles
//     whatever its N, so narrower products would idle the tensor pipe.
//   * The Gram of iteration k+1 is fused into the UPDATE of iteration k: the
//     epilogue writes each chunk of X' into a swizzled shared tile, on which the
//     MMA warp accumulates X' X'^T, and which the producer warp stores to the
//     workspace with a TMA bulk store (in place: a chunk of X' depends only on
//     the same chunk of X and on B; rows >= m and columns >= n are clipped by the
//     store).  A tile is free again once both the Gram and the store have read
//     it.  Iteration 0's Gram reads X0 (written by the momentum kernel) through
//     the ring.
//   * The last UPDATE applies the weight update (or emits U'): each epilogue
//     warp turns its 32 x 32 piece of a chunk around in a private shared
//     buffer, so the weights are read (cp.async, requested before the chunk's
//     accumulator is awaited) and written in whole 128-byte rows of the
//     caller's tensor (columns of U for tall matrices).
//   * The first iteration folds the normalisation s = 1/(||V||_F + eps) into its
//     epilogues (Gram: s^2, UPDATE: s), as the grouped kernel does.
//   * With fuse_prep (bf16 gradients, wide matrices) the first pass over a matrix
//     is also its momentum step ("Muon Optimizer + FSDP", section 背景: M_t =
//     momentum_update(grad) feeds NewtonSchulz): the epilogue warps, idle until
//     the Gram of iteration 0 is done, stream G and M through the shared memory
//     that A, B' and the X' tiles use later, write M_new back, write X0 =
//     bf16(V) to the workspace (for the UPDATE of iteration 0) and into the ring
//     stage the MMA warp builds the Gram from, and sum V^2 for the norm.  G and
//     M are read once, and X0 does not make a round trip through HBM between two
//     kernels.
//
// Roles (one persistent CTA per SM, 576 threads; matrices u = blockIdx.x,
// blockIdx.x + gridDim.x, ...):
//   warp 0     TMA producer: per matrix, X0 for the Gram, then X_k for each UPDATE.
//              During UPDATE k it also stores each X' tile as soon as it is
//              written (polling both; a tile's store half of "free" is given
//              when the next tile is stored), and waits for those stores
//              before loading X_{k+1}.
//   warp 1     tcgen05.mma issuer (M = 128, N = 128; fp32 accumulators in TMEM:
//              Gram 128 columns and three UPDATE buffers of 128, the first of
//              which also takes A A).  Within an UPDATE it issues whichever is
//              ready next: the UPDATE of the next chunk (a ring stage and an
//              accumulator free; its commit releases the stage) or the fused
//              Gram of the next X' tile.
//   warps 2-17 epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31 (rows), the four
//              warps of a lane quadrant split the columns (32 each).  Four
//              warps per SM sub-partition hide the latency of the accumulator
//              and shared-memory reads.  The warps run independently: every
//              hand-off is an mbarrier that each warp arrives on once (count 16).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "small_common.cuh"

namespace muon {
namespace {

constexpr int kThreadsS = 576;
constexpr int kStagesS = 4;
constexpr int kUBufs = 3;                             // UPDATE accumulators (128 TMEM columns each)
constexpr int kXsBufs = 2;                            // X' tiles for the fused Gram and the store
constexpr uint32_t kOffAB = 0;                        // A, then B in place: 2 atom columns
constexpr uint32_t kOffXS = 2 * kTile;                // two X' tiles, or (last iteration) a piece per warp
constexpr uint32_t kXsRegion = kEpiWarps * kWarpBuf;
static_assert(kXsBufs * kChunk <= kXsRegion, "X' tiles fit in the shared region");
constexpr uint32_t kOffRing = kOffXS + kXsRegion;
static_assert(kOffRing % 1024 == 0, "ring stages are 1024-byte aligned");
constexpr size_t kSmemS = kOffRing + (size_t)kStagesS * kChunk + 1024;
// fused momentum: the staging slots lie in the region of A, B' and the X' tiles
// (free while a matrix's first pass runs)
static_assert(kPrepSlots * kPrepSlot <= kOffRing, "the staging slots fit below the ring");
constexpr uint32_t kPrepBar = 1;                       // named barrier of the epilogue warps
constexpr uint32_t kTmemColsS = 512;
constexpr uint32_t kColG = 0, kColU = 128;            // UPDATE buffer u at kColU + 128 u
constexpr uint32_t kColP = kColU;                     // A A, drained before any UPDATE of the iteration
static_assert(kColU + 128 * kUBufs <= kTmemColsS, "accumulators fit in Tensor Memory");

__global__ void __launch_bounds__(kThreadsS, 1) ns_small_kernel(const __grid_constant__ SmallArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full_bar[kStagesS];
  __shared__ __align__(8) uint64_t empty_bar[kStagesS];  // the MMA issuer's commit: its MMAs have read the stage
  __shared__ __align__(8) uint64_t gram_full;            // Gram accumulated (MMA commit)
  __shared__ __align__(8) uint64_t a_ready;              // A in shared memory (epilogue warps)
  __shared__ __align__(8) uint64_t poly_full;            // A A accumulated (MMA commit)
  __shared__ __align__(8) uint64_t b_ready;              // B in shared memory (epilogue warps)
  __shared__ __align__(8) uint64_t u_full[kUBufs];       // UPDATE chunk accumulated (MMA commit)
  __shared__ __align__(8) uint64_t u_empty[kUBufs];      // UPDATE accumulator drained (epilogue warps)
  __shared__ __align__(8) uint64_t xs_full[kXsBufs];     // X' tile written (epilogue warps)
  __shared__ __align__(8) uint64_t xs_empty[kXsBufs];    // X' tile read by the Gram (MMA commit) and the store
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ __align__(8) uint64_t prep_done;            // fused momentum: X0 of the matrix is in the workspace
  __shared__ __align__(8) uint64_t pfull_bar[kStagesS];  // fused momentum: a stage of X0 written (16 warps)
  __shared__ float norm_red[kEpiWarps];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  unsigned* status = &a.status->flags;
  volatile int* abort_p = &abort_flag;
  const int K = a.ns_steps;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesS; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    mbar_init(&gram_full, 1);
    mbar_init(&a_ready, kEpiWarps);
    mbar_init(&poly_full, 1);
    mbar_init(&b_ready, kEpiWarps);
    for (int i = 0; i < kUBufs; ++i) {
      mbar_init(&u_full[i], 1);
      mbar_init(&u_empty[i], kEpiWarps);
    }
    for (int i = 0; i < kXsBufs; ++i) {
      mbar_init(&xs_full[i], kEpiWarps);
      mbar_init(&xs_empty[i], 2);
    }
    mbar_init(&drain_bar, 1);
    mbar_init(&prep_done, kEpiWarps);
    for (int i = 0; i < kStagesS; ++i) mbar_init(&pfull_bar[i], kEpiWarps);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0)
    for (int i = 0; i < a.n_groups; ++i) tma_prefetch_desc(&a.g[i].map_x);
  if (warp == 1) {
    tmem_alloc<1>(&tmem_slot, kTmemColsS);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  start_stagger(a);
  const uint32_t tmem = tmem_slot;
  uint8_t* ring = smem + kOffRing;

  if (warp == 0) {
    // ---------------- TMA producer and X' store ----------------
    // Per matrix the ring carries X0 chunks (Gram of iteration 0), then X_k
    // chunks for UPDATE k = 0 .. K-1.  During UPDATE k < K-1 the producer also
    // stores each X' tile once the epilogue has written it: it polls for a free
    // ring stage (next load) and a written tile (next store) and does whichever
    // is ready.
    int stage = 0;
    uint32_t phase = 0;
    uint32_t xc = 0;  // X' tiles stored so far
    uint32_t pd = 0;  // prep_done phase
    bool ok = true;
    // X is read again every iteration: keep its lines in L2 ahead of streams
    const uint64_t keep = l2_policy_evict_last();
    auto load_chunk = [&](const SmallGroup& G, int b, int j) {
      if (lane == 0) {
        uint8_t* dst = ring + (size_t)stage * kChunk;
        mbar_arrive_expect_tx(&full_bar[stage], kChunk);
        tma_load_3d_hint(dst, &G.map_x, &full_bar[stage], j * kChunkCols, 0, b, keep);
        tma_load_3d_hint(dst + kTile, &G.map_x, &full_bar[stage], j * kChunkCols + kBoxCols, 0, b, keep);
      }
      __syncwarp();
      ring_advance<kStagesS>(stage, phase, 1);
    };
    for (int u = blockIdx.x; ok && u < a.n_units; u += gridDim.x) {
      const UnitRef t = decode_unit(a, u);
      const SmallGroup& G = a.g[t.g];
      const int nch = (G.n + kChunkCols - 1) / kChunkCols;
      for (int pass = 0; ok && pass <= K; ++pass) {
        // serpentine order: odd passes walk the chunks backwards, starting with
        // those the previous pass wrote last, the likeliest to be still in L2
        const bool rev = pass & 1;
        auto chunk = [&](int j) { return rev ? nch - 1 - j : j; };
        if (pass == 0 && a.fuse_prep) {
          // the epilogue warps fill these stages with X0 computed from G and M;
          // UPDATE 0 reads X0 back once all of it is in the workspace
          ring_advance<kStagesS>(stage, phase, nch);
          const bool got = mbar_wait(&prep_done, pd, abort_p, status);
          pd ^= 1u;
          if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
          continue;
        }
        if (pass == 0 || pass == K) {  // no X' to store: plain loads
          for (int j = 0; j < nch; ++j) {
            const bool got = mbar_wait(&empty_bar[stage], phase ^ 1u, abort_p, status);
            if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
            load_chunk(G, t.b, chunk(j));
          }
          continue;
        }
        int jl = 0, js = 0;
        unsigned long long idle_since = 0;
        while (jl < nch || js < nch) {
          bool progressed = false;
          if (jl < nch && poll(&empty_bar[stage], phase ^ 1u)) {
            load_chunk(G, t.b, chunk(jl));
            ++jl;
            progressed = true;
          }
          const int xb = (int)(xc % kXsBufs);
          if (js < jl && poll(&xs_full[xb], (xc / kXsBufs) & 1u)) {
            if (lane == 0) {
              const uint8_t* src = smem + kOffXS + (size_t)xb * kChunk;
              const int cs = chunk(js) * kChunkCols;
              tma_store_3d_hint(&G.map_x, src, cs, 0, t.b, keep);
              if (cs + kBoxCols < G.n) tma_store_3d_hint(&G.map_x, src + kTile, cs + kBoxCols, 0, t.b, keep);
              bulk_commit_group();
              if (js > 0) {  // the previous tile's store has read it: its store half of "free"
                bulk_wait_group_read<1>();
                mbar_arrive(&xs_empty[(xc - 1) % kXsBufs]);
              }
            }
            __syncwarp();
            ++xc;
            ++js;
            progressed = true;
          }
          if (progressed) {
            idle_since = 0;
            continue;
          }
          __nanosleep(32);  // spare the barriers' shared memory while nothing is ready
          bool give_up = false;
          if (lane == 0) {
            const unsigned long long now = globaltimer_ns();
            if (idle_since == 0) idle_since = now;
            if (*abort_p) {
              give_up = true;
            } else if (now - idle_since > kWaitLimitNs) {
              *abort_p = 1;
              atomicOr(status, kStatusWaitTimeout);
              give_up = true;
            }
          }
          if (__shfl_sync(0xffffffffu, give_up, 0)) { ok = false; break; }
        }
        // X_{k+1} complete in the workspace before the next pass loads it
        if (lane == 0 && ok) {
          bulk_wait_group<0>();
          mbar_arrive(&xs_empty[(xc - 1) % kXsBufs]);
        }
        __syncwarp();
      }
    }
    if (lane == 0) {
      bulk_wait_group<0>();
      if (*abort_p) {
        // let loads already issued land before the CTA exits (bounded)
        for (int s = 0; s < kStagesS; ++s)
          (void)mbar_wait(&full_bar[s], phase ^ (s < stage ? 0u : 1u), nullptr, nullptr, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc_sq = make_idesc(1u, 128u, 128u, 0u);   // Gram, A A: both operands K-major
    const uint32_t idesc_up = make_idesc(1u, 128u, 128u, 1u);   // UPDATE: B operand MN-major
    const uint32_t ab = smem_u32(smem + kOffAB);
    const uint32_t xs0 = smem_u32(smem + kOffXS);
    int stage = 0;
    uint32_t phase = 0, ab_phase = 0;
    uint32_t pf_par = 0;      // fused momentum: next parity of pfull_bar[s] in bit s
    uint32_t uc = 0, xc = 0;  // UPDATE chunks and fused-Gram tiles so far
    bool ok = true;
    // K-major descriptor of k-slice kk (16 deep, kk = 0..7) of a 128 x 128 tile
    // made of two 64-column boxes
    auto sq_desc = [&](uint32_t base, int kk) {
      return smem_desc_sw128(base + (uint32_t)(kk >> 2) * kTile + (uint32_t)(kk & 3) * 32u, 16, 1024);
    };
    // X X^T over one 128-column tile (both operands: its rows, K-major)
#ifdef MUON_DEBUG
    const uint32_t smem_lo = smem_u32(smem), smem_hi = smem_lo + (uint32_t)(kSmemS - 1024);
#endif
    auto gram_tile = [&](uint32_t base, bool first) {
#ifdef MUON_DEBUG
      if (!smem_tile_ok(base, kChunk, smem_lo, smem_hi, status, abort_p)) return;
#endif
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t d = sq_desc(base, kk);
        mma<false, 1>(tmem + kColG, d, d, idesc_sq, (first && kk == 0) ? 0u : 1u);
      }
    };
    for (int u = blockIdx.x; ok && u < a.n_units; u += gridDim.x) {
      const UnitRef t = decode_unit(a, u);
      const SmallGroup& G = a.g[t.g];
      const int nch = (G.n + kChunkCols - 1) / kChunkCols;
      // Gram of iteration 0 over X0 chunks from the ring (TMA loads, or written
      // by the epilogue warps when they compute the momentum); the commit
      // releases the stage
      for (int j = 0; j < nch; ++j) {
        bool got;
        if (a.fuse_prep) {
          got = mbar_wait(&pfull_bar[stage], (pf_par >> stage) & 1u, abort_p, status);
          pf_par ^= 1u << stage;
          // complete the stage's full phase too, so that full_bar's phases keep
          // counting ring positions for the TMA-filled passes
          if (got && lane == 0) mbar_arrive(&full_bar[stage]);
        } else {
          got = mbar_wait(&full_bar[stage], phase, abort_p, status);
        }
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
          gram_tile(smem_u32(ring + (size_t)stage * kChunk), j == 0);
          mma_commit<1>(&empty_bar[stage]);
        }
        __syncwarp();
        ring_advance<kStagesS>(stage, phase, 1);
      }
      if (!ok) break;
      if (lane == 0) mma_commit<1>(&gram_full);
      __syncwarp();
      for (int k = 0; ok && k < K; ++k) {
        // A A (A read as A A^T: both operands are the K-major rows of A)
        bool got = mbar_wait(&a_ready, ab_phase, abort_p, status);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t d = sq_desc(ab, kk);
            mma<false, 1>(tmem + kColP, d, d, idesc_sq, kk != 0 ? 1u : 0u);
          }
          mma_commit<1>(&poly_full);
        }
        __syncwarp();
        got = mbar_wait(&b_ready, ab_phase, abort_p, status);
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        tc_fence_after();
        ab_phase ^= 1u;
        const bool fuse = k + 1 < K;
        // UPDATE chunks in order as soon as a ring stage and an accumulator are
        // free; fused-Gram tiles in order as soon as the epilogue has written
        // them.  Lane 0 decides (its view of the barriers), the warp follows.
        int jn = 0, gn = 0;
        unsigned long long idle_since = 0;
        while (jn < nch || (fuse && gn < nch)) {
          bool progressed = false;
          if (jn < nch) {
            const int ub = (int)(uc % kUBufs);
            if (poll(&full_bar[stage], phase) && poll(&u_empty[ub], ((uc / kUBufs) & 1u) ^ 1u)) {
              tc_fence_after();
              if (lane == 0) {
                const uint32_t xb = smem_u32(ring + (size_t)stage * kChunk);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                  // B operand: k rows 16 kk .. +15 of the chunk, MN-major, its two
                  // 64-column boxes one tile apart
                  const uint64_t bd = smem_desc_sw128(xb + (uint32_t)kk * 2048u, kTile, 1024);
                  mma<false, 1>(tmem + kColU + 128u * (uint32_t)ub, sq_desc(ab, kk), bd, idesc_up,
                                kk != 0 ? 1u : 0u);
                }
                mma_commit<1>(&u_full[ub]);
                mma_commit<1>(&empty_bar[stage]);  // free once these MMAs have read it
              }
              __syncwarp();
              ++uc;
              ++jn;
              ring_advance<kStagesS>(stage, phase, 1);
              progressed = true;
            }
          }
          if (fuse && gn < jn) {
            const int xb = (int)(xc % kXsBufs);
            if (poll(&xs_full[xb], (xc / kXsBufs) & 1u)) {
              tc_fence_after();
              if (lane == 0) {
                gram_tile(xs0 + (uint32_t)xb * kChunk, gn == 0);
                mma_commit<1>(&xs_empty[xb]);
              }
              __syncwarp();
              ++xc;
              ++gn;
              progressed = true;
            }
          }
          if (progressed) {
            idle_since = 0;
            continue;
          }
          // nothing ready: give up after the wait limit, or when another role has
          __nanosleep(32);  // spare the barriers' shared memory while nothing is ready
          bool give_up = false;
          if (lane == 0) {
            const unsigned long long now = globaltimer_ns();
            if (idle_since == 0) idle_since = now;
            if (*abort_p) {
              give_up = true;
            } else if (now - idle_since > kWaitLimitNs) {
              *abort_p = 1;
              atomicOr(status, kStatusWaitTimeout);
              give_up = true;
            }
          }
          if (__shfl_sync(0xffffffffu, give_up, 0)) { ok = false; break; }
        }
        if (!ok) break;
        if (fuse) {
          if (lane == 0) mma_commit<1>(&gram_full);
          __syncwarp();
        }
      }
    }
    // every MMA issued by lane 0 has completed before TMEM is freed
    if (lane == 0) {
      mma_commit<1>(&drain_bar);
      (void)mbar_wait(&drain_bar, 0u, nullptr, status);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2..17) ----------------
    // warp w: rows 32 (w % 4) .. +31 (TMEM lanes), columns part * 32 .. +31 of
    // every 128 x 128 tile (A, B, X' and each chunk): pieces (part % 2) * 4 ..
    // +3 of box part / 2
    const int quad = warp & 3;
    const int part = (warp - 2) >> 2;
    const int ew = warp - 2;
    const int r = quad * 32 + lane;                       // row of the matrix (wide form)
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const int box = part >> 1;
    const int p0 = (part & 1) * 4;
    uint8_t* ab = smem + kOffAB + (size_t)box * kTile;    // this warp's box of A / B
    float* wbuf = reinterpret_cast<float*>(smem + kOffXS + (size_t)ew * kWarpBuf);
    uint32_t gp = 0, pp = 0, uc = 0, xc = 0;
    uint32_t pos = 0;  // ring position (fused momentum fills the first pass's stages)
    uint32_t pd = 0;   // prep_done phase
    bool ok = true;
    for (int u = blockIdx.x; u < a.n_units; u += gridDim.x) {
      if (a.fuse_prep) {
        // every epilogue thread arrives here for every matrix (done with the
        // previous one's shared memory), and a warp that gave up a wait stops
        // them all together: the named barriers below are then never left waiting
        __syncwarp();
        ok = bar_and(kPrepBar, kPrepThreads, ok);
      }
      if (!ok) break;
      const UnitRef t = decode_unit(a, u);
      const SmallGroup& G = a.g[t.g];
      const int nch = (G.n + kChunkCols - 1) / kChunkCols;
      const int mat = G.mat_base + t.b;
      float s = 0.f;
      bool bad = false;
      if (a.fuse_prep) {
        ok = __all_sync(0xffffffffu, prep_matrix<kStagesS>(a, G, t.b, mat, smem, smem + 2 * kPrepSlot, ring,
                                                           pfull_bar, empty_bar, &prep_done, norm_red, pos,
                                                           abort_p, status));
        if (!ok) continue;  // the barrier at the top stops every epilogue warp together
        pos += (uint32_t)(nch * K);  // the UPDATE passes' stages, filled by the producer
      } else {
        s = a.scale[mat];
      }
      for (int k = 0; ok && k < K; ++k) {
        // ---- A = (s^2 in iteration 0) X X^T, bf16, into shared memory ----
        ok = __all_sync(0xffffffffu, mbar_wait(&gram_full, gp, abort_p, status));
        gp ^= 1u;
        if (!ok) break;
        tc_fence_after();
        if (k == 0 && a.fuse_prep) {
          // every warp's partial sum was written before its prep_done arrival
          ok = __all_sync(0xffffffffu, mbar_wait(&prep_done, pd, abort_p, status));
          pd ^= 1u;
          if (!ok) break;
          s = prep_scale(a, mat, norm_red, bad);
        }
        {
          const float sa = k == 0 ? s * s : 1.f;
          float v[32];
          tmem_ld_32x32b_x32(tmem + lane_base + kColG + (uint32_t)(part * 32), v);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = sa * v[8 * q + e];
            *reinterpret_cast<uint4*>(ab + sw128(r, p0 + q)) = pack8(w);
          }
        }
        fence_proxy_async_shared();  // read next by the tensor core
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&a_ready);
        // ---- B' = a I + b A + c (A A), in place over A ----
        ok = __all_sync(0xffffffffu, mbar_wait(&poly_full, pp, abort_p, status));
        pp ^= 1u;
        if (!ok) break;
        tc_fence_after();
        {
          float v[32];
          tmem_ld_32x32b_x32(tmem + lane_base + kColP + (uint32_t)(part * 32), v);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4* p = reinterpret_cast<uint4*>(ab + sw128(r, p0 + q));
            float x[8], w[8];
            unpack8(*p, x);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              w[e] = a.coef[k][2] * v[8 * q + e] + a.coef[k][1] * x[e];
              if (quad == part && 8 * q + e == lane) w[e] += a.coef[k][0];  // the diagonal (r, r)
            }
            *p = pack8(w);
          }
        }
        fence_proxy_async_shared();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&b_ready);
        // ---- X' = (s in iteration 0) B' X, chunk by chunk ----
        const bool last = k + 1 == K;
        const float alpha = k == 0 ? s : 1.f;
        ApplyTarget tg{};
        bool vec = false;
        if (last) {
          tg = apply_target(a.apply, mat);
          if (a.fuse_prep) tg.skip = !a.apply.emit && a.apply.skip_nonfinite && bad;
          vec = piece_vec(a.apply, tg);
        }
        for (int j = 0; j < nch; ++j) {
          const int ub = (int)(uc % kUBufs);
          const int xb = (int)(xc % kXsBufs);
          // UPDATE k is the producer's pass k + 1: backwards when k is even
          const int jc = (k & 1) ? j : nch - 1 - j;
          const int64_t c0 = (int64_t)jc * kChunkCols + part * 32;  // this warp's 32 columns
          if (last && j > 0) {
            // the weights of this warp's piece load while the chunk's accumulator
            // is awaited and drained (the buffer's previous piece is stored)
            piece_load(a.apply, tg, vec, G.m, G.n, quad * 32, c0, lane, wbuf);
            cp_async_commit();
          }
          ok = mbar_wait(&u_full[ub], (uc / kUBufs) & 1u, abort_p, status) &&
               (last || mbar_wait(&xs_empty[xb], ((xc / kXsBufs) & 1u) ^ 1u, abort_p, status));
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          if (last && j == 0) {
            // the buffer shares memory with the X' tiles: the previous pass's
            // stores of them completed before the producer loaded this chunk
            piece_load(a.apply, tg, vec, G.m, G.n, quad * 32, c0, lane, wbuf);
            cp_async_commit();
          }
          tc_fence_after();
          float v[32];
          tmem_ld_32x32b_x32(tmem + lane_base + kColU + 128u * (uint32_t)ub + (uint32_t)(part * 32), v);
          if (k == 0) {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] *= alpha;
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&u_empty[ub]);
          if (last) {
            cp_async_wait<0>();
            __syncwarp();
            piece_update(a.apply, tg, vec, lane, v, wbuf);
            __syncwarp();
            piece_store(a.apply, tg, vec, G.m, G.n, quad * 32, c0, lane, wbuf);
            __syncwarp();  // the buffer is refilled for the next chunk
          } else {
            uint8_t* xs = smem + kOffXS + (size_t)xb * kChunk + (size_t)box * kTile;
#pragma unroll
            for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4*>(xs + sw128(r, p0 + q)) = pack8(v + 8 * q);
            fence_proxy_async_shared();  // read next by the tensor core and the TMA store
            __syncwarp();
            if (lane == 0) mbar_arrive(&xs_full[xb]);
            ++xc;
          }
          ++uc;
        }
        if (last) cp_async_wait<0>();
      }
    }
    cp_async_wait<0>();  // no copy into shared memory outlives the CTA (after an abort)
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<1>(tmem, kTmemColsS);
  }
}

}  // namespace

cudaError_t launch_ns_small(const SmallArgs& a, int num_sms, cudaStream_t s) {
  if (a.n_units <= 0) return cudaSuccess;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(ns_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemS);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int grid = a.n_units < num_sms ? a.n_units : num_sms;
  ns_small_kernel<<<grid, kThreadsS, kSmemS, s>>>(a);
  return cudaGetLastError();
}

}  // namespace muon

// Newton-Schulz by the "gram" method for wide matrices of at most 128 rows
// (m <= 128, any n): one CTA takes one matrix through every iteration in a
// single launch, touching X only twice.
//
// The method (DeepSpeed PR "[Muon] CPU offload: pin the momentum and overlap the
// host writeback", section Tests, and DeepSpeed issue "[RFC] ... ZeRO CPU
// Offload", follow-up list, name it; the reading taken is the quintic iteration
// rewritten on the Gram matrix): with A_k = X_k X_k^T and Q_k = a I + b A_k +
// c A_k^2, X_{k+1} = Q_k X_k gives
//   A_{k+1} = Q_k A_k Q_k,   X_K = R_K X_0,   R_{k+1} = Q_k R_k,  R_0 = s I,
// s = 1 / (||V||_F + eps).  Every Q_k, A_k and R_k is a polynomial in A_0, so all
// of them are symmetric and commute: each m x m product is formed as Y Z^T from
// the rows of Y and Z (both tcgen05 operands K-major), like the Gram itself.
//
// Arithmetic: X_0 is bf16 (as in the quintic kernels); A_0 accumulates in fp32.
// The m x m matrices are kept in fp32 and enter each product split into bf16
// high and low parts, Y Z^T ~ Yh Zh^T + Yh Zl^T + Yl Zh^T (fp32 accumulation):
// about 16 bits of each operand, against the 8 of a plain bf16 product.  The
// final U = R X_0 uses Rh X_0 + Rl X_0.  A CPU simulation of exactly these
// roundings against the fp64 oracle gives 1.8e-3 on the per-head inputs (the
// quintic kernels: 8e-3).
//
// Per matrix:
//   first pass   X_0 chunks through the TMA ring (written by the momentum kernel),
//                or computed from G and M by the epilogue warps (fuse_prep, as in
//                the quintic kernel); the MMA warp accumulates X_0 X_0^T.
//   iterations   k = 0 .. K-1: A A, then Q (epilogue), then Q A and Q R, then
//                (Q A) Q -- 3 bf16 products each, 128 x 128 x 128, all on chip;
//                the last iteration forms only A A, Q and Q R.
//   final pass   X_0 chunks through the ring again; U = R X_0 per chunk, applied
//                to the weights (or emitted as U') from the accumulators, as the
//                quintic kernel's last UPDATE does.
//
// Shared memory, in 32 KB units (a 128 x 128 bf16 tile = two 64-column boxes):
//   0-1   momentum staging slots 0, 1 | Q tiles (high, low) | weight-update pieces
//   2-4   ring stages 0-2             | A (or Q A) tiles (high, low) in 2-3
//   5-6   momentum staging slots 2, 3 | R tiles (high, low)
// The ring is idle during the iterations: the producer loads the final pass only
// once the last Q is formed (small_done), when the A tiles have been read.
// Tensor Memory: T0, T1 take A A and the next A in turn, T2 Q A, T3 the Gram and
// then Q R; in the final pass T0-T2 hold U's chunks and T3 the next Gram.
//
// Roles (576 threads): warp 0 TMA producer, warp 1 tcgen05.mma issuer (one
// thread), warps 2-17 epilogue (warp w: TMEM lanes 32 (w % 4) .. +31, columns
// 32 ((w - 2) / 4) .. +31 of each 128 x 128 accumulator).  Every hand-off is an
// mbarrier; every wait is bounded and gives up together with the other roles.
#include "small_common.cuh"

namespace muon {
namespace {

constexpr int kThreadsG = 576;
constexpr int kStagesG = 3;
constexpr int kUBufsG = 3;
constexpr uint32_t kUnit = 2 * kTile;                 // 32 KB: one 128 x 128 bf16 tile
constexpr uint32_t kOffQ = 0;                         // Q high, Q low
constexpr uint32_t kOffRingG = 2 * kUnit;             // ring stages 0-2
constexpr uint32_t kOffA = 2 * kUnit;                 // A (or Q A) high, low
constexpr uint32_t kOffR = 5 * kUnit;                 // R high, low
constexpr size_t kSmemG = 7 * (size_t)kUnit + 1024;
static_assert(kEpiWarps * kWarpBuf <= 2 * kUnit, "weight-update pieces fit in units 0-1");
static_assert(2 * kPrepSlot <= 2 * kUnit, "two staging slots per pair of units");
static_assert(kOffRingG + kStagesG * kChunk <= kOffR, "the ring stays clear of the R tiles");
constexpr uint32_t kTmemColsG = 512;
constexpr uint32_t kColT0 = 0, kColT1 = 128, kColT2 = 256, kColT3 = 384;
constexpr uint32_t kPrepBarG = 1;

// K-major descriptor of k-slice kk (16 deep, kk = 0..7) of a 128 x 128 tile made
// of two 64-column boxes
__device__ __forceinline__ uint64_t tile_desc(uint32_t base, int kk) {
  return smem_desc_sw128(base + (uint32_t)(kk >> 2) * kTile + (uint32_t)(kk & 3) * 32u, 16, 1024);
}

// The warp's 32 x 32 piece of a 128 x 128 fp32 matrix split into bf16 high and
// low tiles: row r, columns 32 part .. +31 (pieces p0 .. p0 + 3 of box `box`).
__device__ __forceinline__ void store_split(uint8_t* hi, uint8_t* lo, int box, int r, int p0, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float h[8], l[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      h[e] = __bfloat162float(__float2bfloat16_rn(v[8 * q + e]));
      l[e] = v[8 * q + e] - h[e];
    }
    *reinterpret_cast<uint4*>(hi + (size_t)box * kTile + sw128(r, p0 + q)) = pack8(h);
    *reinterpret_cast<uint4*>(lo + (size_t)box * kTile + sw128(r, p0 + q)) = pack8(l);
  }
}

__global__ void __launch_bounds__(kThreadsG, 1) ns_gram_kernel(const __grid_constant__ SmallArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  __shared__ __align__(8) uint64_t full_bar[kStagesG];
  __shared__ __align__(8) uint64_t empty_bar[kStagesG];
  __shared__ __align__(8) uint64_t pfull_bar[kStagesG];  // fused momentum: a stage of X_0 written (16 warps)
  __shared__ __align__(8) uint64_t prep_done;            // fused momentum: X_0 in the workspace (16 warps)
  __shared__ __align__(8) uint64_t gram_full;            // X_0 X_0^T accumulated (commit)
  __shared__ __align__(8) uint64_t a_ready;              // A tiles (and at k = 0 the R tiles) written (16)
  __shared__ __align__(8) uint64_t aa_full;              // A A accumulated (commit)
  __shared__ __align__(8) uint64_t q_ready;              // Q tiles written (16)
  __shared__ __align__(8) uint64_t small_done;           // the last Q written: the ring may fill again (16)
  __shared__ __align__(8) uint64_t p2_full;              // Q A accumulated (commit)
  __shared__ __align__(8) uint64_t p2_ready;             // Q A tiles written over the A tiles (16)
  __shared__ __align__(8) uint64_t r_full;               // Q R accumulated (commit)
  __shared__ __align__(8) uint64_t r_ready;              // R tiles written (16)
  __shared__ __align__(8) uint64_t an_full;              // (Q A) Q accumulated (commit)
  __shared__ __align__(8) uint64_t u_full[kUBufsG];      // final pass: a chunk of U accumulated (commit)
  __shared__ __align__(8) uint64_t u_empty[kUBufsG];     // final pass: its accumulator drained (16)
  __shared__ __align__(8) uint64_t drain_bar;
  __shared__ float norm_red[kEpiWarps];
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  unsigned* status = &a.status->flags;
  volatile int* abort_p = &abort_flag;
  const int K = a.ns_steps;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesG; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
      mbar_init(&pfull_bar[s], kEpiWarps);
    }
    mbar_init(&prep_done, kEpiWarps);
    mbar_init(&gram_full, 1);
    mbar_init(&a_ready, kEpiWarps);
    mbar_init(&aa_full, 1);
    mbar_init(&q_ready, kEpiWarps);
    mbar_init(&small_done, kEpiWarps);
    mbar_init(&p2_full, 1);
    mbar_init(&p2_ready, kEpiWarps);
    mbar_init(&r_full, 1);
    mbar_init(&r_ready, kEpiWarps);
    mbar_init(&an_full, 1);
    for (int i = 0; i < kUBufsG; ++i) {
      mbar_init(&u_full[i], 1);
      mbar_init(&u_empty[i], kEpiWarps);
    }
    mbar_init(&drain_bar, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0)
    for (int i = 0; i < a.n_groups; ++i) tma_prefetch_desc(&a.g[i].map_x);
  if (warp == 1) {
    tmem_alloc<1>(&tmem_slot, kTmemColsG);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  start_stagger(a);
  const uint32_t tmem = tmem_slot;
  uint8_t* ring = smem + kOffRingG;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    // Per matrix: X_0 chunks for the Gram (unless the epilogue warps compute
    // them), then -- once the iterations no longer need the A tiles -- X_0 chunks
    // for U = R X_0.
    int stage = 0;
    uint32_t phase = 0, sd = 0;
    bool ok = true;
    const uint64_t keep = l2_policy_evict_last();
    auto load_chunk = [&](const SmallGroup& G, int b, int j) {
      if (lane == 0) {
        uint8_t* dst = ring + (size_t)stage * kChunk;
        mbar_arrive_expect_tx(&full_bar[stage], kChunk);
        tma_load_3d_hint(dst, &G.map_x, &full_bar[stage], j * kChunkCols, 0, b, keep);
        tma_load_3d_hint(dst + kTile, &G.map_x, &full_bar[stage], j * kChunkCols + kBoxCols, 0, b, keep);
      }
      __syncwarp();
      ring_advance<kStagesG>(stage, phase, 1);
    };
    for (int u = blockIdx.x; ok && u < a.n_units; u += gridDim.x) {
      const UnitRef t = decode_unit(a, u);
      const SmallGroup& G = a.g[t.g];
      const int nch = (G.n + kChunkCols - 1) / kChunkCols;
      if (a.fuse_prep) {
        ring_advance<kStagesG>(stage, phase, nch);  // the epilogue warps fill these stages
      } else {
        for (int j = 0; j < nch; ++j) {
          const bool got = mbar_wait(&empty_bar[stage], phase ^ 1u, abort_p, status);
          if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
          load_chunk(G, t.b, j);
        }
        if (!ok) break;
      }
      // the iterations have read the A tiles for the last time (and X_0 is in
      // the workspace: each warp's writes precede its small_done arrival)
      const bool got = mbar_wait(&small_done, sd, abort_p, status);
      sd ^= 1u;
      if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
      for (int j = 0; j < nch; ++j) {
        const bool free = mbar_wait(&empty_bar[stage], phase ^ 1u, abort_p, status);
        if (!__all_sync(0xffffffffu, free)) { ok = false; break; }
        load_chunk(G, t.b, j);
      }
    }
    if (lane == 0 && *abort_p) {
      // let loads already issued land before the CTA exits (bounded)
      for (int s = 0; s < kStagesG; ++s)
        (void)mbar_wait(&full_bar[s], phase ^ (s < stage ? 0u : 1u), nullptr, nullptr, 100000000ull);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    const uint32_t idesc_sq = make_idesc(1u, 128u, 128u, 0u);   // Y Z^T: both operands K-major
    const uint32_t idesc_up = make_idesc(1u, 128u, 128u, 1u);   // R X_0: X_0 MN-major
    const uint32_t qh = smem_u32(smem + kOffQ), ql = qh + kUnit;
    const uint32_t ah = smem_u32(smem + kOffA), al = ah + kUnit;
    const uint32_t rh = smem_u32(smem + kOffR), rl = rh + kUnit;
    int stage = 0;
    uint32_t phase = 0;
    uint32_t pf_par = 0;  // next parity of pfull_bar[s] in bit s
    uint32_t ar = 0, qr = 0, pr = 0, rr = 0;
    uint32_t uc = 0;
    bool ok = true;
#ifdef MUON_DEBUG
    const uint32_t smem_lo = smem_u32(smem), smem_hi = smem_lo + 7 * kUnit;
#endif
    // Y Z^T from the rows of two split tiles, accumulated from zero into `acc`
    auto yzt = [&](uint32_t acc, uint32_t yh, uint32_t yl, uint32_t zh, uint32_t zl) {
#ifdef MUON_DEBUG
      if (!(smem_tile_ok(yh, kUnit, smem_lo, smem_hi, status, abort_p) &&
            smem_tile_ok(yl, kUnit, smem_lo, smem_hi, status, abort_p) &&
            smem_tile_ok(zh, kUnit, smem_lo, smem_hi, status, abort_p) &&
            smem_tile_ok(zl, kUnit, smem_lo, smem_hi, status, abort_p) &&
            MUON_GUARD(acc + 128u <= kTmemColsG, status, abort_p)))
        return;
#endif
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) mma<false, 1>(tmem + acc, tile_desc(yh, kk), tile_desc(zh, kk), idesc_sq, kk ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) mma<false, 1>(tmem + acc, tile_desc(yh, kk), tile_desc(zl, kk), idesc_sq, 1u);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) mma<false, 1>(tmem + acc, tile_desc(yl, kk), tile_desc(zh, kk), idesc_sq, 1u);
    };
    auto wait_all = [&](uint64_t* bar, uint32_t& par) {
      const bool got = mbar_wait(bar, par, abort_p, status);
      par ^= 1u;
      return __all_sync(0xffffffffu, got);
    };
    for (int u = blockIdx.x; ok && u < a.n_units; u += gridDim.x) {
      const UnitRef t = decode_unit(a, u);
      const SmallGroup& G = a.g[t.g];
      const int nch = (G.n + kChunkCols - 1) / kChunkCols;
      // ---- X_0 X_0^T into T3 ----
      for (int j = 0; j < nch; ++j) {
        bool got;
        if (a.fuse_prep) {
          got = mbar_wait(&pfull_bar[stage], (pf_par >> stage) & 1u, abort_p, status);
          pf_par ^= 1u << stage;
          if (got && lane == 0) mbar_arrive(&full_bar[stage]);  // full_bar's phases keep counting positions
        } else {
          got = mbar_wait(&full_bar[stage], phase, abort_p, status);
        }
        if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
        tc_fence_after();
        if (lane == 0) {
          const uint32_t xb = smem_u32(ring + (size_t)stage * kChunk);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t d = tile_desc(xb, kk);
            mma<false, 1>(tmem + kColT3, d, d, idesc_sq, (j == 0 && kk == 0) ? 0u : 1u);
          }
          mma_commit<1>(&empty_bar[stage]);
        }
        __syncwarp();
        ring_advance<kStagesG>(stage, phase, 1);
      }
      if (!ok) break;
      if (lane == 0) mma_commit<1>(&gram_full);
      __syncwarp();
      // ---- the iterations on 128 x 128 matrices ----
      for (int k = 0; ok && k < K; ++k) {
        const bool last = k + 1 == K;
        const uint32_t t_aa = (k & 1) ? kColT1 : kColT0;   // A A now, the next A after Q A Q
        if (!(ok = wait_all(&a_ready, ar))) break;
        tc_fence_after();
        if (lane == 0) {
          yzt(t_aa, ah, al, ah, al);
          mma_commit<1>(&aa_full);
        }
        __syncwarp();
        if (!(ok = wait_all(&q_ready, qr))) break;
        tc_fence_after();
        if (lane == 0 && !last) {
          yzt(kColT2, qh, ql, ah, al);          // Q A
          mma_commit<1>(&p2_full);
        }
        __syncwarp();
        if (k > 0 && !(ok = wait_all(&r_ready, rr))) break;  // R of the previous iteration in its tiles
        tc_fence_after();
        if (lane == 0) {
          yzt(kColT3, qh, ql, rh, rl);          // Q R
          mma_commit<1>(&r_full);
        }
        __syncwarp();
        if (!last) {
          if (!(ok = wait_all(&p2_ready, pr))) break;
          tc_fence_after();
          if (lane == 0) {
            yzt(t_aa, ah, al, qh, ql);          // (Q A) Q, from the Q A tiles
            mma_commit<1>(&an_full);
          }
          __syncwarp();
        }
      }
      if (!ok) break;
      // ---- U = R X_0, chunk by chunk, into T0-T2 ----
      if (!(ok = wait_all(&r_ready, rr))) break;
      tc_fence_after();
      int jn = 0;
      unsigned long long idle_since = 0;
      while (jn < nch) {
        const int ub = (int)(uc % kUBufsG);
        if (poll(&full_bar[stage], phase) && poll(&u_empty[ub], ((uc / kUBufsG) & 1u) ^ 1u)) {
          tc_fence_after();
#ifdef MUON_DEBUG
          const bool stage_ok = smem_tile_ok(smem_u32(ring + (size_t)stage * kChunk), kChunk, smem_lo, smem_hi, status,
                                             abort_p);
#else
          const bool stage_ok = true;
#endif
          if (lane == 0 && stage_ok) {
            const uint32_t xb = smem_u32(ring + (size_t)stage * kChunk);
            const uint32_t acc = tmem + (uint32_t)ub * 128u;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              // B operand: k rows 16 kk .. +15 of the chunk, MN-major, its two
              // 64-column boxes one tile apart
              const uint64_t bd = smem_desc_sw128(xb + (uint32_t)kk * 2048u, kTile, 1024);
              mma<false, 1>(acc, tile_desc(rh, kk), bd, idesc_up, kk ? 1u : 0u);
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t bd = smem_desc_sw128(xb + (uint32_t)kk * 2048u, kTile, 1024);
              mma<false, 1>(acc, tile_desc(rl, kk), bd, idesc_up, 1u);
            }
            mma_commit<1>(&u_full[ub]);
            mma_commit<1>(&empty_bar[stage]);
          }
          __syncwarp();
          ++uc;
          ++jn;
          ring_advance<kStagesG>(stage, phase, 1);
          idle_since = 0;
          continue;
        }
        __nanosleep(32);
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
    }
    // every MMA issued by lane 0 has completed before TMEM is freed
    if (lane == 0) {
      mma_commit<1>(&drain_bar);
      (void)mbar_wait(&drain_bar, 0u, nullptr, status);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2..17) ----------------
    const int quad = warp & 3;
    const int part = (warp - 2) >> 2;
    const int ew = warp - 2;
    const int r = quad * 32 + lane;                       // row of the 128 x 128 matrices
    const uint32_t lane_base = (uint32_t)(quad * 32) << 16;
    const int box = part >> 1;
    const int p0 = (part & 1) * 4;
    uint8_t* q_hi = smem + kOffQ;
    uint8_t* q_lo = q_hi + kUnit;
    uint8_t* a_hi = smem + kOffA;
    uint8_t* a_lo = a_hi + kUnit;
    uint8_t* r_hi = smem + kOffR;
    uint8_t* r_lo = r_hi + kUnit;
    float* wbuf = reinterpret_cast<float*>(smem + (size_t)ew * kWarpBuf);
    uint32_t gp = 0, aap = 0, p2p = 0, rp = 0, anp = 0, pd = 0, uc = 0;
    uint32_t pos = 0;  // ring position (fused momentum fills the first pass's stages)
    bool ok = true;
    auto wait_all = [&](uint64_t* bar, uint32_t& par) {
      const bool got = mbar_wait(bar, par, abort_p, status);
      par ^= 1u;
      return __all_sync(0xffffffffu, got);
    };
    auto tld = [&](uint32_t col, float (&v)[32]) {
      tmem_ld_32x32b_x32(tmem + lane_base + col + (uint32_t)(part * 32), v);
    };
    // tiles written by this warp: visible to the tensor core, then the hand-off
    auto handoff = [&](uint64_t* bar) {
      fence_proxy_async_shared();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar);
    };
    for (int u = blockIdx.x; u < a.n_units; u += gridDim.x) {
      if (a.fuse_prep) {
        // every epilogue thread arrives here for every matrix (done with the
        // previous one's shared memory), and a warp that gave up a wait stops
        // them all together
        __syncwarp();
        ok = bar_and(kPrepBarG, kPrepThreads, ok);
      }
      if (!ok) break;
      const UnitRef t = decode_unit(a, u);
      const SmallGroup& G = a.g[t.g];
      const int nch = (G.n + kChunkCols - 1) / kChunkCols;
      const int mat = G.mat_base + t.b;
      float s = 0.f;
      bool bad = false;
      if (a.fuse_prep) {
        ok = __all_sync(0xffffffffu, prep_matrix<kStagesG>(a, G, t.b, mat, smem, smem + kOffR, ring, pfull_bar,
                                                           empty_bar, &prep_done, norm_red, pos, abort_p,
                                                           status));
        if (!ok) continue;  // the barrier at the top stops every epilogue warp together
        pos += (uint32_t)nch;  // the final pass's stages, filled by the producer
      } else {
        s = a.scale[mat];
      }
      // ---- A_0 = s^2 X_0 X_0^T and R_0 = s I into their tiles ----
      if (!(ok = wait_all(&gram_full, gp))) continue;
      tc_fence_after();
      if (a.fuse_prep) {
        // every warp's partial sum was written before its prep_done arrival
        if (!(ok = wait_all(&prep_done, pd))) continue;
        s = prep_scale(a, mat, norm_red, bad);
      }
      const float s2 = s * s;
      {
        float v[32];
        tld(kColT3, v);
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] *= s2;
        store_split(a_hi, a_lo, box, r, p0, v);
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = (quad == part && e == lane) ? s : 0.f;
        store_split(r_hi, r_lo, box, r, p0, v);
      }
      handoff(&a_ready);
      for (int k = 0; ok && k < K; ++k) {
        const bool last = k + 1 == K;
        const uint32_t t_aa = (k & 1) ? kColT1 : kColT0;
        const uint32_t t_a = (k & 1) ? kColT0 : kColT1;  // A_k for k >= 1
        // ---- Q = a I + b A + c A A ----
        if (!(ok = wait_all(&aa_full, aap))) break;
        tc_fence_after();
        {
          float av[32], qv[32];
          tld(k == 0 ? kColT3 : t_a, av);
          tld(t_aa, qv);
          const float ca = a.coef[k][0], cb = a.coef[k][1], cc = a.coef[k][2];
          const float sa = k == 0 ? s2 : 1.f;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            qv[e] = __fmaf_rn(cc, qv[e], cb * (sa * av[e]));
            if (quad == part && e == lane) qv[e] += ca;  // the diagonal (r, r)
          }
          store_split(q_hi, q_lo, box, r, p0, qv);
        }
        handoff(&q_ready);
        if (last && lane == 0) mbar_arrive(&small_done);
        // ---- Q A into the A tiles ----
        if (!last) {
          if (!(ok = wait_all(&p2_full, p2p))) break;
          tc_fence_after();
          float v[32];
          tld(kColT2, v);
          store_split(a_hi, a_lo, box, r, p0, v);
          handoff(&p2_ready);
        }
        // ---- R = Q R into the R tiles ----
        if (!(ok = wait_all(&r_full, rp))) break;
        tc_fence_after();
        {
          float v[32];
          tld(kColT3, v);
          store_split(r_hi, r_lo, box, r, p0, v);
        }
        handoff(&r_ready);
        // ---- the next A = (Q A) Q into the A tiles ----
        if (!last) {
          if (!(ok = wait_all(&an_full, anp))) break;
          tc_fence_after();
          float v[32];
          tld(t_aa, v);
          store_split(a_hi, a_lo, box, r, p0, v);
          handoff(&a_ready);
        }
      }
      if (!ok) continue;
      // ---- final pass: U = R X_0, applied to the weights (or emitted) ----
      ApplyTarget tg = apply_target(a.apply, mat);
      if (a.fuse_prep) tg.skip = !a.apply.emit && a.apply.skip_nonfinite && bad;
      const bool vec = piece_vec(a.apply, tg);
      for (int j = 0; j < nch; ++j) {
        const int ub = (int)(uc % kUBufsG);
        const int64_t c0 = (int64_t)j * kChunkCols + part * 32;  // this warp's 32 columns
        // the weights of this warp's piece load while the chunk's accumulator is
        // awaited (the Q tiles the buffer overlaps were last read by the final Q R)
        piece_load(a.apply, tg, vec, G.m, G.n, quad * 32, c0, lane, wbuf);
        cp_async_commit();
        ok = __all_sync(0xffffffffu, mbar_wait(&u_full[ub], (uc / kUBufsG) & 1u, abort_p, status));
        if (!ok) break;
        tc_fence_after();
        float v[32];
        tld((uint32_t)ub * 128u, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&u_empty[ub]);
        cp_async_wait<0>();
        __syncwarp();
        piece_update(a.apply, tg, vec, lane, v, wbuf);
        __syncwarp();
        piece_store(a.apply, tg, vec, G.m, G.n, quad * 32, c0, lane, wbuf);
        __syncwarp();  // the buffer is refilled for the next chunk
        ++uc;
      }
      cp_async_wait<0>();
    }
    cp_async_wait<0>();  // no copy into shared memory outlives the CTA (after an abort)
  }

  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<1>(tmem, kTmemColsG);
  }
}

}  // namespace

cudaError_t launch_ns_gram(const SmallArgs& a, int num_sms, cudaStream_t s) {
  if (a.n_units <= 0) return cudaSuccess;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(ns_gram_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemG);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int grid = a.n_units < num_sms ? a.n_units : num_sms;
  ns_gram_kernel<<<grid, kThreadsG, kSmemG, s>>>(a);
  return cudaGetLastError();
}

}  // namespace muon

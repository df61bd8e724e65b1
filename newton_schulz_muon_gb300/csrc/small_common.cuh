// Pieces shared by the two Newton-Schulz kernels for wide matrices of at most
// 128 rows (ns_small.cu: the quintic iteration on X; ns_gram.cu: the same
// iteration on the Gram matrix): the 128-byte-swizzled tile layout, bf16
// packing, the weight update applied from the last accumulators in 32 x 32
// pieces, the matrix index of a launch-wide unit, and the momentum computed in a
// matrix's first pass.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "device.cuh"
#include "epilogue.cuh"
#include "kernels.h"
#include "momentum.cuh"

namespace muon {
namespace {

constexpr uint32_t kEpiWarps = 16;
constexpr int kBoxCols = 64;                          // one 128-byte swizzle row of bf16
constexpr int kChunkCols = 2 * kBoxCols;              // columns per ring stage, UPDATE and X' tile
constexpr uint32_t kTile = 128u * 128u;               // one box: 128 rows x 128 bytes = 16 KB
constexpr uint32_t kChunk = 2 * kTile;                // 32 KB
constexpr uint32_t kWarpBuf = 32u * 32u * 4u;         // one warp's 32 x 32 fp32 piece of a chunk
// fused momentum: 32-column quarters of a chunk staged in shared memory, G 128
// rows x 64 bytes, then M 128 rows x 128 bytes, per slot; three quarters in flight
constexpr uint32_t kPrepThreads = kEpiWarps * 32;
constexpr int kPrepCols = 32;
constexpr uint32_t kPrepG = 128u * 64u;                // 8 KB
constexpr uint32_t kPrepSlot = kPrepG + 128u * 128u;   // 24 KB
constexpr int kPrepSlots = 4;
static_assert(kChunkCols == 4 * kPrepCols, "four quarters per chunk");

// Start stagger.  Every CTA of these kernels takes its matrices in the same order
// of phases: X0 streamed in from HBM, iterations that mostly hit the L2, and a
// last pass that streams the weights from and back to HBM.  CTAs that start
// together stay in step, so their HBM-heavy passes coincide and leave HBM idle in
// between.  The CTAs with one matrix fewer than the others (blockIdx.x >=
// stagger_from) start stagger_ns later, which they can spare, so that their
// matrix boundaries fall inside the others' iterations (when every CTA has as
// many matrices, the second half of them waits).  Performance only: no result
// depends on it.  The condition is the same for every thread of a CTA.
__device__ __forceinline__ void start_stagger(const SmallArgs& a) {
  if (a.stagger_ns <= 0 || (int)blockIdx.x < a.stagger_from) return;
  if (threadIdx.x == 0) {
    // bounded by a count as well as by the clock (a few thousand 1 us sleeps at most)
    const unsigned long long t0 = globaltimer_ns();
    for (int i = 0; i < 4096 && globaltimer_ns() - t0 < (unsigned long long)a.stagger_ns; ++i) __nanosleep(1000);
  }
  __syncthreads();
}

// Byte offset of 16-byte piece `piece` (8 bf16) of row r in a 128-byte-swizzled
// tile of 128-byte rows (1024-byte aligned).
__device__ __forceinline__ uint32_t sw128(int r, int piece) {
  return (uint32_t)r * 128u + ((uint32_t)(piece ^ (r & 7)) << 4);
}

__device__ __forceinline__ void unpack8(const uint4& raw, float (&x)[8]) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162*>(&w[h]);
    x[2 * h] = __low2float(p);
    x[2 * h + 1] = __high2float(p);
  }
}

__device__ __forceinline__ uint4 pack8(const float* v) {
  uint4 raw;
  raw.x = pack_bf16x2(v[0], v[1]);
  raw.y = pack_bf16x2(v[2], v[3]);
  raw.z = pack_bf16x2(v[4], v[5]);
  raw.w = pack_bf16x2(v[6], v[7]);
  return raw;
}

// Where the weight update of bucket-local matrix `mat` lands: the matrix's first
// element in the caller's tensor (weights, or the fp32 U' output when emitting),
// the caller's row length, sqrt(max(1, rows/cols)), and whether the matrix is tall
// (U^T lands in W).  Sources: "Muon Optimizer + FSDP", section 背景.
struct ApplyTarget {
  uint8_t* w;
  int64_t ld;
  float sc;
  bool transposed;
  bool skip;
};

__device__ __forceinline__ ApplyTarget apply_target(const ApplyArgs& A, int mat) {
  int lo = 0, hi = A.n_segs - 1;
  while (lo < hi) {  // last run with mat0 <= mat
    const int mid = (lo + hi + 1) >> 1;
    if (A.seg[mid].mat0 <= mat) lo = mid; else hi = mid - 1;
  }
  const ApplySeg& S = A.seg[lo];
  const int64_t esize = (A.emit || A.param_dtype == 0) ? 4 : 2;
  ApplyTarget t;
  t.w = reinterpret_cast<uint8_t*>(S.w) + (int64_t)(mat - S.mat0) * S.stride * esize;
  t.ld = S.cols;
  t.sc = S.shape_scale;
  t.transposed = S.transposed != 0;
  t.skip = !A.emit && A.skip_nonfinite && A.flags[mat];
  return t;
}

// One warp's 32 x 32 piece of a chunk: wide-form rows r0 .. r0+31 and columns
// c0 .. c0+31, held in a shared buffer as element (row i, column e) at word
// i * 32 + (e ^ i), so that both a row of the piece (a lane per column) and a
// column (a lane per row) are read without bank conflicts.
__device__ __forceinline__ int piece_word(int row, int col) { return row * 32 + (col ^ row); }

// Offset in the caller's tensor of the element lane `lane` moves in step i, its
// word in the piece buffer, and whether it exists.  A wide matrix is moved row
// by row, a tall one column by column (a row of W = U^T): lanes always run along
// W's contiguous dimension.
__device__ __forceinline__ bool piece_elem(const ApplyTarget& t, int m, int n, int r0, int64_t c0, int i, int lane,
                                           int64_t& off, int& word) {
  int r;
  int64_t c;
  if (!t.transposed) {
    r = r0 + i;
    c = c0 + lane;
    off = (int64_t)r * t.ld + c;
    word = piece_word(i, lane);
  } else {
    r = r0 + lane;
    c = c0 + i;
    off = c * t.ld + r;
    word = piece_word(lane, i);
  }
  return r < m && c < n;
}

// 16-byte path: a wide matrix with fp32 weights (or the fp32 U' output) whose
// rows are whole 16-byte units (row length, which is n, a multiple of 4, and a
// 16-byte aligned first element).  Step q moves rows 4q .. 4q+3 of the piece,
// eight lanes per row, four columns per lane; in the buffer the 16-byte unit
// (col / 4) of row `row` sits at unit position (col / 4) ^ (row % 8).
__device__ __forceinline__ bool piece_vec(const ApplyArgs& A, const ApplyTarget& t) {
  return !t.transposed && (A.emit || A.param_dtype == 0) && (t.ld & 3) == 0 &&
         (reinterpret_cast<uintptr_t>(t.w) & 15u) == 0;
}

__device__ __forceinline__ int piece_word_vec(int row, int col) {
  return row * 32 + ((((col >> 2) ^ row) & 7) << 2) + (col & 3);
}

// Starts loading the weights of one piece into `buf` (fp32 weights: cp.async;
// bf16 weights: loaded and widened here).  Nothing when emitting or skipping.
__device__ __forceinline__ void piece_load(const ApplyArgs& A, const ApplyTarget& t, bool vec, int m, int n, int r0,
                                           int64_t c0, int lane, float* buf) {
  if (A.emit || t.skip) return;
  if (vec) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = 4 * q + (lane >> 3);
      const int g = lane & 7;
      const int64_t c = c0 + 4 * g;
      if (r0 + i < m && c < n)
        cp_async_16(buf + piece_word_vec(i, 4 * g), reinterpret_cast<const float*>(t.w) + (int64_t)(r0 + i) * t.ld + c);
    }
    return;
  }
  if (A.param_dtype == 0) {
#pragma unroll 8
    for (int i = 0; i < 32; ++i) {
      int64_t off;
      int word;
      if (piece_elem(t, m, n, r0, c0, i, lane, off, word))
        cp_async_4(buf + word, reinterpret_cast<const float*>(t.w) + off);
    }
  } else {
    float v[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      int64_t off;
      int word;
      v[i] = piece_elem(t, m, n, r0, c0, i, lane, off, word)
                 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(t.w)[off]) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      int64_t off;
      int word;
      piece_elem(t, m, n, r0, c0, i, lane, off, word);
      buf[word] = v[i];
    }
  }
}

// Lane = row of the piece, u[e] = U at column e: W <- W - lr (s U + wd W) (or
// U' = s U) in the buffer.
__device__ __forceinline__ float apply_elem(const ApplyArgs& A, const ApplyTarget& t, float u, float w) {
  return A.emit ? t.sc * u : __fmaf_rn(-A.lr, __fmaf_rn(t.sc, u, __fmul_rn(A.wd, w)), w);
}

__device__ __forceinline__ void piece_update(const ApplyArgs& A, const ApplyTarget& t, bool vec, int lane,
                                             const float* u, float* buf) {
  if (t.skip) return;
  if (vec) {
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      float4* p = reinterpret_cast<float4*>(buf + piece_word_vec(lane, 4 * g));
      float4 w = *p;
      w.x = apply_elem(A, t, u[4 * g], w.x);
      w.y = apply_elem(A, t, u[4 * g + 1], w.y);
      w.z = apply_elem(A, t, u[4 * g + 2], w.z);
      w.w = apply_elem(A, t, u[4 * g + 3], w.w);
      *p = w;
    }
    return;
  }
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    float* p = buf + piece_word(lane, e);
    *p = apply_elem(A, t, u[e], *p);
  }
}

// Writes the piece back to the caller's tensor.
__device__ __forceinline__ void piece_store(const ApplyArgs& A, const ApplyTarget& t, bool vec, int m, int n, int r0,
                                            int64_t c0, int lane, const float* buf) {
  if (t.skip) return;
  if (vec) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int i = 4 * q + (lane >> 3);
      const int g = lane & 7;
      const int64_t c = c0 + 4 * g;
      if (r0 + i < m && c < n)
        *reinterpret_cast<float4*>(reinterpret_cast<float*>(t.w) + (int64_t)(r0 + i) * t.ld + c) =
            *reinterpret_cast<const float4*>(buf + piece_word_vec(i, 4 * g));
    }
    return;
  }
  const bool f32 = A.emit || A.param_dtype == 0;
#pragma unroll 8
  for (int i = 0; i < 32; ++i) {
    int64_t off;
    int word;
    if (piece_elem(t, m, n, r0, c0, i, lane, off, word)) {
      if (f32) reinterpret_cast<float*>(t.w)[off] = buf[word];
      else reinterpret_cast<__nv_bfloat16*>(t.w)[off] = __float2bfloat16_rn(buf[word]);
    }
  }
}

struct UnitRef {
  int g, b;
};

// The momentum run holding bucket-local matrix `mat`.
__device__ __forceinline__ const SmallPrepSeg& prep_seg(const SmallArgs& a, int mat) {
  int lo = 0, hi = a.n_psegs - 1;
  while (lo < hi) {  // last run with mat0 <= mat
    const int mid = (lo + hi + 1) >> 1;
    if (a.pseg[mid].mat0 <= mat) lo = mid; else hi = mid - 1;
  }
  return a.pseg[lo];
}

// Debug build: an MMA operand tile of `bytes` at shared address `addr` lies inside
// the CTA's dynamic shared memory [lo, hi).
__device__ __forceinline__ bool smem_tile_ok(uint32_t addr, uint32_t bytes, uint32_t lo, uint32_t hi,
                                             unsigned* status, volatile int* abort) {
  return MUON_GUARD(addr >= lo && addr + bytes <= hi && (addr & 1023u) == 0, status, abort);
}

// Staging slot q % 4 of the fused momentum: slots 0 and 1 from slots01, 2 and 3
// from slots23 (each pair 2 * kPrepSlot contiguous bytes).
__device__ __forceinline__ uint8_t* prep_slot(uint8_t* slots01, uint8_t* slots23, int q) {
  const int sl = q & (kPrepSlots - 1);
  return (sl < 2 ? slots01 : slots23) + (size_t)(sl & 1) * kPrepSlot;
}

// The first pass over matrix `mat` (fuse_prep), by each epilogue warp on its own
// eight rows (warp w: rows 8 w .. 8 w + 7), with no barrier across warps.  Per
// 32-column quarter q of each 128-column chunk the warp copies its rows of G
// (bf16) and M (fp32) into staging slot q % 4 with cp.async, three quarters ahead;
// then each lane takes 8 consecutive elements of one row:
//   M_new = mu M + w G (within 1 ulp), V = mu M_new + w G (Nesterov) or M_new,
// stores M_new in place and X0 = bf16(V) in the workspace, writes bf16(V) into
// the chunk's ring stage (128-byte swizzle, the layout the TMA loads give; rows
// >= m and columns >= n zero) and adds V^2 to its sum.  Each warp arrives on the
// stage's pfull barrier (count 16) when its rows of a chunk are written, and on
// prep_done (count 16) after its last chunk, once X0 is in the workspace.  The
// warp's sum of V^2 is in norm_red[w] before its last pfull arrival, so the Gram
// of iteration 0 being complete implies every partial is there.  `pos` is the
// ring position of the matrix's first chunk, advanced past the chunks filled
// here.  Returns false when a wait was abandoned.
// Staging slots: prep_slot(slots01, slots23, q).  Layout per slot: G row r at r * 64 bytes (16-byte unit u at u * 16); M
// row r at kPrepG + r * 128 bytes with its 16-byte unit u at (u ^ (r & 1)) * 16,
// so that the eight lanes of a shared-memory phase (two rows) hit distinct banks.
template <int kStages>
__device__ __forceinline__ bool prep_matrix(const SmallArgs& a, const SmallGroup& G, int b, int mat,
                                            uint8_t* slots01, uint8_t* slots23, uint8_t* ring, uint64_t* pfull_bar,
                                            uint64_t* empty_bar,
                                            uint64_t* prep_done, float* norm_red, uint32_t& pos,
                                            volatile int* abort_p, unsigned* status) {
  const int et = (int)threadIdx.x - 64;  // 0 .. kPrepThreads - 1
  const int wp = et >> 5, lane = threadIdx.x & 31;
  const SmallPrepSeg& P = prep_seg(a, mat);
  const int64_t moff = (int64_t)(mat - P.mat0) * P.stride;
  const __nv_bfloat16* gmat = reinterpret_cast<const __nv_bfloat16*>(P.g) + moff;
  float* mmat = P.m + moff;
  __nv_bfloat16* xmat = reinterpret_cast<__nv_bfloat16*>(G.x) + (int64_t)b * G.mstride;
  const int m = G.m, n = G.n;
  const int64_t ld = G.ld;
  const int q_end = 4 * ((n + kChunkCols - 1) / kChunkCols);
  const float mu = a.mu, omu = a.omu;
  auto issue = [&](int q) {
    if (q < q_end) {
      uint8_t* sg = prep_slot(slots01, slots23, q);
      uint8_t* sm = sg + kPrepG;
      const int c0 = q * kPrepCols;
      {
        const int row = 8 * wp + (lane >> 2), u = lane & 3, c = c0 + 8 * u;
        if (row < m && c < n) cp_async_16(sg + row * 64 + u * 16, gmat + (int64_t)row * n + c);
      }
#pragma unroll
      for (int it = 0; it < 2; ++it) {
        const int i = it * 32 + lane;
        const int row = 8 * wp + (i >> 3), u = i & 7, c = c0 + 4 * u;
        if (row < m && c < n) cp_async_16(sm + row * 128 + ((u ^ (row & 1)) << 4), mmat + (int64_t)row * n + c);
      }
    }
    cp_async_commit();  // possibly empty: every lane counts the same groups
  };
  issue(0);
  issue(1);
  issue(2);
  const int row = 8 * wp + (lane >> 2), cg = lane & 3;
  float sumsq = 0.f;
  for (int q = 0; q < q_end; ++q) {
    cp_async_wait<2>();  // this lane's copies of quarter q have landed
    const uint32_t stage = pos % (uint32_t)kStages, lap = (pos / (uint32_t)kStages) & 1u;
    if ((q & 3) == 0) {
      // the chunk's ring stage has been read by the MMAs of its previous use
      bool got = true;
      if (lane == 0) got = mbar_wait(&empty_bar[stage], lap ^ 1u, abort_p, status);
      if (!__shfl_sync(0xffffffffu, got, 0)) {
        cp_async_wait<0>();
        return false;
      }
    }
    __syncwarp();  // the warp's copies of q are visible to all its lanes; slot (q + 3) % 4 is free
    issue(q + 3);
    const uint8_t* sg = prep_slot(slots01, slots23, q);
    const uint8_t* sm = sg + kPrepG;
    const int c = q * kPrepCols + 8 * cg;
    float v[8];
    if (row < m && c < n) {
      float g[8];
      unpack8(*reinterpret_cast<const uint4*>(sg + row * 64 + cg * 16), g);
      const float4 m0 = *reinterpret_cast<const float4*>(sm + row * 128 + (((2 * cg) ^ (row & 1)) << 4));
      const float4 m1 = *reinterpret_cast<const float4*>(sm + row * 128 + (((2 * cg + 1) ^ (row & 1)) << 4));
      const float mo[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
      float mn[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        mn[e] = dot2_accurate(mu, mo[e], omu, g[e]);
        v[e] = nesterov_input(a.nesterov, mu, mn[e], omu, g[e]);
        sumsq = __fmaf_rn(v[e], v[e], sumsq);
      }
      float* mp = mmat + (int64_t)row * n + c;
      __stcs(reinterpret_cast<float4*>(mp), make_float4(mn[0], mn[1], mn[2], mn[3]));
      __stcs(reinterpret_cast<float4*>(mp + 4), make_float4(mn[4], mn[5], mn[6], mn[7]));
      *reinterpret_cast<uint4*>(xmat + (int64_t)row * ld + c) = pack8(v);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] = 0.f;
    }
    uint8_t* st = ring + (size_t)stage * kChunk + (size_t)((q >> 1) & 1) * kTile;
    *reinterpret_cast<uint4*>(st + sw128(row, (q & 1) * 4 + cg)) = pack8(v);
    if ((q & 3) == 3) {
      const bool final_chunk = q + 1 == q_end;
      if (final_chunk) {
        const float w = warp_sum(sumsq);
        if (lane == 0) norm_red[wp] = w;
      }
      fence_proxy_async_shared();  // the stage is read by the tensor core
      fence_proxy_async_global();  // X0 is read by the producer's TMA loads
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&pfull_bar[stage]);
        if (final_chunk) mbar_arrive(prep_done);
      }
      ++pos;
    }
  }
  cp_async_wait<0>();
  return true;
}

// s = 1 / (||V||_F + eps) of the matrix whose first pass just completed, from the
// 16 warp partials in a fixed order (fp64), and whether the norm was finite; one
// thread records them and counts a non-finite matrix.
__device__ __forceinline__ float prep_scale(const SmallArgs& a, int mat, const float* norm_red, bool& bad) {
  double tot = 0.0;
#pragma unroll
  for (int i = 0; i < (int)kEpiWarps; ++i) tot += (double)norm_red[i];
  const bool finite = isfinite(tot);
  const float s = finite ? (float)(1.0 / (sqrt(tot) + (double)a.eps)) : 0.f;
  bad = !finite;
  if (threadIdx.x == 64) {
    a.scale[mat] = s;
    a.flags[mat] = finite ? 0 : 1;
    const SmallPrepSeg& P = prep_seg(a, mat);
    P.norm_out[mat - P.mat0] = (float)sqrt(tot);
    if (!finite) atomicAdd(&a.status->nonfinite, 1u);
  }
  return s;
}

__device__ __forceinline__ UnitRef decode_unit(const SmallArgs& a, int u) {
  int g = 0;
  for (int i = 1; i < a.n_groups; ++i)
    if (a.g[i].unit0 <= u) g = i;
  return {g, u - a.g[g].unit0};
}

// Lane 0 tests the barrier phase (non-blocking); the warp gets its answer.
__device__ __forceinline__ bool poll(uint64_t* bar, uint32_t parity) {
  bool ready = false;
  if ((threadIdx.x & 31) == 0) ready = mbar_test_wait(bar, parity);
  return __shfl_sync(0xffffffffu, ready, 0);
}

// Ring position after `n` more stages.
template <int kStages>
__device__ __forceinline__ void ring_advance(int& stage, uint32_t& phase, int n) {
  for (int i = 0; i < n; ++i)
    if (++stage == kStages) { stage = 0; phase ^= 1u; }
}


}  // namespace
}  // namespace muon

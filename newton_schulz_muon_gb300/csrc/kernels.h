// Kernel argument blocks and launchers shared by the host runtime and the
// kernels of libmuon.so.  Arguments travel by value as kernel parameters
// (tensor maps as __grid_constant__), so nothing here is read from the host.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

struct muon_plan_s;

namespace muon {

constexpr int kMaxSegs = 64;     // runs of consecutive matrices of one tensor per bucket
constexpr int kMaxGroups = 4;    // same-shape groups per bucket (one grouped GEMM launch)
constexpr int kPrepTile = 64;    // momentum / apply tiles are 64 x 64 elements

// Workspace header (offset 0): device status word and non-finite counter.
struct DeviceStatus {
  unsigned flags;       // kStatusWaitTimeout, kStatusGuard
  unsigned nonfinite;   // matrices with a non-finite norm since the last muon_sync
};
constexpr unsigned kStatusWaitTimeout = 1u;  // a kernel's bounded wait ran out
constexpr unsigned kStatusGuard = 2u;        // a debug-build range check failed; the access was skipped

// ---------------------------------------------------------------------------
// momentum + prep (one run of `count` matrices of one tensor)
// ---------------------------------------------------------------------------
struct PrepSeg {
  const void* g;         // gradient of the run's first matrix
  float* m;              // fp32 momentum of the run's first matrix (updated in place)
  void* x_hi;            // workspace X0 of the run's first matrix (bf16, or tf32-hi fp32)
  float* x_lo;           // tf32-lo part (3xTF32 mode), else null
  int64_t rows, cols;    // logical shape
  int64_t stride;        // elements between consecutive matrices in g and m
  int64_t x_ld;          // leading dimension of X (wide form m x n)
  int64_t x_mstride;     // elements between consecutive matrices in X
  int64_t block0;        // first tile index of the run in the bucket's tile space
  void* xt_hi;           // 3xTF32: X0^T (n x m) of the run's first matrix, else null
  float* xt_lo;
  int64_t xt_ld;         // leading dimension of X^T
  int64_t xt_mstride;    // elements between consecutive matrices in X^T
  int32_t count;         // matrices in the run
  int32_t transposed;    // 1 when rows > cols: X = V^T
  int32_t tiles_c;       // 64-wide tiles along cols
  int32_t tiles_per_mat; // tiles per matrix
  int32_t mat0;          // bucket-local index of the run's first matrix
  int32_t pad_;
  float* norm_out;       // ||V||_F of the run's first matrix in the plan's norm record
};

struct PrepArgs {
  PrepSeg seg[kMaxSegs];
  int32_t n_segs;
  int32_t n_mats;        // matrices in the bucket
  int64_t total_tiles;
  float mu, omu;         // momentum and its complement (1 for the SGD form)
  int32_t nesterov;
  int32_t grad_dtype;    // 0 fp32, 1 bf16
  int32_t tf32;          // 1: write X0 as tf32 hi/lo fp32 pair
  float eps;
  float* partials;       // one fp32 sum of squares per tile
  float* scale;          // per matrix: 1 / (||V||_F + eps)
  int32_t* flags;        // per matrix: 1 if the norm was not finite
  DeviceStatus* status;
};

// ---------------------------------------------------------------------------
// apply / emit (one run of matrices)
// ---------------------------------------------------------------------------
struct ApplySeg {
  void* w;               // weights (apply) or fp32 U' output (emit) of the first matrix
  const void* u_hi;      // final X of the first matrix (bf16 or tf32-hi fp32)
  const float* u_lo;     // tf32-lo part, or null
  int64_t rows, cols, stride;
  int64_t u_ld, u_mstride;
  int64_t block0;
  int32_t count, transposed, tiles_c, tiles_per_mat, mat0;
  float shape_scale;     // sqrt(max(1, rows/cols))
};

struct ApplyArgs {
  ApplySeg seg[kMaxSegs];
  int32_t n_segs;
  int64_t total_tiles;
  float lr, wd;
  int32_t param_dtype;   // 0 fp32, 1 bf16
  int32_t tf32;
  int32_t emit;          // 1: write U' = shape_scale * U (fp32) instead of updating W
  int32_t skip_nonfinite;
  int32_t unnormalized;  // 1 when no NS iteration ran: U = scale * X0
  const float* scale;
  const int32_t* flags;
};

// ---------------------------------------------------------------------------
// Newton-Schulz GEMMs (tcgen05)
// ---------------------------------------------------------------------------
enum GemmMode : int32_t { kGram = 0, kPoly = 1, kUpdate = 2 };

struct GemmGroup {
  CUtensorMap map_a;     // operand A (K-major, box {64 (k), 128 rows})
  CUtensorMap map_b;     // operand B (K-major box {64, 128} x2, or bf16 UPDATE: MN-major box {64, 64} x4)
  CUtensorMap map_a_lo;  // 3xTF32: low parts (unused in bf16 mode)
  CUtensorMap map_b_lo;
  CUtensorMap map_c;     // bf16 epilogue: output C, box {32, 32}, 64-byte swizzle (TMA stores)
  CUtensorMap map_d;     // bf16 epilogue: POLY's addend A, same box (TMA loads)
  void* c_hi;            // output (bf16 or tf32-hi fp32)
  float* c_lo;           // output tf32-lo part
  const void* d_hi;      // epilogue addend (POLY: A; 3xTF32 UPDATE: X)
  const float* d_lo;
  int64_t c_ld, c_mstride;   // elements
  void* ct_hi;               // 3xTF32 UPDATE: also write the output transposed (X'^T), else null
  float* ct_lo;
  int64_t ct_ld, ct_mstride;
  int32_t M, N, K;           // output rows, cols, reduction length
  int32_t count;             // matrices
  int32_t tiles_m, tiles_n;  // row blocks (kBM * cluster rows) and 256-column blocks of one matrix
  int32_t tiles_per_mat;     // tiles computed per matrix (upper triangle for GRAM/POLY)
  int32_t tile0;             // first launch-wide tile index of this group
  int32_t mat_base;          // bucket-local index of matrix 0 (for the scale array)
  int32_t pad_[3];
};

struct GemmArgs {
  GemmGroup g[kMaxGroups];
  int32_t n_groups;
  int32_t total_tiles;
  int32_t mode;
  int32_t use_scale;      // first iteration: fold 1/(||V||+eps) into the epilogue
  float alpha, beta;      // GRAM: 1, -; POLY: c, b; UPDATE: 1, a (3xTF32) or - (bf16)
  float diag;             // added to the diagonal of the output: bf16 POLY a (B' = a I + B), else 0
  const float* scale;     // per bucket-local matrix
  DeviceStatus* status;
  // tile schedule: cluster c runs tiles sched_units[sched_off[c] .. sched_off[c+1])
  const int32_t* sched_off;
  const int32_t* sched_units;
  int32_t n_clusters;
  // last UPDATE of a step: apply the weight update (or emit U') from the
  // epilogue instead of storing X; `apply` describes the weights per matrix run
  int32_t fuse_apply;
  ApplyArgs apply;
};

// ---------------------------------------------------------------------------
// Newton-Schulz for wide matrices of at most 128 rows (one CTA per matrix, every
// iteration in one launch, bf16)
// ---------------------------------------------------------------------------
struct SmallGroup {
  CUtensorMap map_x;     // X (in place across iterations): box {64 columns, 128 rows}
  void* x;               // bf16 X of matrix 0 of the group in the workspace
  int64_t ld;            // leading dimension of X (elements)
  int64_t mstride;       // elements between consecutive matrices
  int32_t m, n;          // wide form: m <= 128 rows, n columns
  int32_t count;         // matrices
  int32_t unit0;         // first launch-wide matrix index of this group
  int32_t mat_base;      // bucket-local index of matrix 0 (scale, flags, apply)
  int32_t pad_[3];
};

// One run of `count` matrices of one tensor, for the momentum computed inside the
// small-matrix kernel (bf16 gradients, wide matrices, rows of whole 16-byte units).
struct SmallPrepSeg {
  const void* g;         // bf16 gradient of the run's first matrix
  float* m;              // fp32 momentum of the run's first matrix (updated in place)
  int64_t stride;        // elements between consecutive matrices in g and m
  int32_t mat0;          // bucket-local index of the run's first matrix
  int32_t pad_;
  float* norm_out;       // ||V||_F of the run's first matrix in the plan's norm record
};

struct SmallArgs {
  SmallGroup g[kMaxGroups];
  int32_t n_groups;
  int32_t n_units;       // matrices in the launch
  int32_t ns_steps;      // quintic iterations (1 .. MUON_MAX_NS_STEPS)
  float coef[16][3];     // iteration k: (a, b, c) of X' = a X + (b A + c A A) X, A = X X^T
  float* scale;          // per bucket-local matrix: 1 / (||V||_F + eps), folded into iteration 0
                         // (written by the kernel when fuse_prep = 1)
  DeviceStatus* status;
  ApplyArgs apply;       // the last iteration applies the weight update (or emits U')
  // fuse_prep = 1: the kernel's first pass over each matrix computes the momentum
  // (M updated in place), the Newton-Schulz input V, its Frobenius norm and X0 =
  // bf16(V) itself, instead of reading X0 written by the momentum kernel
  int32_t fuse_prep;
  int32_t nesterov;
  float mu, omu;         // momentum and its complement (1 for the SGD form)
  float eps;
  int32_t n_psegs;
  int32_t* flags;        // per bucket-local matrix: 1 if the norm was not finite (fuse_prep)
  SmallPrepSeg pseg[kMaxSegs];
  // start stagger (performance only): CTAs with blockIdx.x >= stagger_from wait
  // stagger_ns after their set-up before taking their first matrix
  int32_t stagger_from;
  int64_t stagger_ns;
};

// GEMM tile shape (bf16): 128 x 256 outputs per CTA, 64-deep k blocks.
constexpr int kBM = 128;
constexpr int kBN = 256;

// launchers (return the launch's cudaError_t)
cudaError_t launch_prep(const PrepArgs& a, cudaStream_t s);
cudaError_t launch_norm(const PrepArgs& a, cudaStream_t s);
cudaError_t launch_apply(const ApplyArgs& a, cudaStream_t s);
// One CTA waiting on a barrier nothing arrives on, for limit_ns, through the
// kernels' bounded wait: records the timeout in *status (the failure-path self-test).
cudaError_t launch_wait_selftest(DeviceStatus* status, unsigned long long limit_ns, cudaStream_t s);
// cluster: 1, or 2 (pairs of vertically adjacent tiles share the B operand);
// GemmGroup::tiles_m counts row blocks of kBM * cluster rows.
cudaError_t launch_gemm(const GemmArgs& a, int num_sms, bool tf32, int cluster, cudaStream_t s);
// Clusters of the GEMM kernel that can be resident at once on this device
// (a.n_clusters must not exceed it).
int gemm_max_clusters(bool tf32, int cluster, int num_sms);
size_t gemm_smem_bytes(bool tf32);
// All iterations of a bucket whose groups all have m <= 128 (bf16 only).
cudaError_t launch_ns_small(const SmallArgs& a, int num_sms, cudaStream_t s);
// The same by the gram method (the iteration on X X^T, X read twice).
cudaError_t launch_ns_gram(const SmallArgs& a, int num_sms, cudaStream_t s);
constexpr int kSmallMaxRows = 128;

// Records `msg` as the calling thread's muon_last_error text and returns `s`.
int32_t set_error(int32_t s, const char* msg);

// The no-allocation path (noalloc.cu).  bind_shared_scratch binds a plan to the
// library's static scratch like muon_plan_bind_workspace, but copies the tile
// schedules on `stream` (ordered after the work already enqueued there) and
// leaves the device status word as it is; plan_id is a process-unique plan
// number; plan_workspace the device memory the plan is bound to (or null).
int32_t bind_shared_scratch(muon_plan_s* p, void* dev_ptr, size_t bytes, cudaStream_t stream);
uint64_t plan_id(const muon_plan_s* p);
const void* plan_workspace(const muon_plan_s* p);

}  // namespace muon

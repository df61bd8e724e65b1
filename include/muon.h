/*
 * muon.h -- C ABI of libmuon.so, the GB300 (sm_103a) Muon optimizer step.
 *
 * One Muon step of a set of 2-D logical matrices: fp32 momentum update with
 * optional Nesterov look-ahead, Frobenius normalisation, five (ns_steps)
 * Newton-Schulz quintic iterations on the full matrix, and the weight update
 *     W <- W - lr * (sqrt(max(1, rows/cols)) * U + wd * W).
 * Sources: "Muon Optimizer + FSDP" (section 背景: M_t = momentum_update(grad),
 * U_t = NewtonSchulz(M_t), W_t = W_t - lr U_t; section 分块通信: micro-buckets of
 * whole matrices, fused [Q;K;V] and [E,out,in] tensors split into logical
 * matrices; section 内存控制方案 items 1-4: bucket cap, one persistent
 * preallocated workspace, bounded in-flight buckets, bf16 buffers with fp32
 * normalisation scalars); DeepSpeed issue "[RFC] Enable Correct and
 * High-Performance Muon Optimizer under ZeRO CPU Offload" (section 2: 5-6
 * Newton-Schulz iterations on full 2-D matrices; section 4.A: shapes and head
 * dimensions carried with the tensors; section 4.D: per-head Muon on
 * interleaved QKV); DeepSpeed PR "[Muon] CPU offload: pin the momentum and
 * overlap the host writeback" (section Changes: pinned momentum, writeback of
 * batch i on a side stream overlapping batch i+1, drained before the host
 * reads).
 *
 * Conventions for every entry point:
 *  - No C++ exception and no CUDA error escapes: each call returns a
 *    muon_status.  0 is success, < 0 an error (nothing was enqueued unless the
 *    text says so), > 0 a warning.
 *  - The caller owns every tensor and the workspace memory; the plan owns only
 *    host metadata, CUDA events and its private streams.  No entry point
 *    allocates device memory.
 *  - "stream" arguments are cudaStream_t values passed as void* (NULL = the
 *    legacy default stream).  Device work is enqueued asynchronously and in
 *    stream order; device-side faults of that work (a bounded wait that ran
 *    out, a non-finite matrix) are reported by muon_sync.
 *  - Matrices are row-major, contiguous within a matrix.  Device pointers
 *    must be 16-byte aligned.
 */
#ifndef MUON_H
#define MUON_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t muon_status;

#define MUON_OK 0
#define MUON_WARN_NONFINITE 1   /* some matrix had a non-finite norm; see muon_sync */
#define MUON_ERR_INVALID (-1)   /* bad argument: null, size, dtype, alignment, count */
#define MUON_ERR_NOT_PINNED (-2) /* offload host buffer is not page-locked */
#define MUON_ERR_NO_WORKSPACE (-3) /* no workspace bound, or it is too small */
#define MUON_ERR_CUDA (-4)      /* a CUDA runtime/driver call failed */
#define MUON_ERR_TIMEOUT (-5)   /* a bounded host wait ran out */
#define MUON_ERR_UNSUPPORTED (-6) /* option not supported by the library or the device */
#define MUON_ERR_DEVICE (-7)    /* a kernel's bounded wait ran out (device status word) */

/* element types */
#define MUON_DTYPE_F32 0
#define MUON_DTYPE_BF16 1

/* Newton-Schulz arithmetic */
#define MUON_NS_BF16 0    /* bf16 operands, fp32 accumulation (tcgen05 kind::f16) */
#define MUON_NS_TF32X3 1  /* fp32 storage, 3xTF32 split products (tcgen05 kind::tf32) */

/* Newton-Schulz kernels */
#define MUON_NS_KERNEL_AUTO 0 /* buckets whose matrices all have m <= 128 (wide form) run every
                                 iteration in one kernel with A and B on chip (bf16 only);
                                 other buckets run three grouped GEMM launches per iteration */
#define MUON_NS_KERNEL_GEMM 1 /* always the grouped GEMM launches */

/* Newton-Schulz method (DeepSpeed PR "[Muon] CPU offload: pin the momentum and
 * overlap the host writeback", section Tests, names a "gram" and a "standard"
 * method; the pages give no more):
 *   STANDARD  X_{k+1} = a X_k + (b A_k + c A_k A_k) X_k with A_k = X_k X_k^T;
 *   GRAM      the same iteration rewritten on the Gram matrix: A_{k+1} = Q_k A_k Q_k,
 *             Q_k = a I + b A_k + c A_k A_k, and U = (Q_{K-1} ... Q_0) X_0, so X is
 *             read twice whatever the iteration count.  Equal in exact arithmetic;
 *             in this library the m x m products are split into bf16 high and low
 *             parts (about 16 bits per operand), so GRAM is also the more accurate.
 *             Only buckets run by the small-matrix kernel (every matrix with
 *             min(rows, cols) <= 128, bf16 arithmetic, ns_kernel AUTO). */
#define MUON_NS_METHOD_STANDARD 0
#define MUON_NS_METHOD_GRAM 1

/* Newton-Schulz iterations per step: ns_steps in [0, MUON_MAX_NS_STEPS] */
#define MUON_MAX_NS_STEPS 16

/* momentum form (the pages name momentum_update without a formula) */
#define MUON_MOMENTUM_EMA 0 /* M <- mu M + (1-mu) G;  Nesterov V = (1-mu) G + mu M */
#define MUON_MOMENTUM_SGD 1 /* M <- mu M + G;         Nesterov V = G + mu M        */

typedef struct muon_plan_s muon_plan_t;

/* One tensor holding `count` logical rows x cols matrices, `stride_elems`
 * elements apart (0 means rows*cols: contiguous [count, rows, cols]).
 * An expert tensor [E, out, in] is {out, in, E, 0}; a fused projection of H
 * heads of D rows is {D, in, H, 0}; a plain matrix is {rows, cols, 1, 0}. */
typedef struct {
  int64_t rows;
  int64_t cols;
  int64_t count;
  int64_t stride_elems;
} muon_shape;

typedef struct {
  float ns_a, ns_b, ns_c;   /* quintic coefficients: X' = a X + (b A + c A A) X */
  float eps;                /* X0 = V / (||V||_F + eps) */
  int32_t ns_precision;     /* MUON_NS_BF16 or MUON_NS_TF32X3 */
  int32_t momentum_form;    /* MUON_MOMENTUM_EMA or MUON_MOMENTUM_SGD */
  int32_t grad_dtype;       /* MUON_DTYPE_BF16 or MUON_DTYPE_F32 */
  int32_t param_dtype;      /* MUON_DTYPE_F32 or MUON_DTYPE_BF16 (weights) */
  int32_t max_inflight;     /* offload: buckets whose writeback may be in flight (1 or 2) */
  int32_t skip_nonfinite;   /* 1: a matrix whose Newton-Schulz input has a non-finite norm
                               leaves its weights untouched (its momentum keeps the
                               non-finite values; muon_sync reports the count) */
  int32_t timing;           /* 1: record per-bucket CUDA events for muon_get_stats */
  int32_t offload;          /* 1: reserve host-link staging slots for muon_offload_step */
  int32_t ns_kernel;        /* MUON_NS_KERNEL_AUTO or MUON_NS_KERNEL_GEMM */
  int32_t offload_zero_copy; /* with offload = 1: 1 makes muon_offload_step's kernels read G and
                                M and write M and U' in the pinned host buffers themselves
                                (mapped into the device's address space; no staging slots,
                                no copy engines, everything on the compute stream); 0 stages
                                each bucket through device slots with copy-engine copies */
  int32_t ns_momentum_fused; /* 1: buckets run by the small-matrix kernel (bf16 gradients, wide
                                matrices, n and matrix strides multiples of 8) compute their
                                momentum, norm and X0 in that kernel's first pass; 0: the
                                momentum kernel runs first */
  int32_t ns_method;         /* MUON_NS_METHOD_STANDARD or MUON_NS_METHOD_GRAM */
  int32_t reserved[2];
} muon_config;

/* Fills *cfg with (3.4445, -4.7750, 2.0315), eps 1e-7, bf16 NS, EMA momentum,
 * bf16 gradients, fp32 weights, max_inflight 1, skip_nonfinite 1, timing 0,
 * offload 0, ns_kernel MUON_NS_KERNEL_AUTO, ns_momentum_fused 0,
 * ns_method MUON_NS_METHOD_STANDARD. */
void muon_config_default(muon_config* cfg);

/* Defines: "Muon Optimizer + FSDP", section 分块通信 (chunked communication:
 * same-shape matrices bucketed together, fused [Q;K;V] and [E,out,in] tensors
 * split into logical matrices first) and section 推荐的分块执行伪代码 (recommended
 * chunked-execution pseudocode: plan_micro_buckets(bucket, cap_bytes, cost_fn));
 * section 内存控制方案 items 1 (a byte cap per micro-bucket) and 6 (same-shape
 * expert buckets across layers); DeepSpeed issue "[RFC] ... ZeRO CPU Offload",
 * section 4.A (shapes and head dimensions carried into the optimizer).
 * Builds the host plan: orients each logical matrix (wide form m x n, m <= n,
 * transposed when rows > cols), groups matrices by (group label, m, n), and
 * packs whole matrices, in order, into micro-buckets whose wide-form bf16 bytes
 * (m*n*2 summed) stay <= bucket_cap_bytes.  A matrix larger than the cap gets a
 * bucket of its own.  bucket_cap_bytes <= 0 puts everything in one bucket.
 *   shapes[n_shapes]: tensor descriptions (copied).
 *   groups: NULL (group by wide shape only) or n_shapes labels; matrices with
 *           different labels never share a bucket.
 *   cfg:    NULL for muon_config_default.
 *   out:    receives the plan; free it with muon_plan_destroy.
 * Pure host work: needs no GPU.  Errors: MUON_ERR_INVALID; MUON_ERR_UNSUPPORTED when
 * cfg->ns_method is GRAM and a bucket is not run by the small-matrix kernel. */
muon_status muon_plan(const muon_shape* shapes, int32_t n_shapes, const int32_t* groups,
                      int64_t bucket_cap_bytes, const muon_config* cfg, muon_plan_t** out);

/* Defines: "Muon Optimizer + FSDP", section 内存控制方案 item 2 (one persistent
 * preallocated workspace reused by every bucket; MuonWorkspace in section
 * 推荐的分块执行伪代码).
 * Device workspace the plan needs (bytes, 256-byte aligned use), including the
 * offload staging slots.  Pure host work. */
muon_status muon_plan_workspace_bytes(const muon_plan_t* plan, size_t* device_bytes);

/* Defines: as muon_plan_workspace_bytes (the caller allocates, the plan reuses).
 * Binds caller-allocated device memory of at least muon_plan_workspace_bytes,
 * 256-byte aligned, on the current device.  Encodes the TMA tensor maps over
 * it and creates the plan's events/streams.  The memory must outlive every
 * enqueued step.  Errors: MUON_ERR_INVALID, MUON_ERR_NO_WORKSPACE, MUON_ERR_CUDA,
 * MUON_ERR_UNSUPPORTED (device is not sm_103). */
muon_status muon_plan_bind_workspace(muon_plan_t* plan, void* dev_ptr, size_t bytes);

/* Per-iteration Newton-Schulz coefficients for later muon_step and
 * muon_offload_step calls on this plan (DeepSpeed issue "[RFC] Enable Correct and
 * High-Performance Muon Optimizer under ZeRO CPU Offload", follow-up list:
 * per-iteration optimised coefficients as an ns_method option).
 *   coeffs[3k], coeffs[3k+1], coeffs[3k+2]: (a_k, b_k, c_k) of iteration k, host
 *   memory, copied; iterations past n_iters reuse the last triple.
 *   n_iters: 1..MUON_MAX_NS_STEPS, or 0 (coeffs may be NULL) to return to the
 *   plan's cfg (ns_a, ns_b, ns_c) for every iteration.
 * Non-finite values and out-of-range n_iters return MUON_ERR_INVALID and leave the
 * plan unchanged.  Not to be called while a step of this plan is being enqueued. */
muon_status muon_set_ns_schedule(muon_plan_t* plan, const float* coeffs, int32_t n_iters);

/* Builds a per-iteration schedule by the greedy minimax construction: iteration
 * k uses the odd quintic p_k(x) = a x + b x^3 + c x^5 minimising max |1 - p_k(x)|
 * over [l_k, safety * u_k], and [l_{k+1}, u_{k+1}] = [1 - E_k, 1 + E_k] with E_k
 * that minimum, from [lower, 1] (singular values after the Frobenius
 * normalisation lie in (0, 1]).  Host only, no device or plan involved.
 *   n_iters: 1..MUON_MAX_NS_STEPS; lower in (0, 1); safety in [1, 2].
 *   coeffs_out[3 n_iters]: (a_k, b_k, c_k), fp32.
 *   err_out[n_iters] (nullable): E_k, the bound |1 - p_k o ... o p_0(x)| <= E_k
 *   for x in [lower, 1]. */
muon_status muon_polar_express_coefficients(int32_t n_iters, double lower, double safety, float* coeffs_out,
                                            double* err_out);

/* Defines: "Muon Optimizer + FSDP", section 背景 (background: M_t =
 * momentum_update(grad), U_t = NewtonSchulz(M_t), W_t = W_t - lr U_t on each full
 * 2-D matrix); DeepSpeed issue "[RFC] ... ZeRO CPU Offload", section 2 (5-6
 * Newton-Schulz iterations on full 2-D weight matrices).
 * One Muon step over every matrix of the plan, enqueued on `stream`.
 *   params[n_mats]:   device pointers, weights (cfg.param_dtype), updated in place.
 *   grads[n_mats]:    device pointers, gradients (cfg.grad_dtype), read only.
 *   momentum[n_mats]: device pointers, fp32 momentum, updated in place.
 *   n_mats:           number of pointers in each array = n_shapes of the plan;
 *                     entry i covers all `count` logical matrices of shapes[i].
 *   lr, mu, wd:       learning rate, momentum, decoupled weight decay.
 *   nesterov:         0 / 1.
 *   ns_steps:         Newton-Schulz iterations (0..16); the pages use 5-6.
 * Arguments are validated before anything is enqueued.  The buffers of one
 * entry must not overlap another entry's.  Returns MUON_OK after enqueueing.
 * The call only launches kernels on `stream` (no host synchronisation, no
 * allocation), so one step can be captured with stream capture into a CUDA
 * graph and replayed: every replay uses the captured pointers, lr, mu, wd and
 * ns_steps, and reads whatever the captured gradient buffers then hold (tested
 * with cfg.timing = 0; one plan's steps, captured or not, must not overlap on
 * the device, since they share its workspace). */
muon_status muon_step(muon_plan_t* plan, void* const* params, const void* const* grads,
                      void* const* momentum, int64_t n_mats, float lr, float mu,
                      int32_t nesterov, float wd, int32_t ns_steps, void* stream);

/* Defines: DeepSpeed PR "[Muon] CPU offload: pin the momentum and overlap the
 * host writeback", sections Motivation (gradient and momentum copied to the
 * device, update and momentum back, every step) and Changes (pinned momentum; the
 * writeback of batch i on a side stream after batch i+1 is queued; at most one
 * batch computed and one in flight; drained before the host reads).
 * Offload step: gradients and fp32 momentum live in page-locked host memory.
 * Per micro-bucket: host->device copy of G and M on a private copy stream,
 * momentum + Newton-Schulz on `compute`, then device->host writeback of the new
 * momentum (into h_momentum) and of the update U' = sqrt(max(1,rows/cols)) * U
 * (fp32, original orientation, into h_update_out) on the side stream `copy`,
 * overlapping the next bucket's Newton-Schulz.  At most cfg.max_inflight
 * buckets are in writeback while one computes.  The host then applies
 * W -= lr * (U' + wd * W) itself.  Blocks until every writeback has landed
 * (the host reads the results next) or timeout_ms passes (MUON_ERR_TIMEOUT).
 * After MUON_ERR_TIMEOUT (or an error once some work was enqueued) the step's
 * device work is still in flight and keeps writing h_momentum and h_update_out:
 * the host must not read or reuse them before synchronising the device, or
 * before a later muon_offload_step of the plan returns MUON_OK (each step waits
 * for the previous step's writebacks before it touches the host buffers).
 *   h_grads / h_momentum / h_update_out [n_mats]: pinned host pointers laid out
 *   like the device tensors of muon_step.  MUON_ERR_NOT_PINNED if any is not
 *   page-locked. */
muon_status muon_offload_step(muon_plan_t* plan, const void* const* h_grads,
                              void* const* h_momentum, void* const* h_update_out,
                              int64_t n_mats, float mu, int32_t nesterov, int32_t ns_steps,
                              void* compute, void* copy, int64_t timeout_ms);

/* Defines: DeepSpeed PR "[Muon] CPU offload: pin the momentum and overlap the
 * host writeback", section Changes (writebacks drained before the host reads);
 * the injection itself is this library's, for testing the failure path on the
 * host without faulting a device.
 * Makes the `nth` host-link copy (0-based, in enqueue order: per bucket the
 * gradient and momentum uploads, then the momentum and update writebacks) of the
 * plan's next muon_offload_step report a failure instead of being enqueued, as if
 * cudaMemcpy2DAsync had returned an error: that step returns MUON_ERR_CUDA after
 * enqueueing the work before it, and the injection is cleared.  nth = -1 clears
 * it.  Work already enqueued still completes; the plan's next offload step waits
 * for it.  Pure host state.  Errors: MUON_ERR_INVALID (NULL plan, nth < -1). */
muon_status muon_inject_copy_failure(muon_plan_t* plan, int64_t nth);

/* muon_step for callers that cannot allocate device memory: code running inside
 * an allocator or memory-pool callback (which must not re-enter the allocator),
 * a runtime that has given all device memory to its own pool, a plugin host that
 * forbids device allocations.  The sources describe no such variant; it has no
 * counterpart there.
 * Same arguments and results as muon_step, but no workspace is bound by the
 * caller: the step runs in a file-scope device array of the library
 * (muon_noalloc_scratch_bytes(), 64 MiB), which every GPU that loads the library
 * holds until exit.  The entry point allocates nothing (no cudaMalloc/cudaFree,
 * no allocating library routine).
 *   - The first call on a device, with that device current, looks up the array's
 *     address (cudaGetSymbolAddress); make it before any stream capture.
 *   - The array remembers the plan it was last bound to.  A call with another
 *     plan re-binds it: tensor maps encoded on the host, and the plan's tile
 *     schedules copied into the array on `stream`, after the work already
 *     enqueued there (the copy may block the host while the driver stages it).
 *     Calls with the same plan bind nothing.
 *   - The device status word in the array starts at zero and is shared by every
 *     plan that runs in it: calls never clear it, so it keeps counting
 *     (non-finite matrices, bounded waits that ran out) until muon_sync on any
 *     of those plans reads and clears it.
 *   - Plans whose workspace exceeds the array: MUON_ERR_NO_WORKSPACE.
 *   - All calls share the array and it keeps the last call's contents: calls
 *     whose device work overlaps race on it.  Enqueue them on one stream, or make
 *     each call's stream wait for the previous call's work. */
muon_status muon_step_noalloc(muon_plan_t* plan, void* const* params, const void* const* grads,
                              void* const* momentum, int64_t n_mats, float lr, float mu,
                              int32_t nesterov, float wd, int32_t ns_steps, void* stream);

/* Size in bytes of the static array muon_step_noalloc works in. */
size_t muon_noalloc_scratch_bytes(void);

/* Defines: DeepSpeed issue "[RFC] ... ZeRO CPU Offload", section 5 (overflow
 * skipping named among the interactions of the step); the status word itself is
 * this library's.
 * Waits for `stream`, then reads and clears the device status word written by
 * the kernels: MUON_ERR_DEVICE if a kernel's bounded wait ran out,
 * MUON_WARN_NONFINITE (with *n_nonfinite set) if a matrix norm was not finite,
 * else MUON_OK.  n_nonfinite may be NULL. */
muon_status muon_sync(muon_plan_t* plan, void* stream, int64_t* n_nonfinite);

/* Self-test of the device failure path.  Enqueues on `stream` one CTA that waits
 * on an mbarrier nothing arrives on, through the same bounded wait the
 * Newton-Schulz kernels use, and gives up after limit_us microseconds (1 ..
 * 1000000).  The timeout is recorded in the plan's device status word, so the
 * next muon_sync returns MUON_ERR_DEVICE (and clears it); nothing faults and the
 * context stays usable.  Errors: MUON_ERR_INVALID (NULL plan, limit out of range),
 * MUON_ERR_NO_WORKSPACE, MUON_ERR_CUDA. */
muon_status muon_selftest_wait_timeout(muon_plan_t* plan, int64_t limit_us, void* stream);

/* Defines: "Muon Optimizer + FSDP", section 需要记录的指标 (metrics to log per
 * Muon bucket: key, logical shape, tensor counts, bytes, workspace bytes).
 * Plan layout, for logging and tests (pure host). */
typedef struct {
  int64_t n_tensors;
  int64_t n_matrices;
  int64_t n_groups;        /* distinct (label, m, n) */
  int64_t n_buckets;
  int64_t max_bucket_matrices;
  int64_t max_bucket_bytes; /* wide-form bf16 bytes of the largest bucket */
  size_t workspace_bytes;
} muon_plan_info;
muon_status muon_get_plan_info(const muon_plan_t* plan, muon_plan_info* info);

/* Defines: as muon_get_plan_info, per bucket.
 * Bucket b: number of matrices, wide-form bf16 bytes, same-shape groups in it,
 * the (m, n) of its first group, whether its Newton-Schulz iterations run in the
 * single small-matrix kernel (1: every group has m <= 128, bf16 arithmetic,
 * ns_kernel AUTO) or as grouped GEMM launches (0), and whether that kernel also
 * computes the bucket's momentum in its first pass over each matrix when a step
 * runs at least one iteration (1: bf16 gradients, every matrix wide, n and the
 * matrix stride multiples of 8; 0: a separate momentum kernel runs first). */
typedef struct {
  int64_t n_matrices;
  int64_t bytes;
  int64_t n_groups;
  int64_t m, n;
  int64_t ns_single_kernel;
  int64_t momentum_in_ns_kernel;
} muon_bucket_info;
muon_status muon_get_bucket_info(const muon_plan_t* plan, int64_t b, muon_bucket_info* info);

/* Defines: "Muon Optimizer + FSDP", section 需要记录的指标 (per-bucket times:
 * newton_schulz_time_ms and the transfer times around it).
 * Timings of the last step (cfg.timing = 1), summed over buckets, in ms:
 * prep (momentum kernel), ns (all Newton-Schulz GEMMs), apply, h2d, d2h and the
 * whole step; plus bytes moved over the host link.  Synchronizes the events. */
typedef struct {
  double prep_ms, ns_ms, apply_ms, h2d_ms, d2h_ms, step_ms;
  int64_t h2d_bytes, d2h_bytes;
  int64_t n_buckets;
} muon_stats;
muon_status muon_get_stats(const muon_plan_t* plan, muon_stats* out);

/* Defines: "Muon Optimizer + FSDP", section 需要记录的指标 (metrics to log per
 * Muon bucket: its logical shape, tensor count, full bytes, estimated
 * Newton-Schulz workspace bytes, newton_schulz_time_ms and the transfer times and
 * bytes around it).
 * Bucket b: its shape and sizes (pure host), the host-link bytes it moved in the
 * last offload step (0 after muon_step), and, with cfg.timing = 1, the times of
 * its phases in the last step in ms (waits for that step's events).  prep_ms is 0
 * when the small-matrix kernel computed the momentum (it is then part of ns_ms). */
typedef struct {
  int64_t n_matrices, n_groups;
  int64_t m, n;                  /* wide form of its first group */
  int64_t bytes;                 /* wide-form bf16 bytes of its matrices */
  int64_t ns_workspace_bytes;    /* its Newton-Schulz region in the workspace */
  double prep_ms, ns_ms, apply_ms, h2d_ms, d2h_ms;
  int64_t h2d_bytes, d2h_bytes;
} muon_bucket_stats;
muon_status muon_get_bucket_stats(const muon_plan_t* plan, int64_t b, muon_bucket_stats* out);

/* Defines: "Muon Optimizer + FSDP", section 需要记录的指标 (what to log to tell
 * where the step's numbers come from); the quantity is the Frobenius norm the
 * Newton-Schulz normalisation divides by.
 * Copies ||V||_F of every matrix's Newton-Schulz input in the plan's last step
 * (V the Nesterov look-ahead or the new momentum, before the bf16 cast) into
 * out[n], n = the plan's matrix count, in tensor order (shapes[0]'s `count`
 * matrices first).  A non-finite norm is reported as it came out (inf or NaN).
 * Waits for `stream`.  Errors: MUON_ERR_INVALID, MUON_ERR_NO_WORKSPACE,
 * MUON_ERR_CUDA. */
muon_status muon_get_input_norms(const muon_plan_t* plan, float* out, int64_t n, void* stream);

/* Text of the last error reported by an entry point on the calling thread
 * (empty string if none).  Valid until that thread's next call. */
const char* muon_last_error(void);

/* Static description of a status code. */
const char* muon_status_string(muon_status s);

/* Frees the plan's host memory, events and streams (not the workspace). */
void muon_plan_destroy(muon_plan_t* plan);

#ifdef __cplusplus
}
#endif
#endif /* MUON_H */

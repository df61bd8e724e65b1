// Host runtime of libmuon.so: the C ABI declared in include/muon.h.
//
//  * planner   -- logical matrices of fused tensors ("Muon Optimizer + FSDP",
//                 section 分块通信: qkv = [Q;K;V] and experts [E,out,in] are split
//                 into logical matrices; DeepSpeed issue #8463 section 4.A: shapes
//                 and head dimensions carried into the optimizer), wide orientation,
//                 same-shape groups across layers (section 内存控制方案 item 6), and
//                 micro-buckets of whole matrices under a byte cap (section 分块通信
//                 and item 1).
//  * workspace -- one persistent region sized for the largest micro-bucket and
//                 reused by every bucket through offsets (item 2, "preallocate and
//                 reuse"); the caller allocates it, the plan never does.
//  * step      -- per bucket: momentum prep, norm finalize, ns_steps x (GRAM, POLY,
//                 UPDATE), apply; all stream-ordered, no host synchronisation.
//  * offload   -- DeepSpeed PR "[Muon] CPU offload: pin the momentum and overlap
//                 the host writeback", section Changes: pinned host momentum and
//                 gradients, host->device copy per bucket, writeback of bucket i on
//                 a side stream while bucket i+1 computes, at most max_inflight
//                 buckets in flight, drained before the host reads.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <new>
#include <string>
#include <thread>
#include <tuple>
#include <vector>

#include <nvtx3/nvToolsExt.h>

#include "kernels.h"
#include "muon.h"

using namespace muon;

namespace {

thread_local std::string g_last_error;

muon_status fail(muon_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
muon_status fail(muon_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

muon_status cuda_fail(cudaError_t e, const char* what) {
  return fail(MUON_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// NVTX range around the host-side enqueue of a step and of each of its buckets,
// so that a profiler's timeline names them ("Muon Optimizer + FSDP", section
// 需要记录的指标: per-bucket records).  A no-op unless a tool is attached.
struct NvtxRange {
  explicit NvtxRange(const char* fmt, ...) __attribute__((format(printf, 2, 3))) {
    char buf[96];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    nvtxRangePushA(buf);
  }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

constexpr size_t kAlign = 1024;
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
inline int64_t round_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }
inline int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct TensorInfo {
  int64_t rows, cols, count, stride;
  int64_t m, n;
  bool transposed;
  int label;
  int group;
};

struct Run {  // matrices [first, first+count) of tensor `tensor`
  int tensor;
  int64_t first, count;
};

struct BGroup {
  int group;
  int64_t m, n, count;
  int64_t mat_base;      // bucket-local index of the group's first matrix
  int64_t ld_n, ld_m;    // leading dimensions in the workspace
  std::vector<Run> runs;
  // byte offsets inside the NS region (hi parts; lo parts and X^T for 3xTF32)
  size_t off_x[2], off_a, off_b;
  size_t off_x_lo[2], off_a_lo, off_b_lo;
  size_t off_xt[2], off_xt_lo[2];
  int64_t ld_t;          // leading dimension of X^T (n x m)
  // tensor maps encoded at bind time (lo parts: 3xTF32 only)
  CUtensorMap kx[2], mx[2], ka, kb;
  CUtensorMap kx_lo[2], mx_lo[2], ka_lo, kb_lo;
  CUtensorMap kxt[2], kxt_lo[2];
  CUtensorMap ex[2], ea, eb;  // bf16 GEMM epilogue boxes of 32 x 32 (64-byte swizzle)
};

struct Bucket {
  std::vector<BGroup> groups;
  int64_t n_mats = 0, bytes = 0, elems = 0;
  int n_runs = 0;
  int64_t prep_tiles = 0;
  size_t ns_bytes = 0;
  // per GEMM phase: tile schedule (byte offset in the schedule region, clusters)
  size_t sched_off[3] = {0, 0, 0};
  int32_t sched_clusters[3] = {0, 0, 0};
};

// Shape of one grouped GEMM launch of a bucket: cluster size, groups in launch
// order (longest reduction first), tiles per matrix and k blocks per group.
struct LaunchShape {
  int cluster = 1;
  std::vector<size_t> order;
  std::vector<int64_t> tiles_per_mat, kblocks, M, N, K;
  int64_t total = 0;
};

struct BucketEvents {
  cudaEvent_t start = nullptr, prep = nullptr, ns = nullptr, apply = nullptr, h2d = nullptr,
              d2h_start = nullptr, d2h = nullptr;
};

}  // namespace

struct muon_plan_s {
  muon_config cfg;
  int64_t cap = 0;
  std::vector<TensorInfo> tensors;
  int n_groups = 0;
  std::vector<Bucket> buckets;
  int64_t n_matrices = 0;
  // layout
  size_t off_status = 0, off_scale = 0, off_flags = 0, off_partials = 0, off_ns = 0, off_stage = 0;
  size_t off_norms = 0;               // ||V||_F of every matrix (tensor order) in the last step
  std::vector<int64_t> tensor_first;  // index of each tensor's first matrix in that order
  size_t off_sched = 0, sched_bytes = 0;
  size_t ns_bytes = 0, slot_bytes = 0, ws_bytes = 0;
  int n_slots = 0;
  int64_t max_mats = 0, max_tiles = 0, max_elems = 0;
  // binding
  uint8_t* ws = nullptr;
  size_t ws_size = 0;
  int device = -1;
  int num_sms = 0;
  cudaStream_t h2d_stream = nullptr, d2h_stream = nullptr;
  std::vector<BucketEvents> events;
  std::vector<cudaEvent_t> slot_h2d, slot_comp, slot_d2h;
  cudaEvent_t step_start = nullptr, step_end = nullptr;
  bool offload_last = false;
  int64_t last_h2d_bytes = 0, last_d2h_bytes = 0;
  std::vector<int64_t> bucket_h2d_bytes, bucket_d2h_bytes;  // per bucket, last offload step
  // per-iteration (a, b, c) set by muon_set_ns_schedule; empty: cfg's for every iteration
  std::vector<float> ns_sched;
  // offload: recorded after the last writeback of each step, waited on by the next
  // step's streams (a step that returned MUON_ERR_TIMEOUT may still be in flight)
  cudaEvent_t offload_done = nullptr;
  // host-link copy failure injection (muon_inject_copy_failure): the index, in the
  // next offload step, of the copy reported as failed (-1: none)
  int64_t fail_copy_at = -1;
  // process-unique id (never reused, unlike the plan's address)
  uint64_t id = 0;
  // the tile schedules as uploaded by the last bind (host copy kept for stream-ordered re-uploads)
  std::vector<int32_t> sched_host;
};

namespace {

size_t elem_size_ns(const muon_config& c) { return c.ns_precision == MUON_NS_TF32X3 ? 4 : 2; }
size_t grad_size(const muon_config& c) { return c.grad_dtype == MUON_DTYPE_BF16 ? 2 : 4; }
size_t param_size(const muon_config& c) { return c.param_dtype == MUON_DTYPE_BF16 ? 2 : 4; }

// ---------------------------------------------------------------------------
// TMA tensor maps (driver entry point fetched through the runtime)
// ---------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn) return fn;
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  fn = reinterpret_cast<EncodeTiledFn>(p);
  return fn;
}

// [count][rows][ld] array of `esize`-byte elements; logical (cols, rows, count).
bool encode_map(CUtensorMap* map, void* base, size_t esize, int64_t cols, int64_t rows, int64_t count,
                int64_t ld, uint32_t box_x, uint32_t box_y,
                CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)count};
  const cuuint64_t strides[2] = {(cuuint64_t)(ld * esize), (cuuint64_t)(ld * rows * esize)};
  const cuuint32_t box[3] = {box_x, box_y, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  CUresult r = fn(map, dt, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// planning
// ---------------------------------------------------------------------------
void layout_bucket(Bucket& b, const muon_config& cfg) {
  const size_t es = elem_size_ns(cfg);
  const bool tf32 = cfg.ns_precision == MUON_NS_TF32X3;
  size_t off = 0;
  for (BGroup& g : b.groups) {
    g.ld_n = round_up(g.n, 8);
    g.ld_m = round_up(g.m, 8);
    const size_t xb = (size_t)g.count * g.m * g.ld_n * es;
    const size_t ab = (size_t)g.count * g.m * g.ld_m * es;
    for (int i = 0; i < 2; ++i) { g.off_x[i] = off; off = align_up(off + xb, kAlign); }
    g.off_a = off; off = align_up(off + ab, kAlign);
    g.off_b = off; off = align_up(off + ab, kAlign);
    g.ld_t = round_up(g.m, 8);
    if (tf32) {
      const size_t tb = (size_t)g.count * g.n * g.ld_t * es;
      for (int i = 0; i < 2; ++i) { g.off_x_lo[i] = off; off = align_up(off + xb, kAlign); }
      g.off_a_lo = off; off = align_up(off + ab, kAlign);
      g.off_b_lo = off; off = align_up(off + ab, kAlign);
      for (int i = 0; i < 2; ++i) { g.off_xt[i] = off; off = align_up(off + tb, kAlign); }
      for (int i = 0; i < 2; ++i) { g.off_xt_lo[i] = off; off = align_up(off + tb, kAlign); }
    } else {
      g.off_x_lo[0] = g.off_x_lo[1] = g.off_a_lo = g.off_b_lo = 0;
      g.off_xt[0] = g.off_xt[1] = g.off_xt_lo[0] = g.off_xt_lo[1] = 0;
    }
  }
  b.ns_bytes = off;
}

int64_t tiles_of(int64_t rows, int64_t cols) { return cdiv(rows, kPrepTile) * cdiv(cols, kPrepTile); }

// Row blocks of kBM * cluster rows touching the upper triangle, per 256-column block.
int64_t sym_tiles_per_mat(int64_t M, int cluster) {
  const int64_t rb = (int64_t)kBM * cluster;
  const int64_t tm = cdiv(M, rb), tn = cdiv(M, kBN);
  int64_t total = 0;
  for (int64_t bj = 0; bj < tn; ++bj) total += std::min(tm, (bj * kBN + kBN - 1) / rb + 1);
  return total;
}

LaunchShape launch_shape(const Bucket& b, int mode, bool tf32) {
  LaunchShape L;
  L.cluster = 2;  // pairs of CTAs share the B operand unless a group is one 128-row tile high
  for (const BGroup& g : b.groups)
    if (g.m <= kBM) L.cluster = 1;
  L.order.resize(b.groups.size());
  for (size_t i = 0; i < L.order.size(); ++i) L.order[i] = i;
  std::stable_sort(L.order.begin(), L.order.end(), [&](size_t x, size_t y) {
    const int64_t kx = mode == kGram ? b.groups[x].n : b.groups[x].m;
    const int64_t ky = mode == kGram ? b.groups[y].n : b.groups[y].m;
    return kx > ky;
  });
  const int64_t bk = tf32 ? 32 : 64;
  for (size_t gi : L.order) {
    const BGroup& g = b.groups[gi];
    const int64_t M = g.m, N = mode == kUpdate ? g.n : g.m, K = mode == kGram ? g.n : g.m;
    const int64_t tpm = mode == kUpdate ? cdiv(M, (int64_t)kBM * L.cluster) * cdiv(N, kBN)
                                        : sym_tiles_per_mat(M, L.cluster);
    L.M.push_back(M);
    L.N.push_back(N);
    L.K.push_back(K);
    L.tiles_per_mat.push_back(tpm);
    L.kblocks.push_back(cdiv(K, bk));
    L.total += tpm * g.count;
  }
  return L;
}

// Longest-processing-time assignment of the launch's tiles to `clusters`
// clusters: tiles by cost (k blocks plus an epilogue allowance), longest first,
// each to the least-loaded cluster.  Output: offsets[clusters + 1], units[total].
void lpt_schedule(const Bucket& b, const LaunchShape& L, int mode, int clusters, std::vector<int32_t>& out) {
  const int64_t epi = mode == kGram ? 2 : 3;
  std::vector<std::pair<int64_t, int32_t>> units;  // (cost, tile)
  units.reserve(L.total);
  int64_t t = 0;
  for (size_t i = 0; i < L.order.size(); ++i) {
    const int64_t n = L.tiles_per_mat[i] * b.groups[L.order[i]].count;
    for (int64_t j = 0; j < n; ++j) units.emplace_back(L.kblocks[i] + epi, (int32_t)(t + j));
    t += n;
  }
  std::stable_sort(units.begin(), units.end(),
                   [](const std::pair<int64_t, int32_t>& x, const std::pair<int64_t, int32_t>& y) {
                     return x.first > y.first;
                   });
  std::vector<std::vector<int32_t>> per(clusters);
  // min-heap on (load, cluster id): ties go to the lowest id, so the result is deterministic
  std::vector<std::pair<int64_t, int32_t>> heap;
  for (int c = 0; c < clusters; ++c) heap.emplace_back(0, c);
  auto cmp = [](const std::pair<int64_t, int32_t>& x, const std::pair<int64_t, int32_t>& y) {
    return x.first != y.first ? x.first > y.first : x.second > y.second;
  };
  std::make_heap(heap.begin(), heap.end(), cmp);
  for (const auto& u : units) {
    std::pop_heap(heap.begin(), heap.end(), cmp);
    auto& top = heap.back();
    per[top.second].push_back(u.second);
    top.first += u.first;
    std::push_heap(heap.begin(), heap.end(), cmp);
  }
  out.clear();
  out.reserve(clusters + 1 + units.size());
  int32_t off = 0;
  for (int c = 0; c < clusters; ++c) {
    out.push_back(off);
    off += (int32_t)per[c].size();
  }
  out.push_back(off);
  for (int c = 0; c < clusters; ++c) out.insert(out.end(), per[c].begin(), per[c].end());
}

constexpr int kMaxClusters = 256;  // bound on resident clusters, for the schedule region's size

muon_status build_plan(muon_plan_t* p, const muon_shape* shapes, int32_t n, const int32_t* labels) {
  std::map<std::tuple<int, int64_t, int64_t>, int> gid;
  for (int i = 0; i < n; ++i) {
    const muon_shape& s = shapes[i];
    if (s.rows <= 0 || s.cols <= 0 || s.count <= 0)
      return fail(MUON_ERR_INVALID, "shape %d: rows, cols and count must be >= 1", i);
    if (s.rows > (1 << 20) || s.cols > (1 << 20))
      return fail(MUON_ERR_INVALID, "shape %d: rows/cols above 2^20 are not supported", i);
    const int64_t stride = s.stride_elems ? s.stride_elems : s.rows * s.cols;
    if (stride < s.rows * s.cols)
      return fail(MUON_ERR_INVALID, "shape %d: stride_elems smaller than rows*cols", i);
    TensorInfo t;
    t.rows = s.rows; t.cols = s.cols; t.count = s.count; t.stride = stride;
    t.transposed = s.rows > s.cols;
    t.m = std::min(s.rows, s.cols);
    t.n = std::max(s.rows, s.cols);
    t.label = labels ? labels[i] : 0;
    auto key = std::make_tuple(t.label, t.m, t.n);
    auto it = gid.find(key);
    if (it == gid.end()) it = gid.emplace(key, (int)gid.size()).first;
    t.group = it->second;
    p->tensors.push_back(t);
    p->n_matrices += s.count;
  }
  p->n_groups = (int)gid.size();

  // order: group (first appearance), tensor, matrix; pack whole matrices greedily
  std::vector<int> order;
  for (int g = 0; g < p->n_groups; ++g)
    for (int i = 0; i < n; ++i)
      if (p->tensors[i].group == g) order.push_back(i);

  Bucket cur;
  auto close = [&]() {
    if (cur.n_mats > 0) p->buckets.push_back(cur);
    cur = Bucket();
  };
  for (int ti : order) {
    const TensorInfo& t = p->tensors[ti];
    const int64_t mb = t.m * t.n * 2;  // wide-form bf16 bytes
    for (int64_t j = 0; j < t.count; ++j) {
      bool fits = cur.n_mats == 0;
      if (!fits) {
        const BGroup& last = cur.groups.back();
        const bool same_group = last.group == t.group;
        const bool same_label = p->tensors[last.runs.back().tensor].label == t.label;
        const bool new_run = !(same_group && last.runs.back().tensor == ti &&
                               last.runs.back().first + last.runs.back().count == j);
        fits = same_label && (p->cap <= 0 || cur.bytes + mb <= p->cap) &&
               (same_group || (int)cur.groups.size() < kMaxGroups) &&
               (!new_run || cur.n_runs < kMaxSegs);
      }
      if (!fits) close();
      if (cur.groups.empty() || cur.groups.back().group != t.group) {
        BGroup g;
        g.group = t.group; g.m = t.m; g.n = t.n; g.count = 0; g.mat_base = cur.n_mats;
        cur.groups.push_back(g);
      }
      BGroup& g = cur.groups.back();
      if (g.runs.empty() || g.runs.back().tensor != ti || g.runs.back().first + g.runs.back().count != j) {
        g.runs.push_back(Run{ti, j, 0});
        cur.n_runs++;
      }
      g.runs.back().count++;
      g.count++;
      cur.n_mats++;
      cur.bytes += mb;
      cur.elems += t.rows * t.cols;
      cur.prep_tiles += tiles_of(t.rows, t.cols);
    }
  }
  close();

  // layout of the workspace
  size_t ns_max = 0;
  for (Bucket& b : p->buckets) {
    layout_bucket(b, p->cfg);
    ns_max = std::max(ns_max, b.ns_bytes);
    p->max_mats = std::max(p->max_mats, b.n_mats);
    p->max_tiles = std::max(p->max_tiles, b.prep_tiles);
    p->max_elems = std::max(p->max_elems, b.elems);
  }
  size_t off = 0;
  p->off_status = off; off = align_up(off + sizeof(DeviceStatus), kAlign);
  p->off_scale = off; off = align_up(off + (size_t)p->max_mats * 4, kAlign);
  p->off_flags = off; off = align_up(off + (size_t)p->max_mats * 4, kAlign);
  p->off_partials = off; off = align_up(off + (size_t)p->max_tiles * 4, kAlign);
  p->off_norms = off; off = align_up(off + (size_t)p->n_matrices * 4, kAlign);
  p->tensor_first.assign(p->tensors.size(), 0);
  for (size_t i = 1; i < p->tensors.size(); ++i)
    p->tensor_first[i] = p->tensor_first[i - 1] + p->tensors[i - 1].count;
  p->bucket_h2d_bytes.assign(p->buckets.size(), 0);
  p->bucket_d2h_bytes.assign(p->buckets.size(), 0);
  p->off_ns = off; off = align_up(off + ns_max, kAlign);
  p->ns_bytes = ns_max;
  // tile schedules, one per bucket and GEMM phase: offsets (clusters + 1) and tiles
  size_t sched = 0;
  const bool tf32 = p->cfg.ns_precision == MUON_NS_TF32X3;
  for (Bucket& b : p->buckets)
    for (int mode = kGram; mode <= kUpdate; ++mode) {
      b.sched_off[mode] = sched;
      sched += (size_t)(launch_shape(b, mode, tf32).total + kMaxClusters + 1) * sizeof(int32_t);
      sched = align_up(sched, 256);
    }
  p->off_sched = off; off = align_up(off + sched, kAlign);
  p->sched_bytes = sched;
  if (p->cfg.offload && !p->cfg.offload_zero_copy) {
    p->n_slots = std::max(1, std::min(2, (int)p->cfg.max_inflight)) + 1;
    p->slot_bytes = align_up((size_t)p->max_elems * grad_size(p->cfg), kAlign) +
                    2 * align_up((size_t)p->max_elems * 4, kAlign);
    p->off_stage = off;
    off += (size_t)p->n_slots * p->slot_bytes;
  }
  p->ws_bytes = align_up(off, kAlign);
  return MUON_OK;
}

// ---------------------------------------------------------------------------
// kernel argument assembly
// ---------------------------------------------------------------------------
template <typename T>
T* at(const muon_plan_t* p, size_t off) { return reinterpret_cast<T*>(p->ws + off); }

struct RunPtrs {  // where a run's G / M / W (or U') live for this call
  const void* g;
  float* m;
  void* w;
  int64_t stride;  // elements between consecutive matrices at those pointers
};

// Fills PrepArgs for bucket b; ptr(ti, first) gives the run's pointers.
template <typename F>
void make_prep_args(const muon_plan_t* p, const Bucket& b, F ptr, float mu, int nesterov, PrepArgs& a) {
  std::memset(&a, 0, sizeof(a));
  const bool tf32 = p->cfg.ns_precision == MUON_NS_TF32X3;
  const size_t es = elem_size_ns(p->cfg);
  int si = 0;
  int64_t tile = 0;
  for (const BGroup& g : b.groups) {
    int64_t mat = g.mat_base;
    for (const Run& r : g.runs) {
      const TensorInfo& t = p->tensors[r.tensor];
      PrepSeg& s = a.seg[si++];
      RunPtrs rp = ptr(r);
      s.g = rp.g;
      s.m = rp.m;
      const int64_t xoff = (mat - g.mat_base) * g.m * g.ld_n;
      s.x_hi = p->ws + p->off_ns + g.off_x[0] + xoff * es;
      s.x_lo = tf32 ? reinterpret_cast<float*>(p->ws + p->off_ns + g.off_x_lo[0]) + xoff : nullptr;
      s.rows = t.rows; s.cols = t.cols;
      s.stride = rp.stride;
      s.x_ld = g.ld_n;
      s.x_mstride = g.m * g.ld_n;
      s.block0 = tile;
      if (tf32) {
        const int64_t toff = (mat - g.mat_base) * g.n * g.ld_t;
        s.xt_hi = reinterpret_cast<float*>(p->ws + p->off_ns + g.off_xt[0]) + toff;
        s.xt_lo = reinterpret_cast<float*>(p->ws + p->off_ns + g.off_xt_lo[0]) + toff;
        s.xt_ld = g.ld_t;
        s.xt_mstride = g.n * g.ld_t;
      }
      s.count = (int32_t)r.count;
      s.transposed = t.transposed ? 1 : 0;
      s.tiles_c = (int32_t)cdiv(t.cols, kPrepTile);
      s.tiles_per_mat = (int32_t)tiles_of(t.rows, t.cols);
      s.mat0 = (int32_t)mat;
      s.norm_out = at<float>(p, p->off_norms) + p->tensor_first[r.tensor] + r.first;
      tile += r.count * s.tiles_per_mat;
      mat += r.count;
    }
  }
  a.n_segs = si;
  a.n_mats = (int32_t)b.n_mats;
  a.total_tiles = tile;
  const bool sgd = p->cfg.momentum_form == MUON_MOMENTUM_SGD;
  a.mu = mu;
  a.omu = sgd ? 1.0f : 1.0f - mu;
  a.nesterov = nesterov ? 1 : 0;
  a.grad_dtype = p->cfg.grad_dtype;
  a.tf32 = tf32 ? 1 : 0;
  a.eps = p->cfg.eps;
  a.partials = at<float>(p, p->off_partials);
  a.scale = at<float>(p, p->off_scale);
  a.flags = at<int32_t>(p, p->off_flags);
  a.status = at<DeviceStatus>(p, p->off_status);
}

template <typename F>
void make_apply_args(const muon_plan_t* p, const Bucket& b, F ptr, int final_buf, float lr, float wd,
                     int emit, int ns_steps, ApplyArgs& a) {
  std::memset(&a, 0, sizeof(a));
  const bool tf32 = p->cfg.ns_precision == MUON_NS_TF32X3;
  const size_t es = elem_size_ns(p->cfg);
  int si = 0;
  int64_t tile = 0;
  for (const BGroup& g : b.groups) {
    int64_t mat = g.mat_base;
    for (const Run& r : g.runs) {
      const TensorInfo& t = p->tensors[r.tensor];
      ApplySeg& s = a.seg[si++];
      RunPtrs rp = ptr(r);
      s.w = rp.w;
      const int64_t xoff = (mat - g.mat_base) * g.m * g.ld_n;
      s.u_hi = p->ws + p->off_ns + g.off_x[final_buf] + xoff * es;
      s.u_lo = tf32 ? reinterpret_cast<const float*>(p->ws + p->off_ns + g.off_x_lo[final_buf]) + xoff : nullptr;
      s.rows = t.rows; s.cols = t.cols;
      s.stride = rp.stride;
      s.u_ld = g.ld_n;
      s.u_mstride = g.m * g.ld_n;
      s.block0 = tile;
      s.count = (int32_t)r.count;
      s.transposed = t.transposed ? 1 : 0;
      s.tiles_c = (int32_t)cdiv(t.cols, kPrepTile);
      s.tiles_per_mat = (int32_t)tiles_of(t.rows, t.cols);
      s.mat0 = (int32_t)mat;
      s.shape_scale = (float)std::sqrt(std::max(1.0, (double)t.rows / (double)t.cols));
      tile += r.count * s.tiles_per_mat;
      mat += r.count;
    }
  }
  a.n_segs = si;
  a.total_tiles = tile;
  a.lr = lr;
  a.wd = wd;
  a.param_dtype = p->cfg.param_dtype;
  a.tf32 = tf32 ? 1 : 0;
  a.emit = emit;
  a.skip_nonfinite = p->cfg.skip_nonfinite;
  a.unnormalized = ns_steps == 0 ? 1 : 0;
  a.scale = at<float>(p, p->off_scale);
  a.flags = at<int32_t>(p, p->off_flags);
}

// A bucket whose matrices all have at most 128 rows in the wide form.
bool small_bucket(const Bucket& b) {
  if (b.groups.empty() || b.groups.size() > (size_t)kMaxGroups) return false;
  for (const BGroup& g : b.groups)
    if (g.m > kSmallMaxRows) return false;
  return true;
}

bool uses_small_kernel(const muon_config& c, const Bucket& b) {
  return c.ns_precision == MUON_NS_BF16 && c.ns_kernel == MUON_NS_KERNEL_AUTO && small_bucket(b);
}

// Whether the small-matrix kernel computes the bucket's momentum in its first pass
// instead of the momentum kernel: bf16 gradients, every matrix wide (no transpose),
// and rows of G and M that are whole 16-byte units at 16-byte aligned offsets
// (n and the matrix stride multiples of 8 elements).
bool fuses_momentum(const muon_plan_t* p, const Bucket& b, int ns_steps) {
  if (!p->cfg.ns_momentum_fused || ns_steps <= 0 || !uses_small_kernel(p->cfg, b) ||
      p->cfg.grad_dtype != MUON_DTYPE_BF16)
    return false;
  for (const BGroup& g : b.groups) {
    if (g.n % 8 != 0) return false;
    for (const Run& r : g.runs) {
      const TensorInfo& t = p->tensors[r.tensor];
      if (t.transposed || t.stride % 8 != 0) return false;
    }
  }
  return true;
}

// Every iteration of a small-matrix bucket in one launch (X updated in place in
// the workspace's first X buffer), the weight update fused into the last one.
// (a, b, c) of Newton-Schulz iteration k: the plan's schedule (its last triple
// past its end), else the configuration's.
void ns_coeffs(const muon_plan_t* p, int k, float out[3]) {
  if (p->ns_sched.empty()) {
    out[0] = p->cfg.ns_a;
    out[1] = p->cfg.ns_b;
    out[2] = p->cfg.ns_c;
    return;
  }
  const int n = (int)(p->ns_sched.size() / 3);
  const int i = k < n ? k : n - 1;
  for (int j = 0; j < 3; ++j) out[j] = p->ns_sched[3 * i + j];
}

static_assert(sizeof(SmallArgs::coef) / sizeof(SmallArgs::coef[0]) == MUON_MAX_NS_STEPS,
              "one coefficient triple per possible iteration");

muon_status enqueue_ns_small(muon_plan_t* p, const Bucket& b, int ns_steps, cudaStream_t st,
                             const ApplyArgs& fused, const PrepArgs* prep) {
  SmallArgs sa;
  std::memset(&sa, 0, sizeof(sa));
  std::vector<size_t> order(b.groups.size());
  for (size_t i = 0; i < order.size(); ++i) order[i] = i;
  // longer matrices first, so the last matrices handed out are the short ones
  std::stable_sort(order.begin(), order.end(), [&](size_t x, size_t y) { return b.groups[x].n > b.groups[y].n; });
  int32_t units = 0;
  for (size_t gi = 0; gi < order.size(); ++gi) {
    const BGroup& g = b.groups[order[gi]];
    SmallGroup& G = sa.g[gi];
    G.map_x = g.kx[0];
    G.x = p->ws + p->off_ns + g.off_x[0];
    G.ld = g.ld_n;
    G.mstride = g.m * g.ld_n;
    G.m = (int32_t)g.m;
    G.n = (int32_t)g.n;
    G.count = (int32_t)g.count;
    G.unit0 = units;
    G.mat_base = (int32_t)g.mat_base;
    units += (int32_t)g.count;
  }
  sa.n_groups = (int32_t)order.size();
  sa.n_units = units;
  {
    // start stagger (small_common.cuh): ~3 us per 128-column chunk of the widest
    // matrix, about a third of a matrix's time in the quintic kernel and half in
    // the gram kernel (1728 per-head matrices of 20 chunks: fastest between 45 and
    // 60 us; two or three stagger groups were no faster than one).  The CTAs with
    // one matrix fewer wait; when every CTA has as many matrices, the second half
    // waits (1824 matrices, 12 per CTA: 4% faster all the same), but only from four
    // matrices per CTA on, where the wait is a small part of a CTA's time; a single
    // wave of matrices is not staggered.
    const int32_t grid = units < p->num_sms ? units : p->num_sms;
    int64_t max_n = 0;
    for (const BGroup& g : b.groups) max_n = std::max<int64_t>(max_n, g.n);
    const int64_t chunks = (max_n + 127) / 128;
    sa.stagger_from = units <= grid                     ? INT32_MAX
                      : units % grid                    ? units % grid
                      : units >= 4 * (int64_t)grid      ? grid / 2
                                                        : INT32_MAX;
    sa.stagger_ns = std::min<int64_t>(200000, 3000 * chunks);
  }
  sa.ns_steps = ns_steps;
  for (int k = 0; k < ns_steps && k < MUON_MAX_NS_STEPS; ++k) ns_coeffs(p, k, sa.coef[k]);
  sa.scale = at<float>(p, p->off_scale);
  sa.status = at<DeviceStatus>(p, p->off_status);
  sa.apply = fused;
  if (prep) {  // the momentum of the bucket, computed in the kernel's first pass
    sa.fuse_prep = 1;
    sa.nesterov = prep->nesterov;
    sa.mu = prep->mu;
    sa.omu = prep->omu;
    sa.eps = prep->eps;
    sa.flags = prep->flags;
    sa.n_psegs = prep->n_segs;
    for (int i = 0; i < prep->n_segs; ++i) {
      sa.pseg[i].g = prep->seg[i].g;
      sa.pseg[i].m = prep->seg[i].m;
      sa.pseg[i].stride = prep->seg[i].stride;
      sa.pseg[i].mat0 = prep->seg[i].mat0;
      sa.pseg[i].norm_out = prep->seg[i].norm_out;
    }
  }
  cudaError_t e = p->cfg.ns_method == MUON_NS_METHOD_GRAM ? launch_ns_gram(sa, p->num_sms, st)
                                                           : launch_ns_small(sa, p->num_sms, st);
  if (e != cudaSuccess) return cuda_fail(e, "small-matrix Newton-Schulz launch");
  return MUON_OK;
}

// `prep`: the bucket's momentum arguments when the small-matrix kernel computes the
// momentum itself (fuses_momentum), else null (the momentum kernel has run).
muon_status enqueue_ns(muon_plan_t* p, const Bucket& b, int ns_steps, cudaStream_t st,
                       const ApplyArgs* fused = nullptr, const PrepArgs* prep = nullptr) {
  const muon_config& c = p->cfg;
  const bool tf32 = c.ns_precision == MUON_NS_TF32X3;
  if (fused && ns_steps > 0 && uses_small_kernel(c, b)) return enqueue_ns_small(p, b, ns_steps, st, *fused, prep);
  LaunchShape shapes[3];
  for (int mode = kGram; mode <= kUpdate; ++mode) shapes[mode] = launch_shape(b, mode, tf32);
  for (int it = 0; it < ns_steps; ++it) {
    const int cur = it & 1, nxt = cur ^ 1;
    for (int mode = kGram; mode <= kUpdate; ++mode) {
      const LaunchShape& L = shapes[mode];
      GemmArgs ga;
      std::memset(&ga, 0, sizeof(ga));
      ga.mode = mode;
      ga.n_groups = (int32_t)b.groups.size();
      ga.use_scale = it == 0 && mode != kPoly ? 1 : 0;
      // bf16: the a X term rides in B' = a I + b A + c A A (POLY adds a on the
      // diagonal), so UPDATE is the plain product B' X; 3xTF32 adds a X in UPDATE
      float co[3];
      ns_coeffs(p, it, co);
      ga.alpha = mode == kPoly ? co[2] : 1.0f;
      ga.beta = mode == kPoly ? co[1] : (mode == kUpdate && tf32 ? co[0] : 0.0f);
      ga.diag = mode == kPoly && !tf32 ? co[0] : 0.0f;
      ga.scale = at<float>(p, p->off_scale);
      ga.status = at<DeviceStatus>(p, p->off_status);
      const int32_t* sched = reinterpret_cast<const int32_t*>(p->ws + p->off_sched + b.sched_off[mode]);
      ga.n_clusters = b.sched_clusters[mode];
      if (fused && mode == kUpdate && it == ns_steps - 1) {
        ga.fuse_apply = 1;
        ga.apply = *fused;
      }
      ga.sched_off = sched;
      ga.sched_units = sched + ga.n_clusters + 1;
      int tiles = 0;
      for (size_t gi = 0; gi < L.order.size(); ++gi) {
        const BGroup& g = b.groups[L.order[gi]];
        GemmGroup& G = ga.g[gi];
        uint8_t* ns = p->ws + p->off_ns;
        G.count = (int32_t)g.count;
        G.mat_base = (int32_t)g.mat_base;
        auto lo = [&](size_t off) { return tf32 ? reinterpret_cast<float*>(ns + off) : nullptr; };
        if (mode == kGram) {
          G.map_a = g.kx[cur]; G.map_b = g.kx[cur];
          if (tf32) { G.map_a_lo = g.kx_lo[cur]; G.map_b_lo = g.kx_lo[cur]; }
          if (!tf32) G.map_c = g.ea;
          G.c_hi = ns + g.off_a; G.c_lo = lo(g.off_a_lo);
          G.d_hi = nullptr; G.d_lo = nullptr;
          G.c_ld = g.ld_m; G.c_mstride = g.m * g.ld_m;
        } else if (mode == kPoly) {
          G.map_a = g.ka; G.map_b = g.ka;
          if (tf32) { G.map_a_lo = g.ka_lo; G.map_b_lo = g.ka_lo; }
          if (!tf32) { G.map_c = g.eb; G.map_d = g.ea; }
          G.c_hi = ns + g.off_b; G.c_lo = lo(g.off_b_lo);
          G.d_hi = ns + g.off_a; G.d_lo = lo(g.off_a_lo);
          G.c_ld = g.ld_m; G.c_mstride = g.m * g.ld_m;
        } else {
          G.map_a = g.kb; G.map_b = g.mx[cur];
          if (tf32) {
            // 3xTF32 reads the rows of X^T (K-major) and writes X'^T as well
            G.map_a_lo = g.kb_lo;
            G.map_b = g.kxt[cur]; G.map_b_lo = g.kxt_lo[cur];
            G.ct_hi = ns + g.off_xt[nxt]; G.ct_lo = lo(g.off_xt_lo[nxt]);
            G.ct_ld = g.ld_t; G.ct_mstride = g.n * g.ld_t;
          }
          if (!tf32) G.map_c = g.ex[nxt];
          G.c_hi = ns + g.off_x[nxt]; G.c_lo = lo(g.off_x_lo[nxt]);
          G.d_hi = ns + g.off_x[cur]; G.d_lo = lo(g.off_x_lo[cur]);
          G.c_ld = g.ld_n; G.c_mstride = g.m * g.ld_n;
        }
        G.M = (int32_t)L.M[gi];
        G.N = (int32_t)L.N[gi];
        G.K = (int32_t)L.K[gi];
        G.tiles_m = (int32_t)cdiv(L.M[gi], (int64_t)kBM * L.cluster);
        G.tiles_n = (int32_t)cdiv(L.N[gi], kBN);
        G.tiles_per_mat = (int32_t)L.tiles_per_mat[gi];
        G.tile0 = tiles;
        tiles += G.tiles_per_mat * G.count;
      }
      ga.total_tiles = tiles;
      cudaError_t e = launch_gemm(ga, p->num_sms, tf32, L.cluster, st);
      if (e != cudaSuccess) return cuda_fail(e, "Newton-Schulz GEMM launch");
    }
  }
  return MUON_OK;
}

muon_status check_device_ptr(const void* ptr, const char* what, int i) {
  if (ptr == nullptr) return fail(MUON_ERR_INVALID, "%s[%d] is NULL", what, i);
  if (reinterpret_cast<uintptr_t>(ptr) & 15u) return fail(MUON_ERR_INVALID, "%s[%d] is not 16-byte aligned", what, i);
  return MUON_OK;
}

muon_status check_pinned(const void* ptr, const char* what, int i) {
  if (ptr == nullptr) return fail(MUON_ERR_INVALID, "%s[%d] is NULL", what, i);
  cudaPointerAttributes attr;
  cudaError_t e = cudaPointerGetAttributes(&attr, ptr);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(MUON_ERR_NOT_PINNED, "%s[%d] is not page-locked host memory", what, i);
  }
  if (attr.type != cudaMemoryTypeHost)
    return fail(MUON_ERR_NOT_PINNED, "%s[%d] is not page-locked host memory", what, i);
  return MUON_OK;
}

float elapsed(cudaEvent_t a, cudaEvent_t b) {
  float ms = 0.f;
  if (a && b && cudaEventElapsedTime(&ms, a, b) == cudaSuccess) return ms;
  cudaGetLastError();
  return 0.f;
}

}  // namespace

int32_t muon::set_error(int32_t s, const char* msg) { return fail(s, "%s", msg); }

// ===========================================================================
// C ABI
// ===========================================================================
extern "C" {

const char* muon_last_error(void) { return g_last_error.c_str(); }

void muon_config_default(muon_config* cfg) {
  if (!cfg) return;
  std::memset(cfg, 0, sizeof(*cfg));
  cfg->ns_a = 3.4445f;
  cfg->ns_b = -4.7750f;
  cfg->ns_c = 2.0315f;
  cfg->eps = 1e-7f;
  cfg->ns_precision = MUON_NS_BF16;
  cfg->momentum_form = MUON_MOMENTUM_EMA;
  cfg->grad_dtype = MUON_DTYPE_BF16;
  cfg->param_dtype = MUON_DTYPE_F32;
  cfg->max_inflight = 1;
  cfg->skip_nonfinite = 1;
  cfg->timing = 0;
  cfg->offload = 0;
  cfg->ns_kernel = MUON_NS_KERNEL_AUTO;
  cfg->ns_momentum_fused = 0;
}

muon_status muon_plan(const muon_shape* shapes, int32_t n_shapes, const int32_t* groups, int64_t bucket_cap_bytes,
                      const muon_config* cfg, muon_plan_t** out) {
  if (!out) return fail(MUON_ERR_INVALID, "out is NULL");
  *out = nullptr;
  if (!shapes || n_shapes <= 0) return fail(MUON_ERR_INVALID, "need at least one shape");
  muon_config c;
  if (cfg) c = *cfg; else muon_config_default(&c);
  if (c.ns_precision != MUON_NS_BF16 && c.ns_precision != MUON_NS_TF32X3)
    return fail(MUON_ERR_INVALID, "ns_precision must be MUON_NS_BF16 or MUON_NS_TF32X3");
  if (c.momentum_form != MUON_MOMENTUM_EMA && c.momentum_form != MUON_MOMENTUM_SGD)
    return fail(MUON_ERR_INVALID, "momentum_form must be EMA or SGD");
  if (c.grad_dtype != MUON_DTYPE_BF16 && c.grad_dtype != MUON_DTYPE_F32)
    return fail(MUON_ERR_INVALID, "grad_dtype must be BF16 or F32");
  if (c.param_dtype != MUON_DTYPE_BF16 && c.param_dtype != MUON_DTYPE_F32)
    return fail(MUON_ERR_INVALID, "param_dtype must be BF16 or F32");
  if (!(c.eps >= 0.f) || !std::isfinite(c.ns_a) || !std::isfinite(c.ns_b) || !std::isfinite(c.ns_c))
    return fail(MUON_ERR_INVALID, "eps must be >= 0 and coefficients finite");
  if (c.max_inflight < 1 || c.max_inflight > 2) return fail(MUON_ERR_INVALID, "max_inflight must be 1 or 2");
  if (c.ns_kernel != MUON_NS_KERNEL_AUTO && c.ns_kernel != MUON_NS_KERNEL_GEMM)
    return fail(MUON_ERR_INVALID, "ns_kernel must be AUTO or GEMM");
  if (c.ns_momentum_fused != 0 && c.ns_momentum_fused != 1)
    return fail(MUON_ERR_INVALID, "ns_momentum_fused must be 0 or 1");
  if (c.ns_method != MUON_NS_METHOD_STANDARD && c.ns_method != MUON_NS_METHOD_GRAM)
    return fail(MUON_ERR_INVALID, "ns_method must be STANDARD or GRAM");
  muon_plan_t* p = new (std::nothrow) muon_plan_t();
  if (!p) return fail(MUON_ERR_INVALID, "out of host memory");
  static std::atomic<uint64_t> next_id{1};
  p->id = next_id.fetch_add(1);
  p->cfg = c;
  p->cap = bucket_cap_bytes;
  muon_status s = build_plan(p, shapes, n_shapes, groups);
  if (s == MUON_OK && c.ns_method == MUON_NS_METHOD_GRAM)
    for (size_t b = 0; b < p->buckets.size(); ++b)
      if (!uses_small_kernel(c, p->buckets[b])) {
        s = fail(MUON_ERR_UNSUPPORTED,
                 "the gram method runs in the small-matrix kernel only: bucket %zu has a matrix with "
                 "min(rows, cols) > 128, or the configuration is not bf16 with ns_kernel AUTO", b);
        break;
      }
  if (s != MUON_OK) {
    delete p;
    return s;
  }
  *out = p;
  return MUON_OK;
}

muon_status muon_plan_workspace_bytes(const muon_plan_t* plan, size_t* device_bytes) {
  if (!plan || !device_bytes) return fail(MUON_ERR_INVALID, "NULL argument");
  *device_bytes = plan->ws_bytes;
  return MUON_OK;
}

muon_status muon_get_plan_info(const muon_plan_t* plan, muon_plan_info* info) {
  if (!plan || !info) return fail(MUON_ERR_INVALID, "NULL argument");
  std::memset(info, 0, sizeof(*info));
  info->n_tensors = (int64_t)plan->tensors.size();
  info->n_matrices = plan->n_matrices;
  info->n_groups = plan->n_groups;
  info->n_buckets = (int64_t)plan->buckets.size();
  for (const Bucket& b : plan->buckets) {
    info->max_bucket_matrices = std::max(info->max_bucket_matrices, b.n_mats);
    info->max_bucket_bytes = std::max(info->max_bucket_bytes, b.bytes);
  }
  info->workspace_bytes = plan->ws_bytes;
  return MUON_OK;
}

muon_status muon_set_ns_schedule(muon_plan_t* plan, const float* coeffs, int32_t n_iters) {
  if (!plan) return fail(MUON_ERR_INVALID, "NULL plan");
  if (n_iters < 0 || n_iters > MUON_MAX_NS_STEPS) return fail(MUON_ERR_INVALID, "n_iters must be in [0, %d]", MUON_MAX_NS_STEPS);
  if (n_iters > 0 && !coeffs) return fail(MUON_ERR_INVALID, "NULL coefficients");
  for (int i = 0; i < 3 * n_iters; ++i)
    if (!std::isfinite(coeffs[i])) return fail(MUON_ERR_INVALID, "coefficient %d is not finite", i);
  plan->ns_sched.assign(coeffs ? coeffs : nullptr, coeffs ? coeffs + 3 * n_iters : nullptr);
  return MUON_OK;
}

muon_status muon_get_bucket_info(const muon_plan_t* plan, int64_t b, muon_bucket_info* info) {
  if (!plan || !info) return fail(MUON_ERR_INVALID, "NULL argument");
  if (b < 0 || b >= (int64_t)plan->buckets.size()) return fail(MUON_ERR_INVALID, "bucket index out of range");
  const Bucket& k = plan->buckets[b];
  info->n_matrices = k.n_mats;
  info->bytes = k.bytes;
  info->n_groups = (int64_t)k.groups.size();
  info->m = k.groups[0].m;
  info->n = k.groups[0].n;
  info->ns_single_kernel = uses_small_kernel(plan->cfg, k) ? 1 : 0;
  info->momentum_in_ns_kernel = fuses_momentum(plan, k, 1) ? 1 : 0;
  return MUON_OK;
}

}  // extern "C"

namespace {

// Binds `p` to `dev_ptr`: tensor maps, tile schedules, streams and events.
// stream == nullptr (muon_plan_bind_workspace): the schedules are uploaded and the
// status word cleared synchronously.  Otherwise (the shared static scratch): the
// schedules are copied on `stream`, after the work already enqueued there, and
// the status word is left alone.
muon_status bind_impl(muon_plan_t* p, void* dev_ptr, size_t bytes, cudaStream_t stream, bool stream_ordered) {
  if (!p || !dev_ptr) return fail(MUON_ERR_INVALID, "NULL argument");
  if (reinterpret_cast<uintptr_t>(dev_ptr) & 255u) return fail(MUON_ERR_INVALID, "workspace must be 256-byte aligned");
  if (bytes < p->ws_bytes)
    return fail(MUON_ERR_NO_WORKSPACE, "workspace of %zu bytes is smaller than the %zu the plan needs", bytes,
                p->ws_bytes);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int major = 0, minor = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (major != 10 || minor != 3)
    return fail(MUON_ERR_UNSUPPORTED, "libmuon is built for sm_103a; device is sm_%d%d", major, minor);
  cudaPointerAttributes attr;
  e = cudaPointerGetAttributes(&attr, dev_ptr);
  if (e != cudaSuccess || attr.type != cudaMemoryTypeDevice) {
    cudaGetLastError();
    return fail(MUON_ERR_INVALID, "workspace is not device memory");
  }
  if (!get_encode_fn()) return fail(MUON_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  p->ws = static_cast<uint8_t*>(dev_ptr);
  p->ws_size = bytes;
  p->device = dev;
  p->num_sms = sms;
  const size_t es = elem_size_ns(p->cfg);
  const bool tf32 = p->cfg.ns_precision == MUON_NS_TF32X3;
  const uint32_t kbox = tf32 ? 32 : 64;  // 128-byte rows
  for (Bucket& b : p->buckets) {
    for (BGroup& g : b.groups) {
      uint8_t* ns = p->ws + p->off_ns;
      bool ok = true;
      for (int i = 0; i < 2; ++i) {
        ok &= encode_map(&g.kx[i], ns + g.off_x[i], es, g.n, g.m, g.count, g.ld_n, kbox, 128);
        ok &= encode_map(&g.mx[i], ns + g.off_x[i], es, g.n, g.m, g.count, g.ld_n, kbox, kbox);
      }
      ok &= encode_map(&g.ka, ns + g.off_a, es, g.m, g.m, g.count, g.ld_m, kbox, 128);
      ok &= encode_map(&g.kb, ns + g.off_b, es, g.m, g.m, g.count, g.ld_m, kbox, 128);
      if (!tf32) {
        // the epilogue's 32 x 32 chunks: 64-byte rows, swizzled like its staging
        const CUtensorMapSwizzle sw = CU_TENSOR_MAP_SWIZZLE_64B;
        for (int i = 0; i < 2; ++i)
          ok &= encode_map(&g.ex[i], ns + g.off_x[i], es, g.n, g.m, g.count, g.ld_n, 32, 32, sw);
        ok &= encode_map(&g.ea, ns + g.off_a, es, g.m, g.m, g.count, g.ld_m, 32, 32, sw);
        ok &= encode_map(&g.eb, ns + g.off_b, es, g.m, g.m, g.count, g.ld_m, 32, 32, sw);
      }
      if (tf32) {
        for (int i = 0; i < 2; ++i) {
          ok &= encode_map(&g.kx_lo[i], ns + g.off_x_lo[i], es, g.n, g.m, g.count, g.ld_n, kbox, 128);
          ok &= encode_map(&g.mx_lo[i], ns + g.off_x_lo[i], es, g.n, g.m, g.count, g.ld_n, kbox, kbox);
        }
        ok &= encode_map(&g.ka_lo, ns + g.off_a_lo, es, g.m, g.m, g.count, g.ld_m, kbox, 128);
        ok &= encode_map(&g.kb_lo, ns + g.off_b_lo, es, g.m, g.m, g.count, g.ld_m, kbox, 128);
        for (int i = 0; i < 2; ++i) {  // X^T: n rows of m
          ok &= encode_map(&g.kxt[i], ns + g.off_xt[i], es, g.m, g.n, g.count, g.ld_t, kbox, 128);
          ok &= encode_map(&g.kxt_lo[i], ns + g.off_xt_lo[i], es, g.m, g.n, g.count, g.ld_t, kbox, 128);
        }
      }
      if (!ok) return fail(MUON_ERR_CUDA, "cuTensorMapEncodeTiled rejected a workspace tensor map");
    }
  }
  {
    // tile schedules for this device's number of resident clusters
    std::vector<int32_t> host(p->sched_bytes / sizeof(int32_t), 0), one;
    for (Bucket& b : p->buckets)
      for (int mode = kGram; mode <= kUpdate; ++mode) {
        const LaunchShape L = launch_shape(b, mode, tf32);
        int clusters = gemm_max_clusters(tf32, L.cluster, p->num_sms);
        if (clusters <= 0 || clusters > kMaxClusters)
          return fail(MUON_ERR_CUDA, "could not size the GEMM grid (%d resident clusters)", clusters);
        if (L.total < clusters) clusters = (int)std::max<int64_t>(L.total, 1);
        lpt_schedule(b, L, mode, clusters, one);
        std::copy(one.begin(), one.end(), host.begin() + b.sched_off[mode] / sizeof(int32_t));
        b.sched_clusters[mode] = clusters;
      }
    p->sched_host.swap(host);
    e = stream_ordered ? cudaMemcpyAsync(p->ws + p->off_sched, p->sched_host.data(), p->sched_bytes,
                                         cudaMemcpyHostToDevice, stream)
                       : cudaMemcpy(p->ws + p->off_sched, p->sched_host.data(), p->sched_bytes,
                                    cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "schedule upload");
  }
  if (!p->h2d_stream) {
    e = cudaStreamCreateWithFlags(&p->h2d_stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamCreate");
    e = cudaStreamCreateWithFlags(&p->d2h_stream, cudaStreamNonBlocking);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamCreate");
    p->events.resize(p->buckets.size());
    for (BucketEvents& ev : p->events) {
      cudaEvent_t* all[] = {&ev.start, &ev.prep, &ev.ns, &ev.apply, &ev.h2d, &ev.d2h_start, &ev.d2h};
      for (cudaEvent_t* x : all)
        if ((e = cudaEventCreate(x)) != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
    }
    const int slots = std::max(p->n_slots, 1);
    p->slot_h2d.resize(slots); p->slot_comp.resize(slots); p->slot_d2h.resize(slots);
    for (int i = 0; i < slots; ++i) {
      cudaEventCreateWithFlags(&p->slot_h2d[i], cudaEventDisableTiming);
      cudaEventCreateWithFlags(&p->slot_comp[i], cudaEventDisableTiming);
      cudaEventCreateWithFlags(&p->slot_d2h[i], cudaEventDisableTiming);
    }
    cudaEventCreate(&p->step_start);
    cudaEventCreate(&p->step_end);
    cudaEventCreateWithFlags(&p->offload_done, cudaEventDisableTiming);
  }
  if (!stream_ordered) {
    e = cudaMemset(p->ws + p->off_status, 0, sizeof(DeviceStatus));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();  // done before any stream's next kernel
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(status)");
  }
  return MUON_OK;
}

}  // namespace

int32_t muon::bind_shared_scratch(muon_plan_t* p, void* dev_ptr, size_t bytes, cudaStream_t stream) {
  return bind_impl(p, dev_ptr, bytes, stream, true);
}

uint64_t muon::plan_id(const muon_plan_t* p) { return p ? p->id : 0; }

const void* muon::plan_workspace(const muon_plan_t* p) { return p ? p->ws : nullptr; }

extern "C" {

muon_status muon_plan_bind_workspace(muon_plan_t* p, void* dev_ptr, size_t bytes) {
  return bind_impl(p, dev_ptr, bytes, nullptr, false);
}

muon_status muon_step(muon_plan_t* p, void* const* params, const void* const* grads, void* const* momentum,
                      int64_t n_mats, float lr, float mu, int32_t nesterov, float wd, int32_t ns_steps, void* stream) {
  if (!p) return fail(MUON_ERR_INVALID, "plan is NULL");
  if (!p->ws) return fail(MUON_ERR_NO_WORKSPACE, "no workspace bound");
  if (!params || !grads || !momentum) return fail(MUON_ERR_INVALID, "pointer array is NULL");
  if (n_mats != (int64_t)p->tensors.size())
    return fail(MUON_ERR_INVALID, "n_mats %lld != %zu tensors in the plan", (long long)n_mats, p->tensors.size());
  if (ns_steps < 0 || ns_steps > MUON_MAX_NS_STEPS) return fail(MUON_ERR_INVALID, "ns_steps must be in [0, %d]", MUON_MAX_NS_STEPS);
  if (!std::isfinite(lr) || !std::isfinite(mu) || !std::isfinite(wd)) return fail(MUON_ERR_INVALID, "lr, mu, wd must be finite");
  for (int i = 0; i < n_mats; ++i) {
    muon_status s;
    if ((s = check_device_ptr(params[i], "params", i)) != MUON_OK) return s;
    if ((s = check_device_ptr(grads[i], "grads", i)) != MUON_OK) return s;
    if ((s = check_device_ptr(momentum[i], "momentum", i)) != MUON_OK) return s;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const bool timing = p->cfg.timing != 0;
  const size_t gs = grad_size(p->cfg), ps = param_size(p->cfg);
  std::fill(p->bucket_h2d_bytes.begin(), p->bucket_h2d_bytes.end(), 0);
  std::fill(p->bucket_d2h_bytes.begin(), p->bucket_d2h_bytes.end(), 0);
  NvtxRange step_range("muon_step: %zu buckets", p->buckets.size());
  if (timing) cudaEventRecord(p->step_start, st);
  for (size_t bi = 0; bi < p->buckets.size(); ++bi) {
    const Bucket& b = p->buckets[bi];
    NvtxRange bucket_range("muon bucket %zu: %lld matrices, %lld x %lld", bi, (long long)b.n_mats,
                           (long long)b.groups[0].m, (long long)b.groups[0].n);
    auto ptrs = [&](const Run& r) {
      const TensorInfo& t = p->tensors[r.tensor];
      RunPtrs rp;
      rp.g = static_cast<const uint8_t*>(grads[r.tensor]) + (size_t)r.first * t.stride * gs;
      rp.m = static_cast<float*>(momentum[r.tensor]) + (size_t)r.first * t.stride;
      rp.w = static_cast<uint8_t*>(params[r.tensor]) + (size_t)r.first * t.stride * ps;
      rp.stride = t.stride;
      return rp;
    };
    PrepArgs pa;
    make_prep_args(p, b, ptrs, mu, nesterov, pa);
    const bool fuse = fuses_momentum(p, b, ns_steps);
    if (timing) cudaEventRecord(p->events[bi].start, st);
    cudaError_t e;
    if (!fuse) {
      e = launch_prep(pa, st);
      if (e != cudaSuccess) return cuda_fail(e, "momentum_prep launch");
      e = launch_norm(pa, st);
      if (e != cudaSuccess) return cuda_fail(e, "norm_finalize launch");
    }
    if (timing) cudaEventRecord(p->events[bi].prep, st);
    // the weight update runs in the last UPDATE's epilogue; with no iteration, in its own kernel
    ApplyArgs aa;
    make_apply_args(p, b, ptrs, ns_steps & 1, lr, wd, 0, ns_steps, aa);
    muon_status s = enqueue_ns(p, b, ns_steps, st, ns_steps > 0 ? &aa : nullptr, fuse ? &pa : nullptr);
    if (s != MUON_OK) return s;
    if (timing) cudaEventRecord(p->events[bi].ns, st);
    if (ns_steps == 0) {
      e = launch_apply(aa, st);
      if (e != cudaSuccess) return cuda_fail(e, "apply launch");
    }
    if (timing) cudaEventRecord(p->events[bi].apply, st);
  }
  if (timing) cudaEventRecord(p->step_end, st);
  p->offload_last = false;
  p->last_h2d_bytes = p->last_d2h_bytes = 0;
  return MUON_OK;
}

namespace {

// The device address of pinned host memory (the same address under unified
// addressing when the allocation is mapped, as cudaHostAlloc memory is).
muon_status mapped(const void* host, const char* what, int i, const void** dev) {
  void* d = nullptr;
  cudaError_t e = cudaHostGetDevicePointer(&d, const_cast<void*>(host), 0);
  if (e != cudaSuccess || d == nullptr) {
    cudaGetLastError();
    return fail(MUON_ERR_NOT_PINNED, "%s[%d] is pinned but not mapped into the device's address space", what, i);
  }
  *dev = d;
  return MUON_OK;
}

// Zero-copy offload: per bucket, the momentum kernel reads G and M from host
// memory over the host link and writes M back there, Newton-Schulz runs on the
// device, and the last UPDATE's epilogue writes U' into the host buffer; all on
// the compute stream, drained before returning.
muon_status offload_zero_copy(muon_plan_t* p, const void* const* h_grads, void* const* h_momentum,
                              void* const* h_update_out, float mu, int32_t nesterov, int32_t ns_steps,
                              cudaStream_t cs, int64_t timeout_ms) {
  const size_t gs = grad_size(p->cfg);
  const bool timing = p->cfg.timing != 0;
  const int n = (int)p->tensors.size();
  std::vector<const void*> dg(n), dm(n), du(n);
  for (int i = 0; i < n; ++i) {
    muon_status s;
    if ((s = mapped(h_grads[i], "h_grads", i, &dg[i])) != MUON_OK) return s;
    if ((s = mapped(h_momentum[i], "h_momentum", i, &dm[i])) != MUON_OK) return s;
    if ((s = mapped(h_update_out[i], "h_update_out", i, &du[i])) != MUON_OK) return s;
  }
  int64_t h2d_bytes = 0, d2h_bytes = 0;
  std::fill(p->bucket_h2d_bytes.begin(), p->bucket_h2d_bytes.end(), 0);
  std::fill(p->bucket_d2h_bytes.begin(), p->bucket_d2h_bytes.end(), 0);
  cudaError_t e;
  // after the previous step's kernels, even if that step returned before they finished
  cudaStreamWaitEvent(cs, p->offload_done, 0);
  if (timing) cudaEventRecord(p->step_start, cs);
  for (size_t bi = 0; bi < p->buckets.size(); ++bi) {
    const Bucket& b = p->buckets[bi];
    auto ptrs = [&](const Run& r) {
      const TensorInfo& t = p->tensors[r.tensor];
      RunPtrs rp;
      rp.g = static_cast<const uint8_t*>(dg[r.tensor]) + (size_t)r.first * t.stride * gs;
      rp.m = const_cast<float*>(static_cast<const float*>(dm[r.tensor])) + (size_t)r.first * t.stride;
      rp.w = const_cast<float*>(static_cast<const float*>(du[r.tensor])) + (size_t)r.first * t.stride;
      rp.stride = t.stride;
      return rp;
    };
    for (const BGroup& g : b.groups)
      for (const Run& r : g.runs) {
        const TensorInfo& t = p->tensors[r.tensor];
        h2d_bytes += r.count * t.rows * t.cols * (int64_t)(gs + 4);
        d2h_bytes += r.count * t.rows * t.cols * 8;
        p->bucket_h2d_bytes[bi] += r.count * t.rows * t.cols * (int64_t)(gs + 4);
        p->bucket_d2h_bytes[bi] += r.count * t.rows * t.cols * 8;
      }
    if (timing) {
      cudaEventRecord(p->events[bi].start, cs);
      cudaEventRecord(p->events[bi].prep, cs);
    }
    PrepArgs pa;
    make_prep_args(p, b, ptrs, mu, nesterov, pa);
    if ((e = launch_prep(pa, cs)) != cudaSuccess) return cuda_fail(e, "momentum_prep launch");
    if ((e = launch_norm(pa, cs)) != cudaSuccess) return cuda_fail(e, "norm_finalize launch");
    if (timing) cudaEventRecord(p->events[bi].h2d, cs);
    ApplyArgs aa;
    make_apply_args(p, b, ptrs, ns_steps & 1, 0.f, 0.f, 1, ns_steps, aa);
    muon_status s = enqueue_ns(p, b, ns_steps, cs, ns_steps > 0 ? &aa : nullptr);
    if (s != MUON_OK) return s;
    if (timing) cudaEventRecord(p->events[bi].ns, cs);
    if (ns_steps == 0 && (e = launch_apply(aa, cs)) != cudaSuccess) return cuda_fail(e, "emit launch");
    if (timing) {
      cudaEventRecord(p->events[bi].apply, cs);
      cudaEventRecord(p->events[bi].d2h_start, cs);
      cudaEventRecord(p->events[bi].d2h, cs);
    }
  }
  if (timing) cudaEventRecord(p->step_end, cs);
  cudaEvent_t done = p->offload_done;
  e = cudaEventRecord(done, cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  // drain: the host reads the results next
  const auto t0 = std::chrono::steady_clock::now();
  for (;;) {
    e = cudaEventQuery(done);
    if (e == cudaSuccess) break;
    if (e != cudaErrorNotReady) return cuda_fail(e, "zero-copy offload step");
    if (std::chrono::steady_clock::now() - t0 > std::chrono::milliseconds(timeout_ms))
      return fail(MUON_ERR_TIMEOUT, "zero-copy offload step did not finish within %lld ms", (long long)timeout_ms);
    std::this_thread::sleep_for(std::chrono::microseconds(50));
  }
  p->offload_last = true;
  p->last_h2d_bytes = h2d_bytes;
  p->last_d2h_bytes = d2h_bytes;
  return MUON_OK;
}

}  // namespace

muon_status muon_offload_step(muon_plan_t* p, const void* const* h_grads, void* const* h_momentum,
                              void* const* h_update_out, int64_t n_mats, float mu, int32_t nesterov,
                              int32_t ns_steps, void* compute, void* copy, int64_t timeout_ms) {
  if (!p) return fail(MUON_ERR_INVALID, "plan is NULL");
  if (!p->ws) return fail(MUON_ERR_NO_WORKSPACE, "no workspace bound");
  if (!p->cfg.offload || (!p->cfg.offload_zero_copy && p->n_slots < 2))
    return fail(MUON_ERR_NO_WORKSPACE, "plan was made without cfg.offload = 1 (no staging slots)");
  if (!h_grads || !h_momentum || !h_update_out) return fail(MUON_ERR_INVALID, "pointer array is NULL");
  if (n_mats != (int64_t)p->tensors.size())
    return fail(MUON_ERR_INVALID, "n_mats %lld != %zu tensors in the plan", (long long)n_mats, p->tensors.size());
  if (ns_steps < 0 || ns_steps > MUON_MAX_NS_STEPS) return fail(MUON_ERR_INVALID, "ns_steps must be in [0, %d]", MUON_MAX_NS_STEPS);
  if (timeout_ms <= 0) return fail(MUON_ERR_INVALID, "timeout_ms must be > 0");
  for (int i = 0; i < n_mats; ++i) {
    muon_status s;
    if ((s = check_pinned(h_grads[i], "h_grads", i)) != MUON_OK) return s;
    if ((s = check_pinned(h_momentum[i], "h_momentum", i)) != MUON_OK) return s;
    if ((s = check_pinned(h_update_out[i], "h_update_out", i)) != MUON_OK) return s;
  }
  cudaStream_t cs = static_cast<cudaStream_t>(compute);
  if (p->cfg.offload_zero_copy) return offload_zero_copy(p, h_grads, h_momentum, h_update_out, mu, nesterov, ns_steps,
                                                         cs, timeout_ms);
  cudaStream_t ds = copy ? static_cast<cudaStream_t>(copy) : p->d2h_stream;
  cudaStream_t hs = p->h2d_stream;
  const size_t gs = grad_size(p->cfg);
  const bool timing = p->cfg.timing != 0;
  int64_t h2d_bytes = 0, d2h_bytes = 0;
  std::fill(p->bucket_h2d_bytes.begin(), p->bucket_h2d_bytes.end(), 0);
  std::fill(p->bucket_d2h_bytes.begin(), p->bucket_d2h_bytes.end(), 0);
  cudaError_t e;
  if (timing) cudaEventRecord(p->step_start, cs);
  // the host buffers must not be touched by the previous step any more: its
  // compute (the stream's earlier work) and its writebacks, which are still in
  // flight if it returned MUON_ERR_TIMEOUT or an error
  e = cudaEventRecord(p->slot_h2d[0], cs);
  if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
  cudaStreamWaitEvent(hs, p->slot_h2d[0], 0);
  cudaStreamWaitEvent(hs, p->offload_done, 0);
  cudaStreamWaitEvent(cs, p->offload_done, 0);
  int64_t copy_index = 0;  // host-link copies enqueued so far (failure injection)
  const int64_t fail_at = p->fail_copy_at;
  p->fail_copy_at = -1;
  auto injected = [&]() { return copy_index++ == fail_at; };
  // a failure after some buckets' work was enqueued: later steps still wait for it
  auto enqueue_fail = [&](cudaError_t err, const char* what) {
    cudaEventRecord(p->offload_done, ds);
    if (err == cudaSuccess)
      return fail(MUON_ERR_CUDA, "%s: injected failure of host-link copy %lld", what, (long long)fail_at);
    return cuda_fail(err, what);
  };
  NvtxRange step_range("muon_offload_step: %zu buckets", p->buckets.size());
  for (size_t bi = 0; bi < p->buckets.size(); ++bi) {
    const Bucket& b = p->buckets[bi];
    NvtxRange bucket_range("muon offload bucket %zu: %lld matrices, %lld x %lld", bi, (long long)b.n_mats,
                           (long long)b.groups[0].m, (long long)b.groups[0].n);
    const int slot = (int)(bi % p->n_slots);
    uint8_t* sbase = p->ws + p->off_stage + (size_t)slot * p->slot_bytes;
    uint8_t* sg = sbase;
    float* sm = reinterpret_cast<float*>(sbase + align_up((size_t)p->max_elems * gs, kAlign));
    float* su = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(sm) + align_up((size_t)p->max_elems * 4, kAlign));
    if (bi >= (size_t)p->n_slots) cudaStreamWaitEvent(hs, p->slot_d2h[slot], 0);
    if (timing) cudaEventRecord(p->events[bi].start, hs);
    // host -> device: G and M of every run, packed contiguously in bucket order
    std::vector<std::tuple<const Run*, int64_t>> run_off;
    int64_t eoff = 0;
    for (const BGroup& g : b.groups)
      for (const Run& r : g.runs) {
        const TensorInfo& t = p->tensors[r.tensor];
        const int64_t me = t.rows * t.cols;
        const uint8_t* hg = static_cast<const uint8_t*>(h_grads[r.tensor]) + (size_t)r.first * t.stride * gs;
        const uint8_t* hm = static_cast<const uint8_t*>(h_momentum[r.tensor]) + (size_t)r.first * t.stride * 4;
        if (injected()) return enqueue_fail(cudaSuccess, "host->device copy");
        e = cudaMemcpy2DAsync(sg + (size_t)eoff * gs, me * gs, hg, t.stride * gs, me * gs, r.count,
                              cudaMemcpyHostToDevice, hs);
        if (e == cudaSuccess && injected()) return enqueue_fail(cudaSuccess, "host->device copy");
        if (e == cudaSuccess)
          e = cudaMemcpy2DAsync(sm + eoff, me * 4, hm, t.stride * 4, me * 4, r.count, cudaMemcpyHostToDevice, hs);
        if (e != cudaSuccess) return enqueue_fail(e, "host->device copy");
        h2d_bytes += r.count * me * (int64_t)(gs + 4);
        p->bucket_h2d_bytes[bi] += r.count * me * (int64_t)(gs + 4);
        run_off.emplace_back(&r, eoff);
        eoff += r.count * me;
      }
    cudaEventRecord(p->slot_h2d[slot], hs);
    if (timing) cudaEventRecord(p->events[bi].h2d, hs);
    cudaStreamWaitEvent(cs, p->slot_h2d[slot], 0);
    // compute: prep (reads the staged G/M, writes M_new in place), NS, emit U'
    auto stage_ptrs = [&](const Run& r) {
      RunPtrs rp;
      int64_t off = 0;
      for (auto& ro : run_off)
        if (std::get<0>(ro) == &r) off = std::get<1>(ro);
      rp.g = sg + (size_t)off * gs;
      rp.m = sm + off;
      rp.w = su + off;
      rp.stride = p->tensors[r.tensor].rows * p->tensors[r.tensor].cols;
      return rp;
    };
    PrepArgs pa;
    make_prep_args(p, b, stage_ptrs, mu, nesterov, pa);
    const bool fuse = fuses_momentum(p, b, ns_steps);
    if (timing) cudaEventRecord(p->events[bi].prep, cs);  // marks compute start for this bucket
    if (!fuse) {
      if ((e = launch_prep(pa, cs)) != cudaSuccess) return cuda_fail(e, "momentum_prep launch");
      if ((e = launch_norm(pa, cs)) != cudaSuccess) return cuda_fail(e, "norm_finalize launch");
    }
    ApplyArgs aa;
    make_apply_args(p, b, stage_ptrs, ns_steps & 1, 0.f, 0.f, 1, ns_steps, aa);
    muon_status s = enqueue_ns(p, b, ns_steps, cs, ns_steps > 0 ? &aa : nullptr, fuse ? &pa : nullptr);
    if (s != MUON_OK) return s;
    if (timing) cudaEventRecord(p->events[bi].ns, cs);
    if (ns_steps == 0 && (e = launch_apply(aa, cs)) != cudaSuccess) return cuda_fail(e, "emit launch");
    cudaEventRecord(p->slot_comp[slot], cs);
    if (timing) cudaEventRecord(p->events[bi].apply, cs);
    // device -> host writeback on the side stream
    cudaStreamWaitEvent(ds, p->slot_comp[slot], 0);
    if (timing) cudaEventRecord(p->events[bi].d2h_start, ds);
    for (auto& ro : run_off) {
      const Run& r = *std::get<0>(ro);
      const int64_t off = std::get<1>(ro);
      const TensorInfo& t = p->tensors[r.tensor];
      const int64_t me = t.rows * t.cols;
      uint8_t* hm = static_cast<uint8_t*>(h_momentum[r.tensor]) + (size_t)r.first * t.stride * 4;
      uint8_t* hu = static_cast<uint8_t*>(h_update_out[r.tensor]) + (size_t)r.first * t.stride * 4;
      if (injected()) return enqueue_fail(cudaSuccess, "device->host copy");
      e = cudaMemcpy2DAsync(hm, t.stride * 4, sm + off, me * 4, me * 4, r.count, cudaMemcpyDeviceToHost, ds);
      if (e == cudaSuccess && injected()) return enqueue_fail(cudaSuccess, "device->host copy");
      if (e == cudaSuccess)
        e = cudaMemcpy2DAsync(hu, t.stride * 4, su + off, me * 4, me * 4, r.count, cudaMemcpyDeviceToHost, ds);
      if (e != cudaSuccess) return enqueue_fail(e, "device->host copy");
      d2h_bytes += r.count * me * 8;
      p->bucket_d2h_bytes[bi] += r.count * me * 8;
    }
    cudaEventRecord(p->slot_d2h[slot], ds);
    if (timing) cudaEventRecord(p->events[bi].d2h, ds);
  }
  if (timing) cudaEventRecord(p->step_end, ds);
  cudaEventRecord(p->offload_done, ds);  // ds carries every bucket's writeback, in order
  // drain: the host reads the results next
  const auto t0 = std::chrono::steady_clock::now();
  for (int sidx = 0; sidx < p->n_slots && sidx < (int)p->buckets.size(); ++sidx) {
    for (;;) {
      e = cudaEventQuery(p->slot_d2h[sidx]);
      if (e == cudaSuccess) break;
      if (e != cudaErrorNotReady) return cuda_fail(e, "writeback");
      if (std::chrono::steady_clock::now() - t0 > std::chrono::milliseconds(timeout_ms))
        return fail(MUON_ERR_TIMEOUT, "writeback did not finish within %lld ms", (long long)timeout_ms);
      std::this_thread::sleep_for(std::chrono::microseconds(50));
    }
  }
  p->offload_last = true;
  p->last_h2d_bytes = h2d_bytes;
  p->last_d2h_bytes = d2h_bytes;
  return MUON_OK;
}

muon_status muon_inject_copy_failure(muon_plan_t* p, int64_t nth) {
  if (!p) return fail(MUON_ERR_INVALID, "plan is NULL");
  if (nth < -1) return fail(MUON_ERR_INVALID, "nth must be >= -1");
  p->fail_copy_at = nth;
  return MUON_OK;
}

muon_status muon_sync(muon_plan_t* p, void* stream, int64_t* n_nonfinite) {
  if (!p) return fail(MUON_ERR_INVALID, "plan is NULL");
  if (n_nonfinite) *n_nonfinite = 0;
  if (!p->ws) return fail(MUON_ERR_NO_WORKSPACE, "no workspace bound");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  // read and clear on `stream`, and wait for both: a memset on the legacy stream
  // may still be pending when later work starts on a non-blocking stream
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DeviceStatus ds;
  e = cudaMemcpyAsync(&ds, p->ws + p->off_status, sizeof(ds), cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  e = cudaMemsetAsync(p->ws + p->off_status, 0, sizeof(ds), st);
  if (e != cudaSuccess) return cuda_fail(e, "status clear");
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  if (n_nonfinite) *n_nonfinite = ds.nonfinite;
  if (ds.flags & kStatusGuard)
    return fail(MUON_ERR_DEVICE, "a device range check found an index out of range and skipped the access "
                "(status 0x%x)", ds.flags);
  if (ds.flags) return fail(MUON_ERR_DEVICE, "a kernel gave up a bounded wait (status 0x%x)", ds.flags);
  if (ds.nonfinite) return MUON_WARN_NONFINITE;
  return MUON_OK;
}

muon_status muon_selftest_wait_timeout(muon_plan_t* p, int64_t limit_us, void* stream) {
  if (!p) return fail(MUON_ERR_INVALID, "plan is NULL");
  if (limit_us < 1 || limit_us > 1000000) return fail(MUON_ERR_INVALID, "limit_us must be in [1, 1000000]");
  if (!p->ws) return fail(MUON_ERR_NO_WORKSPACE, "no workspace bound");
  cudaError_t e = launch_wait_selftest(at<DeviceStatus>(p, p->off_status), (unsigned long long)limit_us * 1000ull,
                                       static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "self-test launch");
  return MUON_OK;
}

muon_status muon_get_stats(const muon_plan_t* p, muon_stats* out) {
  if (!p || !out) return fail(MUON_ERR_INVALID, "NULL argument");
  std::memset(out, 0, sizeof(*out));
  if (!p->cfg.timing) return fail(MUON_ERR_INVALID, "plan was made with timing = 0");
  if (!p->step_end) return fail(MUON_ERR_NO_WORKSPACE, "no workspace bound");
  cudaError_t e = cudaEventSynchronize(p->step_end);
  if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
  for (size_t i = 0; i < p->buckets.size(); ++i) {
    const BucketEvents& ev = p->events[i];
    if (p->offload_last) {
      out->h2d_ms += elapsed(ev.start, ev.h2d);
      out->ns_ms += elapsed(ev.prep, ev.ns);
      out->apply_ms += elapsed(ev.ns, ev.apply);
      out->d2h_ms += elapsed(ev.d2h_start, ev.d2h);
    } else {
      out->prep_ms += elapsed(ev.start, ev.prep);
      out->ns_ms += elapsed(ev.prep, ev.ns);
      out->apply_ms += elapsed(ev.ns, ev.apply);
    }
  }
  out->step_ms = elapsed(p->step_start, p->step_end);
  out->h2d_bytes = p->last_h2d_bytes;
  out->d2h_bytes = p->last_d2h_bytes;
  out->n_buckets = (int64_t)p->buckets.size();
  return MUON_OK;
}

muon_status muon_get_bucket_stats(const muon_plan_t* p, int64_t b, muon_bucket_stats* out) {
  if (!p || !out) return fail(MUON_ERR_INVALID, "NULL argument");
  if (b < 0 || b >= (int64_t)p->buckets.size()) return fail(MUON_ERR_INVALID, "bucket index out of range");
  std::memset(out, 0, sizeof(*out));
  const Bucket& k = p->buckets[b];
  out->n_matrices = k.n_mats;
  out->n_groups = (int64_t)k.groups.size();
  out->m = k.groups[0].m;
  out->n = k.groups[0].n;
  out->bytes = k.bytes;
  out->ns_workspace_bytes = (int64_t)k.ns_bytes;
  out->h2d_bytes = p->bucket_h2d_bytes[b];
  out->d2h_bytes = p->bucket_d2h_bytes[b];
  if (!p->cfg.timing) return MUON_OK;
  if (!p->step_end) return fail(MUON_ERR_NO_WORKSPACE, "no workspace bound");
  cudaError_t e = cudaEventSynchronize(p->step_end);
  if (e != cudaSuccess) return cuda_fail(e, "cudaEventSynchronize");
  const BucketEvents& ev = p->events[b];
  if (p->offload_last) {
    out->h2d_ms = elapsed(ev.start, ev.h2d);
    out->ns_ms = elapsed(ev.prep, ev.ns);
    out->apply_ms = elapsed(ev.ns, ev.apply);
    out->d2h_ms = elapsed(ev.d2h_start, ev.d2h);
  } else {
    out->prep_ms = elapsed(ev.start, ev.prep);
    out->ns_ms = elapsed(ev.prep, ev.ns);
    out->apply_ms = elapsed(ev.ns, ev.apply);
  }
  return MUON_OK;
}

muon_status muon_get_input_norms(const muon_plan_t* p, float* out, int64_t n, void* stream) {
  if (!p || !out) return fail(MUON_ERR_INVALID, "NULL argument");
  if (n != p->n_matrices) return fail(MUON_ERR_INVALID, "n %lld != %lld matrices in the plan", (long long)n,
                                      (long long)p->n_matrices);
  if (!p->ws) return fail(MUON_ERR_NO_WORKSPACE, "no workspace bound");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(out, p->ws + p->off_norms, (size_t)n * sizeof(float), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "norm read");
  return MUON_OK;
}

const char* muon_status_string(muon_status s) {
  switch (s) {
    case MUON_OK: return "ok";
    case MUON_WARN_NONFINITE: return "warning: non-finite matrix norm";
    case MUON_ERR_INVALID: return "invalid argument";
    case MUON_ERR_NOT_PINNED: return "host buffer is not page-locked";
    case MUON_ERR_NO_WORKSPACE: return "no or too small workspace";
    case MUON_ERR_CUDA: return "CUDA error";
    case MUON_ERR_TIMEOUT: return "timed out";
    case MUON_ERR_UNSUPPORTED: return "unsupported";
    case MUON_ERR_DEVICE: return "device-side bounded wait ran out";
    default: return "unknown status";
  }
}

void muon_plan_destroy(muon_plan_t* p) {
  if (!p) return;
  if (p->h2d_stream) {
    for (BucketEvents& ev : p->events) {
      cudaEvent_t all[] = {ev.start, ev.prep, ev.ns, ev.apply, ev.h2d, ev.d2h_start, ev.d2h};
      for (cudaEvent_t x : all)
        if (x) cudaEventDestroy(x);
    }
    for (auto v : {&p->slot_h2d, &p->slot_comp, &p->slot_d2h})
      for (cudaEvent_t x : *v)
        if (x) cudaEventDestroy(x);
    if (p->step_start) cudaEventDestroy(p->step_start);
    if (p->step_end) cudaEventDestroy(p->step_end);
    if (p->offload_done) cudaEventDestroy(p->offload_done);
    cudaStreamDestroy(p->h2d_stream);
    cudaStreamDestroy(p->d2h_stream);
  }
  delete p;
}

}  // extern "C"

// muon_step_noalloc: the Muon step for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc or any allocating library routine: code
// that runs inside a host-side allocator or memory-pool callback, a runtime that
// has handed all device memory to its own pool before the optimizer is created,
// or a plugin environment that forbids device allocations.  For them this entry
// point runs muon_step with its workspace taken from a fixed, file-scope device
// array that the library owns (kScratchBytes below), instead of a caller-bound
// workspace.  Every GPU that loads the library holds that array until the
// process exits.
//
// Set-up: the first call on a device (with that device current) looks up the
// array's device address with cudaGetSymbolAddress and caches it; make that
// first call before any stream capture.
//
// Binding: the array remembers, per device, which plan it was last bound to.  A
// call with that same plan binds nothing and goes straight to muon_step.  A call
// with another plan re-binds: its tensor maps are encoded on the host and its
// tile schedules are copied into the array on the caller's `stream`, so the copy
// lands after the work already enqueued there (it may block the host while the
// driver stages it from pageable memory).  The device status word at the start of
// the array is zero when the library loads and is never cleared here: it is
// shared by every plan that runs in the array and keeps counting (non-finite
// matrices, bounded waits that ran out) until muon_sync on any of those plans
// reads and clears it.
//
// All calls share the one array and it keeps the last call's contents, so calls
// whose device work overlaps race on it: enqueue them on one stream, or make each
// call's stream wait for the previous call's work.
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"
#include "muon.h"

namespace {

constexpr size_t kScratchBytes = 64ull << 20;  // 64 MiB

__device__ __align__(256) unsigned char g_muon_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
struct DeviceScratch {
  void* ptr = nullptr;    // device address of g_muon_scratch on this device
  uint64_t owner = 0;     // id of the plan last bound to it (0: none)
};
DeviceScratch g_scratch[kMaxDevices];
std::mutex g_scratch_mu;

}  // namespace

extern "C" {

size_t muon_noalloc_scratch_bytes(void) { return kScratchBytes; }

muon_status muon_step_noalloc(muon_plan_t* plan, void* const* params, const void* const* grads,
                              void* const* momentum, int64_t n_mats, float lr, float mu, int32_t nesterov,
                              float wd, int32_t ns_steps, void* stream) {
  if (!plan) return muon::set_error(MUON_ERR_INVALID, "plan is NULL");
  size_t need = 0;
  muon_status s = muon_plan_workspace_bytes(plan, &need);
  if (s != MUON_OK) return s;
  if (need > kScratchBytes)
    return muon::set_error(MUON_ERR_NO_WORKSPACE,
                           "muon_step_noalloc: the plan needs more workspace than the 64 MiB static scratch");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return muon::set_error(MUON_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return muon::set_error(MUON_ERR_UNSUPPORTED, "device ordinal out of range");
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    DeviceScratch& d = g_scratch[dev];
    if (d.ptr == nullptr) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_muon_scratch);
      if (e != cudaSuccess || p == nullptr)
        return muon::set_error(MUON_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");
      d.ptr = p;
    }
    const bool bound = d.owner == muon::plan_id(plan) && muon::plan_workspace(plan) == d.ptr;
    if (!bound) {
      d.owner = 0;
      s = muon::bind_shared_scratch(plan, d.ptr, kScratchBytes, static_cast<cudaStream_t>(stream));
      if (s != MUON_OK) return s;
      d.owner = muon::plan_id(plan);
    }
  }
  return muon_step(plan, params, grads, momentum, n_mats, lr, mu, nesterov, wd, ns_steps, stream);
}

}  // extern "C"

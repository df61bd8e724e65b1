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
// first call before any stream capture.  Each call then binds the plan to the
// array (encoding its tensor maps and clearing the device status word, which
// must start at zero) and enqueues muon_step.  All calls share the one array and
// it keeps the last call's contents: calls whose work overlaps on the GPU race
// on it, so serialise them (one stream, or wait between calls).
#include <cuda_runtime.h>

#include <mutex>

#include "kernels.h"
#include "muon.h"

namespace {

constexpr size_t kScratchBytes = 64ull << 20;  // 64 MiB

__device__ __align__(256) unsigned char g_muon_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
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
  void* ptr = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_muon_scratch);
      if (e != cudaSuccess || p == nullptr)
        return muon::set_error(MUON_ERR_CUDA, "cudaGetSymbolAddress of the static scratch failed");
      g_scratch_ptr[dev] = p;
    }
    ptr = g_scratch_ptr[dev];
  }
  s = muon_plan_bind_workspace(plan, ptr, kScratchBytes);
  if (s != MUON_OK) return s;
  return muon_step(plan, params, grads, momentum, n_mats, lr, mu, nesterov, wd, ns_steps, stream);
}

}  // extern "C"

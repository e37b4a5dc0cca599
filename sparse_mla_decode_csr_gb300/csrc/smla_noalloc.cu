// smla_decode_noalloc: smla_decode with its split-KV workspace in a fixed
// device array of this library rather than in caller memory.  It serves
// callers that may not allocate device memory at call time (a serving loop
// inside another runtime's memory pool, a hot path where a cudaMalloc would
// synchronise or stall other work).  Nothing here allocates: the array is
// static storage of the library's module, found once per device with
// cudaGetSymbolAddress, and the decode itself goes through smla_decode.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "smla.h"
#include "smla_internal.h"

namespace {

// The scratch every smla_decode_noalloc call on a device shares.
static __device__ __align__(256) unsigned char g_noalloc_scratch[SMLA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_address[kMaxDevices];  // device address of g_noalloc_scratch, per device

// Device address of the scratch array on the current device; looked up on
// the first call for that device (the host-side name of a __device__ array is
// not a device address).
int scratch_on_current_device(void** address) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SMLA_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_address[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // the failed lookup is reported through the status
      return SMLA_ERR_DEVICE;
    }
    g_scratch_address[dev] = p;
  }
  *address = g_scratch_address[dev];
  return SMLA_OK;
}

}  // namespace

extern "C" int smla_decode_noalloc(const smla_decode_params* params, void* stream) {
  // every argument check runs before anything is enqueued (the ticket clear below included)
  int rc = smla::check_decode_params(params);
  if (rc != SMLA_OK) return rc;
  if (params->n_q == 0) return SMLA_OK;
  rc = smla_device_check();
  if (rc != SMLA_OK) return rc;
  smla_plan_info plan{};
  rc = smla_plan(params, 0, &plan);
  if (rc != SMLA_OK) return rc;
  if (plan.workspace_bytes < 0 || uint64_t(plan.workspace_bytes) > SMLA_NOALLOC_SCRATCH_BYTES)
    return SMLA_ERR_WORKSPACE;
  void* scratch = nullptr;
  rc = scratch_on_current_device(&scratch);
  if (rc != SMLA_OK) return rc;
  if ((plan.kernel == SMLA_KERNEL_CUDA_CORE || plan.kernel == SMLA_KERNEL_TENSOR_CORE_FP8) &&
      plan.workspace_bytes > 0) {
    // per-row ticket counters at the start of the workspace must start at zero
    if (cudaMemsetAsync(scratch, 0, size_t(params->n_q) * 2 * sizeof(int32_t),
                        static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return SMLA_ERR_LAUNCH;
  }
  return smla_decode(params, scratch, SMLA_NOALLOC_SCRATCH_BYTES, stream);
}

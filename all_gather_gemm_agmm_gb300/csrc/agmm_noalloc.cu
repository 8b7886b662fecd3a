// agmm_noalloc.cu -- an allocation-free variant of the unfused path.
//
// Some callers cannot allocate device memory at the point where they run the
// all-gather matmul: code under a framework allocator that has reserved the
// device's memory for itself (an outside cudaMalloc can fail or fragment that
// pool), and latency-critical loops where cudaMalloc's and cudaFree's
// implicit device synchronisation is unacceptable.  agmm_run_unfused_noalloc
// serves them: its scratch (status words, the gathered [P*m_per_device, k]
// buffer and the split-tail counters and partials) lives in one file-scope
// device array of AGMM_STATIC_SCRATCH_BYTES, which every GPU that loads this
// library holds until the process exits.  The array's device address is
// looked up once per device and kept; a device reset invalidates it.
#include <cuda_runtime.h>

#include <mutex>

#include "agmm.h"
#include "kernel_params.h"

struct agmm_plan_s;

namespace agmm {
agmm_status_t set_last_error(agmm_status_t status, const char* message);
agmm_status_t run_unfused_on_scratch(agmm_plan_s* plan, const void* const* x_shards, const void* y, void* o,
                                     int my_id, void* scratch, size_t scratch_bytes, cudaStream_t s);
}  // namespace agmm

namespace {

static __device__ __align__(256) unsigned char g_agmm_static_scratch[AGMM_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the static scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address comes from
// cudaGetSymbolAddress, once per device, with that device current.
agmm_status_t scratch_on_current_device(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return agmm::set_last_error(AGMM_ERR_CUDA, cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return agmm::set_last_error(AGMM_ERR_UNSUPPORTED, "device ordinal too large");
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_agmm_static_scratch);
    if (e != cudaSuccess || p == nullptr)
      return agmm::set_last_error(AGMM_ERR_CUDA, e != cudaSuccess ? cudaGetErrorString(e)
                                                                  : "static scratch has no device address");
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return AGMM_OK;
}

}  // namespace

extern "C" agmm_status_t agmm_run_unfused_noalloc(agmm_plan_t plan, const void* const* x_shards, const void* y,
                                                  void* o, int my_id, void* stream) {
  if (!plan) return agmm::set_last_error(AGMM_ERR_INVALID_ARG, "plan is NULL");
  void* scratch = nullptr;
  agmm_status_t st = scratch_on_current_device(&scratch);
  if (st != AGMM_OK) return st;
  return agmm::run_unfused_on_scratch(plan, x_shards, y, o, my_id, scratch, AGMM_STATIC_SCRATCH_BYTES,
                                      static_cast<cudaStream_t>(stream));
}

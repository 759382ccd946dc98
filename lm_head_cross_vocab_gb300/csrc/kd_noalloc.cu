// Forward entry point for callers that have no way to allocate device memory.
//
// kd_fwd needs scratch space (the split-vocabulary partial records, a label
// count, per-token buffers for outputs the caller skips) and normally takes it
// from a caller-provided workspace.  Some callers cannot provide one: a host
// program that embeds this library as a plugin but owns every device buffer
// itself and hands out only the tensors of the step, or a runtime that must
// not call cudaMalloc while it runs (cudaMalloc can synchronise the device and
// can fail half way through a step).  kd_fwd_static_scratch serves them from
// a fixed array that lives in the library's own device image.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/kd.h"

namespace {

constexpr size_t kScratchBytes = KD_STATIC_SCRATCH_BYTES;

// The scratch itself: every GPU that loads the library holds it until exit.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_scratch on the current device.  In host code the name
// g_scratch is only a host-side stand-in, so the address is looked up once per
// device (with that device current) and cached.
kd_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KD_ERR_NO_DEVICE;
  if (!kd_device_supported(dev)) return KD_ERR_NO_DEVICE;
  if (dev < 0 || dev >= kMaxDevices) return KD_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) return KD_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return KD_OK;
}

}  // namespace

extern "C" kd_status kd_fwd_static_scratch(const kd_problem* problem, const kd_inputs* inputs,
                                           float* ce_s, float* ce_t, float* kl, float* stats,
                                           float* loss, uint32_t* dev_status, void* stream) {
  size_t need = 0;
  kd_status st = kd_workspace_size(problem, &need, nullptr);
  if (st != KD_OK) return st;
  if (need > kScratchBytes) return KD_ERR_WORKSPACE;  // problem too large for the fixed array
  void* scratch = nullptr;
  st = scratch_address(&scratch);
  if (st != KD_OK) return st;
  // kd_fwd clears the part of the scratch that must start at zero (the label
  // count) on the stream before any kernel reads it; everything else it writes
  // before reading.
  return kd_fwd(problem, inputs, ce_s, ce_t, kl, stats, loss, dev_status, scratch, kScratchBytes,
                stream);
}

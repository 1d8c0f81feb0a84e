// Allocation-free variant of the backward path: the same kernels as fabwd_preprocess +
// fabwd_run, with their scratch (workspace) in a fixed-size array that this library owns in
// device memory instead of a caller-provided buffer.
//
// Why it exists: some callers cannot call cudaMalloc at the point where they run the backward.
// Examples are code running under a host framework that owns every byte of device memory
// through its own pool (a foreign cudaMalloc there can fail or fragment the pool), and
// latency-critical loops whose rules forbid any allocation after start-up.  They still own and
// pass the inputs and outputs; only the scratch moves into the library.
#include "../../include/fabwd.h"
#include "fabwd_internal.cuh"

#include <cuda_runtime.h>

#include <mutex>

namespace {

constexpr size_t kStaticWorkspaceBytes = FABWD_STATIC_WORKSPACE_BYTES;  // per GPU that loads the library

// The scratch itself.  Host code must not pass this name to a kernel: on the host it is only a
// stand-in symbol, so its device address is looked up with cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_workspace[kStaticWorkspaceBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_address[kMaxDevices] = {};

// Device address of g_static_workspace on the current device, looked up once per device.
fabwd_status static_workspace_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FABWD_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_address[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_workspace) != cudaSuccess || !ptr) return FABWD_ERR_CUDA;
    g_address[dev] = ptr;
  }
  *out = g_address[dev];
  return FABWD_OK;
}

}  // namespace

extern "C" fabwd_status fabwd_run_static_workspace(const fabwd_params* p, void* stream) {
  size_t need = 0;
  fabwd_status s = fabwd_workspace_size(p, &need);
  if (s != FABWD_OK) return s;
  if (need > kStaticWorkspaceBytes) return FABWD_ERR_WORKSPACE;  // problem too large for the fixed scratch
  void* ws = nullptr;
  if ((s = static_workspace_address(&ws)) != FABWD_OK) return s;
  // fabwd_preprocess clears what must start at zero (the dq accumulator and the status word).
  if ((s = fabwd_preprocess(p, ws, kStaticWorkspaceBytes, stream)) != FABWD_OK) return s;
  return fabwd_run(p, ws, kStaticWorkspaceBytes, stream);
}


extern "C" size_t fabwd_static_workspace_capacity(void) { return kStaticWorkspaceBytes; }

extern "C" fabwd_status fabwd_static_workspace_status(void* stream, uint32_t* device_status) {
  if (!device_status) return FABWD_ERR_NULLPTR;
  void* ws = nullptr;
  fabwd_status s = static_workspace_address(&ws);
  if (s != FABWD_OK) return s;
  return fabwd_read_device_status(ws, kStaticWorkspaceBytes, stream, device_status);
}

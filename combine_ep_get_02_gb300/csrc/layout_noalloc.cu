// Dispatch layout for callers that cannot allocate device memory.
//
// Some callers are handed only their input and output buffers and may not
// allocate device memory themselves: plugins of inference engines that own the
// whole device-memory budget, or code on a latency-critical path where
// cudaMalloc (which can synchronise the device, or fail under a fixed memory
// budget) is not allowed. They cannot provide the workspace that
// ep_get_dispatch_layout needs. This entry point runs the same three layout
// kernels with their scratch in a fixed-size array that lives in the library
// itself: every GPU that loads the library holds kNoAllocScratchBytes of it
// until the process exits.
//
// Host code cannot use the array's name as a device address (in host code it
// names a host-side stand-in), so the first call on each device, with that
// device current, looks the address up with cudaGetSymbolAddress and keeps it.
// Make that first call before any stream capture. All calls on a device share
// the one array and see what the previous call left there; the parts that
// must start at zero (the error bits and the scan's arrival counter) are
// cleared on the stream at the start of every call. Two calls whose work
// overlaps on the GPU (different streams, no ordering) race on the array.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr size_t kNoAllocScratchBytes = EP_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_layout_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mutex;  // guards the per-device address cache
void* g_scratch_addr[kMaxDevices] = {};

// Device address of this device's scratch array; looked up once per device.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_layout_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace ep

using namespace ep;

extern "C" int ep_get_dispatch_layout_noalloc(const ep_config_t* cfg, const int64_t* topk_idx,
                                              const ep_layout_t* layout, void* stream) {
  Geometry g;
  int st = make_geometry(cfg, &g);
  if (st != EP_OK) return st;
  const Workspace w = workspace_layout(g);
  if (w.total > kNoAllocScratchBytes) return EP_ERR_WORKSPACE;  // too large for the fixed array
  void* ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return EP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // error bits and arrival counter start at zero on every call
  if (cudaMemsetAsync(ws, 0, 256, s) != cudaSuccess) return EP_ERR_CUDA;
  return ep_get_dispatch_layout(cfg, topk_idx, layout, ws, w.total, stream);
}

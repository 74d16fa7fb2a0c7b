// Dispatch layout for callers that cannot allocate device memory.
//
// Some callers are handed only their input and output buffers and may not
// allocate device memory themselves: plugins of inference engines that own the
// whole device-memory budget, or code on a latency-critical path where
// cudaMalloc (which can synchronise the device, or fail under a fixed memory
// budget) is not allowed. They cannot provide the workspace that
// ep_get_dispatch_layout needs. This entry point runs the same layout (the
// cluster kernel, plus the two expanded-layout kernels when expanding) with its
// scratch in a fixed-size array that lives in the library itself: every GPU
// that loads the library holds kNoAllocScratchBytes of it until the process
// exits.
//
// Host code cannot use the array's name as a device address (in host code it
// names a host-side stand-in), so the first call in each CUDA context, with
// that context current, looks the address up with cudaGetSymbolAddress and
// keeps it together with the context's ID; a later call in another context
// (after a device reset, say) looks it up again. Make the first call before
// any stream capture. All calls on a device share the one array and see what
// the previous call left there; the parts that must start at zero (the error
// bits and the scan's arrival counter) are cleared on the stream at the start
// of every call, once its arguments have been checked. Two calls whose work
// overlaps on the GPU (different streams, no ordering) race on the array.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr size_t kNoAllocScratchBytes = EP_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_layout_scratch[kNoAllocScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct Cached {
  unsigned long long ctx_id;  // context the address belongs to (0: none yet)
  void* addr;
};

std::mutex g_scratch_mutex;  // guards the driver entry points and the cache
Cached g_scratch[kMaxDevices] = {};
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// ID of the current context (unique for the life of the process), 0 if there
// is none or the driver cannot say. Caller holds g_scratch_mutex.
unsigned long long current_context_id() {
  if (g_ctx_get_current == nullptr || g_ctx_get_id == nullptr) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return 0;
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return 0;
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f);
  }
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array in the current context; looked up once
// per context.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  Cached& c = g_scratch[dev];
  const unsigned long long id = current_context_id();
  if (c.addr == nullptr || id == 0 || id != c.ctx_id) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_layout_scratch);  // makes the device's context current if needed
    if (err != cudaSuccess) return err;
    c.addr = p;
    c.ctx_id = current_context_id();
  }
  *out = c.addr;
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
  // refuse bad arguments before anything touches the shared array
  if ((st = check_layout_args(g, topk_idx, layout)) != EP_OK) return st;
  void* ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return EP_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // error bits and arrival counter start at zero on every call
  if (cudaMemsetAsync(ws, 0, 256, s) != cudaSuccess) return EP_ERR_CUDA;
  return ep_get_dispatch_layout(cfg, topk_idx, layout, ws, w.total, stream);
}

extern "C" int ep_check_error_noalloc(void* stream) {
  void* ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) return EP_ERR_CUDA;
  return ep_check_error(ws, stream);
}

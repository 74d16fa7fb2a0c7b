// Diagnostic for the bounded waits of the bulk-copy dispatch: one warp runs the
// dispatch's abort sequence on purpose. It starts a real bulk load (so a copy
// is in flight), waits with a small limit on a second mbarrier that nothing
// ever completes, gives up, drains the load with the normal limit, and latches
// kErrTimeout in the workspace, the way the dispatch does when one of its waits
// runs out. The host then reads EP_ERR_TIMEOUT from ep_check_error and the
// context stays usable.
#include "ep_device.cuh"
#include "ep_get.h"
#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr int kWaitProbeBytes = 4096;

__global__ void __launch_bounds__(32) wait_timeout_kernel(const uint8_t* __restrict__ src, int bytes,
                                                          uint32_t rounds, uint32_t* err) {
  __shared__ __align__(128) uint8_t stage[kWaitProbeBytes];
  __shared__ __align__(8) uint64_t bar[2];  // 0: never completed, 1: the real load
  if (threadIdx.x != 0) return;
  const uint32_t never = smem_addr(&bar[0]), loaded = smem_addr(&bar[1]);
  mbar_init(never);
  mbar_init(loaded);
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  const bool in_flight = src != nullptr && bytes > 0;
  if (in_flight) bulk_load(smem_addr(stage), src, static_cast<uint32_t>(bytes), loaded);
  bool ok = mbar_wait(never, 0u, rounds);  // nobody arrives: gives up after `rounds`
  // as the dispatch: never leave with a load still writing shared memory
  if (in_flight && !mbar_wait(loaded, 0u, kBulkWaitLimit)) ok = false;
  bulk_wait_all();
  if (!ok) atomicOr(err, kErrTimeout);
}

}  // namespace
}  // namespace ep

extern "C" int ep_diag_wait_timeout(void* workspace, const void* src, int32_t bytes, uint32_t rounds,
                                    void* stream) {
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return EP_ERR_WORKSPACE;
  if (bytes < 0 || bytes > ep::kWaitProbeBytes || bytes % 16 != 0 || rounds > (1u << 20) ||
      (bytes > 0 && (src == nullptr || (reinterpret_cast<uintptr_t>(src) & 15) != 0)))
    return EP_ERR_INVALID_ARG;
  // the device error word sits at offset 0 of the workspace header
  ep::wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint8_t*>(src), bytes, rounds, static_cast<uint32_t*>(workspace));
  return cudaGetLastError() == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

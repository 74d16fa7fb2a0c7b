// Diagnostic row copy with fan-out: every source row is read once and written to
// a run of consecutive destination rows, the run lengths following a rational
// fan-out num/den. Reads and writes are both sequential streams, so at the byte
// counts and read:write ratio of a dispatch this copy is the ceiling a
// one-read, many-write scatter can reach on this memory system. Two methods, the
// two the dispatch uses: 16-byte register loads and stores (one warp per row,
// four chunks in flight per lane), or bulk copies through shared memory (one
// lane of a warp loads the row into a stage and stores it to each destination
// row; two stages per warp, one CTA of four warps per SM).
#include "ep_get.h"
#include "ep_device.cuh"
#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr int kFanThreads = 256;
constexpr int kFanWarps = kFanThreads / 32;
constexpr int kFanUnroll = 4;

__global__ void __launch_bounds__(kFanThreads)
    fanout_copy_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t rows,
                       int chunks, int64_t num, int64_t den) {
  const int lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kFanWarps;
  const size_t row_bytes = static_cast<size_t>(chunks) * 16;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * kFanWarps + (threadIdx.x >> 5); r < rows;
       r += nwarps) {
    // row r fills destination rows [floor(r*num/den), floor((r+1)*num/den))
    const int64_t first = r * num / den, last = (r + 1) * num / den;
    const uint8_t* s = src + static_cast<size_t>(r) * row_bytes;
    for (int c0 = 0; c0 < chunks; c0 += 32 * kFanUnroll) {
      uint4 v[kFanUnroll];
#pragma unroll
      for (int u = 0; u < kFanUnroll; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < chunks) v[u] = ld_stream16(s + static_cast<size_t>(c) * 16);
      }
      for (int64_t d = first; d < last; ++d) {
        uint8_t* o = dst + static_cast<size_t>(d) * row_bytes;
#pragma unroll
        for (int u = 0; u < kFanUnroll; ++u) {
          const int c = c0 + u * 32 + lane;
          if (c < chunks) st16(o + static_cast<size_t>(c) * 16, v[u]);
        }
      }
    }
  }
}

constexpr int kFanBulkWarps = 4;
constexpr int kFanBulkStageMax = 16384;  // rows up to this many bytes

__global__ void __launch_bounds__(kFanBulkWarps * 32)
    fanout_bulk_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int64_t rows, int row_bytes,
                       int64_t num, int64_t den) {
  extern __shared__ __align__(128) uint8_t stage_mem[];
  __shared__ __align__(8) uint64_t bar[kFanBulkWarps][2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gwarp = static_cast<int64_t>(blockIdx.x) * kFanBulkWarps + warp;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kFanBulkWarps;
  const uint32_t st0 = smem_addr(stage_mem + static_cast<size_t>(warp) * 2 * row_bytes);
  const uint32_t bar0 = smem_addr(&bar[warp][0]);
  auto st_addr = [&](int s) { return st0 + static_cast<uint32_t>(s * row_bytes); };
  auto bar_addr = [&](int s) { return bar0 + static_cast<uint32_t>(s * sizeof(uint64_t)); };
  if (lane == 0) {
    mbar_init(bar_addr(0));
    mbar_init(bar_addr(1));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  uint32_t parity = 0, pending = 0;
  auto load_row = [&](int64_t r, int s) {
    if (lane == 0) {
      bulk_wait_reads();  // the stores that last read stage s are done with it
      bulk_load(st_addr(s), src + static_cast<size_t>(r) * row_bytes, static_cast<uint32_t>(row_bytes),
                bar_addr(s));
    }
    pending |= 1u << s;
  };
  int stage = 0;
  if (gwarp < rows) load_row(gwarp, 0);
  for (int64_t r = gwarp; r < rows; r += nwarps) {
    if (r + nwarps < rows) load_row(r + nwarps, stage ^ 1);
    int landed = 1;
    if (lane == 0) landed = mbar_wait(bar_addr(stage), (parity >> stage) & 1u, kBulkWaitLimit);
    if (!__shfl_sync(kFullMask, landed, 0)) break;
    parity ^= 1u << stage;
    pending &= ~(1u << stage);
    if (lane == 0) {
      for (int64_t d = r * num / den; d < (r + 1) * num / den; ++d)
        bulk_store(dst + static_cast<size_t>(d) * row_bytes, st_addr(stage), static_cast<uint32_t>(row_bytes));
      bulk_commit();
    }
    stage ^= 1;
  }
  if (lane == 0) {
    // never leave with a load still writing this warp's stages; a wait that gives
    // up (never seen) leaves dst incomplete, which the caller sees in the data
    for (int s = 0; s < 2; ++s)
      if ((pending >> s) & 1u) (void)mbar_wait(bar_addr(s), (parity >> s) & 1u, kBulkWaitLimit);
    bulk_wait_all();
  }
}

}  // namespace
}  // namespace ep

extern "C" int ep_diag_copy_fanout(const void* src, void* dst, int64_t rows, int32_t row_bytes,
                                   int32_t fan_num, int32_t fan_den, int32_t num_sms, int32_t method,
                                   void* stream) {
  if (rows < 0 || rows > (int64_t{1} << 40) || row_bytes <= 0 || row_bytes % 16 != 0 || fan_num < 0 ||
      fan_num > (1 << 20) || fan_den < 1 || num_sms < 0 || (method != 0 && method != 1))
    return EP_ERR_INVALID_ARG;
  if (method == 1 && row_bytes > ep::kFanBulkStageMax) return EP_ERR_UNSUPPORTED;
  if (rows == 0 || fan_num == 0) return EP_OK;
  if (src == nullptr || dst == nullptr || (reinterpret_cast<uintptr_t>(src) & 15) != 0 ||
      (reinterpret_cast<uintptr_t>(dst) & 15) != 0)
    return EP_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int sms = num_sms;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return EP_ERR_CUDA;
  }
  if (method == 1) {
    const size_t smem = static_cast<size_t>(ep::kFanBulkWarps) * 2 * row_bytes;
    if (cudaFuncSetAttribute(ep::fanout_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
      return EP_ERR_CUDA;
    int64_t ctas = sms;  // one CTA of four warps per SM, as the dispatch
    const int64_t need = (rows + ep::kFanBulkWarps - 1) / ep::kFanBulkWarps;
    if (ctas > need) ctas = need;
    ep::fanout_bulk_kernel<<<static_cast<unsigned>(ctas), ep::kFanBulkWarps * 32, smem, s>>>(
        static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), rows, row_bytes, fan_num, fan_den);
    return cudaGetLastError() == cudaSuccess ? EP_OK : EP_ERR_CUDA;
  }
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ep::fanout_copy_kernel, ep::kFanThreads, 0) !=
      cudaSuccess)
    return EP_ERR_CUDA;
  int64_t ctas = static_cast<int64_t>(sms) * (per_sm < 1 ? 1 : per_sm);
  const int64_t need = (rows + ep::kFanWarps - 1) / ep::kFanWarps;
  if (ctas > need) ctas = need;
  ep::fanout_copy_kernel<<<static_cast<unsigned>(ctas), ep::kFanThreads, 0, s>>>(
      static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), rows, row_bytes / 16, fan_num,
      fan_den);
  return cudaGetLastError() == cudaSuccess ? EP_OK : EP_ERR_CUDA;
}

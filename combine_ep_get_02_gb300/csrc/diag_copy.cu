// Diagnostic row copy with fan-out: every source row is read once and written to
// a run of consecutive destination rows, the run lengths following a rational
// fan-out num/den. Reads and writes are both sequential streams, so at the byte
// counts and read:write ratio of a dispatch this copy is the ceiling a
// one-read, many-write scatter can reach on this memory system. It uses the
// dispatch's access instructions (16-byte non-allocating loads, 16-byte stores,
// one warp per row, four chunks in flight per lane).
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

}  // namespace
}  // namespace ep

extern "C" int ep_diag_copy_fanout(const void* src, void* dst, int64_t rows, int32_t row_bytes,
                                   int32_t fan_num, int32_t fan_den, int32_t num_sms, void* stream) {
  if (rows < 0 || rows > (int64_t{1} << 40) || row_bytes <= 0 || row_bytes % 16 != 0 || fan_num < 0 ||
      fan_num > (1 << 20) || fan_den < 1 || num_sms < 0)
    return EP_ERR_INVALID_ARG;
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

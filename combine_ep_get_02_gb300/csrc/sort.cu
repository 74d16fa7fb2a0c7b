// The post-hoc deterministic sort of the comparison path.
//
// Before PR #753 the sender took its destination slot with an atomicAdd, so the
// rows of a source inside a destination's receive buffer came in the order the
// warps won the race; EPHandle.deterministic_sort then sorted the received
// tokens by source token and permuted every order-dependent tensor (PR #753,
// Motivation). Here: one CTA per (destination, row block) segment sorts the
// segment's source-token keys with a bitonic sort in shared memory, then its
// warps copy each row and its sidecars to the sorted position of a second
// receive buffer. The rows make one full extra round trip through memory,
// which is the cost the kernel-side slots remove.
#include <climits>

#include "ep_device.cuh"
#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kSortThreads = 512;
constexpr int kSortWarps = kSortThreads / 32;

__global__ void __launch_bounds__(kSortThreads) sort_kernel(SortArgs a) {
  extern __shared__ int32_t sm[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int d = blockIdx.x / a.R, rb = blockIdx.x % a.R;
  const int src = a.n_so == 1 ? rb : (rb % a.n_so) * a.n_su + rb / a.n_so;
  const int n = min(a.send_counters[src * a.R + d], a.M);
  if (n <= 0) return;
  int P = 1;
  while (P < n) P <<= 1;
  int32_t* key = sm;
  int32_t* val = sm + P;
  const int64_t base = static_cast<int64_t>(d) * a.region_rows + static_cast<int64_t>(rb) * a.M;
  const int md_stride = a.K + 2;
  for (int i = tid; i < P; i += kSortThreads) {
    key[i] = i < n ? a.in_md[(base + i) * md_stride + 1] : INT_MAX;  // field 1: source token
    val[i] = i;
  }
  __syncthreads();
  for (int k = 2; k <= P; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < P; i += kSortThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const bool ascending = (i & k) == 0;
          const int ki = key[i], kj = key[ixj];
          if ((ki > kj) == ascending) {
            key[i] = kj;
            key[ixj] = ki;
            const int v = val[i];
            val[i] = val[ixj];
            val[ixj] = v;
          }
        }
      }
      __syncthreads();
    }
  }
  // row i of the sorted segment comes from row val[i] of the received one
  const int nchunk = a.row_bytes >> 4;
  for (int i = warp; i < n; i += kSortWarps) {
    const int64_t from = base + val[i], to = base + i;
    const uint8_t* src_row = a.in_x + from * a.row_bytes;
    uint8_t* dst_row = a.out_x + to * a.row_bytes;
    for (int c0 = 0; c0 < nchunk; c0 += 32 * 4) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < nchunk) v[u] = ld_stream16(src_row + (static_cast<size_t>(c) << 4));
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < nchunk) st16(dst_row + (static_cast<size_t>(c) << 4), v[u]);
      }
    }
    if (a.in_sf != nullptr)
      for (int g = lane; g < a.SW; g += 32) a.out_sf[to * a.SW + g] = a.in_sf[from * a.SW + g];
    if (lane < a.K) {
      a.out_idx[to * a.K + lane] = a.in_idx[from * a.K + lane];
      a.out_w[to * a.K + lane] = a.in_w[from * a.K + lane];
    }
    for (int f = lane; f < md_stride; f += 32) a.out_md[to * md_stride + f] = a.in_md[from * md_stride + f];
  }
}

}  // namespace

cudaError_t launch_sort(const Geometry& g, const SortArgs& a, cudaStream_t stream) {
  int P = 1;
  while (P < g.M) P <<= 1;
  const size_t smem = 2 * sizeof(int32_t) * P;
  cudaError_t err;
  if (smem > 48 * 1024 &&
      (err = cudaFuncSetAttribute(sort_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(smem))) != cudaSuccess)
    return err;
  sort_kernel<<<g.R * g.R, kSortThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace ep

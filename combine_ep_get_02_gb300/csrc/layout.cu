// Dispatch layout: per-block counts, a grid-wide scan, then per-lane slots.
//
// The slot of a (token, destination) entry is the destination row block of its
// source rank times num_max_tokens_per_rank plus the source's running count of
// deduplicated entries to that destination in token order (PR #753, Approach).
// A running count is a prefix sum over tokens, so it is computed as one:
//   1. layout_count_kernel: each CTA takes a block of 256 tokens of one source
//      and counts, per destination and per expert, how many of its tokens go
//      there (warp ballots; one thread per token).
//   2. layout_scan_kernel: one CTA per source turns the block counts into
//      exclusive per-block bases and totals; the last CTA to arrive does the
//      cross-source part (receive counts and their prefix sums, per-expert
//      block starts of the expanded layout).
//   3. layout_slot_kernel: each CTA re-derives its tokens' destination sets and
//      adds the in-block rank (ballot prefix within the warp, then warp prefix
//      within the block) to the block base.
// Every value is a pure function of topk_idx: the three grids and the number
// of CTAs only change who computes what, never the result.
#include "ep_device.cuh"
#include "ep_internal.cuh"

namespace ep {

namespace {

// Row block of source s inside every destination region (R blocks of M rows).
__device__ __forceinline__ int row_block(int s, int n_so, int n_su) {
  return n_so == 1 ? s : (s % n_su) * n_so + s / n_su;
}

// The CTA's tokens' top-k values, staged transposed ([k][token]) as int32:
// -1 masked, -2 out of range (an error), else the expert.
__device__ __forceinline__ void stage_topk(const LayoutArgs& a, int s, int b, int32_t* se) {
  const int t0 = b * kBlockTokens;
  const int nt = min(kBlockTokens, a.T - t0);
  const int64_t base = (static_cast<int64_t>(s) * a.T + t0) * a.K;
  const int n = nt * a.K;
  for (int i = threadIdx.x; i < n; i += kLayoutThreads) {
    const int64_t e = a.topk_idx[base + i];
    const int t = i / a.K, k = i - t * a.K;
    se[k * kBlockTokens + t] = (e >= -1 && e < a.E) ? static_cast<int32_t>(e) : -2;
  }
}

// Destination of lane k of this thread's token, or -1 (masked or invalid).
// In the expanded layout a repeat of an earlier lane's expert is invalid.
__device__ __forceinline__ int lane_dst(const LayoutArgs& a, const int32_t* se, int k, int tid,
                                        bool* bad) {
  const int e = se[k * kBlockTokens + tid];
  if (e < 0) {
    if (e == -2) *bad = true;
    return -1;
  }
  if (a.expand) {
    for (int j = 0; j < k; ++j) {
      if (se[j * kBlockTokens + tid] == e) {
        *bad = true;
        return -1;
      }
    }
  }
  return e / a.L;
}

}  // namespace

// ---- pass 1: per-block counts ----------------------------------------------
__global__ void __launch_bounds__(kLayoutThreads) layout_count_kernel(LayoutArgs a) {
  extern __shared__ int32_t smem[];
  int32_t* se = smem;                              // [K][256]
  int32_t* hist = se + a.K * kBlockTokens;         // [E]
  __shared__ int32_t warp_cnt[kLayoutWarps][kMaxRanks];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int e = tid; e < a.E; e += kLayoutThreads) hist[e] = 0;

  const int units = a.R * a.NB;
  bool bad = false;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int s = u / a.NB, b = u - s * a.NB;
    __syncthreads();  // previous unit done with se / hist / warp_cnt
    stage_topk(a, s, b, se);
    __syncthreads();
    const bool live = b * kBlockTokens + tid < a.T;
    uint64_t dmask = 0;
    if (live) {
      for (int k = 0; k < a.K; ++k) {
        const int d = lane_dst(a, se, k, tid, &bad);
        if (d >= 0) {
          dmask |= 1ull << d;
          atomicAdd(&hist[se[k * kBlockTokens + tid]], 1);
        }
      }
    }
    for (int d = 0; d < a.R; ++d) {
      const unsigned bal = __ballot_sync(kFullMask, (dmask >> d) & 1);
      if (lane == 0) warp_cnt[warp][d] = __popc(bal);
    }
    __syncthreads();
    const int64_t blk = static_cast<int64_t>(s) * a.NB + b;
    for (int d = tid; d < a.R; d += kLayoutThreads) {
      int c = 0;
      for (int w = 0; w < kLayoutWarps; ++w) c += warp_cnt[w][d];
      a.blk_cnt[blk * a.R + d] = c;
    }
    for (int e = tid; e < a.E; e += kLayoutThreads) {
      a.blk_cnt_e[blk * a.E + e] = hist[e];
      hist[e] = 0;
    }
  }
  if (bad) atomicOr(a.err, kErrBadTopk);
}

// ---- grid-wide scan ---------------------------------------------------------
// grid = R CTAs (one per source); the last CTA to finish does the cross-source part.
__global__ void __launch_bounds__(kLayoutThreads) layout_scan_kernel(LayoutArgs a) {
  extern __shared__ int32_t smem[];
  __shared__ bool s_last;
  const int tid = threadIdx.x;
  const int s = blockIdx.x;
  const int R = a.R, NB = a.NB, E = a.E;

  // per destination: exclusive per-block bases (absolute rows in the region) and totals
  const int rb = row_block(s, a.n_so, a.n_su);
  for (int d = tid; d < R; d += kLayoutThreads) {
    int acc = 0;
    for (int b = 0; b < NB; ++b) {
      const int64_t i = (static_cast<int64_t>(s) * NB + b) * R + d;
      const int c = a.blk_cnt[i];
      a.blk_base[i] = rb * a.M + acc;
      acc += c;
    }
    a.num_tokens_per_rank[s * R + d] = acc;
    a.recv_cnt[d * R + s] = acc;
  }
  // per expert: totals, and (expanded) exclusive per-block prefixes within the source
  for (int e = tid; e < E; e += kLayoutThreads) {
    int acc = 0;
    for (int b = 0; b < NB; ++b) {
      const int64_t i = (static_cast<int64_t>(s) * NB + b) * E + e;
      const int c = a.blk_cnt_e[i];
      if (a.expand) a.blk_base_e[i] = acc;
      acc += c;
    }
    a.num_tokens_per_expert[s * E + e] = acc;
  }

  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(a.done, 1u) == static_cast<unsigned>(gridDim.x) - 1u;
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  // receive counts: inclusive prefix over row blocks (block i holds source src(i))
  for (int d = tid; d < R; d += kLayoutThreads) {
    int acc = 0;
    for (int i = 0; i < R; ++i) {
      const int src = a.n_so == 1 ? i : (i % a.n_so) * a.n_su + i / a.n_so;
      acc += ld_cg(a.recv_cnt + d * R + src);
      a.recv_psum[d * R + i] = acc;
    }
  }

  if (a.expand) {
    int32_t* s_blk = smem;         // [E]: block start of expert e inside its region
    int32_t* s_size = smem + E;    // [R]: region sizes
    const int L = a.L;
    for (int e = tid; e < E; e += kLayoutThreads) {
      int n = 0;
      for (int src = 0; src < R; ++src) n += ld_cg(a.num_tokens_per_expert + src * E + e);
      a.exp_cnt[e] = n;
      s_blk[e] = n;
    }
    __syncthreads();
    for (int d = tid; d < R; d += kLayoutThreads) {
      int base = 0;
      for (int j = 0; j < L; ++j) {
        const int n = s_blk[d * L + j];
        a.exp_base[d * (L + 1) + j] = base;
        s_blk[d * L + j] = base;
        base += (n + a.align - 1) / a.align * a.align;
      }
      a.exp_base[d * (L + 1) + L] = base;
      s_size[d] = base;
    }
    __syncthreads();
    if (tid == 0) {
      int acc = 0;
      for (int d = 0; d < R; ++d) {
        a.exp_region[d] = acc;
        acc += s_size[d];
      }
      a.exp_region[R] = acc;
    }
    // per (source, expert, block): block start + earlier sources' lanes + earlier blocks'
    for (int e = tid; e < E; e += kLayoutThreads) {
      int off = s_blk[e];
      for (int src = 0; src < R; ++src) {
        for (int b = 0; b < NB; ++b) {
          const int64_t i = (static_cast<int64_t>(src) * NB + b) * E + e;
          a.blk_base_e[i] = ld_cg(a.blk_base_e + i) + off;
        }
        off += ld_cg(a.num_tokens_per_expert + src * E + e);
      }
    }
  }
  if (tid == 0) *a.done = 0u;  // ready for the next call
}

// ---- pass 2: per-lane slots ---------------------------------------------------
__global__ void __launch_bounds__(kLayoutThreads) layout_slot_kernel(LayoutArgs a) {
  extern __shared__ int32_t smem[];
  int32_t* se = smem;                                                 // [K][256]
  uint32_t* ebits = reinterpret_cast<uint32_t*>(se + a.K * kBlockTokens);  // [8][E] (expand)
  __shared__ uint32_t bal_d[kLayoutWarps][kMaxRanks];
  __shared__ int32_t base_d[kLayoutWarps][kMaxRanks];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const unsigned lt = lanemask_lt();
  if (a.expand)
    for (int i = tid; i < kLayoutWarps * a.E; i += kLayoutThreads) ebits[i] = 0;

  const int units = a.R * a.NB;
  for (int u = blockIdx.x; u < units; u += gridDim.x) {
    const int s = u / a.NB, b = u - s * a.NB;
    __syncthreads();
    stage_topk(a, s, b, se);
    __syncthreads();
    const int t = b * kBlockTokens + tid;
    const bool live = t < a.T;
    bool bad = false;
    uint64_t dmask = 0;
    if (live) {
      for (int k = 0; k < a.K; ++k) {
        const int d = lane_dst(a, se, k, tid, &bad);
        if (d >= 0) {
          dmask |= 1ull << d;
          if (a.expand) atomicOr(&ebits[warp * a.E + se[k * kBlockTokens + tid]], 1u << lane);
        }
      }
    }
    for (int d = 0; d < a.R; ++d) {
      const unsigned bal = __ballot_sync(kFullMask, (dmask >> d) & 1);
      if (lane == 0) bal_d[warp][d] = bal;
    }
    __syncthreads();
    const int64_t blk = static_cast<int64_t>(s) * a.NB + b;
    for (int d = tid; d < a.R; d += kLayoutThreads) {
      int base = a.blk_base[blk * a.R + d];
      for (int w = 0; w < kLayoutWarps; ++w) {
        base_d[w][d] = base;
        base += __popc(bal_d[w][d]);
      }
    }
    __syncthreads();
    if (live) {
      const int64_t tok = static_cast<int64_t>(s) * a.T + t;
      for (int k = 0; k < a.K; ++k) {
        const int d = lane_dst(a, se, k, tid, &bad);
        int slot = -1, pos = -1;
        if (d >= 0) {
          slot = base_d[warp][d] + __popc(bal_d[warp][d] & lt);
          if (a.expand) {
            const int e = se[k * kBlockTokens + tid];
            pos = a.blk_base_e[blk * a.E + e] + __popc(ebits[warp * a.E + e] & lt);
            for (int w = 0; w < warp; ++w) pos += __popc(ebits[w * a.E + e]);
          }
        }
        a.slot_map[tok * a.K + k] = slot;
        if (a.expand) a.exp_pos[tok * a.K + k] = pos;
      }
      uint8_t* row = a.is_token_in_rank + tok * a.R;
      if ((a.R & 3) == 0) {
        for (int d = 0; d < a.R; d += 4) {
          const uint32_t v = static_cast<uint32_t>((dmask >> d) & 1) |
                             static_cast<uint32_t>((dmask >> (d + 1)) & 1) << 8 |
                             static_cast<uint32_t>((dmask >> (d + 2)) & 1) << 16 |
                             static_cast<uint32_t>((dmask >> (d + 3)) & 1) << 24;
          *reinterpret_cast<uint32_t*>(row + d) = v;
        }
      } else {
        for (int d = 0; d < a.R; ++d) row[d] = static_cast<uint8_t>((dmask >> d) & 1);
      }
    }
    if (a.expand) {
      __syncthreads();
      for (int i = tid; i < kLayoutWarps * a.E; i += kLayoutThreads) ebits[i] = 0;
    }
  }
}

cudaError_t launch_layout(const Geometry& g, const LayoutArgs& a, int num_prologue_sms,
                          cudaStream_t stream) {
  const int units = g.R * g.NB;
  int ctas = num_prologue_sms > 0 ? num_prologue_sms : kMaxPrologueCtas;
  ctas = ctas > kMaxPrologueCtas ? kMaxPrologueCtas : ctas;
  ctas = units < ctas ? units : ctas;
  const size_t se_bytes = sizeof(int32_t) * g.K * kBlockTokens;
  const size_t count_smem = se_bytes + sizeof(int32_t) * g.E;
  const size_t slot_smem = se_bytes + (g.expand ? sizeof(uint32_t) * kLayoutWarps * g.E : 0);
  const size_t scan_smem = g.expand ? sizeof(int32_t) * (g.E + g.R) : 0;
  cudaError_t err;
  // only requests above the default 48 KB need the opt-in attribute
  if (count_smem > 48 * 1024 &&
      (err = cudaFuncSetAttribute(layout_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(count_smem))) != cudaSuccess)
    return err;
  if (slot_smem > 48 * 1024 &&
      (err = cudaFuncSetAttribute(layout_slot_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  static_cast<int>(slot_smem))) != cudaSuccess)
    return err;
  if (ctas > 0) {
    layout_count_kernel<<<ctas, kLayoutThreads, count_smem, stream>>>(a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  layout_scan_kernel<<<g.R, kLayoutThreads, scan_smem, stream>>>(a);
  if ((err = cudaGetLastError()) != cudaSuccess) return err;
  if (ctas > 0) {
    layout_slot_kernel<<<ctas, kLayoutThreads, slot_smem, stream>>>(a);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
  }
  return cudaSuccess;
}

}  // namespace ep

// Dispatch layout: per-warp counts, a scan across the CTAs of each source rank,
// then per-lane slots.
//
// The slot of a (token, destination) entry is the row block of its source rank
// times num_max_tokens_per_rank plus the source's running count of
// deduplicated entries to that destination in token order (PR #753,
// Approach). A row block belongs to one source only, so the running count is a
// prefix sum over that source's own tokens: no information crosses sources.
//
// layout_kernel: one thread-block cluster per source rank (up to 8 CTAs, each a
// contiguous range of the source's tokens, one thread per token per round):
//   pass 1  each warp counts, per destination, the tokens that reach it
//           (ballot + popc), and each CTA counts its lanes per expert;
//   scan    after a cluster barrier every CTA adds up the counts of the CTAs
//           before it through distributed shared memory: its base per
//           destination (and, expanded, per expert);
//   pass 2  warp prefix of the ballots plus the running base gives each lane's
//           slot; the expanded layout ranks a lane among its expert's lanes with
//           per-warp bitmaps of the tokens (source-local position).
// layout_rows_kernel computes the same for top-k <= 8 (row form, and the
// expanded positions while their per-(round, warp) tables fit in shared
// memory), with every lane in registers and the counts pushed to the cluster
// peers instead of read from them (its own comment below).
// The last CTA of the grid to finish (a counter in the workspace, no waiting)
// turns the receive counts into their prefix sums, and the destinations'
// totals into the first packed row of each destination.
// Expanded layout only, two more kernels: layout_expert_scan_kernel scans the
// per-source expert counts down each expert's column (cross-source offsets and
// per-expert totals); layout_expand_kernel derives the block starts and region
// offsets and moves every source-local position to its final row.
// Every value is a pure function of topk_idx; the grid shape only changes who
// computes what.
#include <cooperative_groups.h>

#include "ep_device.cuh"
#include "ep_internal.cuh"

namespace cg = cooperative_groups;

namespace ep {

namespace {

// e / L for 0 <= e, L <= 4096 as a multiply-high by ceil(2^32 / L), exact in
// that range; magic == 0 stands for L == 1.
__device__ __forceinline__ int div_l(int e, uint32_t magic) {
  return magic == 0 ? e : static_cast<int>(__umulhi(static_cast<uint32_t>(e), magic));
}

__device__ __forceinline__ bool aligned16(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15) == 0;
}

// 32x32 bit-matrix transpose across a warp: on entry lane i holds row i (bit c
// of x is M[i][c]); on exit lane c holds column c (bit i is M[i][c]), i.e. what
// __ballot_sync would return for predicate "bit c of my row" -- for all 32
// columns with five exchanges instead of 32 ballots. Each step swaps the
// off-diagonal blocks of every 2j x 2j block: the upper lane keeps its left
// columns and takes its partner's left columns, the lower lane the right ones.
__device__ __forceinline__ uint32_t warp_transpose32(uint32_t x, int lane) {
  constexpr uint32_t kLeft[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    const int j = 16 >> step;
    const uint32_t m = kLeft[step];
    const uint32_t y = __shfl_xor_sync(kFullMask, x, j);
    x = (lane & j) ? ((x & ~m) | ((y & ~m) >> j)) : ((x & m) | ((y & m) << j));
  }
  return x;
}

// Row block of source s inside every destination region (R blocks of M rows).
__device__ __forceinline__ int row_block(int s, int n_so, int n_su) {
  return n_so == 1 ? s : (s % n_su) * n_so + s / n_su;
}

// One token's top-k entries as stored (int64), read with 16-byte loads when the
// rows allow it; nothing is read for a token past the end.
template <int KMAX>
__device__ __forceinline__ void load_lanes(const LayoutArgs& a, int64_t tok, bool live, int64_t (&v)[KMAX]) {
  const int64_t* p = a.topk_idx + tok * a.K;
#pragma unroll
  for (int k = 0; k < KMAX; ++k) v[k] = -1;
  if (live && a.topk_vec) {
#pragma unroll
    for (int k = 0; k < KMAX; k += 2) {
      if (k < a.K) {
        const longlong2 q = __ldg(reinterpret_cast<const longlong2*>(p + k));
        v[k] = q.x;
        v[k + 1] = q.y;
      }
    }
  } else if (live) {
#pragma unroll
    for (int k = 0; k < KMAX; ++k)
      if (k < a.K) v[k] = __ldg(p + k);
  }
}

// One token's top-k lanes in registers: expert per lane, -1 when masked or
// invalid. Values outside [-1, E) are errors; in the expanded layout so is a
// repeat of an earlier lane's expert. Returns the destination-rank mask.
template <int KMAX>
__device__ __forceinline__ uint64_t decode_lanes(const LayoutArgs& a, const int64_t (&v)[KMAX], bool live,
                                                 int (&e)[KMAX], bool* bad) {
  uint64_t dmask = 0;
#pragma unroll
  for (int k = 0; k < KMAX; ++k) {
    e[k] = -1;
    if (live && k < a.K) {
      const int64_t x = v[k];
      if (x >= 0 && x < a.E) e[k] = static_cast<int>(x);
      else if (x != -1) *bad = true;
    }
  }
  if (a.expand) {
#pragma unroll
    for (int k = 1; k < KMAX; ++k) {
#pragma unroll
      for (int j = 0; j < k; ++j) {
        if (e[k] >= 0 && e[j] == e[k]) {
          e[k] = -1;
          *bad = true;
        }
      }
    }
  }
#pragma unroll
  for (int k = 0; k < KMAX; ++k)
    if (e[k] >= 0) dmask |= 1ull << div_l(e[k], a.l_magic);
  return dmask;
}

template <int KMAX>
__device__ __forceinline__ uint64_t load_token(const LayoutArgs& a, int64_t tok, bool live, int (&e)[KMAX],
                                               bool* bad) {
  int64_t v[KMAX];
  load_lanes<KMAX>(a, tok, live, v);
  return decode_lanes<KMAX>(a, v, live, e, bad);
}

// Count this CTA in: called by one thread after a CTA barrier that follows the
// CTA's writes of the receive counts (recv_cnt, by each source's last CTA). A
// release atomic: it publishes those writes without waiting for its result;
// the result says at the CTA's end whether it was the last to count in.
__device__ __forceinline__ uint32_t count_in(const LayoutArgs& a) { return atomic_add_release(a.done, 1u); }

// The end of every layout CTA: the last CTA to count in (thread 0 holds the
// counter's old value) reads the counter once more with acquire semantics,
// which makes every other CTA's published receive counts visible, turns them
// into their prefix sums over the row blocks and the first packed row of each
// destination, then returns the counter to zero.
template <int THREADS>
__device__ __forceinline__ void finish_receive_sums(const LayoutArgs& a, uint32_t old, int32_t* s_tot,
                                                    bool* s_last) {
  constexpr int WARPS = THREADS / 32;
  constexpr int kDests = (kMaxRanks + WARPS - 1) / WARPS, kChunks = (kMaxRanks + 31) / 32;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = a.R;
  if (tid == 0) {
    const bool last = old == gridDim.x - 1u;
    if (last) ld_acquire(a.done);
    *s_last = last;
  }
  __syncthreads();
  if (!*s_last) return;
  // warp w scans destinations w, w + WARPS, ...: every count it needs is
  // loaded first (row block j holds source src(j)), then one inclusive scan
  // over the row blocks per destination, 32 at a time
  int v[kDests][kChunks];
#pragma unroll
  for (int i = 0; i < kDests; ++i) {
    const int d = warp + i * WARPS;
#pragma unroll
    for (int ch = 0; ch < kChunks; ++ch) {
      const int j = ch * 32 + lane;
      v[i][ch] = 0;
      if (d < R && j < R) {
        const int q = a.so_magic == 0 ? 0 : static_cast<int>(__umulhi(static_cast<uint32_t>(j), a.so_magic));
        const int src = a.n_so == 1 ? j : (j - q * a.n_so) * a.n_su + q;
        v[i][ch] = ld_cg(a.recv_cnt + d * R + src);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kDests; ++i) {
    const int d = warp + i * WARPS;
    if (d >= R) break;
    int carry = 0;
#pragma unroll
    for (int ch = 0; ch < kChunks; ++ch) {
      const int j = ch * 32 + lane;
      int x = v[i][ch];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(kFullMask, x, o);
        if (lane >= o) x += u;
      }
      x += carry;
      if (j < R) a.recv_psum[d * R + j] = x;
      carry = __shfl_sync(kFullMask, x, 31);
    }
    if (lane == 0) s_tot[d] = carry;
  }
  // packed receive rows: destination d starts after everything the
  // destinations before it receive
  if (a.recv_region != nullptr) {
    __syncthreads();
    if (warp == 0) {
      int carry = 0;
      for (int d0 = 0; d0 < R; d0 += 32) {
        const int d = d0 + lane;
        const int n = d < R ? s_tot[d] : 0;
        int x = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int u = __shfl_up_sync(kFullMask, x, o);
          if (lane >= o) x += u;
        }
        if (d < R) a.recv_region[d] = carry + x - n;
        carry += __shfl_sync(kFullMask, x, 31);
      }
      if (lane == 0) a.recv_region[R] = carry;
    }
  }
  if (tid == 0) *a.done = 0u;  // ready for the next call
}

}  // namespace

// dynamic shared memory: cnt_e [E] | run_e [E] (expand) | ebits [WARPS][E] (expand)
template <int KMAX, int THREADS>
__global__ void __launch_bounds__(THREADS) layout_kernel(LayoutArgs a) {
  constexpr int WARPS = THREADS / 32;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ int32_t smem[];
  int32_t* cnt_e = smem;
  int32_t* run_e = cnt_e + a.E;
  uint32_t* ebits = reinterpret_cast<uint32_t*>(run_e + a.E);
  __shared__ int32_t cnt_d[kMaxRanks];
  __shared__ int32_t run_d[kMaxRanks];
  __shared__ uint32_t bal[WARPS][kMaxRanks];
  __shared__ int32_t wbase[WARPS][kMaxRanks];
  __shared__ int32_t s_tot[kMaxRanks];
  __shared__ bool s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const unsigned lt = lanemask_lt();
  const int R = a.R, E = a.E;
  const int s = blockIdx.x / a.C;
  const int c = static_cast<int>(cluster.block_rank());
  const int t_begin = min(a.T, c * a.TB), t_end = min(a.T, t_begin + a.TB);
  const int64_t tok_base = static_cast<int64_t>(s) * a.T;

  pdl_launch_dependents();
  for (int e = tid; e < E; e += THREADS) cnt_e[e] = 0;
  if (a.expand)
    for (int i = tid; i < WARPS * E; i += THREADS) ebits[i] = 0;
  if (tid < R) cnt_d[tid] = 0;
  __syncthreads();
  pdl_wait();

  // ---- pass 1: this CTA's counts per destination and per expert
  bool bad = false;
  // the first round's lanes stay in registers for pass 2 (with up to 8 lanes a
  // token; wider tokens are loaded again)
  constexpr bool kKeep = KMAX <= 8;
  int e_first[kKeep ? KMAX : 1];
  uint64_t dmask_first = 0;
  {
    int e[KMAX];
    int t = t_begin + tid;
    uint64_t dmask = load_token<KMAX>(a, tok_base + t, t < t_end, e, &bad);
    if constexpr (kKeep) {
#pragma unroll
      for (int k = 0; k < KMAX; ++k) e_first[k] = e[k];
      dmask_first = dmask;
    }
    for (int t0 = t_begin; t0 < t_end; t0 += THREADS) {
      // the next round's lanes are in flight while this round is counted
      int en[KMAX];
      const int tn = t + THREADS;
      const uint64_t dn = load_token<KMAX>(a, tok_base + tn, tn < t_end, en, &bad);
#pragma unroll
      for (int k = 0; k < KMAX; ++k)
        if (e[k] >= 0) atomicAdd(&cnt_e[e[k]], 1);
      // lane d: the warp's tokens that reach destination d (and d + 32)
      const uint32_t col_lo = warp_transpose32(static_cast<uint32_t>(dmask), lane);
      if (lane < R && col_lo != 0) atomicAdd(&cnt_d[lane], __popc(col_lo));
      if (R > 32) {
        const uint32_t col_hi = warp_transpose32(static_cast<uint32_t>(dmask >> 32), lane);
        if (lane + 32 < R && col_hi != 0) atomicAdd(&cnt_d[lane + 32], __popc(col_hi));
      }
#pragma unroll
      for (int k = 0; k < KMAX; ++k) e[k] = en[k];
      dmask = dn;
      t = tn;
    }
  }
  if (bad) atomicOr(a.err, kErrBadTopk);
  cluster.sync();

  // ---- scan across the cluster: counts of the CTAs before this one
  const int rb = row_block(s, a.n_so, a.n_su);
  for (int d = tid; d < R; d += THREADS) {
    int base = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q < c) base += cluster.map_shared_rank(cnt_d, q)[d];
    run_d[d] = rb * a.M + base;
    if (c == a.C - 1) {  // the source's totals
      const int total = base + cnt_d[d];
      a.num_tokens_per_rank[s * R + d] = total;
      a.recv_cnt[d * R + s] = total;
    }
  }
  for (int e = tid; e < E; e += THREADS) {
    int base = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q < c) base += cluster.map_shared_rank(cnt_e, q)[e];
    if (a.expand) run_e[e] = base;
    if (c == a.C - 1) a.num_tokens_per_expert[s * E + e] = base + cnt_e[e];
  }
  // other CTAs may still read this CTA's counts: they are left untouched, and
  // the CTA waits for the whole cluster before it exits
  cluster.barrier_arrive();
  __syncthreads();
  uint32_t arrived = 0;
  if (tid == 0) arrived = count_in(a);

  // ---- pass 2: slots (and source-local expanded positions)
  {
    int e[KMAX];
    bool unused = false;
    int t = t_begin + tid;
    uint64_t dmask;
    if constexpr (kKeep) {
#pragma unroll
      for (int k = 0; k < KMAX; ++k) e[k] = e_first[k];
      dmask = dmask_first;
    } else {
      dmask = load_token<KMAX>(a, tok_base + t, t < t_end, e, &unused);
    }
    for (int t0 = t_begin; t0 < t_end; t0 += THREADS) {
      const bool live = t < t_end;
      int en[KMAX];
      const int tn = t + THREADS;
      const uint64_t dn = load_token<KMAX>(a, tok_base + tn, tn < t_end, en, &unused);
      if (a.expand) {
#pragma unroll
        for (int k = 0; k < KMAX; ++k)
          if (e[k] >= 0) atomicOr(&ebits[warp * E + e[k]], 1u << lane);
      }
      // lane d stores the warp's ballot of destination d (and d + 32)
      const uint32_t col_lo = warp_transpose32(static_cast<uint32_t>(dmask), lane);
      if (lane < R) bal[warp][lane] = col_lo;
      if (R > 32) {
        const uint32_t col_hi = warp_transpose32(static_cast<uint32_t>(dmask >> 32), lane);
        if (lane + 32 < R) bal[warp][lane + 32] = col_hi;
      }
      __syncthreads();
      for (int d = tid; d < R; d += THREADS) {
        int r = run_d[d];
#pragma unroll
        for (int w = 0; w < WARPS; ++w) {
          wbase[w][d] = r;
          r += __popc(bal[w][d]);
        }
        run_d[d] = r;
      }
      __syncthreads();
      if (live) {
        const int64_t tok = tok_base + t;
        int slot[KMAX], pos[KMAX];
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
          slot[k] = -1;
          pos[k] = -1;
          if (e[k] >= 0) {
            const int d = div_l(e[k], a.l_magic);
            slot[k] = wbase[warp][d] + __popc(bal[warp][d] & lt);
            // checked builds: the slot stays inside this source's row block
            if (!row_in_bounds(slot[k] - static_cast<int64_t>(rb) * a.M, a.M, a.err)) slot[k] = -1;
            if (a.expand) {
              int p = run_e[e[k]] + __popc(ebits[warp * E + e[k]] & lt);
              for (int w = 0; w < warp; ++w) p += __popc(ebits[w * E + e[k]]);
              pos[k] = p;
            }
          }
        }
        int32_t* srow = a.slot_map + tok * a.K;
        int32_t* prow = a.expand ? a.exp_pos + tok * a.K : nullptr;
        if (a.K == KMAX && (KMAX & 3) == 0 && aligned16(srow) && (prow == nullptr || aligned16(prow))) {
#pragma unroll
          for (int k = 0; k < KMAX; k += 4) {
            *reinterpret_cast<int4*>(srow + k) = make_int4(slot[k], slot[k + 1], slot[k + 2], slot[k + 3]);
            if (prow) *reinterpret_cast<int4*>(prow + k) = make_int4(pos[k], pos[k + 1], pos[k + 2], pos[k + 3]);
          }
        } else {
#pragma unroll
          for (int k = 0; k < KMAX; ++k) {
            if (k < a.K) {
              srow[k] = slot[k];
              if (prow) prow[k] = pos[k];
            }
          }
        }
        uint8_t* row = a.is_token_in_rank + tok * R;
        if ((R & 3) == 0) {
          for (int d = 0; d < R; d += 4) {
            const uint32_t v = static_cast<uint32_t>((dmask >> d) & 1) |
                               static_cast<uint32_t>((dmask >> (d + 1)) & 1) << 8 |
                               static_cast<uint32_t>((dmask >> (d + 2)) & 1) << 16 |
                               static_cast<uint32_t>((dmask >> (d + 3)) & 1) << 24;
            *reinterpret_cast<uint32_t*>(row + d) = v;
          }
        } else {
          for (int d = 0; d < R; ++d) row[d] = static_cast<uint8_t>((dmask >> d) & 1);
        }
      }
      if (a.expand) {
        __syncthreads();
        for (int x = tid; x < E; x += THREADS) {
          int n = 0;
          for (int w = 0; w < WARPS; ++w) {
            n += __popc(ebits[w * E + x]);
            ebits[w * E + x] = 0;
          }
          run_e[x] += n;
        }
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < KMAX; ++k) e[k] = en[k];
      dmask = dn;
      t = tn;
    }
  }

  cluster.barrier_wait();
  finish_receive_sums<THREADS>(a, arrived, s_tot, &s_last);
}

// Top-k <= 8, row form or expanded: the same counts, slots and source-local
// expanded positions as layout_kernel, reorganised for latency.
//  - Each CTA (256 threads) holds every round of its tokens' lanes in
//    registers; all routing rows are requested at once (and prefetched to L2
//    before the wait for the previous kernel).
//  - Pass 1 records each (round, warp)'s token count per destination and,
//    expanded, a bitmap per (round, warp, expert) of the warp's tokens with a
//    lane on that expert. The CTA then pushes its counts into its cluster
//    peers' shared memory: its destination counts to every later CTA of the
//    source, and its per-expert counts to the CTA that totals that expert (row
//    form) or to every later CTA (expanded, whose positions need the prefix).
//    After one cluster barrier every sum a CTA needs is in its own shared
//    memory.
//  - One CTA barrier turns the (round, warp) counts into bases, so pass 2 runs
//    without barriers: a lane's rank among its warp's tokens to destination d
//    is the popcount below it of column d of the warp's destination bit matrix
//    (fetched from lane d with a shuffle); its rank among the lanes on expert e
//    is the popcount below it of the warp's bitmap for e. The CTA counts itself
//    in before pass 2 (see count_in).
// No CTA reads another's shared memory after the barrier, so none waits for its
// peers before it exits.
//
// dynamic shared memory: cnt_e [E] | row form: in_e [C][EB]; expanded: in_e
// [C][E], ebits [RW][E], ebase [RW][E]
template <int ROUNDS, bool EXPAND>
__global__ void __launch_bounds__(kRowsThreads, 1) layout_rows_kernel(LayoutArgs a) {
  constexpr int THREADS = kRowsThreads, WARPS = THREADS / 32, KMAX = 8;
  constexpr int RW = ROUNDS * WARPS;  // (round, warp) pairs
  cg::cluster_group cluster = cg::this_cluster();
  const int R = a.R, E = a.E, C = a.C, EB = a.EB;
  extern __shared__ int32_t smem[];
  int32_t* cnt_e = smem;                                  // this CTA's lanes per expert
  int32_t* in_e = smem + E;                               // peers' per-expert counts
  uint32_t* ebits = reinterpret_cast<uint32_t*>(in_e + C * E);  // expanded only
  int32_t* ebase = in_e + C * E + RW * E;                 // expanded only
  __shared__ int32_t in_d[8][kMaxRanks];  // [q][d]: CTA q's tokens to d (q < this CTA; own at q == c)
  __shared__ int32_t wcnt[RW][kMaxRanks];  // counts of each (round, warp), then their bases
  __shared__ int32_t s_tot[kMaxRanks];
  __shared__ bool s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const unsigned lt = lanemask_lt();
  const int s = blockIdx.x / C;
  const int c = static_cast<int>(cluster.block_rank());
  const int t_begin = min(a.T, c * a.TB), t_end = min(a.T, t_begin + a.TB);
  const int64_t tok_base = static_cast<int64_t>(s) * a.T;

  pdl_launch_dependents();
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    const int t = t_begin + r * THREADS + tid;
    if (t < t_end) prefetch_l2(a.topk_idx + (tok_base + t) * a.K);
  }
  // every CTA of the cluster has started before any writes to a peer's shared
  // memory (the matching wait comes after pass 1)
  cluster_arrive_relaxed();
  if constexpr (EXPAND) {
    for (int i = tid; i < RW * E; i += THREADS) ebits[i] = 0u;
  } else {
    for (int e = tid; e < E; e += THREADS) cnt_e[e] = 0;
  }
  __syncthreads();
  pdl_wait();

  // ---- pass 1: every round's lanes at once, counted per (round, warp,
  // destination) and per expert (expanded: as per-(round, warp) bitmaps)
  bool bad = false;
  int e[ROUNDS][KMAX];
  uint64_t dmask[ROUNDS];
  uint32_t col_lo[ROUNDS], col_hi[ROUNDS];
  {
    int64_t v[ROUNDS][KMAX];
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
      const int t = t_begin + r * THREADS + tid;
      load_lanes<KMAX>(a, tok_base + t, t < t_end, v[r]);
    }
#pragma unroll
    for (int r = 0; r < ROUNDS; ++r) {
      const int t = t_begin + r * THREADS + tid;
      dmask[r] = decode_lanes<KMAX>(a, v[r], t < t_end, e[r], &bad);
    }
  }
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      if (e[r][k] >= 0) {
        if constexpr (EXPAND) atomicOr(&ebits[(r * WARPS + warp) * E + e[r][k]], 1u << lane);
        else atomicAdd(&cnt_e[e[r][k]], 1);
      }
    }
    // lane d: the warp's tokens that reach destination d (and d + 32)
    col_lo[r] = warp_transpose32(static_cast<uint32_t>(dmask[r]), lane);
    if (lane < R) wcnt[r * WARPS + warp][lane] = __popc(col_lo[r]);
    col_hi[r] = 0;
    if (R > 32) {
      col_hi[r] = warp_transpose32(static_cast<uint32_t>(dmask[r] >> 32), lane);
      if (lane + 32 < R) wcnt[r * WARPS + warp][lane + 32] = __popc(col_hi[r]);
    }
  }
  if (bad) atomicOr(a.err, kErrBadTopk);
  __syncthreads();

  // ---- push the counts to the peers, then one cluster barrier
  cluster_wait();
  for (int d = tid; d < R; d += THREADS) {
    int n = 0;
#pragma unroll
    for (int rw = 0; rw < RW; ++rw) n += wcnt[rw][d];
    in_d[c][d] = n;
    for (int q = c + 1; q < C; ++q) cluster.map_shared_rank(&in_d[0][0], q)[c * kMaxRanks + d] = n;
  }
  if constexpr (EXPAND) {
    for (int x = tid; x < E; x += THREADS) {
      int n = 0;
#pragma unroll
      for (int rw = 0; rw < RW; ++rw) n += __popc(ebits[rw * E + x]);
      cnt_e[x] = n;
      for (int q = c + 1; q < C; ++q) cluster.map_shared_rank(in_e, q)[c * E + x] = n;
    }
  } else {
    for (int q = 0; q < C; ++q) {
      int32_t* dst = (q == c ? in_e : cluster.map_shared_rank(in_e, q)) + c * EB;
      for (int j = tid; j < EB; j += THREADS) {
        const int x = q * EB + j;
        if (x < E) dst[j] = cnt_e[x];
      }
    }
  }
  cluster.sync();

  // ---- bases: this CTA's (round, warp) counts become their first slots (and
  // expanded, their first source-local positions)
  const int rb = row_block(s, a.n_so, a.n_su);
  for (int d = tid; d < R; d += THREADS) {
    int base = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q)
      if (q < c) base += in_d[q][d];
    if (c == C - 1) {  // the source's totals
      const int total = base + in_d[c][d];
      a.num_tokens_per_rank[s * R + d] = total;
      a.recv_cnt[d * R + s] = total;
    }
    int run = rb * a.M + base;
#pragma unroll
    for (int rw = 0; rw < RW; ++rw) {
      const int n = wcnt[rw][d];
      wcnt[rw][d] = run;
      run += n;
    }
  }
  if constexpr (EXPAND) {
    for (int x = tid; x < E; x += THREADS) {
      int run = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q)
        if (q < c) run += in_e[q * E + x];
      if (c == C - 1) a.num_tokens_per_expert[s * E + x] = run + cnt_e[x];
#pragma unroll
      for (int rw = 0; rw < RW; ++rw) {
        ebase[rw * E + x] = run;
        run += __popc(ebits[rw * E + x]);
      }
    }
  } else {
    // this CTA's share of the source's per-expert totals
    for (int j = tid; j < EB; j += THREADS) {
      const int x = c * EB + j;
      if (x < E) {
        int n = 0;
#pragma unroll
        for (int q = 0; q < 8; ++q)
          if (q < C) n += in_e[q * EB + j];
        a.num_tokens_per_expert[s * E + x] = n;
      }
    }
  }
  __syncthreads();
  uint32_t arrived = 0;
  if (tid == 0) arrived = count_in(a);

  // ---- pass 2: slots (and source-local positions), no barriers
#pragma unroll
  for (int r = 0; r < ROUNDS; ++r) {
    const int t = t_begin + r * THREADS + tid;
    const int rw = r * WARPS + warp;
    int slot[KMAX], pos[KMAX];
#pragma unroll
    for (int k = 0; k < KMAX; ++k) {
      const int d = e[r][k] >= 0 ? div_l(e[r][k], a.l_magic) : 0;
      uint32_t col = __shfl_sync(kFullMask, col_lo[r], d & 31);  // every lane takes part
      if (R > 32) {
        const uint32_t hi = __shfl_sync(kFullMask, col_hi[r], d & 31);
        if (d >= 32) col = hi;
      }
      slot[k] = -1;
      pos[k] = -1;
      if (e[r][k] >= 0) {
        slot[k] = wcnt[rw][d] + __popc(col & lt);
        // checked builds: the slot stays inside this source's row block
        if (!row_in_bounds(slot[k] - static_cast<int64_t>(rb) * a.M, a.M, a.err)) slot[k] = -1;
        if constexpr (EXPAND) pos[k] = ebase[rw * E + e[r][k]] + __popc(ebits[rw * E + e[r][k]] & lt);
      }
    }
    if (t < t_end) {
      const int64_t tok = tok_base + t;
      int32_t* srow = a.slot_map + tok * a.K;
      int32_t* prow = EXPAND ? a.exp_pos + tok * a.K : nullptr;
      if (a.K == KMAX && aligned16(srow) && (!EXPAND || aligned16(prow))) {
        *reinterpret_cast<int4*>(srow) = make_int4(slot[0], slot[1], slot[2], slot[3]);
        *reinterpret_cast<int4*>(srow + 4) = make_int4(slot[4], slot[5], slot[6], slot[7]);
        if constexpr (EXPAND) {
          *reinterpret_cast<int4*>(prow) = make_int4(pos[0], pos[1], pos[2], pos[3]);
          *reinterpret_cast<int4*>(prow + 4) = make_int4(pos[4], pos[5], pos[6], pos[7]);
        }
      } else {
#pragma unroll
        for (int k = 0; k < KMAX; ++k) {
          if (k < a.K) {
            srow[k] = slot[k];
            if constexpr (EXPAND) prow[k] = pos[k];
          }
        }
      }
      uint8_t* row = a.is_token_in_rank + tok * R;
      if ((R & 15) == 0 && aligned16(row)) {
        for (int d = 0; d < R; d += 16) {
          uint32_t w[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t m = static_cast<uint32_t>(dmask[r] >> (d + 4 * i)) & 15u;
            w[i] = (m & 1u) | (m & 2u) << 7 | (m & 4u) << 14 | (m & 8u) << 21;
          }
          *reinterpret_cast<uint4*>(row + d) = make_uint4(w[0], w[1], w[2], w[3]);
        }
      } else if ((R & 3) == 0) {
        for (int d = 0; d < R; d += 4) {
          const uint32_t m = static_cast<uint32_t>(dmask[r] >> d) & 15u;
          *reinterpret_cast<uint32_t*>(row + d) = (m & 1u) | (m & 2u) << 7 | (m & 4u) << 14 | (m & 8u) << 21;
        }
      } else {
        for (int d = 0; d < R; ++d) row[d] = static_cast<uint8_t>((dmask[r] >> d) & 1);
      }
    }
  }

  finish_receive_sums<THREADS>(a, arrived, s_tot, &s_last);
}

// Expanded layout, step 2: for 32 experts per CTA, the exclusive prefix of the
// per-source counts down each expert's column (lanes of that expert from lower
// source ranks) and the column totals.
__global__ void __launch_bounds__(kLayoutThreads) layout_expert_scan_kernel(LayoutArgs a) {
  constexpr int kCols = 32, kGroups = kLayoutThreads / kCols;
  __shared__ int32_t part[kGroups][kCols];
  pdl_launch_dependents();
  pdl_wait();
  const int ci = threadIdx.x % kCols, g = threadIdx.x / kCols;
  const int e = blockIdx.x * kCols + ci;
  const int R = a.R, E = a.E;
  const int per = (R + kGroups - 1) / kGroups;
  const int s0 = min(R, g * per), s1 = min(R, s0 + per);
  int v[(kMaxRanks + kGroups - 1) / kGroups];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < (kMaxRanks + kGroups - 1) / kGroups; ++i) {
    v[i] = (s0 + i < s1 && e < E) ? __ldg(a.num_tokens_per_expert + (s0 + i) * E + e) : 0;
    sum += v[i];
  }
  part[g][ci] = sum;
  __syncthreads();
  int acc = 0;
  for (int q = 0; q < g; ++q) acc += part[q][ci];
  if (e < E) {
#pragma unroll
    for (int i = 0; i < (kMaxRanks + kGroups - 1) / kGroups; ++i) {
      if (s0 + i < s1) a.exp_off[(s0 + i) * E + e] = acc;
      acc += v[i];
    }
    if (g == kGroups - 1) a.exp_cnt[e] = acc;
  }
}

// Expanded layout, step 3: block starts (aligned) and region offsets, then
// each lane's final row = block start + lower sources' lanes + source-local rank.
__global__ void __launch_bounds__(kLayoutThreads) layout_expand_kernel(LayoutArgs a) {
  extern __shared__ int32_t smem[];
  int32_t* blk = smem;              // [E]: block start of each expert inside its region
  int32_t* off = smem + a.E;        // [E]: this source's cross-source offsets
  __shared__ int32_t size_d[kMaxRanks];
  const int tid = threadIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  const int s = blockIdx.x / a.C, c = blockIdx.x % a.C;
  const int E = a.E, L = a.L, R = a.R;
  for (int e = tid; e < E; e += kLayoutThreads) {
    blk[e] = __ldg(a.exp_cnt + e);
    off[e] = __ldg(a.exp_off + s * E + e);
  }
  __syncthreads();
  for (int d = tid; d < R; d += kLayoutThreads) {
    int base = 0;
    for (int j = 0; j < L; ++j) {
      const int n = blk[d * L + j];
      blk[d * L + j] = base;
      base += (n + a.align - 1) / a.align * a.align;
    }
    size_d[d] = base;
  }
  __syncthreads();
  if (blockIdx.x == 0) {  // the tables themselves
    for (int e = tid; e < E; e += kLayoutThreads) a.exp_base[(e / L) * (L + 1) + e % L] = blk[e];
    for (int d = tid; d < R; d += kLayoutThreads) a.exp_base[d * (L + 1) + L] = size_d[d];
    if (tid == 0) {
      int acc = 0;
      for (int d = 0; d < R; ++d) {
        a.exp_region[d] = acc;
        acc += size_d[d];
      }
      a.exp_region[R] = acc;
    }
  }
  const int t_begin = min(a.T, c * a.TB), t_end = min(a.T, t_begin + a.TB);
  const int64_t i0 = (static_cast<int64_t>(s) * a.T + t_begin) * a.K;
  const int64_t i1 = (static_cast<int64_t>(s) * a.T + t_end) * a.K;
  // four lanes in flight per thread: positions and experts load together
  constexpr int kU = 4;
  for (int64_t i = i0 + tid; i < i1; i += kU * kLayoutThreads) {
    int p[kU];
    int64_t ev[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      const int64_t j = i + u * kLayoutThreads;
      p[u] = j < i1 ? a.exp_pos[j] : -1;
      ev[u] = j < i1 ? __ldg(a.topk_idx + j) : 0;
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) {
      if (p[u] >= 0) {  // a placed lane: its expert is valid
        const int e = static_cast<int>(ev[u]);
        int row = p[u] + blk[e] + off[e];
        // checked builds: the row stays inside its destination's region
        if (!row_in_bounds(row, size_d[e / L], a.err)) row = -1;
        a.exp_pos[i + u * kLayoutThreads] = row;
      }
    }
  }
}

namespace {

// One thread-block cluster of a.C CTAs per source rank (a plain grid when a.C is 1).
template <typename Kernel>
cudaError_t launch_clusters(Kernel kernel, const Geometry& g, const LayoutArgs& a, int threads, size_t smem,
                            cudaStream_t stream) {
  cudaError_t err;
  if (smem > 32 * 1024 &&
      (err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem))) !=
          cudaSuccess)
    return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(g.R * a.C));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(a.C);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  // one CTA per source needs no cluster (each CTA is its own); the cluster
  // attribute costs ~0.7 us of launch on GB300
  cfg.numAttrs = a.C == 1 ? 1 : 2;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <bool EXPAND>
cudaError_t launch_rows(int rounds, const Geometry& g, const LayoutArgs& a, size_t smem, cudaStream_t stream) {
  if (rounds <= 1) return launch_clusters(layout_rows_kernel<1, EXPAND>, g, a, kRowsThreads, smem, stream);
  if (rounds <= 2) return launch_clusters(layout_rows_kernel<2, EXPAND>, g, a, kRowsThreads, smem, stream);
  return launch_clusters(layout_rows_kernel<4, EXPAND>, g, a, kRowsThreads, smem, stream);
}

template <int KMAX, int THREADS>
cudaError_t launch_main(const Geometry& g, const LayoutArgs& a, cudaStream_t stream) {
  const size_t smem = sizeof(int32_t) * g.E +
                      (g.expand ? sizeof(int32_t) * (g.E + static_cast<size_t>(THREADS / 32) * g.E) : 0);
  return launch_clusters(layout_kernel<KMAX, THREADS>, g, a, THREADS, smem, stream);
}

}  // namespace

cudaError_t launch_layout(const Geometry& g, const LayoutArgs& args, int num_prologue_sms,
                          cudaStream_t stream) {
  LayoutArgs a = args;
  // One thread per token and round in CTAs of 256 threads, as many per source
  // as make rounds of 256 tokens, at most 8 (a portable cluster; on GB300 a
  // 16th cluster of 512-thread CTAs started about 7 us after the others).
  // Top-k <= 8 with at most four rounds a CTA runs the register kernel (the
  // expanded layout too, while its per-(round, warp) expert tables fit in
  // shared memory); otherwise the general kernel, which loads the rounds in
  // turn. Always within the prologue budget of 2 CTAs per requested SM, and at
  // least one CTA per source.
  const int threads = kRowsThreads;
  const int sms = num_prologue_sms > 0 ? (num_prologue_sms < kMaxPrologueCtas ? num_prologue_sms
                                                                               : kMaxPrologueCtas)
                                       : kMaxPrologueCtas;
  int C = (g.T + threads - 1) / threads;
  C = C < 1 ? 1 : (C > 8 ? 8 : C);
  const int budget = (2 * sms) / g.R;
  if (C > budget) C = budget < 1 ? 1 : budget;
  a.C = C;
  a.TB = (g.T + C - 1) / C;
  a.l_magic = g.L == 1 ? 0u : static_cast<uint32_t>((0x100000000ull + g.L - 1) / g.L);
  a.so_magic = g.n_so == 1 ? 0u : static_cast<uint32_t>((0x100000000ull + g.n_so - 1) / g.n_so);
  a.EB = (g.E + C - 1) / C;
  const int rounds = (a.TB + threads - 1) / threads;
  const int rt = rounds <= 1 ? 1 : (rounds <= 2 ? 2 : 4);  // the kernel's rounds
  const size_t smem_rows =
      sizeof(int32_t) * (g.expand ? static_cast<size_t>(g.E) * (1 + C + 2 * rt * (kRowsThreads / 32))
                                  : g.E + static_cast<size_t>(C) * a.EB);
  int dev = 0, smem_optin = 0;
  cudaError_t qerr;
  if ((qerr = cudaGetDevice(&dev)) != cudaSuccess ||
      (qerr = cudaDeviceGetAttribute(&smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
    return qerr;
  // the register kernel's static shared memory stays under 12 KB
  const bool rows = g.K <= 8 && rounds <= 4 && smem_rows + 12 * 1024 <= static_cast<size_t>(smem_optin);
  cudaError_t err;
  if (rows)
    err = g.expand ? launch_rows<true>(rt, g, a, smem_rows, stream) : launch_rows<false>(rt, g, a, smem_rows, stream);
  else
    err = g.K <= 8 ? launch_main<8, 256>(g, a, stream) : launch_main<32, 256>(g, a, stream);
  if (err != cudaSuccess) return err;
  if (g.expand) {
    if ((err = launch_chained(layout_expert_scan_kernel, dim3((g.E + 31) / 32), dim3(kLayoutThreads), 0, stream,
                              a)) != cudaSuccess)
      return err;
    const size_t smem2 = 2 * sizeof(int32_t) * g.E;
    if (smem2 > 32 * 1024 &&
        (err = cudaFuncSetAttribute(layout_expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem2))) != cudaSuccess)
      return err;
    if ((err = launch_chained(layout_expand_kernel, dim3(g.R * C), dim3(kLayoutThreads), smem2, stream, a)) !=
        cudaSuccess)
      return err;
  }
  return cudaSuccess;
}

}  // namespace ep

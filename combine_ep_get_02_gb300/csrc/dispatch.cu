// Dispatch: scatter every source token's hidden row into the receive rows of
// its deduplicated destinations, with the row's sidecars.
//
// One warp owns one source token at a time: it reads the row once (16-byte
// loads, each lane a strided set of chunks), optionally casts it to FP8-e4m3
// in registers, and stores it to each destination row; the slots come from the
// layout (PR #753, Approach: the kernel replays precomputed slots instead of
// racing for them). When tokens are fewer than two per warp, a token is split
// into column ranges and each range is its own work unit. A persistent grid
// sized to the SMs works through the units; in the row form it takes them from
// a work queue in the workspace (a token's cost grows with its number of
// destinations, so a static share would leave the launch waiting on its
// heaviest warps).
// Lanes 0..K-1 carry the token's top-k lanes; the small sidecar rows (routing
// of the lanes to each destination and the source metadata) are written by the
// whole warp.
// This register path carries the fused cast always, and rows that travel
// unchanged when copy_path asks for it or the input is small; larger unchanged
// inputs go to the bulk-copy kernel in dispatch_bulk.cu.
#include "dispatch_common.cuh"
#include "ep_device.cuh"
#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kWarps = kCopyThreads / 32;
constexpr int kUnroll = 4;     // 16-byte chunks in flight per lane (row copy)
constexpr int kCastUnits = 4;  // 16-column units in flight per lane (cast)

enum Kind { kCopyRow = 0, kCastRow = 1 };

// The cast keeps more bytes in flight per warp with two CTAs per SM (up to 128
// registers a thread) than with more, smaller-register CTAs; the row copy runs
// three CTAs per SM (up to 85 registers: four, at 64, spilled).
template <int kKind, bool kExpand, bool kAtomic = false>
__global__ void __launch_bounds__(kCopyThreads, kKind == kCastRow ? 2 : 3) dispatch_kernel(DispatchArgs a) {
  __shared__ int64_t s_row[kWarps][kMaxTopk];               // hidden destination rows
  __shared__ float s_sf[kWarps][kMaxScaleGroups];           // this token's FP8 scales
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gwarp = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  pdl_launch_dependents();
  pdl_wait();

  // The warp's work units in turn (from the work queue in the row form): a unit
  // is one token's column range (a.splits ranges a token; more than one only
  // when tokens are too few to keep every warp busy). The next unit's routing
  // loads, and the one after it is taken, while this unit's columns stream.
  const int64_t units = a.num_tokens * a.splits;
  // a unit's token: with more than one range a token there are fewer than
  // 2^31 units (the split is only taken for a few thousand tokens)
  auto token_of = [&](int64_t u) -> int64_t {
    if (u >= units) return a.num_tokens;
    return a.splits == 1 ? u : static_cast<int64_t>(static_cast<uint32_t>(u) / static_cast<uint32_t>(a.splits));
  };
  UnitStream us = start_units(gwarp, nwarps, units, !kExpand);
  RawLane next = fetch_lane(a, token_of(us.cur), lane, kExpand, kAtomic);
  while (us.cur < units) {
    const int64_t tok = token_of(us.cur);
    const int part = static_cast<int>(us.cur - tok * a.splits);
    const int s = static_cast<int>(tok / a.T);
    const int t = static_cast<int>(tok - static_cast<int64_t>(s) * a.T);
    const RawLane cur = next;
    const int64_t after = take_unit(us, a.queue, lane);
    next = fetch_lane(a, token_of(us.nxt), lane, kExpand, kAtomic);
    // this unit's 16-byte chunks (row copy) or 16-column units (cast)
    const int n_items = kKind == kCopyRow ? a.in_row_bytes >> 4 : a.H >> 4;
    const int i_begin = part * a.split_len, i_end = min(n_items, i_begin + a.split_len);
    // the first loads go out before the token's destinations are resolved:
    // their addresses depend on the token alone
    const uint8_t* src = a.x + tok * a.in_row_bytes;
    uint4 v[kKind == kCopyRow ? kUnroll : 2 * kCastUnits];
    if (kKind == kCopyRow) {
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = i_begin + u * 32 + lane;
        if (c < i_end) v[u] = ld_stream16(src + (static_cast<size_t>(c) << 4));
      }
    } else {
#pragma unroll
      for (int r = 0; r < kCastUnits; ++r) {
        const int u = i_begin + r * 32 + lane;
        if (u < i_end) {
          v[2 * r] = ld_stream16(src + (static_cast<size_t>(u) << 5));
          v[2 * r + 1] = ld_stream16(src + (static_cast<size_t>(u) << 5) + 16);
        }
      }
    }
    const TokenLanes ln = lanes_of(a, cur, tok, lane, kExpand, kAtomic);
    const int nh = hidden_rows(a, ln, lane, kExpand, s_row[warp]);

    if (kKind == kCopyRow) {
      // the row's bytes unchanged (bf16 -> bf16, or pre-cast e4m3 -> e4m3)
      for (int c0 = i_begin; c0 < i_end; c0 += 32 * kUnroll) {
        if (c0 > i_begin) {
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < i_end) v[u] = ld_stream16(src + (static_cast<size_t>(c) << 4));
          }
        }
        for (int j = 0; j < nh; ++j) {
          uint8_t* dst = a.recv_x + s_row[warp][j] * a.out_row_bytes;
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < i_end) st16(dst + (static_cast<size_t>(c) << 4), v[u]);
          }
        }
      }
      if (a.x_sf != nullptr && part == 0) {  // pre-cast FP8: the scale words travel verbatim
        const float* ssrc = a.x_sf + tok * a.SW;
        for (int g = lane; g < a.SW; g += 32) {
          const float v = ssrc[g];
          for (int j = 0; j < nh; ++j) a.recv_sf[s_row[warp][j] * a.SW + g] = v;
        }
      }
    } else {
      // bf16 -> e4m3 with one fp32 scale per 128 columns. A lane owns 16 columns
      // (32 bytes in, 16 bytes out); 8 consecutive lanes form one 128-column group.
      // A unit's range starts on a multiple of 128 units (16 groups, 4 packed
      // scale words), so no group or scale word spans two units.
      for (int u0 = i_begin; u0 < i_end; u0 += 32 * kCastUnits) {
        if (u0 > i_begin) {
#pragma unroll
          for (int r = 0; r < kCastUnits; ++r) {
            const int u = u0 + r * 32 + lane;
            if (u < i_end) {
              v[2 * r] = ld_stream16(src + (static_cast<size_t>(u) << 5));
              v[2 * r + 1] = ld_stream16(src + (static_cast<size_t>(u) << 5) + 16);
            }
          }
        }
#pragma unroll
        for (int r = 0; r < kCastUnits; ++r) {
          const int u = u0 + r * 32 + lane;
          if (u0 + r * 32 >= i_end) continue;  // warp-uniform
          const CastUnit cu = cast_unit(v[2 * r], v[2 * r + 1], u < i_end, a.sf_pack);
          const uint4 q = cu.q;
          if (u < i_end) {
            if ((lane & 7) == 0) {
              if (a.sf_pack) reinterpret_cast<uint8_t*>(s_sf[warp])[u >> 3] = cu.sf_byte;
              else s_sf[warp][u >> 3] = cu.sf;
            }
            for (int j = 0; j < nh; ++j)
              st16(a.recv_x + s_row[warp][j] * a.out_row_bytes + (static_cast<size_t>(u) << 4), q);
          }
        }
      }
      __syncwarp();
      // this unit's groups [g_begin, g_end) (the last unit's end rounds up to the
      // row's last group, and, packed, its last word)
      const int g_begin = i_begin >> 3, g_end = (i_end + 7) >> 3;
      if (a.sf_pack) {  // four exponent bytes per word; bytes past the last group are 0
        const uint8_t* b = reinterpret_cast<const uint8_t*>(s_sf[warp]);
        for (int wd = (g_begin >> 2) + lane; wd < (g_end + 3) >> 2; wd += 32) {
          uint32_t v = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (4 * wd + i < a.G) v |= static_cast<uint32_t>(b[4 * wd + i]) << (8 * i);
          for (int j = 0; j < nh; ++j) reinterpret_cast<uint32_t*>(a.recv_sf)[s_row[warp][j] * a.SW + wd] = v;
        }
      } else {
        for (int g = g_begin + lane; g < g_end; g += 32) {
          const float v = s_sf[warp][g];
          for (int j = 0; j < nh; ++j) a.recv_sf[s_row[warp][j] * a.G + g] = v;
        }
      }
    }

    if (part == 0) write_sidecars(a, ln, s, t, lane, kExpand);
    __syncwarp();  // s_row / s_sf are rewritten by the next token
    advance_units(us, after);
  }
  leave_queue(us, a.queue, lane);

  if (kExpand && a.zero_padding)
    zero_padding_rows(a, gwarp, nwarps, lane, kKind == kCastRow || a.x_sf != nullptr);
}

template <int kKind, bool kExpand, bool kAtomic = false>
cudaError_t launch_one(const DispatchArgs& args, int num_sms, cudaStream_t stream) {
  auto kern = dispatch_kernel<kKind, kExpand, kAtomic>;
  int per_sm = resident_ctas(reinterpret_cast<const void*>(kern), kCopyThreads, 0);
  if (per_sm < 0) return cudaErrorUnknown;
  if (per_sm < 1) per_sm = 1;
  DispatchArgs a = args;
  int64_t ctas = static_cast<int64_t>(num_sms) * per_sm;
  // Fewer than two tokens a warp: split each token into column ranges (whole
  // lane sweeps) until there are, so that every warp has bytes in flight. The
  // atomic-slot path takes one slot per token and is never split.
  const int n_items = kKind == kCopyRow ? a.in_row_bytes >> 4 : a.H >> 4;
  const int sweep = 32 * (kKind == kCopyRow ? kUnroll : kCastUnits);
  const int max_splits = (n_items + sweep - 1) / sweep;
  int64_t want = a.num_tokens > 0 ? (2 * ctas * kWarps + a.num_tokens - 1) / a.num_tokens : 1;
  if (kAtomic || want < 1) want = 1;
  if (want > max_splits) want = max_splits;
  a.split_len = static_cast<int>(((n_items + want - 1) / want + sweep - 1) / sweep * sweep);
  if (a.split_len < sweep) a.split_len = sweep;
  a.splits = (n_items + a.split_len - 1) / a.split_len;
  if (a.splits < 1) a.splits = 1;
  const int64_t units = a.num_tokens * a.splits;
  const int64_t need = ((a.zero_padding && a.E > units ? a.E : units) + kWarps - 1) / kWarps;
  if (ctas > need) ctas = need;
  if (ctas < 1) return cudaSuccess;
  return launch_chained(kern, dim3(static_cast<unsigned>(ctas)), dim3(kCopyThreads), 0, stream, a);
}

}  // namespace

cudaError_t launch_dispatch(const Geometry& g, const DispatchArgs& a, int num_sms,
                            cudaStream_t stream) {
  const bool cast = !g.x_fp8 && g.recv_fp8;
  if (cast) {
    return g.expand ? launch_one<kCastRow, true>(a, num_sms, stream)
                    : launch_one<kCastRow, false>(a, num_sms, stream);
  }
  // Unchanged rows: bulk copies pay off once the input streams from DRAM; on small
  // (L2-resident, latency-bound) inputs the register path has more rows in flight.
  const bool bulk = g.copy_path == 2 ||
                    (g.copy_path == 0 && a.num_tokens * a.in_row_bytes >= kBulkAutoMinBytes);
  if (bulk) return launch_dispatch_bulk(g, a, num_sms, stream);
  return g.expand ? launch_one<kCopyRow, true>(a, num_sms, stream)
                  : launch_one<kCopyRow, false>(a, num_sms, stream);
}

cudaError_t launch_dispatch_atomic(const Geometry& g, const DispatchArgs& a, int num_sms,
                                   cudaStream_t stream) {
  const bool cast = !g.x_fp8 && g.recv_fp8;
  return cast ? launch_one<kCastRow, false, true>(a, num_sms, stream)
              : launch_one<kCopyRow, false, true>(a, num_sms, stream);
}

}  // namespace ep

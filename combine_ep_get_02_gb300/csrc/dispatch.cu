// Dispatch: scatter every source token's hidden row into the receive rows of
// its deduplicated destinations, with the row's sidecars.
//
// One warp owns one source token at a time: it reads the row once (16-byte
// loads, each lane a strided set of chunks), optionally casts it to FP8-e4m3
// in registers, and stores it to each destination row; the slots come from the
// layout (PR #753, Approach: the kernel replays precomputed slots instead of
// racing for them). A persistent grid sized to the SMs works through the
// tokens; in the row form it takes them from a work queue in the workspace (a
// token's cost grows with its number of destinations, so a static share would
// leave the launch waiting on its heaviest warps).
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
// registers a thread) than with more, smaller-register CTAs; the row copy fits
// four CTAs per SM.
template <int kKind, bool kExpand, bool kAtomic = false>
__global__ void __launch_bounds__(kCopyThreads, kKind == kCastRow ? 2 : 4) dispatch_kernel(DispatchArgs a) {
  __shared__ int64_t s_row[kWarps][kMaxTopk];               // hidden destination rows
  __shared__ float s_sf[kWarps][kMaxScaleGroups];           // this token's FP8 scales
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gwarp = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  pdl_launch_dependents();
  pdl_wait();

  // the warp's tokens in turn (from the work queue in the row form): the next
  // token's routing loads, and the one after it is taken, while this token's
  // row streams
  UnitStream us = start_units(gwarp, nwarps, a.num_tokens, !kExpand);
  RawLane next = fetch_lane(a, us.cur, lane, kExpand, kAtomic);
  while (us.cur < a.num_tokens) {
    const int64_t tok = us.cur;
    const int s = static_cast<int>(tok / a.T);
    const int t = static_cast<int>(tok - static_cast<int64_t>(s) * a.T);
    const RawLane cur = next;
    const int64_t after = take_unit(us, a.queue, lane);
    next = fetch_lane(a, us.nxt, lane, kExpand, kAtomic);
    // the row's first loads go out before its destinations are resolved: its
    // address depends on the token alone
    const uint8_t* src = a.x + tok * a.in_row_bytes;
    uint4 v[kKind == kCopyRow ? kUnroll : 2 * kCastUnits];
    if (kKind == kCopyRow) {
      const int nchunk = a.in_row_bytes >> 4;
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int c = u * 32 + lane;
        if (c < nchunk) v[u] = ld_stream16(src + (static_cast<size_t>(c) << 4));
      }
    } else {
      const int nunit = a.H >> 4;
#pragma unroll
      for (int r = 0; r < kCastUnits; ++r) {
        const int u = r * 32 + lane;
        if (u < nunit) {
          v[2 * r] = ld_stream16(src + (static_cast<size_t>(u) << 5));
          v[2 * r + 1] = ld_stream16(src + (static_cast<size_t>(u) << 5) + 16);
        }
      }
    }
    const TokenLanes ln = lanes_of(a, cur, tok, lane, kExpand, kAtomic);
    const int nh = hidden_rows(a, ln, lane, kExpand, s_row[warp]);

    if (kKind == kCopyRow) {
      // the row's bytes unchanged (bf16 -> bf16, or pre-cast e4m3 -> e4m3)
      const int nchunk = a.in_row_bytes >> 4;
      for (int c0 = 0; c0 < nchunk; c0 += 32 * kUnroll) {
        if (c0 > 0) {
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < nchunk) v[u] = ld_stream16(src + (static_cast<size_t>(c) << 4));
          }
        }
        for (int j = 0; j < nh; ++j) {
          uint8_t* dst = a.recv_x + s_row[warp][j] * a.out_row_bytes;
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < nchunk) st16(dst + (static_cast<size_t>(c) << 4), v[u]);
          }
        }
      }
      if (a.x_sf != nullptr) {  // pre-cast FP8: the scale words travel verbatim
        const float* ssrc = a.x_sf + tok * a.SW;
        for (int g = lane; g < a.SW; g += 32) {
          const float v = ssrc[g];
          for (int j = 0; j < nh; ++j) a.recv_sf[s_row[warp][j] * a.SW + g] = v;
        }
      }
    } else {
      // bf16 -> e4m3 with one fp32 scale per 128 columns. A lane owns 16 columns
      // (32 bytes in, 16 bytes out); 8 consecutive lanes form one 128-column group.
      const int nunit = a.H >> 4;  // multiple of 8
      for (int u0 = 0; u0 < nunit; u0 += 32 * kCastUnits) {
        if (u0 > 0) {
#pragma unroll
          for (int r = 0; r < kCastUnits; ++r) {
            const int u = u0 + r * 32 + lane;
            if (u < nunit) {
              v[2 * r] = ld_stream16(src + (static_cast<size_t>(u) << 5));
              v[2 * r + 1] = ld_stream16(src + (static_cast<size_t>(u) << 5) + 16);
            }
          }
        }
#pragma unroll
        for (int r = 0; r < kCastUnits; ++r) {
          const int u = u0 + r * 32 + lane;
          if (u0 + r * 32 >= nunit) continue;  // warp-uniform
          const CastUnit cu = cast_unit(v[2 * r], v[2 * r + 1], u < nunit, a.sf_pack);
          const uint4 q = cu.q;
          if (u < nunit) {
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
      if (a.sf_pack) {  // four exponent bytes per word; bytes past the last group are 0
        const uint8_t* b = reinterpret_cast<const uint8_t*>(s_sf[warp]);
        for (int wd = lane; wd < a.SW; wd += 32) {
          uint32_t v = 0;
#pragma unroll
          for (int i = 0; i < 4; ++i)
            if (4 * wd + i < a.G) v |= static_cast<uint32_t>(b[4 * wd + i]) << (8 * i);
          for (int j = 0; j < nh; ++j) reinterpret_cast<uint32_t*>(a.recv_sf)[s_row[warp][j] * a.SW + wd] = v;
        }
      } else {
        for (int g = lane; g < a.G; g += 32) {
          const float v = s_sf[warp][g];
          for (int j = 0; j < nh; ++j) a.recv_sf[s_row[warp][j] * a.G + g] = v;
        }
      }
    }

    write_sidecars(a, ln, s, t, lane, kExpand);
    __syncwarp();  // s_row / s_sf are rewritten by the next token
    advance_units(us, after);
  }
  leave_queue(us, a.queue, lane);

  if (kExpand && a.zero_padding)
    zero_padding_rows(a, gwarp, nwarps, lane, kKind == kCastRow || a.x_sf != nullptr);
}

template <int kKind, bool kExpand, bool kAtomic = false>
cudaError_t launch_one(const DispatchArgs& a, int num_sms, cudaStream_t stream) {
  auto kern = dispatch_kernel<kKind, kExpand, kAtomic>;
  int per_sm = resident_ctas(reinterpret_cast<const void*>(kern), kCopyThreads, 0);
  if (per_sm < 0) return cudaErrorUnknown;
  if (per_sm < 1) per_sm = 1;
  int64_t ctas = static_cast<int64_t>(num_sms) * per_sm;
  const int64_t need = ((a.zero_padding && a.E > a.num_tokens ? a.E : a.num_tokens) + kWarps - 1) / kWarps;
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

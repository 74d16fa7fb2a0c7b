// Dispatch: scatter every source token's hidden row into the receive rows of
// its deduplicated destinations, with the row's sidecars.
//
// One warp owns one source token at a time: it reads the row once (16-byte
// loads, each lane a strided set of chunks), optionally casts it to FP8-e4m3
// in registers, and stores it to each destination row; the slots come from the
// layout (PR #753, Approach: the kernel replays precomputed slots instead of
// racing for them). Tokens are spread over a persistent grid sized to the SMs.
// Lanes 0..K-1 carry the token's top-k lanes and write the small sidecar rows
// (routing of the lanes to that destination and the source metadata).
#include "ep_device.cuh"
#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kWarps = kCopyThreads / 32;
constexpr int kUnroll = 4;     // 16-byte chunks in flight per lane (row copy)
constexpr int kCastUnits = 4;  // 16-column units in flight per lane (cast)

enum Kind { kCopyRow = 0, kCastRow = 1 };

struct TokenLanes {
  int e, d, slot, pos;
  int row;  // receive row of the lane's deduplicated entry inside its destination region
  float w;
  unsigned vmask;  // valid lanes
  unsigned rmask;  // first lane per destination (deduplicated entries)
};

// The raw routing of top-k lane `lane` of a token, loaded one token ahead.
struct RawLane {
  int64_t e;
  int slot, pos;
  float w;
};

__device__ __forceinline__ RawLane fetch_lane(const DispatchArgs& a, int64_t tok, int lane, bool expand,
                                              bool atomic) {
  RawLane r;
  r.e = -1;
  r.slot = -1;
  r.pos = -1;
  r.w = 0.f;
  if (tok < a.num_tokens && lane < a.K) {
    const int64_t i = tok * a.K + lane;
    r.e = __ldg(a.topk_idx + i);
    if (!atomic) r.slot = __ldg(a.slot_map + i);
    r.w = __ldg(a.topk_w + i);
    if (expand) r.pos = __ldg(a.exp_pos + i);
  }
  return r;
}

// Lane k < K: the token's k-th top-k lane. Invalid lanes get a distinct
// negative d so that they never group with anything. With `atomic` (the
// prior-art comparison path) there is no layout: the first lane to each
// destination takes the next row of the source's block with an atomicAdd on
// the (source, destination) counter, so the order inside a block depends on
// which warp gets there first (PR #753, Motivation).
__device__ __forceinline__ TokenLanes lanes_of(const DispatchArgs& a, const RawLane& raw, int64_t tok,
                                               int lane, bool expand, bool atomic) {
  TokenLanes L;
  L.slot = raw.slot;
  L.pos = raw.pos;
  L.w = raw.w;
  L.e = (raw.e >= 0 && raw.e < a.E) ? static_cast<int>(raw.e) : -1;
  const bool valid = L.e >= 0 && (atomic || (expand ? L.pos >= 0 : L.slot >= 0));
  L.d = valid ? L.e / a.L : -1 - lane;
  const unsigned same = __match_any_sync(kFullMask, L.d);
  L.vmask = __ballot_sync(kFullMask, valid);
  L.rmask = __ballot_sync(kFullMask, valid && (same & lanemask_lt()) == 0);
  if (atomic) {
    const int s = static_cast<int>(tok / a.T);
    const int rb = a.n_so == 1 ? s : (s % a.n_su) * a.n_so + s / a.n_su;
    int mine = -1;
    if ((L.rmask >> lane) & 1) mine = rb * a.M + atomicAdd(a.send_counters + s * a.R + L.d, 1);
    L.slot = __shfl_sync(kFullMask, mine, __ffs(same) - 1);
    if (!valid) L.slot = -1;
  }
  L.row = (valid && !expand) ? recv_row_of_slot(L.slot, L.d, a.R, a.M, a.compact, a.recv_psum) : -1;
  return L;
}

template <int kKind, bool kExpand, bool kAtomic = false>
__global__ void __launch_bounds__(kCopyThreads) dispatch_kernel(DispatchArgs a) {
  __shared__ int64_t s_row[kWarps][kMaxTopk];               // hidden destination rows
  __shared__ float s_sf[kWarps][kMaxScaleGroups];           // this token's FP8 scales
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const unsigned lt = lanemask_lt();
  const int64_t gwarp = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;

  // the next token's routing loads while this token's row streams
  RawLane next = fetch_lane(a, gwarp, lane, kExpand, kAtomic);
  for (int64_t tok = gwarp; tok < a.num_tokens; tok += nwarps) {
    const int s = static_cast<int>(tok / a.T);
    const int t = static_cast<int>(tok - static_cast<int64_t>(s) * a.T);
    const RawLane cur = next;
    next = fetch_lane(a, tok + nwarps, lane, kExpand, kAtomic);
    const TokenLanes ln = lanes_of(a, cur, tok, lane, kExpand, kAtomic);
    const unsigned hmask = kExpand ? ln.vmask : ln.rmask;
    if ((hmask >> lane) & 1) {
      const int64_t row = kExpand ? static_cast<int64_t>(a.exp_region[ln.d]) + ln.pos
                                  : static_cast<int64_t>(ln.d) * a.region_rows + ln.row;
      s_row[warp][__popc(hmask & lt)] = row;
    }
    __syncwarp();
    const int nh = __popc(hmask);

    if (kKind == kCopyRow) {
      // the row's bytes unchanged (bf16 -> bf16, or pre-cast e4m3 -> e4m3)
      const uint8_t* src = a.x + tok * a.in_row_bytes;
      const int nchunk = a.in_row_bytes >> 4;
      for (int c0 = 0; c0 < nchunk; c0 += 32 * kUnroll) {
        uint4 v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int c = c0 + u * 32 + lane;
          if (c < nchunk) v[u] = ld_stream16(src + (static_cast<size_t>(c) << 4));
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
      const uint8_t* src = a.x + tok * a.in_row_bytes;
      const int nunit = a.H >> 4;  // multiple of 8
      for (int u0 = 0; u0 < nunit; u0 += 32 * kCastUnits) {
        uint4 lo[kCastUnits], hi[kCastUnits];
#pragma unroll
        for (int r = 0; r < kCastUnits; ++r) {
          const int u = u0 + r * 32 + lane;
          if (u < nunit) {
            lo[r] = ld_stream16(src + (static_cast<size_t>(u) << 5));
            hi[r] = ld_stream16(src + (static_cast<size_t>(u) << 5) + 16);
          }
        }
#pragma unroll
        for (int r = 0; r < kCastUnits; ++r) {
          const int u = u0 + r * 32 + lane;
          if (u0 + r * 32 >= nunit) continue;  // warp-uniform
          float f[16];
          const uint32_t wv[8] = {lo[r].x, lo[r].y, lo[r].z, lo[r].w, hi[r].x, hi[r].y, hi[r].z, hi[r].w};
          float amax = 0.f;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const float2 p = bf16x2_to_f32x2(u < nunit ? wv[i] : 0u);
            f[2 * i] = p.x;
            f[2 * i + 1] = p.y;
            amax = fmaxf(amax, fmaxf(fabsf(p.x), fabsf(p.y)));
          }
          amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 1));
          amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 2));
          amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 4));
          amax = fmaxf(amax, 1e-4f);
          // fp32 scale: inv = 448/amax. Packed: the smallest 2^e >= amax/448, read off
          // amax's exponent and mantissa (amax = m*2^k; e = k-8, or k-7 when m > 1.75).
          const uint32_t ab = __float_as_uint(amax);
          const int e2 = static_cast<int>(ab >> 23) - 127 - 8 + ((ab & 0x7FFFFFu) > 0x600000u ? 1 : 0);
          const float inv = a.sf_pack ? __uint_as_float(static_cast<uint32_t>(127 - e2) << 23)
                                      : __fdiv_rn(448.0f, amax);
          uint4 q;
          q.x = f32x2_to_e4m3x2(__fmul_rn(f[0], inv), __fmul_rn(f[1], inv)) |
                f32x2_to_e4m3x2(__fmul_rn(f[2], inv), __fmul_rn(f[3], inv)) << 16;
          q.y = f32x2_to_e4m3x2(__fmul_rn(f[4], inv), __fmul_rn(f[5], inv)) |
                f32x2_to_e4m3x2(__fmul_rn(f[6], inv), __fmul_rn(f[7], inv)) << 16;
          q.z = f32x2_to_e4m3x2(__fmul_rn(f[8], inv), __fmul_rn(f[9], inv)) |
                f32x2_to_e4m3x2(__fmul_rn(f[10], inv), __fmul_rn(f[11], inv)) << 16;
          q.w = f32x2_to_e4m3x2(__fmul_rn(f[12], inv), __fmul_rn(f[13], inv)) |
                f32x2_to_e4m3x2(__fmul_rn(f[14], inv), __fmul_rn(f[15], inv)) << 16;
          if (u < nunit) {
            if ((lane & 7) == 0) {
              if (a.sf_pack) reinterpret_cast<uint8_t*>(s_sf[warp])[u >> 3] = static_cast<uint8_t>(e2 + 127);
              else s_sf[warp][u >> 3] = __fdiv_rn(amax, 448.0f);
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
          for (int j = 0; j < nh; ++j)
            reinterpret_cast<uint32_t*>(a.recv_sf)[s_row[warp][j] * a.SW + wd] = v;
        }
      } else {
        for (int g = lane; g < a.G; g += 32) {
          const float v = s_sf[warp][g];
          for (int j = 0; j < nh; ++j) a.recv_sf[s_row[warp][j] * a.G + g] = v;
        }
      }
    }

    // sidecar rows of each deduplicated destination (row form). Metadata field
    // f = 2 + k carries lane k's expanded row; with K up to 32 there are up to 34
    // fields, so a lane writes fields lane and lane + 32.
    if (a.recv_idx != nullptr || a.recv_w != nullptr || a.recv_md != nullptr) {
      const int f0_d = __shfl_sync(kFullMask, ln.d, (lane - 2) & 31);   // lane f-2 for f = lane
      const int f0_pos = __shfl_sync(kFullMask, ln.pos, (lane - 2) & 31);
      const int f1_d = __shfl_sync(kFullMask, ln.d, (lane + 30) & 31);  // f = lane + 32
      const int f1_pos = __shfl_sync(kFullMask, ln.pos, (lane + 30) & 31);
      unsigned m = ln.rmask;
      while (m) {
        const int rl = __ffs(m) - 1;
        m &= m - 1;
        const int dj = __shfl_sync(kFullMask, ln.d, rl);
        const int row = __shfl_sync(kFullMask, kExpand ? ln.slot : ln.row, rl);
        const int64_t mrow = static_cast<int64_t>(dj) * a.region_rows + row;
        if (lane < a.K) {
          const bool on = ln.d == dj;
          if (a.recv_idx) a.recv_idx[mrow * a.K + lane] = on ? static_cast<int64_t>(ln.e - dj * a.L) : -1;
          if (a.recv_w) a.recv_w[mrow * a.K + lane] = on ? ln.w : 0.f;
        }
        if (a.recv_md) {
          int32_t* md = a.recv_md + mrow * (a.K + 2);
          if (lane < a.K + 2) {
            int v;
            if (lane == 0) v = s;
            else if (lane == 1) v = t;
            else v = (kExpand && f0_d == dj) ? f0_pos : -1;
            md[lane] = v;
          }
          if (lane + 32 < a.K + 2) md[lane + 32] = (kExpand && f1_d == dj) ? f1_pos : -1;
        }
      }
    }
    __syncwarp();  // s_row / s_sf are rewritten by the next token
  }

  // expanded blocks padded to expert_alignment: zero the rows after each
  // expert's lanes up to the next block start (and their scales)
  if (kExpand && a.zero_padding) {
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    const int nchunk = a.out_row_bytes >> 4;
    for (int64_t blk = gwarp; blk < a.E; blk += nwarps) {
      const int d = static_cast<int>(blk / a.L), j = static_cast<int>(blk % a.L);
      const int64_t region = a.exp_region[d];
      const int64_t first = region + a.exp_base[d * (a.L + 1) + j] + a.exp_cnt[blk];
      const int64_t end = region + a.exp_base[d * (a.L + 1) + j + 1];
      for (int64_t row = first; row < end; ++row) {
        uint8_t* dst = a.recv_x + row * a.out_row_bytes;
        for (int c = lane; c < nchunk; c += 32) st16(dst + (static_cast<size_t>(c) << 4), zero);
        if (kKind == kCastRow || a.x_sf != nullptr)
          for (int g = lane; g < a.SW; g += 32) a.recv_sf[row * a.SW + g] = 0.f;
      }
    }
  }
}

template <int kKind, bool kExpand, bool kAtomic = false>
cudaError_t launch_one(const DispatchArgs& a, int num_sms, cudaStream_t stream) {
  auto kern = dispatch_kernel<kKind, kExpand, kAtomic>;
  int per_sm = 0;
  cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kCopyThreads, 0);
  if (err != cudaSuccess) return err;
  if (per_sm < 1) per_sm = 1;
  int64_t ctas = static_cast<int64_t>(num_sms) * per_sm;
  const int64_t need = ((a.zero_padding && a.E > a.num_tokens ? a.E : a.num_tokens) + kWarps - 1) / kWarps;
  if (ctas > need) ctas = need;
  if (ctas < 1) return cudaSuccess;
  kern<<<static_cast<unsigned>(ctas), kCopyThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_dispatch(const Geometry& g, const DispatchArgs& a, int num_sms,
                            cudaStream_t stream) {
  const bool cast = !g.x_fp8 && g.recv_fp8;
  if (cast) {
    return g.expand ? launch_one<kCastRow, true>(a, num_sms, stream)
                    : launch_one<kCastRow, false>(a, num_sms, stream);
  }
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

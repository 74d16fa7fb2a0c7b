// Per-token pieces shared by the dispatch kernels: a token's top-k lanes, the
// per-128-column FP8 cast of 16 columns, the sidecar rows, and the zeroing of
// alignment padding rows.
#pragma once

#include "ep_device.cuh"
#include "ep_internal.cuh"

namespace ep {
namespace {

struct TokenLanes {
  int e, d, slot, pos;
  int64_t row;  // row of the lane's deduplicated entry in the receive tensors (the
                // sidecars, and recv_x unless expanded); -1 for an invalid lane
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
  L.row = valid ? entry_row(a, L.d, L.slot, a.err) : -1;
  return L;
}

// The receive rows of recv_x a token's row goes to, gathered into s_row (one
// per deduplicated entry, or per valid lane when expanded) in lane order;
// returns how many. A row that may not be written (a packed row past the
// capacity, or in checked builds one outside the buffer) is left out and its
// error latched.
__device__ __forceinline__ int hidden_rows(const DispatchArgs& a, const TokenLanes& ln, int lane, bool expand,
                                           int64_t* s_row) {
  const unsigned hmask = expand ? ln.vmask : ln.rmask;
  int64_t row = -1;
  if ((hmask >> lane) & 1) {
    row = expand ? static_cast<int64_t>(a.exp_region[ln.d]) + ln.pos : ln.row;
    if (!row_usable(row, a.recv_rows, a.compact == 2, a.err)) row = -1;
  }
  const unsigned keep = __ballot_sync(kFullMask, row >= 0);
  if (row >= 0) s_row[__popc(keep & lanemask_lt())] = row;
  __syncwarp();
  return __popc(keep);
}

// One lane's 16 columns of a 128-column group (8 consecutive lanes form a
// group; all 32 lanes must call this together). fp32 scales: amax/448 and the
// product with the rounded reciprocal 448/amax. Packed scales: the smallest
// power of two 2^e >= amax/448, read off amax's exponent and mantissa
// (amax = m*2^k: e = k-8, or k-7 when m > 1.75), and the exact product with
// 2^-e. Both round each product to fp32, then to e4m3 (nearest even,
// saturating).
struct CastUnit {
  uint4 q;          // the 16 e4m3 codes
  float sf;         // fp32 scale of the group
  uint8_t sf_byte;  // packed scale byte e + 127
};

__device__ __forceinline__ CastUnit cast_unit(const uint4& lo, const uint4& hi, bool in_range, int sf_pack) {
  float f[16];
  const uint32_t wv[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 p = bf16x2_to_f32x2(in_range ? wv[i] : 0u);
    f[2 * i] = p.x;
    f[2 * i + 1] = p.y;
    amax = fmaxf(amax, fmaxf(fabsf(p.x), fabsf(p.y)));
  }
  amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 4));
  amax = fmaxf(amax, 1e-4f);
  const uint32_t ab = __float_as_uint(amax);
  const int e2 = static_cast<int>(ab >> 23) - 127 - 8 + ((ab & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  const float inv = sf_pack ? __uint_as_float(static_cast<uint32_t>(127 - e2) << 23) : __fdiv_rn(448.0f, amax);
  CastUnit c;
  c.q.x = f32x2_to_e4m3x2(__fmul_rn(f[0], inv), __fmul_rn(f[1], inv)) |
          f32x2_to_e4m3x2(__fmul_rn(f[2], inv), __fmul_rn(f[3], inv)) << 16;
  c.q.y = f32x2_to_e4m3x2(__fmul_rn(f[4], inv), __fmul_rn(f[5], inv)) |
          f32x2_to_e4m3x2(__fmul_rn(f[6], inv), __fmul_rn(f[7], inv)) << 16;
  c.q.z = f32x2_to_e4m3x2(__fmul_rn(f[8], inv), __fmul_rn(f[9], inv)) |
          f32x2_to_e4m3x2(__fmul_rn(f[10], inv), __fmul_rn(f[11], inv)) << 16;
  c.q.w = f32x2_to_e4m3x2(__fmul_rn(f[12], inv), __fmul_rn(f[13], inv)) |
          f32x2_to_e4m3x2(__fmul_rn(f[14], inv), __fmul_rn(f[15], inv)) << 16;
  c.sf = sf_pack ? 0.f : __fdiv_rn(amax, 448.0f);
  c.sf_byte = static_cast<uint8_t>(e2 + 127);
  return c;
}

// Sidecar rows of a token with top-k <= 8, all entries at once: lanes 4i..4i+3
// write entry i (the i-th deduplicated destination, in lane order), each lane
// two of its K routing values and three of its 2 + K metadata fields; the
// token's lanes' experts, destinations, weights and positions come by shuffle.
__device__ __forceinline__ void write_sidecars_k8(const DispatchArgs& a, const TokenLanes& ln, int s, int t,
                                                  int lane, bool kExpand) {
  const int K = a.K;
  const int n = __popc(ln.rmask);
  const int i = lane >> 2, q = lane & 3;
  const bool active = i < n;
  const int ri = active ? static_cast<int>(__fns(ln.rmask, 0, i + 1)) : 0;  // lane of entry i
  const int di = __shfl_sync(kFullMask, ln.d, ri);
  const int64_t mrow = __shfl_sync(kFullMask, ln.row, ri);
  // packed rows past the capacity (and, checked builds, rows outside the
  // buffer) are skipped; one lane per entry reports it
  const bool ok = active && row_usable(mrow, a.side_rows, a.compact == 2, q == 0 ? a.err : nullptr);
  const int k0 = 2 * q, k1 = 2 * q + 1;
  const int e0 = __shfl_sync(kFullMask, ln.e, k0), e1 = __shfl_sync(kFullMask, ln.e, k1);
  const int d0 = __shfl_sync(kFullMask, ln.d, k0), d1 = __shfl_sync(kFullMask, ln.d, k1);
  const float w0 = __shfl_sync(kFullMask, ln.w, k0), w1 = __shfl_sync(kFullMask, ln.w, k1);
  if (ok && a.recv_idx) {
    int64_t* r = a.recv_idx + mrow * K;
    if (k0 < K) r[k0] = d0 == di ? static_cast<int64_t>(e0 - di * a.L) : -1;
    if (k1 < K) r[k1] = d1 == di ? static_cast<int64_t>(e1 - di * a.L) : -1;
  }
  if (ok && a.recv_w) {
    float* r = a.recv_w + mrow * K;
    if (k0 < K) r[k0] = d0 == di ? w0 : 0.f;
    if (k1 < K) r[k1] = d1 == di ? w1 : 0.f;
  }
  if (a.recv_md) {
    int32_t* md = a.recv_md + mrow * (K + 2);
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int f = q + 4 * j;  // field f = 2 + k carries lane k's expanded row
      const int src = (f - 2) & 31;
      const int dk = __shfl_sync(kFullMask, ln.d, src);
      const int pk = kExpand ? __shfl_sync(kFullMask, ln.pos, src) : -1;
      if (ok && f < K + 2) md[f] = f == 0 ? s : (f == 1 ? t : ((kExpand && dk == di) ? pk : -1));
    }
  }
}

// Sidecar rows of each deduplicated destination of a token (row form): the
// routing of the lanes to that destination and the source metadata.
__device__ __forceinline__ void write_sidecars(const DispatchArgs& a, const TokenLanes& ln, int s, int t,
                                               int lane, bool kExpand) {
  if (a.recv_idx == nullptr && a.recv_w == nullptr && a.recv_md == nullptr) return;
  if (a.K <= 8) {
    write_sidecars_k8(a, ln, s, t, lane, kExpand);
    return;
  }
  // top-k above 8: one deduplicated destination at a time. Metadata field
  // f = 2 + k carries lane k's expanded row; with K up to 32 there are up to 34
  // fields, so a lane writes fields lane and lane + 32.
  const int f0_d = __shfl_sync(kFullMask, ln.d, (lane - 2) & 31);   // lane f-2 for f = lane
  const int f0_pos = __shfl_sync(kFullMask, ln.pos, (lane - 2) & 31);
  const int f1_d = __shfl_sync(kFullMask, ln.d, (lane + 30) & 31);  // f = lane + 32
  const int f1_pos = __shfl_sync(kFullMask, ln.pos, (lane + 30) & 31);
  unsigned m = ln.rmask;
  while (m) {
    const int rl = __ffs(m) - 1;
    m &= m - 1;
    const int dj = __shfl_sync(kFullMask, ln.d, rl);
    const int64_t mrow = __shfl_sync(kFullMask, ln.row, rl);
    // packed rows past the capacity (and, checked builds, rows outside the
    // buffer) are skipped; the same for every lane
    if (!row_usable(mrow, a.side_rows, a.compact == 2, lane == 0 ? a.err : nullptr)) continue;
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

// Expanded blocks padded to expert_alignment: zero the rows after each
// expert's lanes up to the next block start (and their scales). Warp gwarp of
// nwarps takes experts gwarp, gwarp + nwarps, ...
__device__ __forceinline__ void zero_padding_rows(const DispatchArgs& a, int64_t gwarp, int64_t nwarps,
                                                  int lane, bool with_scales) {
  const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
  const int nchunk = a.out_row_bytes >> 4;
  for (int64_t blk = gwarp; blk < a.E; blk += nwarps) {
    const int d = static_cast<int>(blk / a.L), j = static_cast<int>(blk % a.L);
    const int64_t region = a.exp_region[d];
    const int64_t first = region + a.exp_base[d * (a.L + 1) + j] + a.exp_cnt[blk];
    const int64_t end = region + a.exp_base[d * (a.L + 1) + j + 1];
    if (end > first && !row_in_bounds(end - 1, a.recv_rows, lane == 0 ? a.err : nullptr)) continue;
    for (int64_t row = first; row < end; ++row) {
      uint8_t* dst = a.recv_x + row * a.out_row_bytes;
      for (int c = lane; c < nchunk; c += 32) st16(dst + (static_cast<size_t>(c) << 4), zero);
      if (with_scales)
        for (int g = lane; g < a.SW; g += 32) a.recv_sf[row * a.SW + g] = 0.f;
    }
  }
}

}  // namespace
}  // namespace ep

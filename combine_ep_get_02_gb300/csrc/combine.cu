// Combine: gather each source token's expert-output rows and reduce them with
// the token's top-k weights.
//
// out[s][t] = bf16_rn(acc), acc = +0, then for k in lane order over the valid
// lanes acc = fma(w_k, y[row of lane k], acc) in fp32. The order of the fused
// multiply-adds is fixed, so the result is bitwise reproducible and equal to
// the sequential definition. One warp owns one token; each lane owns 8
// columns (one 16-byte chunk) per step and keeps the loads of all K rows of
// two steps in flight before it reduces.
#include "ep_device.cuh"
#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kWarps = kCopyThreads / 32;

template <bool kExpand, int kMaxK, int kSteps>
__global__ void __launch_bounds__(kCopyThreads) combine_kernel(CombineArgs a) {
  __shared__ const uint16_t* s_ptr[kWarps][kMaxK];
  __shared__ float s_w[kWarps][kMaxK];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kWarps;
  const int nchunk = a.H >> 3;  // 8 bf16 per chunk
  pdl_launch_dependents();
  pdl_wait();

  // A work unit is one token's column range (a token is split into a.splits
  // ranges of a.split_chunks 16-byte chunks when tokens are too few to keep
  // every warp busy to the end). In the row form warps take units from the
  // workspace's work queue (a token's cost follows its number of distinct
  // rows); expanded units keep a fixed share. Lane k of the warp carries top-k
  // lane k of the unit's token; the next unit is taken, and its routing
  // (expert, slot or position, weight) loaded, while the current unit's rows
  // stream.
  const int64_t units = a.num_tokens * a.splits;
  int64_t e_next = -1;
  int r_next = -1;
  float w_next = 0.f;
  auto load_raw = [&](int64_t unit) {
    e_next = -1;
    r_next = -1;
    w_next = 0.f;
    if (unit < units && lane < a.K) {
      const int64_t i = (unit / a.splits) * a.K + lane;
      e_next = __ldg(a.topk_idx + i);
      r_next = __ldg((kExpand ? a.exp_pos : a.slot_map) + i);
      w_next = __ldg(a.topk_w + i);
    }
  };
  const int64_t gwarp = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  UnitStream us = start_units(gwarp, nwarps, units, !kExpand);
  load_raw(us.cur);
  while (us.cur < units) {
    const int64_t unit = us.cur;
    const int64_t tok = unit / a.splits;
    const int c_begin = static_cast<int>(unit - tok * a.splits) * a.split_chunks;
    const int c_end = min(nchunk, c_begin + a.split_chunks);
    const int64_t e = e_next;
    const int r = r_next;
    const float w_cur = w_next;
    const int64_t after = take_unit(us, a.queue, lane);
    load_raw(us.nxt);
    if (lane < kMaxK) {
      const uint16_t* p = nullptr;
      float w = 0.f;
      if (e >= 0 && e < a.E && r >= 0) {
        const int d = static_cast<int>(e) / a.L;
        const int64_t row = kExpand ? static_cast<int64_t>(a.exp_region[d]) + r : entry_row(a, d, r, a.err);
        // a packed row past the capacity was never received: the lane is left
        // out and kErrOverflow latched (checked builds: rows outside y too)
        if (row_usable(row, a.y_rows, a.compact == 2, a.err)) {
          p = a.y + row * a.H;
          w = w_cur;
        }
      }
      s_ptr[warp][lane] = p;
      s_w[warp][lane] = w;
    }
    __syncwarp();
    const uint16_t* ptr[kMaxK];
    float wk[kMaxK];
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
      ptr[k] = s_ptr[warp][k];
      wk[k] = s_w[warp][k];
    }
    uint16_t* orow = a.out + tok * a.H;
    for (int c0 = c_begin + lane; c0 < c_end; c0 += 32 * kSteps) {
      uint4 v[kSteps][kMaxK];
#pragma unroll
      for (int h = 0; h < kSteps; ++h) {
        const int c = c0 + h * 32;
#pragma unroll
        for (int k = 0; k < kMaxK; ++k)
          if (ptr[k] != nullptr && c < c_end) v[h][k] = ld_ro16(ptr[k] + (static_cast<size_t>(c) << 3));
      }
#pragma unroll
      for (int h = 0; h < kSteps; ++h) {
        const int c = c0 + h * 32;
        if (c >= c_end) continue;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
#pragma unroll
        for (int k = 0; k < kMaxK; ++k) {
          if (ptr[k] == nullptr) continue;
          const uint32_t wv[4] = {v[h][k].x, v[h][k].y, v[h][k].z, v[h][k].w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = bf16x2_to_f32x2(wv[i]);
            acc[2 * i] = __fmaf_rn(wk[k], f.x, acc[2 * i]);
            acc[2 * i + 1] = __fmaf_rn(wk[k], f.y, acc[2 * i + 1]);
          }
        }
        uint4 o;
        o.x = f32x2_to_bf16x2(acc[0], acc[1]);
        o.y = f32x2_to_bf16x2(acc[2], acc[3]);
        o.z = f32x2_to_bf16x2(acc[4], acc[5]);
        o.w = f32x2_to_bf16x2(acc[6], acc[7]);
        st16(orow + (static_cast<size_t>(c) << 3), o);
      }
    }
    __syncwarp();  // s_ptr / s_w are rewritten by the next unit
    advance_units(us, after);
  }
  leave_queue(us, a.queue, lane);
}

template <bool kExpand, int kMaxK, int kSteps>
cudaError_t launch_one(const CombineArgs& args, int num_sms, cudaStream_t stream) {
  auto kern = combine_kernel<kExpand, kMaxK, kSteps>;
  int per_sm = resident_ctas(reinterpret_cast<const void*>(kern), kCopyThreads, 0);
  if (per_sm < 0) return cudaErrorUnknown;
  if (per_sm < 1) per_sm = 1;
  CombineArgs a = args;
  // Split tokens into column ranges until every warp gets about 16 units, so
  // that the last wave is short; a range is a whole number of lane sweeps, at
  // least two (a one-sweep range pays its routing loads for too few bytes)
  // unless two-sweep ranges would leave warps without a unit.
  const int64_t warps = static_cast<int64_t>(num_sms) * per_sm * kWarps;
  const int nchunk = a.H >> 3;
  const int sweep = 32 * kSteps;
  int max_splits = (nchunk + 2 * sweep - 1) / (2 * sweep);
  if (a.num_tokens * max_splits < warps) max_splits = (nchunk + sweep - 1) / sweep;
  int64_t want = a.num_tokens > 0 ? (16 * warps + a.num_tokens - 1) / a.num_tokens : 1;
  if (want > max_splits) want = max_splits;
  if (want < 1) want = 1;
  a.split_chunks = static_cast<int>(((nchunk + want - 1) / want + sweep - 1) / sweep * sweep);
  a.splits = (nchunk + a.split_chunks - 1) / a.split_chunks;
  if (a.splits < 1) a.splits = 1;
  int64_t ctas = static_cast<int64_t>(num_sms) * per_sm;
  const int64_t need = (a.num_tokens * a.splits + kWarps - 1) / kWarps;
  if (ctas > need) ctas = need;
  if (ctas < 1) return cudaSuccess;
  return launch_chained(kern, dim3(static_cast<unsigned>(ctas)), dim3(kCopyThreads), 0, stream, a);
}

}  // namespace

cudaError_t launch_combine(const Geometry& g, const CombineArgs& a, int num_sms,
                           cudaStream_t stream) {
  if (g.K <= 8)
    return g.expand ? launch_one<true, 8, 2>(a, num_sms, stream)
                    : launch_one<false, 8, 2>(a, num_sms, stream);
  if (g.K <= 16)
    return g.expand ? launch_one<true, 16, 1>(a, num_sms, stream)
                    : launch_one<false, 16, 1>(a, num_sms, stream);
  return g.expand ? launch_one<true, 32, 1>(a, num_sms, stream)
                  : launch_one<false, 32, 1>(a, num_sms, stream);
}

}  // namespace ep

// Dispatch of rows that travel unchanged (bf16 -> bf16, or pre-cast e4m3 ->
// e4m3) with the Blackwell bulk-copy engine instead of per-lane stores.
//
// One warp owns one source token at a time, as in the register path: its lanes
// read the routing, place the destination rows and write the sidecars. The
// hidden row goes through shared memory: one elected lane issues a bulk copy
// (cp.async.bulk, completion counted on an mbarrier) of the row into a stage
// buffer, then one bulk copy from the stage to each destination row. Each warp
// has two stages, so the next row (or the next piece of a long row) loads while
// the current one is being stored. No lane touches the row's bytes.
//
// Every wait on an mbarrier is bounded: past the limit the kernel latches
// kErrTimeout in the workspace, lets its copies finish and returns.
#include "dispatch_common.cuh"
#include "ep_device.cuh"
#include "ep_internal.cuh"

namespace ep {

namespace {

constexpr int kBulkWarps = kBulkThreads / 32;
constexpr int kBulkStages = 2;
// One CTA (four warps, four rows in flight) per SM: on GB300 more concurrent
// row streams measured slower (2-6% on 4K-14K-byte rows), not faster.
constexpr int kBulkMaxCtasPerSm = 1;
static_assert(kBulkThreads / 32 * 2 * kBulkStageMax <= 160 * 1024, "bulk stages exceed shared memory");

template <bool kExpand>
__global__ void __launch_bounds__(kBulkThreads) dispatch_bulk_kernel(DispatchArgs a, int stage_bytes) {
  extern __shared__ __align__(128) uint8_t stage_mem[];
  __shared__ __align__(8) uint64_t bar[kBulkWarps][kBulkStages];
  __shared__ int64_t s_row[kBulkWarps][kMaxTopk];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gwarp = static_cast<int64_t>(blockIdx.x) * kBulkWarps + warp;
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * kBulkWarps;
  const int row_bytes = a.in_row_bytes;  // == out_row_bytes for an unchanged row
  const int pieces = (row_bytes + stage_bytes - 1) / stage_bytes;

  // shared-memory addresses of stage s and of its barrier
  const uint32_t st0 = smem_addr(stage_mem + static_cast<size_t>(warp) * kBulkStages * stage_bytes);
  const uint32_t bar0 = smem_addr(&bar[warp][0]);
  auto st_addr = [&](int s) { return st0 + static_cast<uint32_t>(s * stage_bytes); };
  auto bar_addr = [&](int s) { return bar0 + static_cast<uint32_t>(s * sizeof(uint64_t)); };
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < kBulkStages; ++s) mbar_init(bar_addr(s));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  pdl_launch_dependents();
  pdl_wait();

  // pieces run (token, 0..pieces-1) for the warp's tokens in turn (in the row
  // form its fixed two, then those it takes from the work queue); consecutive
  // pieces alternate between the two stages.
  // All lanes keep the same bookkeeping; lane 0 issues the copies.
  uint32_t parity = 0;   // bit s: parity of stage s's next completion
  uint32_t pending = 0;  // bit s: a load into stage s is in flight
  auto load_piece = [&](int64_t tok, int piece, int s) {
    if (lane == 0) {
      const int off = piece * stage_bytes;
      const int n = min(stage_bytes, row_bytes - off);
      bulk_wait_reads();  // the stores of the piece that last used a stage are done with it
      bulk_load(st_addr(s), a.x + tok * row_bytes + off, static_cast<uint32_t>(n), bar_addr(s));
    }
    pending |= 1u << s;
  };

  bool ok = true;
  int stage = 0;
  UnitStream us = start_units(gwarp, nwarps, a.num_tokens, !kExpand);
  if (us.cur < a.num_tokens) load_piece(us.cur, 0, 0);
  RawLane next = fetch_lane(a, us.cur, lane, kExpand, false);
  while (us.cur < a.num_tokens) {
    const int64_t tok = us.cur;
    const int s_rank = static_cast<int>(tok / a.T);
    const int t = static_cast<int>(tok - static_cast<int64_t>(s_rank) * a.T);
    const RawLane cur = next;
    const int64_t after = take_unit(us, a.queue, lane);
    next = fetch_lane(a, us.nxt, lane, kExpand, false);
    const TokenLanes ln = lanes_of(a, cur, tok, lane, kExpand, false);
    const int nh = hidden_rows(a, ln, lane, kExpand, s_row[warp]);

    for (int piece = 0; piece < pieces; ++piece) {
      // start the following piece in the other stage
      const bool last = piece + 1 == pieces;
      const int64_t ntok = last ? us.nxt : tok;
      if (ntok < a.num_tokens) load_piece(ntok, last ? 0 : piece + 1, stage ^ 1);
      // store this piece to every destination row once it has landed
      int landed = 1;
      if (lane == 0) landed = mbar_wait(bar_addr(stage), (parity >> stage) & 1u, kBulkWaitLimit);
      landed = __shfl_sync(kFullMask, landed, 0);
      if (!landed) {
        ok = false;
        break;
      }
      parity ^= 1u << stage;
      pending &= ~(1u << stage);
      if (lane == 0) {
        const int off = piece * stage_bytes;
        const uint32_t n = static_cast<uint32_t>(min(stage_bytes, row_bytes - off));
        for (int j = 0; j < nh; ++j) bulk_store(a.recv_x + s_row[warp][j] * a.out_row_bytes + off, st_addr(stage), n);
        bulk_commit();
      }
      stage ^= 1;
    }
    if (!ok) break;

    if (a.x_sf != nullptr) {  // pre-cast FP8: the scale words travel verbatim
      const float* ssrc = a.x_sf + tok * a.SW;
      for (int g = lane; g < a.SW; g += 32) {
        const float v = ssrc[g];
        for (int j = 0; j < nh; ++j) a.recv_sf[s_row[warp][j] * a.SW + g] = v;
      }
    }
    write_sidecars(a, ln, s_rank, t, lane, kExpand);
    __syncwarp();  // s_row is rewritten by the next token
    advance_units(us, after);
  }

  if (lane == 0) {
    // never leave with a load still writing this warp's stages
#pragma unroll
    for (int s = 0; s < kBulkStages; ++s)
      if (((pending >> s) & 1u) && !mbar_wait(bar_addr(s), (parity >> s) & 1u, kBulkWaitLimit)) ok = false;
    bulk_wait_all();
    if (!ok) atomicOr(a.err, kErrTimeout);
  }
  __syncwarp();
  leave_queue(us, a.queue, lane);

  if (kExpand && a.zero_padding) zero_padding_rows(a, gwarp, nwarps, lane, a.x_sf != nullptr);
}

}  // namespace

int dispatch_bulk_stage_bytes(int row_bytes) {
  // whole rows up to kBulkStageMax bytes, else equal 16-byte-multiple pieces
  const int pieces = (row_bytes + kBulkStageMax - 1) / kBulkStageMax;
  return ((row_bytes + pieces - 1) / pieces + 15) & ~15;
}

cudaError_t launch_dispatch_bulk(const Geometry& g, const DispatchArgs& a, int num_sms, cudaStream_t stream) {
  const int stage_bytes = dispatch_bulk_stage_bytes(a.in_row_bytes);
  size_t smem = static_cast<size_t>(kBulkWarps) * kBulkStages * stage_bytes;
  // One CTA per SM, whatever the stage size: the grid is one CTA per SM, and
  // the launch may be placed while the kernel before it drains (see pdl_wait),
  // when SMs with free shared memory could otherwise take several CTAs each
  // and leave others without. So ask for more than half an SM's shared memory.
  int dev = 0, sm_smem = 0;
  cudaError_t qerr;
  if ((qerr = cudaGetDevice(&dev)) != cudaSuccess ||
      (qerr = cudaDeviceGetAttribute(&sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess)
    return qerr;
  const size_t half = static_cast<size_t>(sm_smem) / 2 + 1024;
  if (smem < half) smem = half;
  auto kern = g.expand ? dispatch_bulk_kernel<true> : dispatch_bulk_kernel<false>;
  int per_sm = resident_ctas(reinterpret_cast<const void*>(kern), kBulkThreads, smem);
  if (per_sm < 0) return cudaErrorUnknown;
  if (per_sm > kBulkMaxCtasPerSm) per_sm = kBulkMaxCtasPerSm;
  if (per_sm < 1) per_sm = 1;
  int64_t ctas = static_cast<int64_t>(num_sms) * per_sm;
  const int64_t work = (a.zero_padding && a.E > a.num_tokens) ? a.E : a.num_tokens;
  const int64_t need = (work + kBulkWarps - 1) / kBulkWarps;
  if (ctas > need) ctas = need;
  if (ctas < 1) return cudaSuccess;
  return launch_chained(kern, dim3(static_cast<unsigned>(ctas)), dim3(kBulkThreads), smem, stream, a, stage_bytes);
}

}  // namespace ep

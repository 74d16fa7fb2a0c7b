// Internal declarations shared by the kernels and the C-ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ep_get.h"

namespace ep {

constexpr int kLayoutThreads = 256;  // one thread per token in the layout kernels
constexpr int kRowsThreads = 256;    // the row-form layout kernel's CTA
constexpr int kLayoutWarps = kLayoutThreads / 32;
constexpr int kMaxRanks = 64;
constexpr int kMaxTopk = 32;
constexpr int kMaxExperts = 4096;
constexpr int kMaxScaleGroups = 128;  // FP8 receive: hidden <= 128 * 128
constexpr int kCopyThreads = 256;     // dispatch / combine CTA size (8 warps)
constexpr int kBulkThreads = 128;     // bulk-copy dispatch CTA size (4 warps)
constexpr int kBulkStageMax = 16384;  // bytes of one shared-memory stage of the bulk-copy dispatch
constexpr int64_t kBulkAutoMinBytes = int64_t{32} << 20;  // input rows from which copy_path 0 picks bulk
constexpr int kMaxPrologueCtas = 64;
constexpr int kMaxSortRows = 8192;   // rows of one segment the comparison sort handles

// device error bits latched in the workspace header
constexpr uint32_t kErrBadTopk = 1u;
constexpr uint32_t kErrOverflow = 2u;
constexpr uint32_t kErrTimeout = 4u;  // a bounded wait on a copy gave up
constexpr uint32_t kErrBounds = 8u;   // checked builds: a computed row fell outside its buffer

// Checked builds (-DEP_CHECKED, libep_get_checked.so) test every computed row
// index against its buffer before the access; one outside latches kErrBounds
// and the access is skipped. Ordinary builds compile the tests away.
#ifdef EP_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

// Sizes derived from an ep_config_t that passed validation.
struct Geometry {
  int R, n_so, n_su, E, L, K, T, M, H, G;
  int x_fp8, recv_fp8, expand, align, zero_padding, sf_pack;
  int compact;  // receive rows: 0 at their slots, 1 compact windows, 2 packed back to back
  int copy_path;  // 0 automatic, 1 register copies, 2 bulk copies (rows that travel unchanged)
  int SW;  // 32-bit words of one row's scale sidecar: G, or ceil(G/4) packed
  int64_t region_rows;  // rows of one destination region in the row form: R * M
  int64_t entry_rows;   // rows of the receive tensors holding deduplicated entries (recv_x
                        // unless expanded, and the sidecars): R * R * M, or the packed capacity
  int64_t num_tokens;   // R * T
};

// Byte offsets of the workspace pieces.
struct Workspace {
  size_t err;            // uint32: sticky device error bits
  size_t done;           // uint32: arrival counter of the layout kernel (returns to 0)
  size_t dispatch_queue; // 2 x uint64: the dispatch's work queue (returns to 0)
  size_t combine_queue;  // 2 x uint64: the combine's work queue (returns to 0)
  size_t exp_off;        // int32 [R][E]: lanes of each expert from lower source ranks (expand)
  size_t total;
};

// Dynamic distribution of a kernel's work units (source tokens, or token
// column ranges) over its warps. In the row form a token's cost follows its
// number of distinct destinations (1 to min(K, R)), so a fixed share per warp
// leaves the launch waiting on its heaviest warps; there a warp's first two
// units are fixed (its warp index, then that plus the grid's warps) and after
// those it takes the next unit from a counter in the workspace header. Each
// take is issued one unit before the warp needs it, so the atomic's round trip
// overlaps the current unit. Every warp leaves the queue once, and the last to
// leave (a second counter) returns both counters to zero for the next launch.
// Expanded tokens all carry about K rows; they keep the fixed share (units
// gwarp, gwarp + nwarps, ...), as does a launch whose units fit two per warp.
struct WorkQueue {
  unsigned long long* next;
  unsigned long long* left;
};

Workspace workspace_layout(const Geometry& g);
int make_geometry(const ep_config_t* cfg, Geometry* g);  // returns EP_OK or an error
// The layout's pointer arguments (present, aligned): EP_OK or EP_ERR_INVALID_ARG.
int check_layout_args(const Geometry& g, const int64_t* topk_idx, const ep_layout_t* layout);

struct LayoutArgs {
  const int64_t* topk_idx;
  int32_t* num_tokens_per_rank;
  int32_t* num_tokens_per_expert;
  uint8_t* is_token_in_rank;
  int32_t* slot_map;
  int32_t* recv_cnt;
  int32_t* recv_psum;
  int32_t* recv_region;  // may be null
  int32_t* exp_cnt;
  int32_t* exp_base;
  int32_t* exp_region;
  int32_t* exp_pos;
  uint32_t* err;
  uint32_t* done;
  int32_t* exp_off;
  int R, n_so, n_su, E, L, K, T, M, expand, align;
  int topk_vec;       // topk_idx rows can be read as 16-byte pairs
  uint32_t l_magic;   // e / L == __umulhi(e, l_magic) for e, L < 2^16
  uint32_t so_magic;  // j / n_so == __umulhi(j, so_magic) for j, n_so < 2^16 (0: n_so == 1)
  int C;   // CTAs (one cluster) per source rank
  int TB;  // tokens per CTA
  int EB;  // experts whose per-source totals each CTA of a cluster adds up (row-form kernel)
};

struct DispatchArgs {
  const uint8_t* x;
  const float* x_sf;
  const int64_t* topk_idx;
  const float* topk_w;
  const int32_t* slot_map;
  const int32_t* exp_pos;
  const int32_t* exp_region;
  const int32_t* recv_psum;    // compact and packed receive rows only
  const int32_t* recv_region;  // packed receive rows only
  const int32_t* exp_cnt;    // zero padding only
  const int32_t* exp_base;   // zero padding only
  int32_t* send_counters;    // atomic-slot comparison path only: [R src][R dst]
  uint8_t* recv_x;
  float* recv_sf;
  int64_t* recv_idx;
  float* recv_w;
  int32_t* recv_md;
  uint32_t* err;             // the workspace's device error bits (null: none)
  WorkQueue queue;           // the workspace's dispatch work queue
  int64_t recv_rows;         // rows of recv_x and recv_sf (the capacity when packed)
  int64_t side_rows;         // rows of the sidecar tensors
  int R, E, L, K, T, H, G, M, compact, zero_padding, n_so, n_su, sf_pack;
  int SW;  // 32-bit words of one row's scale sidecar
  int64_t region_rows;
  int64_t num_tokens;
  int in_row_bytes, out_row_bytes;
  int splits;     // register-path work units per token (column ranges); 1 elsewhere
  int split_len;  // 16-byte chunks (row copy) or 16-column units (cast) per range
};

// The post-hoc sort of the comparison path: permutes each (destination, row
// block) segment of a receive buffer into source-token order.
struct SortArgs {
  const uint8_t* in_x;
  const float* in_sf;
  const int64_t* in_idx;
  const float* in_w;
  const int32_t* in_md;
  uint8_t* out_x;
  float* out_sf;
  int64_t* out_idx;
  float* out_w;
  int32_t* out_md;
  const int32_t* send_counters;  // [R src][R dst]: rows each source sent each destination
  int R, K, M, SW, n_so, n_su;
  int64_t region_rows;
  int row_bytes;
};

struct CombineArgs {
  const uint16_t* y;
  const int64_t* topk_idx;
  const float* topk_w;
  const int32_t* slot_map;
  const int32_t* exp_pos;
  const int32_t* exp_region;
  const int32_t* recv_psum;    // compact and packed receive rows only
  const int32_t* recv_region;  // packed receive rows only
  uint16_t* out;
  uint32_t* err;     // the workspace's device error bits
  WorkQueue queue;   // the workspace's combine work queue
  int64_t y_rows;    // rows of y (the capacity when packed)
  int E, L, K, T, H, R, M, compact;
  int splits;        // column ranges per token (work units per token)
  int split_chunks;  // 16-byte chunks per range
  int64_t region_rows;
  int64_t num_tokens;
};

cudaError_t launch_layout(const Geometry& g, const LayoutArgs& a, int num_prologue_sms,
                          cudaStream_t stream);
// Rows that travel unchanged, through shared memory with bulk copies
// (dispatch_bulk.cu); the stage size a row of row_bytes is split into.
cudaError_t launch_dispatch_bulk(const Geometry& g, const DispatchArgs& a, int num_sms, cudaStream_t stream);
int dispatch_bulk_stage_bytes(int row_bytes);
cudaError_t launch_dispatch(const Geometry& g, const DispatchArgs& a, int num_sms,
                            cudaStream_t stream);
cudaError_t launch_dispatch_atomic(const Geometry& g, const DispatchArgs& a, int num_sms,
                                   cudaStream_t stream);
cudaError_t launch_sort(const Geometry& g, const SortArgs& a, cudaStream_t stream);
cudaError_t launch_combine(const Geometry& g, const CombineArgs& a, int num_sms,
                           cudaStream_t stream);

int device_sm_count();

// Launch `kernel` with programmatic stream serialization (see pdl_wait): it may
// be placed on the SMs while the previous kernel on the stream drains; it waits
// for that kernel before it touches global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_chained(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                           Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// Resident CTAs per SM of `kernel` at `threads` threads and `smem` bytes of
// dynamic shared memory on the current device, raising the kernel's dynamic
// shared-memory limit first when smem needs it. Asked of the runtime once per
// (kernel, threads, smem, device) and kept, so a launch pays for neither query
// again; the limit is only ever raised. Returns the count (>= 0) or -1 if a
// runtime call failed.
int resident_ctas(const void* kernel, int threads, size_t smem);

// Row of a deduplicated (token, destination d) entry with row-form slot
// `slot` in the receive tensors (Args: DispatchArgs or CombineArgs):
//   row form  d*R*M + slot;
//   compact   d*R*M + recv_psum[d][rb-1] + slot - rb*M with rb = slot / M (the
//             destination's entries packed from the start of its window in
//             row-block order, PR #690 Direct Recv X; recv_psum[d][-1] = 0);
//   packed    the same with recv_region[d] (the entries of the destinations
//             before d) in place of d*R*M.
// Checked builds test the slot's row block before reading recv_psum: one
// outside [0, R) latches kErrBounds and gives -1.
template <class Args>
__device__ __forceinline__ int64_t entry_row(const Args& a, int d, int slot, uint32_t* err) {
  const int64_t window = static_cast<int64_t>(d) * a.region_rows;
  if (a.compact == 0) return window + slot;
  const int rb = slot / a.M;
  if (kChecked && (slot < 0 || rb >= a.R)) {
    if (err != nullptr) atomicOr(err, kErrBounds);
    return -1;
  }
  const int before = rb == 0 ? 0 : __ldg(a.recv_psum + d * a.R + rb - 1);
  const int64_t base = a.compact == 1 ? window : static_cast<int64_t>(__ldg(a.recv_region + d));
  return base + before + slot - static_cast<int64_t>(rb) * a.M;
}

// The units of one warp in order: `cur` is being worked on, `nxt` comes next
// (known one unit ahead, so its routing can load during `cur`).
struct UnitStream {
  int64_t cur, nxt;
  int64_t nwarps, units;
  bool dynamic;  // units beyond the fixed two per warp come from the queue
};

__device__ __forceinline__ UnitStream start_units(int64_t gwarp, int64_t nwarps, int64_t units, bool queue) {
  return UnitStream{gwarp, gwarp + nwarps, nwarps, units, queue && units > 2 * nwarps};
}

// Issue the take of the unit after `nxt` (all lanes get it); pass the result
// to advance_units once the current unit is done.
__device__ __forceinline__ int64_t take_unit(const UnitStream& u, const WorkQueue& q, int lane) {
  if (!u.dynamic) return u.nxt + u.nwarps;  // the fixed share
  unsigned long long v = 0;
  if (lane == 0) v = atomicAdd(q.next, 1ull);
  return 2 * u.nwarps + static_cast<int64_t>(__shfl_sync(0xFFFFFFFFu, v, 0));
}

__device__ __forceinline__ void advance_units(UnitStream& u, int64_t after) {
  u.cur = u.nxt;
  u.nxt = after;
}

// The calling warp has run out of units and is done with the queue; the last
// of the grid's warps to leave resets it.
__device__ __forceinline__ void leave_queue(const UnitStream& u, const WorkQueue& q, int lane) {
  if (u.dynamic && lane == 0) {
    __threadfence();
    if (atomicAdd(q.left, 1ull) == static_cast<unsigned long long>(u.nwarps) - 1ull) {
      atomicExch(q.next, 0ull);
      atomicExch(q.left, 0ull);
    }
  }
  __syncwarp();
}

// Checked builds: is row inside [0, rows)? If not, latch kErrBounds (when there
// is an error word) and tell the caller to skip the access.
__device__ __forceinline__ bool row_in_bounds(int64_t row, int64_t rows, uint32_t* err) {
  if (!kChecked || (row >= 0 && row < rows)) return true;
  if (err != nullptr) atomicOr(err, kErrBounds);
  return false;
}

// Whether a computed receive row may be accessed. A packed row at or past the
// capacity (`rows`) is an entry that does not fit: it latches kErrOverflow and
// is skipped, in every build (never dropped silently). Checked builds also
// test [0, rows) (kErrBounds); -1 (a row a check already refused) is skipped.
__device__ __forceinline__ bool row_usable(int64_t row, int64_t rows, bool packed, uint32_t* err) {
  if (row < 0) return false;
  if (packed && row >= rows) {
    if (err != nullptr) atomicOr(err, kErrOverflow);
    return false;
  }
  return row_in_bounds(row, rows, err);
}

}  // namespace ep

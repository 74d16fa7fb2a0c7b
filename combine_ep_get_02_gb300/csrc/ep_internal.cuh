// Internal declarations shared by the kernels and the C-ABI layer.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ep_get.h"

namespace ep {

constexpr int kLayoutThreads = 256;  // one thread per token in the layout kernels
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
  int x_fp8, recv_fp8, expand, align, compact, zero_padding, sf_pack;
  int copy_path;  // 0 automatic, 1 register copies, 2 bulk copies (rows that travel unchanged)
  int SW;  // 32-bit words of one row's scale sidecar: G, or ceil(G/4) packed
  int64_t region_rows;  // rows of one destination region in the row form: R * M
  int64_t num_tokens;   // R * T
};

// Byte offsets of the workspace pieces.
struct Workspace {
  size_t err;      // uint32: sticky device error bits
  size_t done;     // uint32: arrival counter of the layout kernel (returns to 0)
  size_t exp_off;  // int32 [R][E]: lanes of each expert from lower source ranks (expand)
  size_t total;
};

Workspace workspace_layout(const Geometry& g);
int make_geometry(const ep_config_t* cfg, Geometry* g);  // returns EP_OK or an error

struct LayoutArgs {
  const int64_t* topk_idx;
  int32_t* num_tokens_per_rank;
  int32_t* num_tokens_per_expert;
  uint8_t* is_token_in_rank;
  int32_t* slot_map;
  int32_t* recv_cnt;
  int32_t* recv_psum;
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
  int C;   // CTAs (one cluster) per source rank
  int TB;  // tokens per CTA
};

struct DispatchArgs {
  const uint8_t* x;
  const float* x_sf;
  const int64_t* topk_idx;
  const float* topk_w;
  const int32_t* slot_map;
  const int32_t* exp_pos;
  const int32_t* exp_region;
  const int32_t* recv_psum;  // compact receive rows only
  const int32_t* exp_cnt;    // zero padding only
  const int32_t* exp_base;   // zero padding only
  int32_t* send_counters;    // atomic-slot comparison path only: [R src][R dst]
  uint8_t* recv_x;
  float* recv_sf;
  int64_t* recv_idx;
  float* recv_w;
  int32_t* recv_md;
  uint32_t* err;             // the workspace's device error bits (null: none)
  int64_t recv_rows;         // rows of recv_x and recv_sf (checked builds)
  int R, E, L, K, T, H, G, M, compact, zero_padding, n_so, n_su, sf_pack;
  int SW;  // 32-bit words of one row's scale sidecar
  int64_t region_rows;
  int64_t num_tokens;
  int in_row_bytes, out_row_bytes;
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
  const int32_t* recv_psum;  // compact receive rows only
  uint16_t* out;
  uint32_t* err;     // the workspace's device error bits
  int64_t y_rows;    // rows of y (checked builds)
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

// Resident CTAs per SM of `kernel` at `threads` threads and `smem` bytes of
// dynamic shared memory on the current device, raising the kernel's dynamic
// shared-memory limit first when smem needs it. Asked of the runtime once per
// (kernel, threads, smem, device) and kept, so a launch pays for neither query
// again; the limit is only ever raised. Returns the count (>= 0) or -1 if a
// runtime call failed.
int resident_ctas(const void* kernel, int threads, size_t smem);

// Receive row inside destination d's region of a row-form slot: the slot, or
// (compact) the exclusive prefix of d's receive counts before the slot's row
// block plus the slot's offset in that block.
__device__ __forceinline__ int recv_row_of_slot(int slot, int d, int R, int M, int compact,
                                                const int32_t* recv_psum) {
  if (!compact) return slot;
  const int rb = slot / M;
  const int before = rb == 0 ? 0 : __ldg(recv_psum + d * R + rb - 1);
  return before + slot - rb * M;
}

// Checked builds: is row inside [0, rows)? If not, latch kErrBounds (when there
// is an error word) and tell the caller to skip the access.
__device__ __forceinline__ bool row_in_bounds(int64_t row, int64_t rows, uint32_t* err) {
  if (!kChecked || (row >= 0 && row < rows)) return true;
  if (err != nullptr) atomicOr(err, kErrBounds);
  return false;
}

}  // namespace ep

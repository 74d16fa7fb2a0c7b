// C ABI: argument validation, workspace layout, launches.
//
// Every host-detectable problem is reported before anything is enqueued
// (PR #690 review: guard unsupported combinations instead of accepting them).
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <vector>

#include "ep_device.cuh"
#include "ep_internal.cuh"

namespace ep {

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

int cuda_status(cudaError_t e) { return e == cudaSuccess ? EP_OK : EP_ERR_CUDA; }

__global__ void diag_e4m3_kernel(uint32_t first, int64_t n, uint8_t* out) {
  const int64_t i0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 2;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * 2;
  for (int64_t i = i0; i < n; i += stride) {
    const float a = __uint_as_float(first + static_cast<uint32_t>(i));
    const float b = __uint_as_float(first + static_cast<uint32_t>(i + 1));
    const uint32_t q = f32x2_to_e4m3x2(a, b);
    out[i] = static_cast<uint8_t>(q & 0xFF);
    if (i + 1 < n) out[i + 1] = static_cast<uint8_t>(q >> 8);
  }
}

__global__ void diag_bf16_kernel(uint32_t first, int64_t n, uint16_t* out) {
  const int64_t i0 = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) * 2;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x * 2;
  for (int64_t i = i0; i < n; i += stride) {
    const float a = __uint_as_float(first + static_cast<uint32_t>(i));
    const float b = __uint_as_float(first + static_cast<uint32_t>(i + 1));
    const uint32_t h = f32x2_to_bf16x2(a, b);
    out[i] = static_cast<uint16_t>(h & 0xFFFF);
    if (i + 1 < n) out[i + 1] = static_cast<uint16_t>(h >> 16);
  }
}

}  // namespace

int resident_ctas(const void* kernel, int threads, size_t smem) {
  struct Known {
    const void* kernel;
    int threads;
    size_t smem;
    int device;
    int ctas;
  };
  struct Limit {  // the largest dynamic shared-memory limit set on a kernel so far
    const void* kernel;
    int device;
    size_t smem;
  };
  static std::mutex mu;
  static std::vector<Known> known;
  static std::vector<Limit> limits;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  std::lock_guard<std::mutex> lock(mu);
  if (smem > 48 * 1024) {  // raise the kernel's limit when this launch needs more; never lower it
    Limit* lim = nullptr;
    for (Limit& l : limits)
      if (l.kernel == kernel && l.device == dev) lim = &l;
    if (lim == nullptr || lim->smem < smem) {
      if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
          cudaSuccess)
        return -1;
      if (lim == nullptr) limits.push_back({kernel, dev, smem});
      else lim->smem = smem;
    }
  }
  for (const Known& e : known)
    if (e.kernel == kernel && e.threads == threads && e.smem == smem && e.device == dev) return e.ctas;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess) return -1;
  known.push_back({kernel, threads, smem, dev, n});
  return n;
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

int make_geometry(const ep_config_t* c, Geometry* g) {
  if (c == nullptr) return EP_ERR_INVALID_ARG;
  if (c->num_scaleout_ranks < 1 || c->num_scaleup_ranks < 1) return EP_ERR_INVALID_ARG;
  const int64_t R = static_cast<int64_t>(c->num_scaleout_ranks) * c->num_scaleup_ranks;
  if (R > kMaxRanks) return EP_ERR_UNSUPPORTED;
  if (c->num_experts < R || c->num_experts % R != 0) return EP_ERR_INVALID_ARG;
  if (c->num_experts > kMaxExperts) return EP_ERR_UNSUPPORTED;
  if (c->num_topk < 1 || c->num_topk > kMaxTopk) return EP_ERR_INVALID_ARG;
  if (c->num_max_tokens_per_rank < 1 || c->num_tokens < 0 ||
      c->num_tokens > c->num_max_tokens_per_rank)
    return EP_ERR_INVALID_ARG;
  if (c->hidden < 8 || c->hidden % 8 != 0) return EP_ERR_INVALID_ARG;
  if ((c->x_dtype != EP_DTYPE_BF16 && c->x_dtype != EP_DTYPE_FP8_E4M3) ||
      (c->recv_dtype != EP_DTYPE_BF16 && c->recv_dtype != EP_DTYPE_FP8_E4M3))
    return EP_ERR_INVALID_ARG;
  const bool fp8 = c->x_dtype == EP_DTYPE_FP8_E4M3 || c->recv_dtype == EP_DTYPE_FP8_E4M3;
  if (fp8 && c->hidden % 128 != 0) return EP_ERR_INVALID_ARG;
  if (fp8 && c->hidden / 128 > kMaxScaleGroups) return EP_ERR_UNSUPPORTED;
  if (c->x_dtype == EP_DTYPE_FP8_E4M3 && c->recv_dtype == EP_DTYPE_BF16) return EP_ERR_UNSUPPORTED;
  if (c->expand != 0 && c->expand != 1) return EP_ERR_INVALID_ARG;
  if (c->expert_alignment < 1) return EP_ERR_INVALID_ARG;
  if (c->num_sms < 0 || c->num_prologue_sms < 0) return EP_ERR_INVALID_ARG;
  if (c->compact_recv < 0 || c->compact_recv > 2 || c->recv_capacity < 0) return EP_ERR_INVALID_ARG;
  if (c->compact_recv && c->expand) return EP_ERR_UNSUPPORTED;  // expanded rows are packed already
  if (c->recv_capacity && c->compact_recv != 2) return EP_ERR_UNSUPPORTED;  // only packed rows take one
  if (c->zero_padding != 0 && c->zero_padding != 1) return EP_ERR_INVALID_ARG;
  if (c->zero_padding && !c->expand) return EP_ERR_UNSUPPORTED;  // only expanded blocks are padded
  if (c->sf_pack != 0 && c->sf_pack != 1) return EP_ERR_INVALID_ARG;
  if (c->sf_pack && c->recv_dtype != EP_DTYPE_FP8_E4M3) return EP_ERR_UNSUPPORTED;
  if (c->copy_path < 0 || c->copy_path > 2) return EP_ERR_INVALID_ARG;
  // 32-bit row indices: rows of one region, lanes, and expanded rows must fit
  const int64_t region_rows = R * c->num_max_tokens_per_rank;
  const int64_t lanes = R * c->num_tokens * c->num_topk;
  const int64_t exp_rows = lanes + static_cast<int64_t>(c->num_experts) * (c->expert_alignment - 1);
  if (region_rows > INT32_MAX || lanes > INT32_MAX || (c->expand && exp_rows > INT32_MAX))
    return EP_ERR_UNSUPPORTED;
  g->R = static_cast<int>(R);
  g->n_so = c->num_scaleout_ranks;
  g->n_su = c->num_scaleup_ranks;
  g->E = c->num_experts;
  g->L = c->num_experts / g->R;
  g->K = c->num_topk;
  g->T = c->num_tokens;
  g->M = c->num_max_tokens_per_rank;
  g->H = c->hidden;
  g->G = c->hidden / 128;
  g->x_fp8 = c->x_dtype == EP_DTYPE_FP8_E4M3;
  g->recv_fp8 = c->recv_dtype == EP_DTYPE_FP8_E4M3;
  g->expand = c->expand;
  g->align = c->expert_alignment;
  g->compact = c->compact_recv;
  if (g->compact == 2)  // every token has at most min(K, R) distinct destinations
    g->entry_rows = c->recv_capacity > 0 ? c->recv_capacity
                                         : R * c->num_tokens * (c->num_topk < R ? c->num_topk : R);
  else
    g->entry_rows = R * region_rows;
  g->zero_padding = c->zero_padding;
  g->sf_pack = c->sf_pack;
  g->copy_path = c->copy_path;
  g->SW = c->sf_pack ? (g->G + 3) / 4 : g->G;
  g->region_rows = region_rows;
  g->num_tokens = R * c->num_tokens;
  return EP_OK;
}

int check_layout_args(const Geometry& g, const int64_t* topk_idx, const ep_layout_t* layout) {
  if (layout == nullptr) return EP_ERR_INVALID_ARG;
  const bool has_tokens = g.T > 0;
  if ((has_tokens && (topk_idx == nullptr || layout->is_token_in_rank == nullptr ||
                      layout->slot_map == nullptr)) ||
      layout->num_tokens_per_rank == nullptr || layout->num_tokens_per_expert == nullptr ||
      layout->recv_cnt == nullptr || layout->recv_psum == nullptr)
    return EP_ERR_INVALID_ARG;
  if (g.expand && (layout->exp_cnt == nullptr || layout->exp_base == nullptr ||
                   layout->exp_region == nullptr || (has_tokens && layout->exp_pos == nullptr)))
    return EP_ERR_INVALID_ARG;
  if (g.compact == 2 && layout->recv_region == nullptr) return EP_ERR_INVALID_ARG;
  if (!aligned(topk_idx, 8) || !aligned(layout->slot_map, 4) ||
      !aligned(layout->is_token_in_rank, 4) || !aligned(layout->num_tokens_per_rank, 4))
    return EP_ERR_INVALID_ARG;
  return EP_OK;
}

Workspace workspace_layout(const Geometry& g) {
  Workspace w;
  w.err = 0;
  w.done = 4;
  w.dispatch_queue = 8;
  w.combine_queue = 24;
  w.exp_off = 256;
  const size_t off_bytes = g.expand ? sizeof(int32_t) * static_cast<size_t>(g.R) * g.E : 0;
  w.total = 256 + ((off_bytes + 255) & ~static_cast<size_t>(255));
  return w;
}

}  // namespace ep

using namespace ep;

namespace {

int check_workspace(const Geometry& g, void* ws, size_t ws_bytes) {
  if (ws == nullptr || !aligned(ws, 256)) return EP_ERR_WORKSPACE;
  if (ws_bytes < workspace_layout(g).total) return EP_ERR_WORKSPACE;
  return EP_OK;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

WorkQueue work_queue(void* ws, size_t off) {
  return WorkQueue{at<unsigned long long>(ws, off), at<unsigned long long>(ws, off + 8)};
}

int sms_or_all(int requested) {
  const int n = device_sm_count();
  if (n <= 0) return -1;
  return (requested > 0 && requested < n) ? requested : n;
}

}  // namespace

extern "C" {

size_t ep_workspace_bytes(const ep_config_t* cfg) {
  Geometry g;
  if (make_geometry(cfg, &g) != EP_OK) return 0;
  return workspace_layout(g).total;
}

int64_t ep_recv_rows(const ep_config_t* cfg) {
  Geometry g;
  if (make_geometry(cfg, &g) != EP_OK) return -1;
  if (g.expand)
    return static_cast<int64_t>(g.R) * g.T * g.K + static_cast<int64_t>(g.E) * (g.align - 1);
  return g.entry_rows;
}

int ep_workspace_init(void* workspace, size_t workspace_bytes, void* stream) {
  if (workspace == nullptr || !aligned(workspace, 256)) return EP_ERR_WORKSPACE;
  return cuda_status(cudaMemsetAsync(workspace, 0, workspace_bytes, static_cast<cudaStream_t>(stream)));
}

int ep_get_dispatch_layout(const ep_config_t* cfg, const int64_t* topk_idx,
                           const ep_layout_t* layout, void* workspace, size_t workspace_bytes,
                           void* stream) {
  Geometry g;
  int st = make_geometry(cfg, &g);
  if (st != EP_OK) return st;
  if ((st = check_workspace(g, workspace, workspace_bytes)) != EP_OK) return st;
  if ((st = check_layout_args(g, topk_idx, layout)) != EP_OK) return st;
  const Workspace w = workspace_layout(g);
  LayoutArgs a;
  a.topk_idx = topk_idx;
  a.num_tokens_per_rank = layout->num_tokens_per_rank;
  a.num_tokens_per_expert = layout->num_tokens_per_expert;
  a.is_token_in_rank = layout->is_token_in_rank;
  a.slot_map = layout->slot_map;
  a.recv_cnt = layout->recv_cnt;
  a.recv_psum = layout->recv_psum;
  a.recv_region = layout->recv_region;
  a.exp_cnt = layout->exp_cnt;
  a.exp_base = layout->exp_base;
  a.exp_region = layout->exp_region;
  a.exp_pos = layout->exp_pos;
  a.err = at<uint32_t>(workspace, w.err);
  a.done = at<uint32_t>(workspace, w.done);
  a.exp_off = at<int32_t>(workspace, w.exp_off);
  a.topk_vec = (g.K % 2 == 0) && aligned(topk_idx, 16);
  a.R = g.R;
  a.n_so = g.n_so;
  a.n_su = g.n_su;
  a.E = g.E;
  a.L = g.L;
  a.K = g.K;
  a.T = g.T;
  a.M = g.M;
  a.expand = g.expand;
  a.align = g.align;
  return cuda_status(launch_layout(g, a, cfg->num_prologue_sms, static_cast<cudaStream_t>(stream)));
}

int ep_dispatch(const ep_config_t* cfg, const ep_layout_t* layout, const void* x,
                const float* x_sf, const int64_t* topk_idx, const float* topk_weights,
                const ep_recv_t* recv, void* workspace, size_t workspace_bytes, void* stream) {
  Geometry g;
  int st = make_geometry(cfg, &g);
  if (st != EP_OK) return st;
  if ((st = check_workspace(g, workspace, workspace_bytes)) != EP_OK) return st;
  if (layout == nullptr || recv == nullptr) return EP_ERR_INVALID_ARG;
  if (g.num_tokens == 0) return EP_OK;
  if (x == nullptr || topk_idx == nullptr || topk_weights == nullptr || layout->slot_map == nullptr ||
      recv->recv_x == nullptr)
    return EP_ERR_INVALID_ARG;
  if (g.x_fp8 != (x_sf != nullptr)) return EP_ERR_INVALID_ARG;
  if (g.recv_fp8 && recv->recv_sf == nullptr) return EP_ERR_INVALID_ARG;
  if (g.expand && (layout->exp_pos == nullptr || layout->exp_region == nullptr))
    return EP_ERR_INVALID_ARG;
  if (g.compact && layout->recv_psum == nullptr) return EP_ERR_INVALID_ARG;
  if (g.compact == 2 && layout->recv_region == nullptr) return EP_ERR_INVALID_ARG;
  if (g.zero_padding && (layout->exp_cnt == nullptr || layout->exp_base == nullptr))
    return EP_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(recv->recv_x, 16) || !aligned(topk_idx, 8) ||
      !aligned(topk_weights, 4) || !aligned(x_sf, 4) || !aligned(recv->recv_sf, 4) ||
      !aligned(recv->recv_topk_idx, 8) || !aligned(recv->recv_topk_weights, 4) ||
      !aligned(recv->recv_src_metadata, 4))
    return EP_ERR_INVALID_ARG;
  const int64_t need_rows = ep_recv_rows(cfg);
  if (recv->recv_x_rows < need_rows) return EP_ERR_INVALID_ARG;
  const int sms = sms_or_all(cfg->num_sms);
  if (sms < 0) return EP_ERR_CUDA;
  DispatchArgs a = {};
  a.x = static_cast<const uint8_t*>(x);
  a.x_sf = x_sf;
  a.topk_idx = topk_idx;
  a.topk_w = topk_weights;
  a.slot_map = layout->slot_map;
  a.exp_pos = layout->exp_pos;
  a.exp_region = layout->exp_region;
  a.recv_psum = layout->recv_psum;
  a.recv_region = layout->recv_region;
  a.exp_cnt = layout->exp_cnt;
  a.exp_base = layout->exp_base;
  a.recv_x = static_cast<uint8_t*>(recv->recv_x);
  a.recv_sf = recv->recv_sf;
  a.recv_idx = recv->recv_topk_idx;
  a.recv_w = recv->recv_topk_weights;
  a.recv_md = recv->recv_src_metadata;
  a.err = at<uint32_t>(workspace, workspace_layout(g).err);
  a.queue = work_queue(workspace, workspace_layout(g).dispatch_queue);
  a.recv_rows = g.expand ? recv->recv_x_rows : need_rows;  // packed: the configured capacity
  a.side_rows = g.entry_rows;
  a.R = g.R;
  a.E = g.E;
  a.L = g.L;
  a.K = g.K;
  a.T = g.T;
  a.H = g.H;
  a.G = g.G;
  a.M = g.M;
  a.compact = g.compact;
  a.zero_padding = g.zero_padding;
  a.sf_pack = g.sf_pack;
  a.SW = g.SW;
  a.region_rows = g.region_rows;
  a.num_tokens = g.num_tokens;
  a.in_row_bytes = g.H * (g.x_fp8 ? 1 : 2);
  a.out_row_bytes = g.H * (g.recv_fp8 ? 1 : 2);
  return cuda_status(launch_dispatch(g, a, sms, static_cast<cudaStream_t>(stream)));
}

int ep_combine(const ep_config_t* cfg, const ep_layout_t* layout, const uint16_t* y,
               const int64_t* topk_idx, const float* topk_weights, uint16_t* out, void* workspace,
               size_t workspace_bytes, void* stream) {
  Geometry g;
  int st = make_geometry(cfg, &g);
  if (st != EP_OK) return st;
  if ((st = check_workspace(g, workspace, workspace_bytes)) != EP_OK) return st;
  if (layout == nullptr) return EP_ERR_INVALID_ARG;
  if (g.num_tokens == 0) return EP_OK;
  if (y == nullptr || out == nullptr || topk_idx == nullptr || topk_weights == nullptr)
    return EP_ERR_INVALID_ARG;
  if (g.expand ? (layout->exp_pos == nullptr || layout->exp_region == nullptr)
               : layout->slot_map == nullptr)
    return EP_ERR_INVALID_ARG;
  if (g.compact && layout->recv_psum == nullptr) return EP_ERR_INVALID_ARG;
  if (g.compact == 2 && layout->recv_region == nullptr) return EP_ERR_INVALID_ARG;
  if (!aligned(y, 16) || !aligned(out, 16) || !aligned(topk_idx, 8) || !aligned(topk_weights, 4))
    return EP_ERR_INVALID_ARG;
  const int sms = sms_or_all(cfg->num_sms);
  if (sms < 0) return EP_ERR_CUDA;
  CombineArgs a;
  a.y = y;
  a.topk_idx = topk_idx;
  a.topk_w = topk_weights;
  a.slot_map = layout->slot_map;
  a.exp_pos = layout->exp_pos;
  a.exp_region = layout->exp_region;
  a.recv_psum = layout->recv_psum;
  a.recv_region = layout->recv_region;
  a.out = out;
  a.err = at<uint32_t>(workspace, workspace_layout(g).err);
  a.queue = work_queue(workspace, workspace_layout(g).combine_queue);
  a.y_rows = ep_recv_rows(cfg);
  a.E = g.E;
  a.L = g.L;
  a.K = g.K;
  a.T = g.T;
  a.H = g.H;
  a.R = g.R;
  a.M = g.M;
  a.compact = g.compact;
  a.region_rows = g.region_rows;
  a.num_tokens = g.num_tokens;
  return cuda_status(launch_combine(g, a, sms, static_cast<cudaStream_t>(stream)));
}

int ep_dispatch_atomic(const ep_config_t* cfg, const void* x, const float* x_sf,
                       const int64_t* topk_idx, const float* topk_weights, const ep_recv_t* recv,
                       int32_t* send_counters, void* workspace, size_t workspace_bytes, void* stream) {
  Geometry g;
  int st = make_geometry(cfg, &g);
  if (st != EP_OK) return st;
  if (g.expand || g.compact || g.zero_padding) return EP_ERR_UNSUPPORTED;
  if ((st = check_workspace(g, workspace, workspace_bytes)) != EP_OK) return st;
  if (recv == nullptr || send_counters == nullptr) return EP_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(send_counters, 0, sizeof(int32_t) * g.R * g.R, s) != cudaSuccess) return EP_ERR_CUDA;
  if (g.num_tokens == 0) return EP_OK;
  if (x == nullptr || topk_idx == nullptr || topk_weights == nullptr || recv->recv_x == nullptr)
    return EP_ERR_INVALID_ARG;
  if (g.x_fp8 != (x_sf != nullptr) || (g.recv_fp8 && recv->recv_sf == nullptr)) return EP_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(recv->recv_x, 16) || !aligned(topk_idx, 8) ||
      !aligned(topk_weights, 4) || !aligned(send_counters, 4))
    return EP_ERR_INVALID_ARG;
  if (recv->recv_x_rows < static_cast<int64_t>(g.R) * g.region_rows) return EP_ERR_INVALID_ARG;
  const int sms = sms_or_all(cfg->num_sms);
  if (sms < 0) return EP_ERR_CUDA;
  DispatchArgs a = {};
  a.x = static_cast<const uint8_t*>(x);
  a.x_sf = x_sf;
  a.topk_idx = topk_idx;
  a.topk_w = topk_weights;
  a.send_counters = send_counters;
  a.err = at<uint32_t>(workspace, workspace_layout(g).err);
  a.queue = work_queue(workspace, workspace_layout(g).dispatch_queue);
  a.recv_x = static_cast<uint8_t*>(recv->recv_x);
  a.recv_sf = recv->recv_sf;
  a.recv_idx = recv->recv_topk_idx;
  a.recv_w = recv->recv_topk_weights;
  a.recv_md = recv->recv_src_metadata;
  a.recv_rows = recv->recv_x_rows;
  a.side_rows = g.entry_rows;
  a.R = g.R;
  a.E = g.E;
  a.L = g.L;
  a.K = g.K;
  a.T = g.T;
  a.H = g.H;
  a.G = g.G;
  a.M = g.M;
  a.n_so = g.n_so;
  a.n_su = g.n_su;
  a.sf_pack = g.sf_pack;
  a.SW = g.SW;
  a.region_rows = g.region_rows;
  a.num_tokens = g.num_tokens;
  a.in_row_bytes = g.H * (g.x_fp8 ? 1 : 2);
  a.out_row_bytes = g.H * (g.recv_fp8 ? 1 : 2);
  return cuda_status(launch_dispatch_atomic(g, a, sms, s));
}

int ep_deterministic_sort(const ep_config_t* cfg, const ep_recv_t* recv,
                          const int32_t* send_counters, const ep_recv_t* sorted, void* stream) {
  Geometry g;
  int st = make_geometry(cfg, &g);
  if (st != EP_OK) return st;
  if (g.expand || g.compact) return EP_ERR_UNSUPPORTED;
  if (g.M > kMaxSortRows) return EP_ERR_UNSUPPORTED;
  if (recv == nullptr || sorted == nullptr || send_counters == nullptr) return EP_ERR_INVALID_ARG;
  const ep_recv_t* bufs[2] = {recv, sorted};
  for (const ep_recv_t* r : bufs) {
    if (r->recv_x == nullptr || r->recv_topk_idx == nullptr || r->recv_topk_weights == nullptr ||
        r->recv_src_metadata == nullptr || (g.recv_fp8 && r->recv_sf == nullptr))
      return EP_ERR_INVALID_ARG;
    if (!aligned(r->recv_x, 16) || !aligned(r->recv_topk_idx, 8) || !aligned(r->recv_sf, 4) ||
        !aligned(r->recv_topk_weights, 4) || !aligned(r->recv_src_metadata, 4))
      return EP_ERR_INVALID_ARG;
    if (r->recv_x_rows < static_cast<int64_t>(g.R) * g.region_rows) return EP_ERR_INVALID_ARG;
  }
  SortArgs a;
  a.in_x = static_cast<const uint8_t*>(recv->recv_x);
  a.in_sf = g.recv_fp8 ? recv->recv_sf : nullptr;
  a.in_idx = recv->recv_topk_idx;
  a.in_w = recv->recv_topk_weights;
  a.in_md = recv->recv_src_metadata;
  a.out_x = static_cast<uint8_t*>(sorted->recv_x);
  a.out_sf = sorted->recv_sf;
  a.out_idx = sorted->recv_topk_idx;
  a.out_w = sorted->recv_topk_weights;
  a.out_md = sorted->recv_src_metadata;
  a.send_counters = send_counters;
  a.R = g.R;
  a.K = g.K;
  a.M = g.M;
  a.SW = g.SW;
  a.n_so = g.n_so;
  a.n_su = g.n_su;
  a.region_rows = g.region_rows;
  a.row_bytes = g.H * (g.recv_fp8 ? 1 : 2);
  return cuda_status(launch_sort(g, a, static_cast<cudaStream_t>(stream)));
}

int ep_check_error(void* workspace, void* stream) {
  if (workspace == nullptr || !aligned(workspace, 256)) return EP_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t bits = 0;
  if (cudaMemcpyAsync(&bits, workspace, sizeof(bits), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return EP_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return EP_ERR_CUDA;
  if (bits != 0) {
    if (cudaMemsetAsync(workspace, 0, sizeof(uint32_t), s) != cudaSuccess) return EP_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return EP_ERR_CUDA;
  }
  if (bits & kErrBadTopk) return EP_ERR_BAD_TOPK;
  if (bits & kErrOverflow) return EP_ERR_OVERFLOW;
  if (bits & kErrTimeout) return EP_ERR_TIMEOUT;
  if (bits & kErrBounds) return EP_ERR_BOUNDS;
  return EP_OK;
}

const char* ep_status_string(int status) {
  switch (status) {
    case EP_OK: return "EP_OK";
    case EP_ERR_INVALID_ARG: return "EP_ERR_INVALID_ARG";
    case EP_ERR_UNSUPPORTED: return "EP_ERR_UNSUPPORTED";
    case EP_ERR_WORKSPACE: return "EP_ERR_WORKSPACE";
    case EP_ERR_CUDA: return "EP_ERR_CUDA";
    case EP_ERR_BAD_TOPK: return "EP_ERR_BAD_TOPK";
    case EP_ERR_OVERFLOW: return "EP_ERR_OVERFLOW";
    case EP_ERR_TIMEOUT: return "EP_ERR_TIMEOUT";
    case EP_ERR_BOUNDS: return "EP_ERR_BOUNDS";
    default: return "EP_ERR_UNKNOWN";
  }
}

int ep_diag_e4m3_of_bits(uint32_t first, int64_t n, uint8_t* out, void* stream) {
  if (n < 0 || (n > 0 && out == nullptr)) return EP_ERR_INVALID_ARG;
  if (n == 0) return EP_OK;
  diag_e4m3_kernel<<<1024, 256, 0, static_cast<cudaStream_t>(stream)>>>(first, n, out);
  return cuda_status(cudaGetLastError());
}

int ep_diag_bf16_of_bits(uint32_t first, int64_t n, uint16_t* out, void* stream) {
  if (n < 0 || (n > 0 && out == nullptr)) return EP_ERR_INVALID_ARG;
  if (n == 0) return EP_OK;
  diag_bf16_kernel<<<1024, 256, 0, static_cast<cudaStream_t>(stream)>>>(first, n, out);
  return cuda_status(cudaGetLastError());
}

}  // extern "C"

/*
 * ep_get.h — C ABI of a single-GPU MoE expert-parallel token dispatch / combine.
 *
 * The EP ranks are logical partitions of one GPU's memory: rank r's tokens are
 * rows [r*T, (r+1)*T) of the inputs, and rank r's receive buffer is region r of
 * the receive tensors. Every move is a device-memory scatter or gather on the
 * caller's stream.
 *
 * Sources (DeepEP issue and pull-request pages):
 *   [P753] PR #753 "Kernel-side deterministic dispatch for the non-expand
 *          layout": Motivation, Approach, "Direct vs hybrid dispatch",
 *          Compatibility, "New API".
 *   [P690] PR #690 "Add Direct Recv X dispatch path": review comments on the
 *          copy epilogue and the buffer sizing; Summary; Implementation.
 *   [P544] PR #544 "Fix duplicate calculation of num_tokens_per_rank" (title,
 *          cited from the footer of issue #647).
 *
 * Conventions for every entry point:
 *   - Pointers named "device" must point to device memory of the current CUDA
 *     device; the caller owns and allocates every buffer, including the
 *     workspace. The library never allocates, frees or synchronises, except
 *     ep_check_error, which synchronises the given stream.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). All work
 *     is enqueued asynchronously on it, in call order. The layout, dispatch and
 *     combine kernels are launched with programmatic stream serialization: one
 *     may be placed on the SMs while the kernel before it drains, but it waits
 *     for that kernel's completion before it reads or writes memory, so stream
 *     order holds as for any launch.
 *   - Returns EP_OK (0) or a negative EP_ERR_* code. Host-detectable errors are
 *     reported before anything is enqueued. Errors found on the device (bad
 *     top-k values; a bounded wait that ran out; in the bounds-checked build
 *     libep_get_checked.so, a row index outside its buffer) are latched in the
 *     workspace and read by ep_check_error.
 *     Unsupported combinations return EP_ERR_UNSUPPORTED; nothing is ever
 *     dropped silently.
 *   - All row pointers must be 16-byte aligned.
 */
#ifndef EP_GET_H_
#define EP_GET_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes -------------------------------------------------------- */
#define EP_OK 0
#define EP_ERR_INVALID_ARG (-1) /* bad size, null or misaligned pointer      */
#define EP_ERR_UNSUPPORTED (-2) /* valid request this library does not do    */
#define EP_ERR_WORKSPACE (-3)   /* workspace missing or smaller than needed  */
#define EP_ERR_CUDA (-4)        /* a CUDA launch or runtime call failed      */
#define EP_ERR_BAD_TOPK (-5)    /* device: top-k value < -1 or >= num_experts,
                                   or a repeated expert in the expanded layout */
#define EP_ERR_OVERFLOW (-6)    /* device: an entry did not fit its receive
                                   buffer: a packed row past recv_capacity
                                   (that entry was not written, and combine
                                   left its lane out)                        */
#define EP_ERR_TIMEOUT (-7)     /* device: a bounded wait for a bulk copy gave
                                   up (the kernel returned early; its
                                   outputs are incomplete)                   */
#define EP_ERR_BOUNDS (-8)      /* device, checked builds only
                                   (libep_get_checked.so): a computed row
                                   index fell outside its buffer; that access
                                   was skipped                               */

/* ---- element types ------------------------------------------------------- */
#define EP_DTYPE_BF16 0
#define EP_DTYPE_FP8_E4M3 1 /* OCP E4M3 ("FN"), fp32 scale per 128 columns */

/* ---- configuration --------------------------------------------------------
 * Ranks: R = num_scaleout_ranks * num_scaleup_ranks; global rank
 * r = scaleout * num_scaleup_ranks + scaleup. num_scaleout_ranks == 1 is the
 * direct layout, > 1 the hybrid row form [P753 "Direct vs hybrid dispatch"].
 * Experts: expert e lives on rank e / (num_experts / R).
 */
typedef struct ep_config {
  int32_t num_scaleout_ranks;      /* >= 1; 1 = direct                           */
  int32_t num_scaleup_ranks;       /* >= 1; R <= 64                              */
  int32_t num_experts;             /* multiple of R                              */
  int32_t num_topk;                /* K, 1..32                                   */
  int32_t num_tokens;              /* T per logical rank, 0..num_max_tokens_per_rank */
  int32_t num_max_tokens_per_rank; /* M >= 1                                     */
  int32_t hidden;                  /* H; multiple of 8 (bf16), of 128 with FP8   */
  int32_t x_dtype;                 /* EP_DTYPE_BF16, or EP_DTYPE_FP8_E4M3 (pre-cast x + x_sf) */
  int32_t recv_dtype;              /* EP_DTYPE_BF16, or EP_DTYPE_FP8_E4M3 (cast inside dispatch
                                      when x is bf16)                            */
  int32_t expand;                  /* 0 = row form, 1 = expanded per-expert blocks */
  int32_t expert_alignment;        /* >= 1: expanded blocks padded to a multiple */
  int32_t num_sms;                 /* SMs for dispatch/combine; 0 = all          */
  int32_t num_prologue_sms;        /* SMs for the layout prologue; 0 = automatic;
                                      capped at 64 [P753 "New API"]. Results never
                                      depend on it.                              */
  int32_t compact_recv;            /* row form only. 0: receive rows at their slots;
                                      1 (compact): each destination's rows packed from
                                      the start of its R*M-row window in row-block
                                      order ([P690] Direct Recv X: the entries of row
                                      block i start at the exclusive prefix
                                      recv_psum[d][i-1] of the receive counts);
                                      2 (packed): the same order with the destinations
                                      back to back in one buffer of recv_capacity rows
                                      (destination d from layout.recv_region[d]), so
                                      the receive tensors hold only what can arrive */
  int32_t zero_padding;            /* expanded only: 1 = dispatch writes zeros into the
                                      rows between each expert's lanes and the next
                                      expert_alignment boundary (and their FP8
                                      scales); 0 = those rows are left untouched  */
  int32_t sf_pack;                 /* FP8 receive only. 0: recv_sf row = G fp32 scales
                                      (amax/448). 1: packed power-of-two scales (a
                                      reading of [P690]'s num_sf_packs, whose format the
                                      pages do not give): per 128 columns one byte
                                      e+127 (UE8M0) with 2^e the smallest power of two
                                      >= amax/448 and q = e4m3(x * 2^-e); four groups
                                      per 32-bit word, group g in byte g%4 of word g/4,
                                      so a row holds ceil(G/4) words. Pre-cast FP8
                                      input then carries x_sf in the same packing.  */
  int32_t copy_path;               /* how dispatch moves rows that travel unchanged
                                      (bf16 -> bf16, pre-cast FP8): 0 = automatic
                                      (bulk copies when the input rows total
                                      at least 32 MiB, register copies below);
                                      1 = 16-byte register loads and stores; 2 = bulk
                                      copies through shared memory. Results never
                                      depend on it; the fused cast ignores it.     */
  int32_t recv_capacity;           /* packed rows only (compact_recv = 2): rows of the
                                      receive tensors; 0 = R*T*min(K, R), the most
                                      that can arrive (every token has at most min(K,R)
                                      destinations). An entry past it is not written
                                      and latches EP_ERR_OVERFLOW; layout.recv_region[R]
                                      gives the exact count after the layout.      */
} ep_config_t;

/* ---- dispatch layout (all device pointers, int32 unless noted) -------------
 * Row form: destination d's region of the receive tensors has R*M rows; source
 * s owns the M rows starting at row_block(s)*M, where row_block(s) = s
 * (direct) or scaleup(s)*num_scaleout_ranks + scaleout(s) (hybrid: segment =
 * source scale-up rank, in-segment offset = source scale-out rank * M + slot)
 * [P753 Approach; "Direct vs hybrid dispatch"].
 */
typedef struct ep_layout {
  int32_t* num_tokens_per_rank;   /* [R src][R dst]: tokens of src reaching dst,
                                     once per token [P544]                      */
  int32_t* num_tokens_per_expert; /* [R src][E]: valid lanes per expert         */
  uint8_t* is_token_in_rank;      /* [R][T][R dst]: 0/1                          */
  int32_t* slot_map;              /* [R][T][K]: row inside the destination region =
                                     row_block(src)*M + the source's running count of
                                     deduplicated entries to that destination in token
                                     order; lanes to the same destination share it;
                                     -1 for masked lanes [P753 Approach]         */
  int32_t* recv_cnt;              /* [R dst][R src] = num_tokens_per_rank transposed */
  int32_t* recv_psum;             /* [R dst][R row blocks]: inclusive prefix sums of
                                     recv_cnt in row-block order [P753 "Direct vs
                                     hybrid dispatch": per-source receive counts] */
  /* expanded layout only (may be NULL when expand == 0): per destination, per
     local expert j, a block of rows holding that expert's lanes in (source rank,
     token) order, padded to expert_alignment; regions concatenated by rank. */
  int32_t* exp_cnt;    /* [R][L]: lanes per (destination, local expert)         */
  int32_t* exp_base;   /* [R][L+1]: block starts inside the region; [L] = size  */
  int32_t* exp_region; /* [R+1]: first row of each region; [R] = total rows     */
  int32_t* exp_pos;    /* [R][T][K]: row of the lane inside its destination's
                          region, -1 for masked lanes                          */
  int32_t* recv_region; /* [R+1] (may be NULL unless compact_recv = 2): first
                           packed row of each destination = the entries all
                           destinations before it receive; [R] = total entries */
} ep_layout_t;

/* ---- receive buffers (device pointers) -------------------------------------
 * Row form: recv_x/recv_sf and the sidecars' rows are indexed d*R*M + slot;
 * compact (compact_recv = 1): d*R*M + recv_psum[d][rb-1] + slot - rb*M with
 * rb = slot / M (recv_psum[d][-1] = 0), so destination d's rows are
 * [d*R*M, d*R*M + sum_s recv_cnt[d][s]); packed (compact_recv = 2):
 * recv_region[d] + recv_psum[d][rb-1] + slot - rb*M, so destination d's rows
 * are [recv_region[d], recv_region[d+1]) and all tensors have ep_recv_rows()
 * rows. Expanded: recv_x and recv_sf rows are indexed exp_region[d] + exp_pos;
 * the sidecars stay in the row form. Rows no entry fills are left untouched.
 * recv_topk_idx, recv_topk_weights and recv_src_metadata may be NULL (not
 * written).
 */
typedef struct ep_recv {
  void* recv_x;                /* [recv_x_rows][H] bf16 or e4m3                 */
  float* recv_sf;              /* [recv_x_rows][H/128] fp32, or [recv_x_rows][ceil(H/512)]
                                  packed words with sf_pack (FP8 receive only)   */
  int64_t* recv_topk_idx;      /* [R][R*M][K] (packed: [ep_recv_rows][K]):
                                  destination-local expert or -1                 */
  float* recv_topk_weights;    /* same rows x K: weight, or 0 off this destination */
  int32_t* recv_src_metadata;  /* same rows x (2+K): {src rank, src token,
                                  dst_tensor_idx[K]}; field 2+k = expanded row of
                                  lane k in this destination's region, else -1
                                  [P690 copy-epilogue review]                   */
  int64_t recv_x_rows;         /* capacity of recv_x in rows, >= ep_recv_rows()  */
} ep_recv_t;

/* Workspace bytes the three entry points need for this configuration (the
 * library's own convention: the pages' buffers are transport windows with no
 * single-GPU counterpart): a 256-byte header (the device error word, the
 * layout's arrival counter, and the work queues from which the dispatch and
 * combine warps take their tokens), plus per-(source, expert) offsets when
 * expanding. The workspace must be zero-filled before its first use
 * (ep_workspace_init or a zeroing allocator); afterwards every kernel returns
 * its counters to zero itself. One workspace serves one stream at a time. */
size_t ep_workspace_bytes(const ep_config_t* cfg);

/* Rows the receive buffer recv_x needs: R*R*M (row form and compact; the
 * per-destination window of [P690]'s buffer sizing times R), recv_capacity or
 * R*T*min(K, R) (packed), or R*T*K + E*(expert_alignment-1) (expanded upper
 * bound). Returns -1 for an invalid configuration. */
int64_t ep_recv_rows(const ep_config_t* cfg);

/* Zero the workspace on `stream` (the library's own convention). */
int ep_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/* Dispatch layout [P753 Motivation, Approach]: turns topk_idx (device, int64
 * [R][T][K]; -1 = masked lane) into the counts, the per-lane slots and, when
 * expanding, the per-expert positions of `layout` (all device outputs). One
 * kernel with a thread-block cluster per source rank: per-warp counts, a scan
 * of the CTAs' counts through distributed shared memory, then per-lane slots;
 * its last CTA writes the receive prefix sums (and recv_region). The expanded
 * layout adds two small kernels (the per-expert scan across sources, then the
 * final positions). The result is a pure function of topk_idx. */
int ep_get_dispatch_layout(const ep_config_t* cfg, const int64_t* topk_idx,
                           const ep_layout_t* layout, void* workspace,
                           size_t workspace_bytes, void* stream);

/* Size of the fixed scratch array used by ep_get_dispatch_layout_noalloc. */
#define EP_NOALLOC_SCRATCH_BYTES (1u << 20)

/* ep_get_dispatch_layout for callers that cannot allocate device memory (for
 * example plugins of inference engines that are handed only their input and
 * output buffers, or latency-critical code where cudaMalloc is not allowed).
 * No counterpart on the DeepEP pages: it is the same layout with the workspace
 * replaced by a fixed array of EP_NOALLOC_SCRATCH_BYTES inside the library,
 * which every GPU that loads the library keeps until the process exits.
 *   - Outputs, layout and errors for invalid arguments are those of
 *     ep_get_dispatch_layout; a configuration whose ep_workspace_bytes exceeds
 *     EP_NOALLOC_SCRATCH_BYTES returns EP_ERR_WORKSPACE.
 *   - Allocates nothing. The first call in a CUDA context (that context
 *     current) looks up the array's device address; make it before any stream
 *     capture. A device reset gives a new context, and the next call looks the
 *     address up again.
 *   - All calls share the array: each call, once its arguments have passed
 *     the checks, clears the array's error bits and counter on `stream`
 *     first; calls that overlap on the GPU race on it.
 *   - Invalid top-k values are treated as masked lanes, as in
 *     ep_get_dispatch_layout, and latched in the array's error word, which
 *     ep_check_error_noalloc reads. */
int ep_get_dispatch_layout_noalloc(const ep_config_t* cfg, const int64_t* topk_idx,
                                   const ep_layout_t* layout, void* stream);

/* ep_check_error for ep_get_dispatch_layout_noalloc (no counterpart on the
 * pages): synchronises `stream`, returns the first device-detected error the
 * allocation-free layout latched in the library's array since the last call
 * (EP_OK if none) and clears it. Allocates nothing; shares the array, and its
 * race with overlapping calls, with ep_get_dispatch_layout_noalloc. */
int ep_check_error_noalloc(void* stream);

/* Dispatch: for every deduplicated (token, destination) entry writes the
 * token's hidden row into the destination's receive rows at its slot (row
 * form) or, expanded, one row per valid lane at its position; plus the
 * sidecars [P753 Approach; P690 Summary/Implementation].
 *   x: device [R][T][H] bf16 (x_dtype BF16) or e4m3 codes (FP8).
 *   x_sf: device [R][T][H/128] fp32, FP8 input only (else NULL).
 *   recv_dtype FP8 with bf16 x casts inside the copy: per 128 columns,
 *   amax = max(max|x|, 1e-4), sf = amax/448, q = e4m3_rn_satfinite(x*(448/amax)).
 *   topk_idx / topk_weights: device [R][T][K] int64 / fp32.
 * `layout` must come from ep_get_dispatch_layout with the same cfg/topk_idx. */
int ep_dispatch(const ep_config_t* cfg, const ep_layout_t* layout, const void* x,
                const float* x_sf, const int64_t* topk_idx, const float* topk_weights,
                const ep_recv_t* recv, void* workspace, size_t workspace_bytes,
                void* stream);

/* Combine: out[s][t] = bf16_rn(acc), acc = +0 then, for k in lane order over
 * the valid lanes, acc = fma(topk_weights[s][t][k], y[row of lane k], acc),
 * in fp32. y: device bf16 expert outputs in the receive layout (row form or
 * compact [R][R*M][H], or expanded [rows][H]), at least ep_recv_rows(cfg)
 * rows; out: device bf16 [R][T][H]. The result is bitwise reproducible. */
int ep_combine(const ep_config_t* cfg, const ep_layout_t* layout, const uint16_t* y,
               const int64_t* topk_idx, const float* topk_weights, uint16_t* out,
               void* workspace, size_t workspace_bytes, void* stream);

/* ---- comparison path: the design PR #753 replaces ----------------------------
 * [P753 Motivation] Before kernel-side slots, a sender took its destination slot
 * with an atomicAdd on a shared counter, so the order of a source's rows inside
 * a destination depended on the race between warps, and EPHandle.deterministic_sort
 * restored a reproducible order afterwards by sorting the received tokens by
 * source token and permuting every order-dependent tensor. These two entry points
 * reproduce that path (row form only, not compact) so it can be measured against
 * ep_get_dispatch_layout + ep_dispatch; after the sort the buffers equal the
 * deterministic dispatch's bit for bit.
 *
 * ep_dispatch_atomic: ep_dispatch without a layout. send_counters: device int32
 * [R src][R dst], zeroed on `stream` by the call, then left holding how many
 * rows each source sent each destination. Rows land in the source's row block
 * of the destination region in race order. The workspace (as for ep_dispatch)
 * carries the work queue that spreads the tokens over the warps. */
int ep_dispatch_atomic(const ep_config_t* cfg, const void* x, const float* x_sf,
                       const int64_t* topk_idx, const float* topk_weights, const ep_recv_t* recv,
                       int32_t* send_counters, void* workspace, size_t workspace_bytes, void* stream);

/* ep_deterministic_sort: sorts every (destination, row block) segment of `recv`
 * (filled by ep_dispatch_atomic; the sidecars must be present: the key is the
 * metadata's source token) and writes rows and sidecars in that order to
 * `sorted` (same shapes). num_max_tokens_per_rank <= 8192. */
int ep_deterministic_sort(const ep_config_t* cfg, const ep_recv_t* recv,
                          const int32_t* send_counters, const ep_recv_t* sorted, void* stream);

/* Synchronises `stream`, returns the first device-detected error latched in
 * the workspace since the last call (EP_OK if none) and clears it. The
 * library's own convention (the pages print and continue on a device error;
 * PR #690's review asks that nothing be dropped silently). */
int ep_check_error(void* workspace, void* stream);

/* Human-readable name of a status code (static storage; the library's own). */
const char* ep_status_string(int status);

/* Diagnostics: the device's fp32 -> e4m3 (round to nearest even, saturating)
 * and fp32 -> bf16 (round to nearest even) conversions used by the kernels,
 * applied to the binary32 bit patterns first .. first+n-1; out is device
 * memory of n bytes / n uint16. */
int ep_diag_e4m3_of_bits(uint32_t first, int64_t n, uint8_t* out, void* stream);
int ep_diag_bf16_of_bits(uint32_t first, int64_t n, uint16_t* out, void* stream);

/* Diagnostic copy for the bandwidth ceiling of a one-read, many-write stream
 * (no counterpart on the pages; the benchmark times it beside the dispatch,
 * whose scatter reads each token row once and writes it to each destination).
 * Row r of `src` (rows x row_bytes, 16-byte aligned) is read once and
 * written to rows floor(r*fan_num/fan_den) .. floor((r+1)*fan_num/fan_den) - 1
 * of `dst` (16-byte aligned, floor(rows*fan_num/fan_den) rows of row_bytes;
 * the caller owns both). Either may be device memory or pinned host memory the
 * device addresses directly (the benchmark times the host link that way). row_bytes: a positive multiple of 16;
 * 0 <= fan_num <= 2^20, fan_den >= 1, 0 <= rows <= 2^40; num_sms: SMs the grid
 * is sized for (0 = all). method 0: 16-byte register loads and stores; method
 * 1: bulk copies through shared memory (row_bytes <= 16384, else
 * EP_ERR_UNSUPPORTED). Returns EP_ERR_INVALID_ARG for any other argument,
 * EP_ERR_CUDA if the launch fails; asynchronous on `stream`. */
int ep_diag_copy_fanout(const void* src, void* dst, int64_t rows, int32_t row_bytes, int32_t fan_num,
                        int32_t fan_den, int32_t num_sms, int32_t method, void* stream);

/* Diagnostic for the bounded waits (no counterpart on the pages): one warp
 * starts a bulk load of `bytes` (0..4096, a multiple of 16) from `src` (device,
 * 16-byte aligned; may be null when bytes is 0), waits at most `rounds`
 * (<= 2^20) try_wait rounds on an mbarrier that nothing completes, drains the
 * load and latches the timeout bit in `workspace` (256-byte aligned), exactly
 * as the bulk-copy dispatch does when a wait runs out; ep_check_error then
 * returns EP_ERR_TIMEOUT. Asynchronous on `stream`. */
int ep_diag_wait_timeout(void* workspace, const void* src, int32_t bytes, uint32_t rounds, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* EP_GET_H_ */

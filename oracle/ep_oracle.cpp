// CPU oracle for MoE token dispatch and combine.
//
// TEST INFRASTRUCTURE ONLY. Plain, slow, single-threaded C++17 that computes
// what the GPU path computes, straight from the definitions, so that the GPU
// results can be compared against it element by element. Only the tests, the
// smoke check and the benchmark's CPU-baseline leg use it; the product path
// never does. It shares no code, header, table or constant with the CUDA
// library.
//
// Sources (DeepEP issue / PR pages):
//   * PR #753 "Kernel-side deterministic dispatch for the non-expand layout",
//     sections Motivation, Approach, "Direct vs hybrid dispatch", Compatibility:
//     destination rank of an expert, per-token deduplication of destination
//     ranks, slot = row_base_idx * num_max_tokens_per_rank + the sender's
//     running count of deduplicated entries to that destination in token
//     order, direct row base = the source's rank, hybrid row form
//     (segment = src scale-up rank, in-segment offset = src scale-out rank *
//     num_max_tokens_per_rank + row-local slot), per-source-rank receive
//     counts with their prefix sums.
//   * PR #690 "Add Direct Recv X dispatch path", review of the copy epilogue:
//     metadata field 2 + lane holds dst_tensor_idx in the expanded layout; FP8
//     scale sidecars travel beside the hidden payload; a payload is never
//     dropped silently. Summary and "Direct Recv X design": the sender writes
//     its rows straight into the receiver's compact recv_x, at the receiver's
//     exclusive prefix of the per-source counts.
//   * Issue #647 footer, PR #544 "Fix duplicate calculation of
//     num_tokens_per_rank": a token counts once per destination rank.
//
// Readings where the pages are silent (each one is listed in the design notes):
//   * dedup keeps the lowest lane per destination rank; every lane to that
//     rank shares its row; "token order" = increasing local token index;
//   * global rank r = scale_out * n_su + scale_up;
//   * topk_idx == -1 is a masked lane; any other value outside [0, E) is an
//     error (BAD_TOPK), as is a repeated expert within one token in the
//     expanded layout; such lanes are then treated as masked;
//   * recv_topk_idx holds the destination-local expert index or -1,
//     recv_topk_weights the weight or 0; metadata = {src rank, src token,
//     dst_tensor_idx x K} with -1 where not expanded;
//   * expanded layout: per destination, per local expert, a block holding the
//     expert's lanes in (source rank, token) order; blocks padded up to
//     expert_alignment; destination regions concatenated in rank order;
//   * FP8: per token and per 128 columns, amax (clamped below at 1e-4),
//     sf = amax / 448, q = e4m3_rn_satfinite(x * (448 / amax));
//   * combine: acc = +0; for k in lane order over valid lanes
//     acc = fma(w_k, y_k, acc); out = bf16_rn(acc);
//   * compact receive rows: each destination's entries from the start of its
//     R*M-row window in row-block order; packed: the same order with the
//     destinations back to back in one buffer of R*T*min(K, R) rows (or a
//     caller's capacity; entries past it are reported as OVERFLOW).
//
// Parity pins for every function here live in the CPU test suite; none is
// unpinned.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

struct Cfg {
  int32_t n_so, n_su, E, K, T, M, H;
  int32_t x_fp8, recv_fp8, expand, align, compact, zero_padding, sf_pack;
  int32_t recv_capacity;  // packed receive rows only: rows the receive tensors hold (0 = the bound)
};

constexpr int kOk = 0;
constexpr int kInvalid = -1;
constexpr int kUnsupported = -2;
constexpr int kBadTopk = -5;
constexpr int kOverflow = -6;

// ---- number formats, from their public definitions ----------------------

// bfloat16 = the upper 16 bits of an IEEE-754 binary32; round to nearest,
// ties to even on the 16 discarded bits.
float bf16_to_f32(uint16_t b) {
  uint32_t u = static_cast<uint32_t>(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

uint16_t f32_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u)  // NaN: keep it a (quiet) NaN
    return static_cast<uint16_t>((u >> 16) | 0x0040u);
  const uint32_t keep_lsb = (u >> 16) & 1u;
  u += 0x7FFFu + keep_lsb;
  return static_cast<uint16_t>(u >> 16);
}

// OCP 8-bit floating point, E4M3 ("FN"): bias 7, no infinities, S.1111.111 is
// NaN, largest finite 1.75 * 2^8 = 448, subnormals m * 2^-9.
float e4m3_to_f32(uint8_t c) {
  const int sign = c >> 7, exp = (c >> 3) & 0xF, man = c & 0x7;
  if (exp == 0xF && man == 0x7) return NAN;
  const double mag = exp == 0 ? std::ldexp(static_cast<double>(man), -9)
                              : std::ldexp(static_cast<double>(8 + man), exp - 10);
  return static_cast<float>(sign ? -mag : mag);
}

// Round to nearest (ties to even); magnitudes beyond the largest finite value
// saturate to +-448 ("satfinite").
uint8_t f32_to_e4m3(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  const uint8_t sign = static_cast<uint8_t>((u >> 24) & 0x80u);
  if (std::isnan(f)) return static_cast<uint8_t>(sign | 0x7F);
  const double a = std::fabs(static_cast<double>(f));
  if (a >= 448.0) return static_cast<uint8_t>(sign | 0x7E);
  if (a < 0.015625) {  // below the smallest normal 2^-6: quantum 2^-9
    const double q = std::nearbyint(a * 512.0);  // 0..8; 8 is the smallest normal
    return static_cast<uint8_t>(sign | static_cast<int>(q));
  }
  int e2;
  std::frexp(a, &e2);  // a = m * 2^e2 with m in [0.5, 1)
  int exp = e2 - 1;    // a in [2^exp, 2^(exp+1)), exp in [-6, 8]
  double q = std::nearbyint(std::ldexp(a, 3 - exp));  // 8..16 quanta of 2^(exp-3)
  if (q == 16.0) {
    q = 8.0;
    exp += 1;
  }
  int code = ((exp + 7) << 3) | (static_cast<int>(q) - 8);
  if (code > 0x7E) code = 0x7E;
  return static_cast<uint8_t>(sign | code);
}

// Per-128-column FP8 cast of one bf16 row.
void cast_row_fp8(const uint16_t* x, int H, uint8_t* q, float* sf) {
  const int G = H / 128;
  for (int g = 0; g < G; ++g) {
    float amax = 0.0f;
    for (int c = 0; c < 128; ++c) amax = std::fmax(amax, std::fabs(bf16_to_f32(x[g * 128 + c])));
    amax = std::fmax(amax, 1e-4f);
    const float scale = amax / 448.0f;
    const float inv = 448.0f / amax;
    sf[g] = scale;
    for (int c = 0; c < 128; ++c) {
      const float v = bf16_to_f32(x[g * 128 + c]) * inv;
      q[g * 128 + c] = f32_to_e4m3(v);
    }
  }
}

// Packed scales (reading of the pages' num_sf_packs, whose format they do not
// give): per 128 columns an unsigned power-of-two exponent byte (UE8M0, value
// 2^(byte - 127)); four groups per 32-bit word, group g in byte g % 4 of word
// g / 4. The scale is the smallest power of two 2^e with amax <= 448 * 2^e
// (amax clamped below at 1e-4), and q = e4m3_rn_satfinite(x * 2^-e).
void cast_row_fp8_ue8m0(const uint16_t* x, int H, uint8_t* q, uint32_t* words) {
  const int G = H / 128;
  std::memset(words, 0, sizeof(uint32_t) * ((G + 3) / 4));
  for (int g = 0; g < G; ++g) {
    float amax = 0.0f;
    for (int c = 0; c < 128; ++c) amax = std::fmax(amax, std::fabs(bf16_to_f32(x[g * 128 + c])));
    amax = std::fmax(amax, 1e-4f);
    int e2;
    std::frexp(static_cast<double>(amax), &e2);
    int e = e2 - 10;  // 448 * 2^(e2 - 10) < 2^(e2 - 1) <= amax: too small, step up
    while (static_cast<double>(amax) > std::ldexp(448.0, e)) ++e;
    words[g / 4] |= static_cast<uint32_t>(e + 127) << (8 * (g % 4));
    const float down = std::ldexp(1.0f, -e);
    for (int c = 0; c < 128; ++c) q[g * 128 + c] = f32_to_e4m3(bf16_to_f32(x[g * 128 + c]) * down);
  }
}

// 32-bit words of one row's scale sidecar: G fp32 scales, or ceil(G/4) packed words.
int sf_words(int H, int sf_pack) {
  const int G = H / 128;
  return sf_pack ? (G + 3) / 4 : G;
}

int ranks(const Cfg& c) { return c.n_so * c.n_su; }

// Row block of source s inside every destination's region (R blocks of M rows).
//   direct: block s;  hybrid: segment su(s) of n_so blocks, then so(s).
int64_t row_block(const Cfg& c, int s) {
  if (c.n_so == 1) return s;
  const int su = s % c.n_su, so = s / c.n_su;
  return static_cast<int64_t>(su) * c.n_so + so;
}

int check_cfg(const Cfg& c) {
  if (c.n_so < 1 || c.n_su < 1 || c.K < 1 || c.K > 32 || c.T < 0 || c.M < 1 || c.H < 1)
    return kInvalid;
  const int R = ranks(c);
  if (c.E < R || c.E % R != 0 || c.T > c.M || c.align < 1) return kInvalid;
  if ((c.x_fp8 || c.recv_fp8) && c.H % 128 != 0) return kInvalid;
  if (c.x_fp8 && !c.recv_fp8) return kUnsupported;
  if (c.compact < 0 || c.compact > 2 || c.recv_capacity < 0) return kInvalid;
  if (c.compact && c.expand) return kUnsupported;
  if (c.recv_capacity && c.compact != 2) return kUnsupported;
  if (c.zero_padding && !c.expand) return kUnsupported;
  if (c.sf_pack && !c.recv_fp8) return kUnsupported;
  return kOk;
}

// Rows of the receive tensors (recv_x, recv_sf, and the sidecars unless
// expanded): R regions of R*M rows (row form and compact), or, packed, the
// capacity (R*T*min(K, R) deduplicated entries at most, or the caller's).
int64_t entry_rows(const Cfg& c) {
  const int64_t R = ranks(c);
  if (c.compact == 2) {
    if (c.recv_capacity > 0) return c.recv_capacity;
    return R * c.T * (c.K < R ? c.K : R);
  }
  return R * R * c.M;
}

// Row of a deduplicated (token, destination d) entry with row-form slot
// `slot` in the receive tensors.
//   row form:  d*R*M + slot (PR #753, Approach: the slot is already the row).
//   compact (PR #690, Direct Recv X): destination d's entries are packed from
//              the start of its R*M-row window in row-block order, so the
//              entries of row block rb follow everything d receives from row
//              blocks before rb (the exclusive prefix of its per-source receive
//              counts): d*R*M + recv_psum[d][rb-1] + slot - rb*M.
//   packed:    the same, with the destinations back to back instead of one
//              window each: recv_region[d] = everything destinations before d
//              receive, in place of d*R*M.
int64_t entry_row(const Cfg& c, int d, int64_t slot, const int32_t* recv_psum, const int32_t* recv_region) {
  const int R = ranks(c);
  const int64_t window = static_cast<int64_t>(d) * R * c.M;
  if (c.compact == 0) return window + slot;
  const int64_t rb = slot / c.M;
  const int64_t before = rb == 0 ? 0 : recv_psum[static_cast<int64_t>(d) * R + rb - 1];
  const int64_t base = c.compact == 1 ? window : recv_region[d];
  return base + before + (slot - rb * c.M);
}

// Lane validity: -1 is masked; anything else outside [0, E) is an error; in
// the expanded layout a repeat of an earlier lane's expert is an error too.
// Invalid lanes are treated as masked afterwards.
bool lane_valid(const Cfg& c, const int64_t* idx_tok, int k, int* status) {
  const int64_t e = idx_tok[k];
  if (e == -1) return false;
  if (e < -1 || e >= c.E) {
    *status = kBadTopk;
    return false;
  }
  if (c.expand) {
    for (int j = 0; j < k; ++j) {
      if (idx_tok[j] == e) {
        *status = kBadTopk;
        return false;
      }
    }
  }
  return true;
}

}  // namespace

extern "C" {

struct orc_cfg {
  int32_t n_so, n_su, E, K, T, M, H;
  int32_t x_fp8, recv_fp8, expand, align, compact, zero_padding, sf_pack, recv_capacity;
};

static Cfg to_cfg(const orc_cfg* p) {
  Cfg c;
  std::memcpy(&c, p, sizeof(Cfg));
  return c;
}

float orc_bf16_to_f32(uint16_t b) { return bf16_to_f32(b); }
uint16_t orc_f32_to_bf16(float f) { return f32_to_bf16(f); }
float orc_e4m3_to_f32(uint8_t c) { return e4m3_to_f32(c); }
uint8_t orc_f32_to_e4m3(float f) { return f32_to_e4m3(f); }

void orc_f32_to_bf16_n(const float* in, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16(in[i]);
}
void orc_f32_to_e4m3_n(const float* in, uint8_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_e4m3(in[i]);
}
// Converts every binary32 bit pattern in [first, first + n) (as uint32).
void orc_e4m3_of_bits(uint32_t first, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) {
    const uint32_t u = first + static_cast<uint32_t>(i);
    float f;
    std::memcpy(&f, &u, 4);
    out[i] = f32_to_e4m3(f);
  }
}
void orc_bf16_of_bits(uint32_t first, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) {
    const uint32_t u = first + static_cast<uint32_t>(i);
    float f;
    std::memcpy(&f, &u, 4);
    out[i] = f32_to_bf16(f);
  }
}
void orc_cast_row_fp8(const uint16_t* x, int H, uint8_t* q, float* sf) { cast_row_fp8(x, H, q, sf); }
void orc_cast_row_fp8_ue8m0(const uint16_t* x, int H, uint8_t* q, uint32_t* words) {
  cast_row_fp8_ue8m0(x, H, q, words);
}

// Number of rows the receive buffer recv_x needs: the expanded upper bound
// R*T*K + E*(align-1), else the rows of the receive tensors (entry_rows).
int64_t orc_recv_rows(const orc_cfg* p) {
  const Cfg c = to_cfg(p);
  const int64_t R = ranks(c);
  if (c.expand) return R * c.T * c.K + static_cast<int64_t>(c.E) * (c.align - 1);
  return entry_rows(c);
}

// Rows of the sidecar tensors (recv_topk_idx, recv_topk_weights,
// recv_src_metadata): the deduplicated entries' rows, R*R*M in the row form,
// compact and expanded layouts, the capacity when packed.
int64_t orc_sidecar_rows(const orc_cfg* p) { return entry_rows(to_cfg(p)); }

// Dispatch layout: counts, per-lane slots and (expanded) positions.
//   num_tokens_per_rank   [R][R]    (src, dst): tokens of src that reach dst, once per token
//   num_tokens_per_expert [R][E]    (src, expert): valid lanes
//   is_token_in_rank      [R][T][R] 0/1
//   slot_map              [R][T][K] row inside the destination's region, -1 if masked
//   recv_cnt              [R][R]    (dst, src) = num_tokens_per_rank transposed
//   recv_psum             [R][R]    (dst, row block i) inclusive prefix of recv_cnt in
//                                   row-block order (block i holds source src_of_block(i))
//   recv_region           [R+1]     (may be null) first packed row of each destination:
//                                   the entries all destinations before it receive; [R] = total
//   exp_cnt [R][L], exp_base [R][L+1], exp_region [R+1], exp_pos [R][T][K] (expanded only)
int orc_layout(const orc_cfg* p, const int64_t* topk_idx, int32_t* num_tokens_per_rank,
               int32_t* num_tokens_per_expert, uint8_t* is_token_in_rank, int32_t* slot_map,
               int32_t* recv_cnt, int32_t* recv_psum, int32_t* recv_region, int32_t* exp_cnt,
               int32_t* exp_base, int32_t* exp_region, int32_t* exp_pos) {
  const Cfg c = to_cfg(p);
  int status = check_cfg(c);
  if (status != kOk) return status;
  const int R = ranks(c), L = c.E / R, K = c.K, T = c.T, M = c.M;

  std::memset(num_tokens_per_rank, 0, sizeof(int32_t) * R * R);
  std::memset(num_tokens_per_expert, 0, sizeof(int32_t) * R * c.E);
  std::memset(is_token_in_rank, 0, static_cast<size_t>(R) * T * R);

  std::vector<int32_t> running(R);  // sender's running count per destination
  std::vector<int64_t> row_of(R);   // this token's row per destination
  for (int s = 0; s < R; ++s) {
    std::fill(running.begin(), running.end(), 0);
    for (int t = 0; t < T; ++t) {
      const int64_t* idx_tok = topk_idx + (static_cast<int64_t>(s) * T + t) * K;
      int32_t* slot_tok = slot_map + (static_cast<int64_t>(s) * T + t) * K;
      std::fill(row_of.begin(), row_of.end(), -1);
      for (int k = 0; k < K; ++k) {
        if (!lane_valid(c, idx_tok, k, &status)) {
          slot_tok[k] = -1;
          continue;
        }
        const int e = static_cast<int>(idx_tok[k]);
        const int d = e / L;
        num_tokens_per_expert[s * c.E + e] += 1;
        if (row_of[d] < 0) {  // first lane to d: this token's dedup entry for d
          if (running[d] >= M) {
            status = kOverflow;
            slot_tok[k] = -1;
            continue;
          }
          row_of[d] = row_block(c, s) * M + running[d];
          running[d] += 1;
          is_token_in_rank[(static_cast<int64_t>(s) * T + t) * R + d] = 1;
          num_tokens_per_rank[s * R + d] += 1;
        }
        slot_tok[k] = static_cast<int32_t>(row_of[d]);
      }
    }
  }

  // receive side: per-source counts and their prefix sums in row-block order
  std::vector<int> src_of_block(R);
  for (int s = 0; s < R; ++s) src_of_block[row_block(c, s)] = s;
  int32_t all = 0;
  for (int d = 0; d < R; ++d) {
    int32_t acc = 0;
    for (int s = 0; s < R; ++s) recv_cnt[d * R + s] = num_tokens_per_rank[s * R + d];
    for (int i = 0; i < R; ++i) {
      acc += recv_cnt[d * R + src_of_block[i]];
      recv_psum[d * R + i] = acc;
    }
    if (recv_region) recv_region[d] = all;
    all += acc;
  }
  if (recv_region) recv_region[R] = all;

  if (c.expand) {
    // per (destination, local expert) totals, aligned block starts, regions
    for (int d = 0; d < R; ++d) {
      exp_base[d * (L + 1)] = 0;
      for (int j = 0; j < L; ++j) {
        int32_t n = 0;
        for (int s = 0; s < R; ++s) n += num_tokens_per_expert[s * c.E + d * L + j];
        exp_cnt[d * L + j] = n;
        const int32_t padded = (n + c.align - 1) / c.align * c.align;
        exp_base[d * (L + 1) + j + 1] = exp_base[d * (L + 1) + j] + padded;
      }
    }
    exp_region[0] = 0;
    for (int d = 0; d < R; ++d) exp_region[d + 1] = exp_region[d] + exp_base[d * (L + 1) + L];
    // positions: inside the expert's block, lanes in (source rank, token) order
    std::vector<int32_t> fill(c.E, 0);
    int dummy = kOk;
    for (int s = 0; s < R; ++s) {
      for (int t = 0; t < T; ++t) {
        const int64_t* idx_tok = topk_idx + (static_cast<int64_t>(s) * T + t) * K;
        int32_t* pos_tok = exp_pos + (static_cast<int64_t>(s) * T + t) * K;
        for (int k = 0; k < K; ++k) {
          if (!lane_valid(c, idx_tok, k, &dummy)) {
            pos_tok[k] = -1;
            continue;
          }
          const int e = static_cast<int>(idx_tok[k]);
          const int d = e / L, j = e % L;
          pos_tok[k] = exp_base[d * (L + 1) + j] + fill[e];
          fill[e] += 1;
        }
      }
    }
  }
  return status;
}

// The receive rows of one source token (s, t), computed from that token's
// inputs and its layout entries (recv_psum for the compact and packed layouts,
// recv_region for the packed one, exp_region when expanded).
//   hid      : the row as received (H bf16 values, or H e4m3 codes)
//   hid_sf   : its scale sidecar (FP8 receive only): G = H/128 fp32 scales, or
//              ceil(G/4) words of packed exponent bytes
//   hid_dst / hid_row : the n_hid (destination, row of recv_x) pairs that
//              receive the hidden row: the entry's row (entry_row), or the
//              expanded row exp_region[d] + position
//   meta_dst / meta_row : the n_meta deduplicated entries: destination and row
//              of the sidecar tensors (entry_row)
//   meta_idx [K][K] int64, meta_w [K][K] fp32, meta_md [K][2+K] int32: the
//              sidecar rows written at meta_row[i]
// Returns n_hid | (n_meta << 8).
int orc_dispatch_token(const orc_cfg* p, int s, int t, const int32_t* slot_tok,
                       const int32_t* pos_tok, const int32_t* recv_psum, const int32_t* recv_region,
                       const int32_t* exp_region, const void* x_row, const float* x_sf_row,
                       const int64_t* idx_tok, const float* w_tok, uint8_t* hid, float* hid_sf,
                       int32_t* hid_dst, int64_t* hid_row, int32_t* meta_dst, int64_t* meta_row,
                       int64_t* meta_idx, float* meta_w, int32_t* meta_md) {
  const Cfg c = to_cfg(p);
  const int R = ranks(c), L = c.E / R, K = c.K, H = c.H;
  (void)R;
  int status = kOk;

  // the row as it is received
  if (c.x_fp8) {
    std::memcpy(hid, x_row, H);
    std::memcpy(hid_sf, x_sf_row, sizeof(uint32_t) * sf_words(H, c.sf_pack));
  } else if (c.recv_fp8 && c.sf_pack) {
    cast_row_fp8_ue8m0(static_cast<const uint16_t*>(x_row), H, hid, reinterpret_cast<uint32_t*>(hid_sf));
  } else if (c.recv_fp8) {
    cast_row_fp8(static_cast<const uint16_t*>(x_row), H, hid, hid_sf);
  } else {
    std::memcpy(hid, x_row, sizeof(uint16_t) * H);
  }

  std::vector<int> lane_d(K, -1);
  for (int k = 0; k < K; ++k)
    if (lane_valid(c, idx_tok, k, &status)) lane_d[k] = static_cast<int>(idx_tok[k]) / L;

  int n_hid = 0, n_meta = 0;
  for (int k = 0; k < K; ++k) {
    const int d = lane_d[k];
    if (d < 0 || slot_tok[k] < 0) continue;
    bool first = true;
    for (int j = 0; j < k; ++j)
      if (lane_d[j] == d && slot_tok[j] >= 0) first = false;
    if (c.expand) {
      hid_dst[n_hid] = d;
      hid_row[n_hid] = static_cast<int64_t>(exp_region[d]) + pos_tok[k];
      ++n_hid;
    }
    if (!first) continue;
    const int64_t row = entry_row(c, d, slot_tok[k], recv_psum, recv_region);
    if (!c.expand) {
      hid_dst[n_hid] = d;
      hid_row[n_hid] = row;
      ++n_hid;
    }
    meta_dst[n_meta] = d;
    meta_row[n_meta] = row;
    int32_t* md = meta_md + static_cast<int64_t>(n_meta) * (2 + K);
    md[0] = s;
    md[1] = t;
    for (int j = 0; j < K; ++j) {
      const bool on_d = lane_d[j] == d;
      meta_idx[n_meta * K + j] = on_d ? idx_tok[j] - static_cast<int64_t>(d) * L : -1;
      meta_w[n_meta * K + j] = on_d ? w_tok[j] : 0.0f;
      md[2 + j] = (c.expand && on_d) ? pos_tok[j] : -1;
    }
    ++n_meta;
  }
  return n_hid | (n_meta << 8);
}

// Full dispatch into caller-provided receive buffers (only filled rows are
// written; the rest are left as they are).
//   recv_x [orc_recv_rows][H] (bf16 or e4m3); recv_sf [orc_recv_rows][sf words] (FP8 only)
//   recv_topk_idx [orc_sidecar_rows][K], recv_topk_weights [orc_sidecar_rows][K],
//   recv_src_metadata [orc_sidecar_rows][2+K]
// recv_psum is needed for the compact and packed layouts, recv_region for the
// packed one. An entry whose packed row is past the capacity is not written and
// the result is OVERFLOW (never dropped silently).
int orc_dispatch(const orc_cfg* p, const int32_t* slot_map, const int32_t* exp_pos,
                 const int32_t* exp_region, const int32_t* exp_cnt, const int32_t* exp_base,
                 const int32_t* recv_psum, const int32_t* recv_region, const void* x, const float* x_sf,
                 const int64_t* topk_idx, const float* topk_weights, void* recv_x,
                 float* recv_sf, int64_t* recv_topk_idx, float* recv_topk_weights,
                 int32_t* recv_src_metadata) {
  const Cfg c = to_cfg(p);
  int status = check_cfg(c);
  if (status != kOk) return status;
  const int R = ranks(c), K = c.K, T = c.T, H = c.H, G = H / 128, SW = sf_words(H, c.sf_pack);
  const int64_t cap = entry_rows(c);
  const size_t in_eb = c.x_fp8 ? 1 : 2, out_eb = c.recv_fp8 ? 1 : 2;

  std::vector<uint8_t> hid(static_cast<size_t>(H) * 2);
  std::vector<float> hid_sf(G > 0 ? G : 1);
  std::vector<int32_t> hid_dst(K), meta_dst(K), meta_md(static_cast<size_t>(K) * (2 + K));
  std::vector<int64_t> hid_row(K), meta_row(K), meta_idx(static_cast<size_t>(K) * K);
  std::vector<float> meta_w(static_cast<size_t>(K) * K);

  for (int s = 0; s < R; ++s) {
    for (int t = 0; t < T; ++t) {
      const int64_t tok = static_cast<int64_t>(s) * T + t;
      for (int k = 0; k < K; ++k) lane_valid(c, topk_idx + tok * K, k, &status);
      const int n = orc_dispatch_token(
          p, s, t, slot_map + tok * K, c.expand ? exp_pos + tok * K : nullptr, recv_psum, recv_region,
          exp_region, static_cast<const uint8_t*>(x) + tok * H * in_eb, x_sf ? x_sf + tok * SW : nullptr,
          topk_idx + tok * K, topk_weights + tok * K, hid.data(), hid_sf.data(), hid_dst.data(),
          hid_row.data(), meta_dst.data(), meta_row.data(), meta_idx.data(), meta_w.data(),
          meta_md.data());
      const int n_hid = n & 0xFF, n_meta = n >> 8;
      for (int i = 0; i < n_hid; ++i) {
        const int64_t row = hid_row[i];
        if (c.compact == 2 && row >= cap) {
          status = kOverflow;
          continue;
        }
        std::memcpy(static_cast<uint8_t*>(recv_x) + row * H * out_eb, hid.data(), H * out_eb);
        if (c.recv_fp8) std::memcpy(recv_sf + row * SW, hid_sf.data(), sizeof(float) * SW);
      }
      for (int i = 0; i < n_meta; ++i) {
        const int64_t row = meta_row[i];
        if (c.compact == 2 && row >= cap) continue;  // reported with the hidden row
        if (recv_topk_idx) std::memcpy(recv_topk_idx + row * K, &meta_idx[i * K], 8 * K);
        if (recv_topk_weights) std::memcpy(recv_topk_weights + row * K, &meta_w[i * K], 4 * K);
        if (recv_src_metadata)
          std::memcpy(recv_src_metadata + row * (2 + K), &meta_md[i * (2 + K)], 4 * (2 + K));
      }
    }
  }
  // expanded blocks padded to expert_alignment: with zero padding, the rows
  // after each expert's lanes up to the next block start are zero (and so are
  // their FP8 scales)
  if (c.expand && c.zero_padding) {
    const int L = c.E / R;
    for (int d = 0; d < R; ++d) {
      for (int j = 0; j < L; ++j) {
        const int64_t first = static_cast<int64_t>(exp_region[d]) + exp_base[d * (L + 1) + j] + exp_cnt[d * L + j];
        const int64_t end = static_cast<int64_t>(exp_region[d]) + exp_base[d * (L + 1) + j + 1];
        for (int64_t row = first; row < end; ++row) {
          std::memset(static_cast<uint8_t*>(recv_x) + row * H * out_eb, 0, H * out_eb);
          if (c.recv_fp8) std::memset(recv_sf + row * SW, 0, sizeof(float) * SW);
        }
      }
    }
  }
  return status;
}

// Row of every top-k lane in the receive tensors, from the layout:
//   hid_rows [R][T][K]  the recv_x row lane k's expert reads: its deduplicated
//                       entry's row (entry_row), or, expanded, exp_region[d] +
//                       its position;
//   side_rows [R][T][K] the sidecar row of its deduplicated entry (entry_row);
// both -1 for a masked or invalid lane and, packed, for an entry past the
// capacity (OVERFLOW is returned then).
int orc_lane_rows(const orc_cfg* p, const int64_t* topk_idx, const int32_t* slot_map,
                  const int32_t* exp_pos, const int32_t* exp_region, const int32_t* recv_psum,
                  const int32_t* recv_region, int64_t* hid_rows, int64_t* side_rows) {
  const Cfg c = to_cfg(p);
  int status = check_cfg(c);
  if (status != kOk) return status;
  const int R = ranks(c), L = c.E / R, K = c.K;
  const int64_t cap = entry_rows(c);
  const int64_t lanes = static_cast<int64_t>(R) * c.T * K;
  for (int64_t i = 0; i < lanes; ++i) {
    const int64_t* idx_tok = topk_idx + i / K * K;
    hid_rows[i] = -1;
    side_rows[i] = -1;
    if (!lane_valid(c, idx_tok, static_cast<int>(i % K), &status) || slot_map[i] < 0) continue;
    const int d = static_cast<int>(topk_idx[i]) / L;
    const int64_t row = entry_row(c, d, slot_map[i], recv_psum, recv_region);
    if (c.compact == 2 && row >= cap) {
      status = kOverflow;
      continue;
    }
    side_rows[i] = row;
    hid_rows[i] = c.expand ? (exp_pos[i] < 0 ? -1 : static_cast<int64_t>(exp_region[d]) + exp_pos[i]) : row;
  }
  return status;
}

// Weighted reduction of one token: rows[k] is the expert-output row lane k
// reads (nullptr for a masked lane). acc starts at +0 and takes one fused
// multiply-add per valid lane in lane order; the result is rounded to bf16.
void orc_combine_token(int K, int H, const uint16_t* const* rows, const float* w, uint16_t* out) {
  for (int h = 0; h < H; ++h) {
    float acc = 0.0f;
    for (int k = 0; k < K; ++k)
      if (rows[k] != nullptr) acc = std::fmaf(w[k], bf16_to_f32(rows[k][h]), acc);
    out[h] = f32_to_bf16(acc);
  }
}

// Combine of n tokens whose lanes' rows were gathered into one compact array:
// lane_rows [n][K] indexes rows of y (-1 = masked lane), w [n][K], out [n][H].
void orc_combine_gathered(int K, int H, int64_t n, const int64_t* lane_rows, const uint16_t* y,
                          const float* w, uint16_t* out) {
  std::vector<const uint16_t*> rows(K);
  for (int64_t i = 0; i < n; ++i) {
    for (int k = 0; k < K; ++k) {
      const int64_t r = lane_rows[i * K + k];
      rows[k] = r < 0 ? nullptr : y + r * H;
    }
    orc_combine_token(K, H, rows.data(), w + i * K, out + i * H);
  }
}

// Full combine: y holds the expert outputs in the receive layout (the rows
// of recv_x: entry_row of each lane's deduplicated entry, or exp_region[d] +
// position when expanded). A lane whose packed row is past the capacity was
// never received: it is left out of the sum and the result is OVERFLOW.
int orc_combine(const orc_cfg* p, const int32_t* slot_map, const int32_t* exp_pos,
                const int32_t* exp_region, const int32_t* recv_psum, const int32_t* recv_region,
                const uint16_t* y, const int64_t* topk_idx, const float* topk_weights, uint16_t* out) {
  const Cfg c = to_cfg(p);
  int status = check_cfg(c);
  if (status != kOk) return status;
  const int R = ranks(c), L = c.E / R, K = c.K, T = c.T, H = c.H;
  const int64_t cap = entry_rows(c);
  std::vector<const uint16_t*> rows(K);
  for (int s = 0; s < R; ++s) {
    for (int t = 0; t < T; ++t) {
      const int64_t tok = static_cast<int64_t>(s) * T + t;
      for (int k = 0; k < K; ++k) {
        rows[k] = nullptr;
        if (!lane_valid(c, topk_idx + tok * K, k, &status)) continue;
        const int d = static_cast<int>(topk_idx[tok * K + k]) / L;
        if ((c.expand ? exp_pos[tok * K + k] : slot_map[tok * K + k]) < 0) continue;
        const int64_t r = c.expand ? static_cast<int64_t>(exp_region[d]) + exp_pos[tok * K + k]
                                   : entry_row(c, d, slot_map[tok * K + k], recv_psum, recv_region);
        if (c.compact == 2 && r >= cap) {
          status = kOverflow;
          continue;
        }
        rows[k] = y + r * H;
      }
      orc_combine_token(K, H, rows.data(), topk_weights + tok * K, out + tok * H);
    }
  }
  return status;
}

}  // extern "C"

// Internal host-side launcher interface between the C ABI (api.cu) and the
// kernel translation units. Arguments are validated by the caller.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "attn.h"

namespace attn {

// Attention mask (attn_mask in attn.h): key j is visible to query row i iff
// it lies in the row's window around i' = i + Nk - Nq (a negative bound is
// absent) or among the first n_global keys, and, when row ranges are given,
// in [row_kv_start[b, i], row_kv_end[b, i]). Default: every key visible.
struct MaskSpec {
  int window_left = -1, window_right = -1, n_global = 0;
  const int* row_kv_start = nullptr;   // [B, Nq] int32, device
  const int* row_kv_end = nullptr;     // [B, Nq] int32, device
  // work per query tile falls along the sequence (causal-like): CTA order
  // puts the heaviest tiles first
  bool varies() const { return window_right >= 0 || window_left >= 0 || row_kv_start != nullptr; }
};

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, Hq, Hkv, Nq, Nk, d;
  float scale;
  int causal;
  attn_dtype dt;
  cudaStream_t stream;
  MaskSpec mask;      // the full mask (causal: window (-1, 0))
};

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dO;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  int B, Hq, Hkv, Nq, Nk, d;
  float scale;
  int causal;
  attn_dtype dt;
  float* row_term;   // D = rowsum(dO ∘ O), [B, Hq, Nq]
  float* dq_acc;     // float32 dQ accumulator, [B, Hq, Nq, d]
  cudaStream_t stream;
  bool zero_dq_acc;  // the preprocess zeroes dq_acc (the passes that add into it)
  MaskSpec mask;     // the full mask (causal: window (-1, 0))
  // Work counter of the persistent dQ pass, zeroed by the preprocess;
  // nullptr when no persistent pass runs.
  int* sched = nullptr;
};

struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, Hq, Hkv, L, d;
  float scale;
  int num_splits;
  float* o_part;     // [B*Hq, S, d]
  float* m_part;     // [B*Hq, S]
  float* l_part;     // [B*Hq, S]
  cudaStream_t stream;
  // Paged cache (block_table != nullptr): k, v are pages
  // [num_pages, Hkv, page_size, d]; request b holds seq_lens[b] keys, key t
  // in page block_table[b * max_pages + t / page_size]. L is unused.
  const int* block_table = nullptr;
  const int* seq_lens = nullptr;
  int num_pages = 0, page_size = 0, max_pages = 0;
  // Sparse index list (sparse): block_table = listed rows [B, max_pages] of
  // the contiguous cache, seq_lens = list lengths, page_size = 1,
  // num_pages = L. T query tokens per request: q, o [B, Hq, T, d].
  bool sparse = false;
  int T = 1;
};

struct MergeArgs {
  const float* o_part;
  const float* m_part;
  const float* l_part;
  void* o;
  float* lse;
  int rows, num_splits, d;
  attn_dtype out_dt;
  cudaStream_t stream;
  // Decode partials (chunk > 0): row r merges only the chunks that hold keys
  // of its request, ceil(n / chunk) of them, with n = seq_lens[r / Hq] (or
  // `len` when seq_lens is null); n outside [0, max_len] counts as 0. With
  // chunk == 0 every row merges all num_splits partials.
  const int* seq_lens = nullptr;
  int Hq = 1, len = 0, max_len = 0, chunk = 0;
};

// Streaming multiprocessors of the current device (cached per device); 0 if
// it cannot be read.
inline int device_sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cached[dev] = n;
  }
  return cached[dev];
}

// Keys per decode chunk: ceil(L / S) for a contiguous cache; for a paged
// cache one length for all requests, the table's capacity over S rounded up
// to whole 32-key stages, so request b uses ceil(n_b / chunk) <= S chunks.
// A sparse index list has chunks of at least 128 entries (four 32-entry
// stages): smaller ones leave each CTA too little work to cover its start.
//
// Paged caches: every CTA pays the same start whatever its chunk (its
// request's length and table entries come back before its first copy can be
// issued, and a chunk past the request's end still pays that round trip to
// learn it is empty), so the chunk doubles while the grid keeps at least
// kDecodeWaves CTAs per resident slot: fewer, longer chunks cover the same
// keys with fewer starts, and enough CTAs stay to balance the last wave.
constexpr int kDecodeWaves = 8;
inline int decode_chunk(const DecodeArgs& a) {
  if (a.block_table == nullptr) return (a.L + a.num_splits - 1) / a.num_splits;
  const long long cap = 1LL * a.max_pages * a.page_size;
  long long c = (cap + a.num_splits - 1) / a.num_splits;
  c = (c + 31) / 32 * 32;
  if (a.sparse) return int(c < 128 ? 128 : c);
  // resident CTAs per SM of the split kernel: 3 with up to 4 query rows per
  // KV head, 2 with 8 (register-bound)
  const long long slots = 1LL * device_sm_count() * (a.Hq <= 4 * a.Hkv ? 3 : 2);
  if (slots <= 0) return int(c);
  while (2 * c < (1LL << 30)) {
    const long long splits = (cap + c - 1) / c, splits2 = (cap + 2 * c - 1) / (2 * c);
    if (splits2 == splits || 1LL * a.B * a.Hkv * splits2 < kDecodeWaves * slots) break;
    c *= 2;
  }
  return int(c);
}

// Chunk indices the split grid covers: the paged cache's ceil(capacity /
// chunk) (<= S; the partials keep the stride S), otherwise S.
inline int decode_grid_splits(const DecodeArgs& a) {
  if (a.block_table == nullptr || a.sparse) return a.num_splits;
  const long long cap = 1LL * a.max_pages * a.page_size;
  const long long c = decode_chunk(a);
  const long long n = (cap + c - 1) / c;
  return int(n < a.num_splits ? n : a.num_splits);
}

// The merge that completes a decode call.
inline MergeArgs decode_merge_args(const DecodeArgs& a) {
  MergeArgs m{a.o_part, a.m_part, a.l_part, a.o, a.lse, a.B * a.Hq * a.T, a.num_splits, a.d,
              ATTN_BF16, a.stream};
  m.seq_lens = a.seq_lens;
  m.Hq = a.Hq * a.T;   // query rows per request
  m.len = a.L;
  m.max_len = a.block_table != nullptr ? a.max_pages * a.page_size : a.L;
  m.chunk = decode_chunk(a);
  return m;
}

// Heads per CTA-order group (grouped_tile_order): with a causal mask, as many
// heads as keep `bytes_per_head` of re-read operands within `budget` bytes
// of L2 (a quarter to a half of its 126 MB); otherwise 1 (head-major).
inline int order_group(bool causal, long long bytes_per_head, long long budget = 32LL << 20) {
  if (!causal || bytes_per_head <= 0) return 1;
  const long long g = budget / bytes_per_head;
  return g < 1 ? 1 : (g > (1 << 20) ? (1 << 20) : int(g));
}

// Workspace carving (bytes, 256-aligned sections).
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// The bf16 d = 128 backward runs its dQ pass as a persistent grid that takes
// work from a counter in the workspace, with no mask, causal, or a window
// under which every query tile sees a key (always so for Nq <= Nk or a
// window open to the right); other masks use one CTA per query tile.
inline bool bwd_persistent(int d, attn_dtype dt, const MaskSpec& m, int Nq, int Nk) {
  if (dt != ATTN_BF16 || d != 128 || m.n_global != 0 || m.row_kv_start != nullptr) return false;
  const bool causal_only = m.window_left < 0 && m.window_right <= 0;
  return causal_only || Nq <= Nk || m.window_right < 0;
}
// (the persistent dQ pass's window form: any window but plain causal)
inline bool bwd_dq_window(const MaskSpec& m) {
  return !(m.window_left < 0 && m.window_right <= 0);
}

cudaError_t launch_fwd_simt(const FwdArgs& a);
cudaError_t launch_fwd_tc(const FwdArgs& a);
cudaError_t launch_fwd_tc64(const FwdArgs& a);
cudaError_t launch_bwd_preprocess(const BwdArgs& a);
cudaError_t launch_bwd_simt(const BwdArgs& a);
cudaError_t launch_bwd_tc(const BwdArgs& a);
cudaError_t launch_bwd_dq(const BwdArgs& a);
cudaError_t launch_bwd_convert(const BwdArgs& a);
cudaError_t launch_decode_split(const DecodeArgs& a);
cudaError_t launch_merge(const MergeArgs& a);

// Per-translation-unit device error words (read and cleared).
uint32_t take_error_fwd_tc();
uint32_t take_error_fwd_tc64();
uint32_t take_error_bwd_tc();
uint32_t take_error_bwd_dq();
uint32_t take_error_decode();

}  // namespace attn

// Internal host-side launcher interface between the C ABI (api.cu) and the
// kernel translation units. Arguments are validated by the caller.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "attn.h"

namespace attn {

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
};

// Workspace carving (bytes, 256-aligned sections).
inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

cudaError_t launch_fwd_simt(const FwdArgs& a);
cudaError_t launch_fwd_tc(const FwdArgs& a);
cudaError_t launch_bwd_preprocess(const BwdArgs& a);
cudaError_t launch_bwd_simt(const BwdArgs& a);
cudaError_t launch_bwd_tc(const BwdArgs& a);
cudaError_t launch_bwd_dq(const BwdArgs& a);
cudaError_t launch_bwd_convert(const BwdArgs& a);
cudaError_t launch_decode_split(const DecodeArgs& a);
cudaError_t launch_merge(const MergeArgs& a);

// Per-translation-unit device error words (read and cleared).
uint32_t take_error_fwd_tc();
uint32_t take_error_bwd_tc();
uint32_t take_error_bwd_dq();
uint32_t take_error_decode();

}  // namespace attn

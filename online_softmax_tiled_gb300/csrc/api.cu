// C ABI entry points: argument validation, workspace carving and dispatch to
// the kernel launchers. Declarations and their documentation: include/attn.h.

#include <stdint.h>

#include "common.cuh"
#include "launchers.h"

using namespace attn;

namespace {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline attn_status from_cuda(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

attn_status check_attention_shapes(int B, int Hq, int Hkv, int Nq, int Nk, int d, int causal,
                                   attn_dtype dt) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Nq <= 0 || Nk <= 0 || d <= 0) return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (causal && Nq > Nk) return ATTN_ERR_INVALID_ARG;
  if (dt != ATTN_F32 && dt != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  // index arithmetic inside the kernels uses 32-bit row counts per head
  if ((long long)B * Hq * Nq > (1LL << 31) || (long long)B * Hkv * Nk > (1LL << 31))
    return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

// Row term D, then 256 bytes for the persistent dQ pass's work counter, then
// the float32 dQ accumulator.
struct BwdLayout {
  size_t row_term, sched, dq_acc, total;
};

BwdLayout bwd_layout(int B, int Hq, int Nq, int d) {
  BwdLayout l;
  const size_t rows = size_t(B) * Hq * Nq;
  l.row_term = 0;
  l.sched = align256(rows * sizeof(float));
  l.dq_acc = l.sched + 256;
  l.total = l.dq_acc + align256(rows * d * sizeof(float));
  return l;
}

// bf16 at d = 128 runs the dQ query-tile pass, which writes dQ directly: only
// the row term and the counter are needed. Every other path also adds dQ
// into the float32 accumulator that follows them.
inline bool bwd_split_dq(int d, attn_dtype dt) { return dt == ATTN_BF16 && d == 128; }

size_t bwd_workspace_need(const BwdLayout& l, int d, attn_dtype dt) {
  return bwd_split_dq(d, dt) ? l.dq_acc : l.total;
}

struct DecodeLayout {
  size_t o_part, m_part, l_part, total;
};

DecodeLayout decode_layout(int B, int Hq, int d, int S) {
  DecodeLayout l;
  const size_t n = size_t(B) * Hq * S;
  l.o_part = 0;
  l.m_part = align256(n * d * sizeof(float));
  l.l_part = l.m_part + align256(n * sizeof(float));
  l.total = l.l_part + align256(n * sizeof(float));
  return l;
}

}  // namespace

extern "C" {

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_MISALIGNED: return "misaligned pointer (16-byte alignment required)";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    case ATTN_ERR_DEVICE_INDEX: return "out-of-range length or page index read on the device";
  }
  return "unknown status";
}

namespace {

inline bool scale_ok(float scale) { return scale > 0.f && scale <= 3.4e38f; }   // rejects NaN too

MaskSpec mask_spec(const attn_mask* m) {
  MaskSpec ms;
  if (m != nullptr) {
    ms.window_left = m->window_left < 0 ? -1 : m->window_left;
    ms.window_right = m->window_right < 0 ? -1 : m->window_right;
    ms.n_global = m->n_global < 0 ? 0 : m->n_global;
    ms.row_kv_start = m->row_kv_start;
    ms.row_kv_end = m->row_kv_end;
  }
  return ms;
}

attn_status check_mask(const attn_mask* m) {
  if (m == nullptr) return ATTN_OK;
  if ((m->row_kv_start == nullptr) != (m->row_kv_end == nullptr)) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(m->row_kv_start) & 3u) ||
      (reinterpret_cast<uintptr_t>(m->row_kv_end) & 3u))
    return ATTN_ERR_MISALIGNED;
  return ATTN_OK;
}

attn_status fwd_common(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int Hq, int Hkv, int Nq, int Nk, int d, float scale, const MaskSpec& ms,
                       attn_dtype dt, void* stream) {
  if (!q || !k || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (!scale_ok(scale)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse && !aligned16(lse)))
    return ATTN_ERR_MISALIGNED;
  const int causal = (ms.window_left < 0 && ms.window_right == 0 && ms.n_global == 0 &&
                      ms.row_kv_start == nullptr) ? 1 : 0;
  FwdArgs a{q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, causal, dt,
            static_cast<cudaStream_t>(stream)};
  a.mask = ms;
  if (dt == ATTN_BF16) return from_cuda(launch_fwd_tc(a));
  return from_cuda(launch_fwd_simt(a));
}

}  // namespace

attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                     int Hq, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                     attn_dtype dt, void* stream) {
  attn_status st = check_attention_shapes(B, Hq, Hkv, Nq, Nk, d, causal, dt);
  if (st != ATTN_OK) return st;
  MaskSpec ms;
  if (causal) ms.window_right = 0;
  return fwd_common(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, ms, dt, stream);
}

attn_status attn_fwd_masked(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale,
                            const attn_mask* mask, attn_dtype dt, void* stream) {
  // any Nq, Nk: rows may see nothing, so the causal Nq <= Nk rule does not apply
  attn_status st = check_attention_shapes(B, Hq, Hkv, Nq, Nk, d, 0, dt);
  if (st != ATTN_OK) return st;
  if ((st = check_mask(mask)) != ATTN_OK) return st;
  return fwd_common(q, k, v, o, lse, B, Hq, Hkv, Nq, Nk, d, scale, mask_spec(mask), dt, stream);
}

size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int d) {
  (void)Hkv;
  (void)Nk;
  if (B <= 0 || Hq <= 0 || Nq <= 0 || d <= 0) return 0;
  return bwd_layout(B, Hq, Nq, d).total;
}

size_t attn_bwd_workspace_size_dt(int B, int Hq, int Hkv, int Nq, int Nk, int d,
                                  attn_dtype dt) {
  (void)Hkv;
  (void)Nk;
  if (B <= 0 || Hq <= 0 || Nq <= 0 || d <= 0) return 0;
  if (dt != ATTN_F32 && dt != ATTN_BF16) return 0;
  return bwd_workspace_need(bwd_layout(B, Hq, Nq, d), d, dt);
}

namespace {

attn_status bwd_common(const void* q, const void* k, const void* v, const void* o,
                       const void* dO, const float* lse, void* dq, void* dk, void* dv, int B,
                       int Hq, int Hkv, int Nq, int Nk, int d, float scale, const MaskSpec& ms,
                       attn_dtype dt, void* workspace, size_t ws_bytes, void* stream) {
  if (!q || !k || !v || !o || !dO || !lse || !dq || !dk || !dv) return ATTN_ERR_INVALID_ARG;
  if (!scale_ok(scale)) return ATTN_ERR_INVALID_ARG;
  const void* ptrs[] = {q, k, v, o, dO, lse, dq, dk, dv};
  for (const void* p : ptrs)
    if (!aligned16(p)) return ATTN_ERR_MISALIGNED;
  const BwdLayout lay = bwd_layout(B, Hq, Nq, d);
  if (!workspace || ws_bytes < bwd_workspace_need(lay, d, dt)) return ATTN_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_ERR_MISALIGNED;
  const bool plain = ms.window_left < 0 && ms.window_right <= 0 && ms.n_global == 0 &&
                     ms.row_kv_start == nullptr;
  // masks with global keys or row ranges on the tensor-core key-tile pass
  // list at most 1024 query tiles (64 rows at d = 128, 128 rows at d = 64)
  // per key tile (windows take their tiles from the bounds)
  const bool listed = ms.n_global != 0 || ms.row_kv_start != nullptr;
  if (listed && dt == ATTN_BF16 && (Nq + (d == 128 ? 64 : 128) - 1) / (d == 128 ? 64 : 128) > 1024)
    return ATTN_ERR_UNSUPPORTED;
  const int causal = (plain && ms.window_right == 0) ? 1 : 0;
  char* ws = static_cast<char*>(workspace);
  BwdArgs a{q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, Nq, Nk, d, scale, causal, dt,
            reinterpret_cast<float*>(ws + lay.row_term), reinterpret_cast<float*>(ws + lay.dq_acc),
            static_cast<cudaStream_t>(stream), true};
  a.mask = ms;
  if (bwd_persistent(d, dt, ms, Nq, Nk)) a.sched = reinterpret_cast<int*>(ws + lay.sched);
  // bf16, d = 128: a key-tile pass (dK, dV) and a query-tile pass (dQ, written
  // in bf16 directly; the float32 accumulator is not used). Otherwise one
  // pass adds dQ into the float32 accumulator, converted at the end.
  const bool split_dq = bwd_split_dq(d, dt);
  a.zero_dq_acc = !split_dq;
  cudaError_t e = launch_bwd_preprocess(a);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  if (split_dq) {
    e = launch_bwd_tc(a);
    if (e != cudaSuccess) return ATTN_ERR_CUDA;
    return from_cuda(launch_bwd_dq(a));
  }
  e = (dt == ATTN_BF16) ? launch_bwd_tc(a) : launch_bwd_simt(a);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  return from_cuda(launch_bwd_convert(a));
}

}  // namespace

attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dO,
                     const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv,
                     int Nq, int Nk, int d, float scale, int causal, attn_dtype dt,
                     void* workspace, size_t ws_bytes, void* stream) {
  attn_status st = check_attention_shapes(B, Hq, Hkv, Nq, Nk, d, causal, dt);
  if (st != ATTN_OK) return st;
  MaskSpec ms;
  if (causal) ms.window_right = 0;
  return bwd_common(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, Nq, Nk, d, scale, ms, dt,
                    workspace, ws_bytes, stream);
}

attn_status attn_bwd_masked(const void* q, const void* k, const void* v, const void* o,
                            const void* dO, const float* lse, void* dq, void* dk, void* dv,
                            int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale,
                            const attn_mask* mask, attn_dtype dt, void* workspace,
                            size_t ws_bytes, void* stream) {
  attn_status st = check_attention_shapes(B, Hq, Hkv, Nq, Nk, d, 0, dt);
  if (st != ATTN_OK) return st;
  if ((st = check_mask(mask)) != ATTN_OK) return st;
  return bwd_common(q, k, v, o, dO, lse, dq, dk, dv, B, Hq, Hkv, Nq, Nk, d, scale,
                    mask_spec(mask), dt, workspace, ws_bytes, stream);
}

size_t attn_decode_workspace_size(int B, int Hq, int d, int num_splits) {
  if (B <= 0 || Hq <= 0 || d <= 0 || num_splits <= 0) return 0;
  return decode_layout(B, Hq, d, num_splits).total;
}

attn_status attn_decode_splitkv(const void* q, const void* k_cache, const void* v_cache, void* o,
                                float* lse, int B, int Hq, int Hkv, int L, int d, float scale,
                                int num_splits, void* workspace, size_t ws_bytes, void* stream) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || L <= 0 || d <= 0 || num_splits <= 0)
    return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !o) return ATTN_ERR_INVALID_ARG;
  if (!(scale == scale)) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return ATTN_ERR_UNSUPPORTED;
  // (eight query heads per KV head run as two CTAs of four: grid rows Hkv·2)
  if (num_splits > 65535 || B > 65535 || 1LL * Hkv * G > 65535) return ATTN_ERR_UNSUPPORTED;
  // work items (request, KV head, chunk) are numbered in 32 bits
  if (1LL * B * Hkv * num_splits > (1LL << 30)) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
      (lse && !aligned16(lse)))
    return ATTN_ERR_MISALIGNED;
  const DecodeLayout lay = decode_layout(B, Hq, d, num_splits);
  if (!workspace || ws_bytes < lay.total) return ATTN_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_ERR_MISALIGNED;
  char* ws = static_cast<char*>(workspace);
  DecodeArgs a{q, k_cache, v_cache, o, lse, B, Hq, Hkv, L, d, scale, num_splits,
               reinterpret_cast<float*>(ws + lay.o_part), reinterpret_cast<float*>(ws + lay.m_part),
               reinterpret_cast<float*>(ws + lay.l_part), static_cast<cudaStream_t>(stream)};
  cudaError_t e = launch_decode_split(a);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  return from_cuda(launch_merge(decode_merge_args(a)));
}

attn_status attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                              const int* block_table, const int* seq_lens, void* o, float* lse,
                              int B, int Hq, int Hkv, int num_pages, int page_size,
                              int max_pages_per_seq, int d, float scale, int num_splits,
                              void* workspace, size_t ws_bytes, void* stream) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || num_pages <= 0 || page_size <= 0 ||
      max_pages_per_seq <= 0 || d <= 0 || num_splits <= 0)
    return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!q || !k_pages || !v_pages || !block_table || !seq_lens || !o) return ATTN_ERR_INVALID_ARG;
  if (!(scale == scale)) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return ATTN_ERR_UNSUPPORTED;
  // (eight query heads per KV head run as two CTAs of four: grid rows Hkv·2)
  if (num_splits > 65535 || B > 65535 || 1LL * Hkv * G > 65535) return ATTN_ERR_UNSUPPORTED;
  // work items (request, KV head, chunk) are numbered in 32 bits
  if (1LL * B * Hkv * num_splits > (1LL << 30)) return ATTN_ERR_UNSUPPORTED;
  // key positions and page row offsets are 32-bit inside the kernel
  if ((long long)max_pages_per_seq * page_size > (1LL << 30) ||
      (long long)num_pages * Hkv * page_size > (1LL << 40))
    return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o) ||
      (lse && !aligned16(lse)) || (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
    return ATTN_ERR_MISALIGNED;
  const DecodeLayout lay = decode_layout(B, Hq, d, num_splits);
  if (!workspace || ws_bytes < lay.total) return ATTN_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_ERR_MISALIGNED;
  char* ws = static_cast<char*>(workspace);
  DecodeArgs a{q, k_pages, v_pages, o, lse, B, Hq, Hkv, 0, d, scale, num_splits,
               reinterpret_cast<float*>(ws + lay.o_part), reinterpret_cast<float*>(ws + lay.m_part),
               reinterpret_cast<float*>(ws + lay.l_part), static_cast<cudaStream_t>(stream)};
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.num_pages = num_pages;
  a.page_size = page_size;
  a.max_pages = max_pages_per_seq;
  cudaError_t e = launch_decode_split(a);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  return from_cuda(launch_merge(decode_merge_args(a)));
}

attn_status attn_decode_sparse(const void* q, const void* k_cache, const void* v_cache,
                               const int* indices, const int* counts, void* o, float* lse, int B,
                               int Hq, int Hkv, int T, int L, int max_idx, int d, float scale,
                               int num_splits, void* workspace, size_t ws_bytes, void* stream) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || T <= 0 || L <= 0 || max_idx <= 0 || d <= 0 ||
      num_splits <= 0)
    return ATTN_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !indices || !counts || !o) return ATTN_ERR_INVALID_ARG;
  if (!(scale == scale)) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  const int G = Hq / Hkv;
  if (G != 1 && G != 2 && G != 4 && G != 8) return ATTN_ERR_UNSUPPORTED;
  if (num_splits > 65535 || B > 65535 || max_idx > (1 << 30)) return ATTN_ERR_UNSUPPORTED;
  // query rows (heads x tokens) and the CTAs over them stay in 32 bits; one
  // CTA row group holds at least one row, so Hkv x G x T bounds the grid rows
  const long long rows = 1LL * Hq * T;
  if (rows * B > (1LL << 30) || 1LL * Hkv * G * T > 65535 ||
      1LL * B * Hkv * G * T * num_splits > (1LL << 30))
    return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
      (lse && !aligned16(lse)) || (reinterpret_cast<uintptr_t>(indices) & 3u) ||
      (reinterpret_cast<uintptr_t>(counts) & 3u))
    return ATTN_ERR_MISALIGNED;
  const DecodeLayout lay = decode_layout(B, int(rows), d, num_splits);
  if (!workspace || ws_bytes < lay.total) return ATTN_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_ERR_MISALIGNED;
  char* ws = static_cast<char*>(workspace);
  DecodeArgs a{q, k_cache, v_cache, o, lse, B, Hq, Hkv, L, d, scale, num_splits,
               reinterpret_cast<float*>(ws + lay.o_part), reinterpret_cast<float*>(ws + lay.m_part),
               reinterpret_cast<float*>(ws + lay.l_part), static_cast<cudaStream_t>(stream)};
  a.block_table = indices;
  a.seq_lens = counts;
  a.num_pages = L;          // a listed row must lie in [0, L)
  a.page_size = 1;
  a.max_pages = max_idx;
  a.sparse = true;
  a.T = T;
  cudaError_t e = launch_decode_split(a);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  return from_cuda(launch_merge(decode_merge_args(a)));
}

attn_status attn_merge_partials(const float* o_part, const float* m_part, const float* l_part,
                                void* o, float* lse, int rows, int num_splits, int d,
                                attn_dtype out_dt, void* stream) {
  if (rows <= 0 || num_splits <= 0 || d <= 0) return ATTN_ERR_INVALID_ARG;
  if (!o_part || !m_part || !l_part || !o) return ATTN_ERR_INVALID_ARG;
  if (out_dt != ATTN_F32 && out_dt != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (d % 4 != 0 || d > 256) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(o_part) || !aligned16(o)) return ATTN_ERR_MISALIGNED;
  MergeArgs m{o_part, m_part, l_part, o, lse, rows, num_splits, d, out_dt,
              static_cast<cudaStream_t>(stream)};
  return from_cuda(launch_merge(m));
}

attn_status attn_sync_status(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  const uint32_t w = take_error_fwd_tc() | take_error_fwd_tc64() | take_error_bwd_tc() |
                     take_error_bwd_dq() | take_error_decode();
  if (w == 0xffffffffu) return ATTN_ERR_CUDA;
  if (w & kErrTimeout) return ATTN_ERR_DEVICE_TIMEOUT;
  if (w & kErrBadIndex) return ATTN_ERR_DEVICE_INDEX;
  return ATTN_OK;
}

}  // extern "C"

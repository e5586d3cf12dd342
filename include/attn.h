/*
 * attn.h — C ABI of the GB300 (sm_103a) tiled exact-attention library.
 *
 * Every entry point computes exact softmax attention
 *     O = softmax(scale · Q Kᵀ) V
 * tile by tile with the online-softmax recurrence, as defined in the
 * "Flash Attention 2" post (ahmadsaeedzaidi.github.io feed), sections
 * "Standard Attention" (the definition) and "Flash Attention 2" (the inner
 * loop: running row max m, running denominator l, accumulator rescaled by
 * exp(m_old - m_new), one division by l at the end). The N×N score matrix
 * never reaches device memory.
 *
 * Conventions shared by all calls
 * -------------------------------
 * Layout. Q, O, dO, dQ are [B, Hq, Nq, d]; K, V, dK, dV are [B, Hkv, Nk, d];
 *   all contiguous, row-major, d innermost. LSE and the backward row term are
 *   [B, Hq, Nq] float32. Decode uses q, o [B, Hq, d] and a KV cache
 *   [B, Hkv, L, d] (the KVCache layout of the KV-compression post on
 *   shreyansh26.github.io: batch, head, sequence, head_dim).
 * GQA. Query head h reads KV head h / (Hq / Hkv) (contiguous groups, as the
 *   KV-compression post's SnapKV code views heads); Hq % Hkv must be 0.
 * LSE. Natural-log logsumexp of the scaled scores of each query row,
 *   LSE = m + ln(l). A row with no visible key has O = 0 and LSE = -inf.
 * Causal. Key j is visible to query i iff j <= i + (Nk - Nq) (bottom-right
 *   alignment; at Nq == Nk this is the lower-triangular mask of the Flash
 *   Attention 2 post, section "Causal masking"). Causal with Nq > Nk is
 *   rejected.
 * Pointers. All tensor pointers are DEVICE pointers owned by the caller.
 *   The library allocates no memory and keeps no per-call state; scratch
 *   space comes from the caller through the *_workspace_size() contract.
 *   bf16 tensors must be 16-byte aligned; float32 tensors 16-byte aligned.
 * Streams. `stream` is a cudaStream_t passed as void* (NULL = the legacy
 *   default stream). All calls are asynchronous on that stream and return
 *   after argument validation and launch. Arguments are validated before
 *   anything is launched; on any error nothing is launched.
 * Device-side waits. Every wait inside a kernel is bounded; a wait that runs
 *   out sets a library error word and the kernel returns. attn_sync_status()
 *   reports that as ATTN_ERR_DEVICE_TIMEOUT.
 * Error word scope. The device error word is one per device for the whole
 *   process: every call and every stream on that device sets the same word,
 *   and attn_sync_status() reports and clears it for whichever caller polls
 *   first. With several streams (or threads) on one device, a timeout or a
 *   bad index raised by work on one stream can therefore be reported to, and
 *   cleared by, a caller that polls another; callers that need to attribute
 *   a device error to a call must poll with no other work in flight.
 */
#ifndef ONLINE_SOFTMAX_TILED_GB300_ATTN_H
#define ONLINE_SOFTMAX_TILED_GB300_ATTN_H

#include <stddef.h>

#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = -1,     /* null pointer, non-positive size, Hq % Hkv != 0, ... */
  ATTN_ERR_UNSUPPORTED = -2,     /* valid but not implemented (head dim, dtype, ...)   */
  ATTN_ERR_MISALIGNED = -3,      /* a tensor pointer is not 16-byte aligned             */
  ATTN_ERR_WORKSPACE = -4,       /* workspace null or smaller than *_workspace_size()   */
  ATTN_ERR_CUDA = -5,            /* a CUDA runtime call or kernel launch failed         */
  ATTN_ERR_DEVICE_TIMEOUT = -6,  /* a bounded device-side wait ran out                  */
  ATTN_ERR_DEVICE_INDEX = -7     /* a length or page index read on the device was out of range */
} attn_status;

typedef enum { ATTN_F32 = 0, ATTN_BF16 = 1 } attn_dtype;

/*
 * Forward pass with the row log-sum-exp.
 *
 * Flash Attention 2 post, section "Flash Attention 2", inner-loop steps 1-5
 * and the final safe normalisation; the saved per-row statistic is the LSE
 * (the attention-residuals kernel lab on manishklach.github.io saves the row
 * max and denominator for the backward; LSE = max + ln(denominator) carries
 * both). Scores are scaled by `scale` (1/sqrt(d) in the ML notes'
 * attention Q&A on haolingpu.github.io); scale must be positive and finite
 * (the kernels take each row maximum before scaling).
 *
 * q [B,Hq,Nq,d], k/v [B,Hkv,Nk,d] in `dt`; o [B,Hq,Nq,d] written in `dt`;
 * lse [B,Hq,Nq] float32 written (may be NULL to skip it).
 * dt = ATTN_BF16: tcgen05 tensor-core path, d in {64, 128}; the probabilities
 *   are rounded to bf16 for the P·V product, all softmax state is float32.
 * dt = ATTN_F32:  float32 FFMA path (no TF32), d in {64, 128}.
 * Returns ATTN_OK or an error listed above; nothing is launched on error.
 */
ATTN_API attn_status attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                     int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                     attn_dtype dt, void* stream);

/*
 * Attention mask.
 *
 * Flash Attention 2 post, section "Causal masking", option A and its "Why":
 * any mask (sliding window, document boundaries, prefix LM, ...) is a
 * 0 / -inf term added to the scores before the online softmax; key tiles no
 * query row of a tile can see are skipped, tiles that straddle a boundary
 * are masked element by element.
 *
 * Query row i (0-based) sits at position i' = i + (Nk - Nq) of the key axis
 * (bottom-right alignment, as for causal). Key j is visible to row i of
 * batch entry b iff
 *     [ (window_left  < 0 || j >= i' - window_left)  and
 *       (window_right < 0 || j <= i' + window_right) ]   (its window)
 *     or j < n_global                                    (global keys)
 *   and, when row_kv_start / row_kv_end are given,
 *     row_kv_start[b*Nq + i] <= j < row_kv_end[b*Nq + i] (its key range).
 * Examples: no mask {-1, -1, 0}; causal {-1, 0, 0}; sliding window of W keys
 * {W-1, 0, 0}; attention sinks plus a window {W-1, 0, n_sink}; prefix LM
 * with a prefix of P tokens {-1, 0, P}; documents packed into one sequence:
 * each row's document as its key range, with {-1, 0, 0} (causal within a
 * document) or {-1, -1, 0}.
 * row_kv_start and row_kv_end: [B, Nq] int32 in device memory, both or
 * neither; values are clipped to [0, Nk]; the same for every head.
 * A row with no visible key gets O = 0, LSE = -inf.
 */
typedef struct {
  int window_left;
  int window_right;
  int n_global;
  const int* row_kv_start;
  const int* row_kv_end;
} attn_mask;

/*
 * attn_fwd under a general mask (see attn_mask). mask == NULL: no mask.
 * Any Nq, Nk > 0 (rows may have no visible key); otherwise as attn_fwd.
 */
ATTN_API attn_status attn_fwd_masked(const void* q, const void* k, const void* v, void* o,
                                     float* lse, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                                     float scale, const attn_mask* mask, attn_dtype dt,
                                     void* stream);

/*
 * Bytes of device scratch attn_bwd needs for any dtype: the row term D
 * [B,Hq,Nq] float32, 256 bytes for a work counter, and a float32 dQ
 * accumulator [B,Hq,Nq,d], each 256-byte aligned. This is the largest
 * need; attn_bwd_workspace_size_dt gives the exact need of one dtype.
 */
ATTN_API size_t attn_bwd_workspace_size(int B, int Hq, int Hkv, int Nq, int Nk, int d);

/*
 * Bytes of device scratch attn_bwd (and attn_bwd_masked) use for dtype `dt`:
 * with dt = ATTN_BF16 and d = 128 only the row term D [B,Hq,Nq] float32
 * (256-byte aligned) and the 256-byte work counter of the dQ pass, which
 * writes dQ directly; otherwise also the float32 dQ accumulator, as
 * attn_bwd_workspace_size. 0 for invalid arguments.
 */
ATTN_API size_t attn_bwd_workspace_size_dt(int B, int Hq, int Hkv, int Nq, int Nk, int d,
                                           attn_dtype dt);

/*
 * Backward pass by recomputation.
 *
 * Flash Attention 2 post, section "Flash Attention 2", "Recomputation in
 * backward pass": S and P are rebuilt tile by tile from Q, K and the saved
 * LSE, P = exp(scale·Q Kᵀ - LSE). The softmax step is the Jacobian-vector
 * product of the softmax-backward note (shreyansh26.github.io), section
 * "Backpropagating Through Softmax": dS = P ∘ (dP - D) with dP = dO Vᵀ and the
 * row term D = rowsum(P ∘ dP), which equals rowsum(dO ∘ O) and is computed
 * that way by a preprocess kernel. Then dV = Pᵀ dO, dK = scale·dSᵀ Q and
 * dQ = scale·dS K. For dt = ATTN_BF16 with d = 128, dK and dV come from a
 * pass over key tiles and dQ from a second pass over query tiles that
 * recomputes S and dP, keeps dQ in tensor memory and writes it once in bf16
 * (each gradient has one writer; the dQ accumulator in the workspace is not
 * used). Otherwise dQ is accumulated across key tiles in float32 in the
 * workspace (the attention-residuals lab reduces multi-writer gradients
 * through float32 atomics) and converted at the end. With GQA, dK and dV of
 * a KV head sum over its query heads.
 *
 * Inputs: q, k, v, o (forward output), dO, lse (forward LSE), all in `dt`
 * except lse (float32). Outputs dq, dk, dv in `dt`, overwritten.
 * workspace: device scratch of at least attn_bwd_workspace_size_dt(..., dt)
 * bytes (attn_bwd_workspace_size() is always enough), 256-byte aligned; its
 * contents on entry do not matter.
 * dt = ATTN_BF16 with d in {64, 128}; ATTN_F32 with d in {64, 128}.
 */
ATTN_API attn_status attn_bwd(const void* q, const void* k, const void* v, const void* o,
                     const void* dO, const float* lse, void* dq, void* dk, void* dv,
                     int B, int Hq, int Hkv, int Nq, int Nk, int d, float scale, int causal,
                     attn_dtype dt, void* workspace, size_t ws_bytes, void* stream);

/*
 * attn_bwd under a general mask (see attn_mask; mask == NULL: no mask): the
 * same mask the forward used, so P is zero on every hidden (row, key) pair
 * and on rows that see no key (LSE = -inf). Any Nq, Nk > 0; with dt =
 * ATTN_BF16 and a mask with global keys or per-row key ranges, Nq is
 * limited to 65536 (d = 128) or 131072 (d = 64): ATTN_ERR_UNSUPPORTED
 * beyond (windows alone have no limit). Otherwise as attn_bwd, with the
 * same workspace.
 */
ATTN_API attn_status attn_bwd_masked(const void* q, const void* k, const void* v, const void* o,
                                     const void* dO, const float* lse, void* dq, void* dk,
                                     void* dv, int B, int Hq, int Hkv, int Nq, int Nk, int d,
                                     float scale, const attn_mask* mask, attn_dtype dt,
                                     void* workspace, size_t ws_bytes, void* stream);

/*
 * Bytes of device scratch attn_decode_splitkv needs: per (b, query head,
 * split) the partial triple (o [d], m, l) in float32, 256-byte aligned.
 */
ATTN_API size_t attn_decode_workspace_size(int B, int Hq, int d, int num_splits);

/*
 * Split-KV decode (query length 1) with an exact merge.
 *
 * ML notes (haolingpu.github.io), split-K kernel notes: the KV axis of each
 * request is cut into `num_splits` chunks processed by independent blocks;
 * each chunk leaves its maximum score m_s, un-normalised denominator
 * l_s = Σ exp(s - m_s) and un-normalised output o_s = Σ exp(s - m_s) v in the
 * workspace; a second kernel rescales every chunk onto the common maximum and
 * merges them exactly, in any order. Chunk s covers keys
 * [s*c, min((s+1)*c, L)), c = ceil(L / num_splits); an empty chunk carries
 * zero mass (attention-residuals lab, "Phase 2").
 *
 * q [B,Hq,d] bf16, k_cache/v_cache [B,Hkv,L,d] bf16; o [B,Hq,d] bf16 written;
 * lse [B,Hq] float32 written (may be NULL). d must be 128 or 64; Hq/Hkv <= 8.
 * workspace: at least attn_decode_workspace_size() bytes, 256-byte aligned.
 */
ATTN_API attn_status attn_decode_splitkv(const void* q, const void* k_cache, const void* v_cache,
                                void* o, float* lse, int B, int Hq, int Hkv, int L, int d,
                                float scale, int num_splits, void* workspace, size_t ws_bytes,
                                void* stream);

/*
 * Paged, variable-length split-KV decode.
 *
 * ML notes (haolingpu.github.io), KV-cache Q&A: the cache is allocated in
 * fixed-size blocks that a per-request block table maps, like pages through
 * a page table (PagedAttention); decode steps of different requests are
 * independent, each reading its own cache. Computes, for every request b
 * with n_b = seq_lens[b] keys, what attn_decode_splitkv computes on the
 * contiguous cache gathered from its pages: key t of request b, KV head g,
 * is row (t % page_size) of head g in page block_table[b*max_pages_per_seq +
 * t / page_size].
 *
 * q [B,Hq,d] bf16; k_pages/v_pages [num_pages, Hkv, page_size, d] bf16;
 * block_table [B, max_pages_per_seq] int32 and seq_lens [B] int32, DEVICE
 * memory (read by the kernel, so both may be written by earlier work on
 * `stream`); o [B,Hq,d] bf16 written; lse [B,Hq] float32 written (may be
 * NULL). Entries of block_table past ceil(n_b / page_size) are not read.
 * page_size >= 1 (a multiple of 32 reads each 32-key step with one copy per
 * tensor; smaller or other sizes with one per page touched); d 64 or 128;
 * Hq/Hkv <= 8.
 * A request with n_b = 0 gets O = 0, LSE = -inf. Chunks have one length for
 * all requests, c = ceil(max_pages_per_seq * page_size / num_splits)
 * rounded up to a multiple of 32 keys, then doubled while the grid keeps
 * at least 8 CTAs per resident CTA slot of the device (B * Hkv *
 * ceil(capacity / c) CTAs; every CTA pays the same start, so a large batch
 * runs fewer, longer chunks); request b uses its own number of splits,
 * ceil(n_b / c) <= num_splits, split s covering keys
 * [s*c, min((s+1)*c, n_b)), so every split carries about the same work
 * whatever the mix of lengths. num_splits is thus the most splits a request
 * uses, and the partials keep that stride.
 * Device-side checks: a length outside [0, max_pages_per_seq*page_size] or
 * a page index outside [0, num_pages) is never dereferenced; the request
 * (for a bad length) or the split holding the bad index gets no keys, and
 * attn_sync_status() reports ATTN_ERR_DEVICE_INDEX.
 * workspace: at least attn_decode_workspace_size(B, Hq, d, num_splits)
 * bytes, 256-byte aligned.
 */
ATTN_API attn_status attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                              const int* block_table, const int* seq_lens, void* o,
                              float* lse, int B, int Hq, int Hkv, int num_pages,
                              int page_size, int max_pages_per_seq, int d, float scale,
                              int num_splits, void* workspace, size_t ws_bytes,
                              void* stream);

/*
 * Sparse-index split-KV decode: T query tokens per request attend over a
 * scattered list of cache rows.
 *
 * ML notes (haolingpu.github.io), sparse-attention split-K notes: the list
 * of KV positions is chosen upstream (an indexer); the kernel gathers the
 * listed rows tile by tile into shared memory, splits the list across
 * blocks and merges the (o, m, l) partials exactly. Reading: one list per
 * request, shared by its T tokens and all heads; a row listed twice counts
 * twice.
 *
 * q [B, Hq, T, d] bf16; k_cache/v_cache [B, Hkv, L, d] bf16; indices
 * [B, max_idx] int32 and counts [B] int32 in DEVICE memory: request b
 * attends over cache rows indices[b*max_idx + e], e < counts[b]; o
 * [B, Hq, T, d] bf16 written; lse [B, Hq, T] float32 written (may be NULL).
 * A request with an empty list gets O = 0, LSE = -inf. The list is cut into
 * chunks of c = ceil(max_idx / num_splits) rounded up to 32 entries and at
 * least 128 (num_splits is the most splits a request uses).
 * Device-side checks: a count outside [0, max_idx] or a listed row outside
 * [0, L) is never dereferenced; the request (bad count) or the chunk
 * holding the bad row gets no keys and attn_sync_status() reports
 * ATTN_ERR_DEVICE_INDEX. d 64 or 128; Hq/Hkv in {1, 2, 4, 8}; any T.
 * workspace: attn_decode_workspace_size(B, Hq * T, d, num_splits) bytes,
 * 256-byte aligned.
 */
ATTN_API attn_status attn_decode_sparse(const void* q, const void* k_cache, const void* v_cache,
                                        const int* indices, const int* counts, void* o,
                                        float* lse, int B, int Hq, int Hkv, int T, int L,
                                        int max_idx, int d, float scale, int num_splits,
                                        void* workspace, size_t ws_bytes, void* stream);

/*
 * The exact (o, m, l) merge on its own (ML notes, split-K notes; the
 * attention-residuals lab, "Phase 2: merge the live partial exactly").
 *
 * o_part [rows, num_splits, d], m_part and l_part [rows, num_splits], all
 * float32, with o un-normalised (o_s = Σ exp(s - m_s) v). Writes
 * o [rows, d] in `out_dt` = Σ_s e^(m_s - m) o_s / Σ_s e^(m_s - m) l_s with
 * m = max_s m_s, and lse [rows] = m + ln(l) (lse may be NULL). A split with
 * m_s = -inf contributes nothing; a row with no mass gets O = 0, LSE = -inf.
 * d must be a multiple of 4 and at most 256.
 */
ATTN_API attn_status attn_merge_partials(const float* o_part, const float* m_part, const float* l_part,
                                void* o, float* lse, int rows, int num_splits, int d,
                                attn_dtype out_dt, void* stream);

/*
 * Split-KV decode without any allocation by the caller.
 *
 * The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory at the point where they decode — for
 * example a serving loop whose memory is partitioned up front and that must
 * not call cudaMalloc after start-up (cudaMalloc can synchronise the device
 * and its latency is unpredictable), or a plugin inside a host program that
 * owns all device memory and exposes no allocator. It computes exactly what
 * attn_decode_splitkv computes, with the same arguments minus the workspace.
 *
 * Scratch: the per-split partials live in one fixed array inside the library
 * of ATTN_DECODE_NOALLOC_SCRATCH_BYTES bytes, which every GPU that loads the
 * library holds until the process exits. A call whose partials need more
 * than that (attn_decode_workspace_size(B, Hq, d, num_splits) larger than
 * ATTN_DECODE_NOALLOC_SCRATCH_BYTES) is rejected with ATTN_ERR_WORKSPACE and
 * nothing is launched.
 *
 * Set-up: the first call on a device looks up that device's address of the
 * array (cudaGetSymbolAddress, with the device current) and caches it; make
 * that first call before any stream capture on the device. The cached
 * address belongs to the device's current context: after cudaDeviceReset()
 * on that device it is stale, and this entry point must not be called again
 * in that process.
 *
 * Sharing: all calls on a device use the same array. Nothing in it needs to
 * start at zero (each call writes every partial it reads), but calls whose
 * kernels overlap on the GPU (different streams without ordering between
 * them) race on the array and give wrong results; order them on one stream.
 */
#define ATTN_DECODE_NOALLOC_SCRATCH_BYTES (24u * 1024u * 1024u)

ATTN_API attn_status attn_decode_splitkv_noalloc(const void* q, const void* k_cache,
                                                 const void* v_cache, void* o, float* lse, int B,
                                                 int Hq, int Hkv, int L, int d, float scale,
                                                 int num_splits, void* stream);

/*
 * Self-test of the bounded device wait (no counterpart on the pages).
 *
 * Launches one warp on `stream` that waits, with the same bounded wait the
 * kernels use, on a barrier nothing ever arrives on, for `limit_us`
 * microseconds (1 .. 1,000,000); then it records a timeout in the device
 * error word and exits. Nothing asynchronous is in flight while it waits, so
 * the context stays usable: a following attn_sync_status() returns
 * ATTN_ERR_DEVICE_TIMEOUT (and clears the word), and later calls run
 * normally. It shows that a wait that runs out reaches the caller as a
 * status instead of a hang. Returns ATTN_ERR_INVALID_ARG for a limit out of
 * range, ATTN_ERR_CUDA if the launch fails, else ATTN_OK.
 */
ATTN_API attn_status attn_selftest_bounded_wait(unsigned int limit_us, void* stream);

/* Static, human-readable name of a status code. */
ATTN_API const char* attn_status_string(attn_status s);

/*
 * Synchronise `stream`, then report (and clear) the library's device error
 * word: ATTN_ERR_DEVICE_TIMEOUT if a bounded device wait ran out since the
 * last check, else ATTN_ERR_DEVICE_INDEX if a paged decode met an
 * out-of-range length or page index; ATTN_ERR_CUDA if the stream reports a
 * CUDA error; else ATTN_OK.
 */
ATTN_API attn_status attn_sync_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* ONLINE_SOFTMAX_TILED_GB300_ATTN_H */

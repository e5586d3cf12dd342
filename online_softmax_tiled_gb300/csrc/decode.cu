// Split-KV decode and the exact (o, m, l) merge.
//
// ML notes (haolingpu.github.io), split-K kernel notes: the KV axis of one
// request is cut into S chunks so that more blocks run at once; each chunk
// leaves its maximum score m_s, un-normalised denominator
// l_s = Σ exp(s - m_s) and un-normalised output o_s = Σ exp(s - m_s) v in
// global scratch, and a second kernel rescales every chunk by exp(m_s - m)
// onto the common maximum m and merges them exactly, in any order. A chunk
// with no keys carries zero mass (attention-residuals kernel lab,
// manishklach.github.io, "Phase 2"): it is simply left out of the merge.
//
// Split kernel. Decode is bound by reading the KV cache once (about 4 flops
// per byte), so it runs on the FMA pipes, not the tensor cores. One CTA owns
// (request b, KV head g, chunk s) and the G = Hq/Hkv query heads that share
// that KV head (up to four; with eight, two CTAs of four read the same
// keys), so every K/V byte is read from HBM once per CTA group. K and V
// rows of the chunk stream through a 4-stage shared-memory ring filled by
// bulk asynchronous copies (each stage is a contiguous run of rows, so one
// copy per tensor per stage). Eight consecutive lanes own one key: lane
// `sub` holds dims {64v + 8sub .. 64v + 8sub + 7}, so a warp's 16-byte
// shared loads cover whole 128-byte rows without bank conflicts. Each 8-lane
// group runs its own online softmax over its keys; the 16 groups of the CTA
// are merged with the same exact rule at the end (the four groups of a warp
// by shuffles, then the four warps through shared memory).
//
// Paged, variable-length decode (ML notes, KV-cache Q&A: the cache lives in
// fixed-size blocks reached through a per-request block table, as pages
// through a page table): the same kernel with request b's length read from
// seq_lens[b] and key t read from page block_table[b][t / page_size].
// Chunks have one length c for all requests (the table's capacity over the
// split count, rounded up to 32 keys, doubled while the grid keeps eight
// CTAs per resident slot: decode_chunk), so request b uses its own number of
// splits, ceil(n_b / c), every non-empty chunk carries about the same work
// and the CTAs of chunks past a request's end return at once (the merge
// reads only a request's own chunks). A CTA fetches its request's length and
// all block-table entries of its chunk in one round of independent loads,
// keeps the entries in shared memory and range-checks every one before any
// page is read. Each 32-key stage is filled by one bulk copy per page it
// touches (rows are 128 or 256 bytes, so every row start is 16-byte
// aligned); chunks start on multiples of 32 keys, so with 32 | page_size
// that is one copy per tensor, as for a contiguous cache.
//
// Sparse-index decode (ML notes, sparse-attention split-K notes: the kernel
// gathers the listed KV rows into shared memory tile by tile): the same
// kernel over one list of cache rows per request, each 32-row stage filled
// by tile::gather4 tensor copies of four listed rows each (a 2-D view of the
// cache, one row per box), issued by 16 lanes of warp 0 at once.

#include <mutex>

#include "common.cuh"
#include "launchers.h"
#include "tma_host.h"

namespace attn {

ATTN_DEFINE_ERROR_WORD(take_error_decode)

namespace {

constexpr int kThreads = 128;     // 4 warps, 16 key groups of 8 lanes
constexpr int kStageKeys = 32;    // keys per pipeline stage
constexpr int kStages = 4;
constexpr int kChunkPagesCached = 256;   // block-table entries of a chunk kept in shared memory
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// End of a chunk, shared by both split kernels so that they round alike.
// Each 8-lane group holds (m, l, o) relative to its own reference. The four
// groups of a warp (lanes 8 apart hold the same dimensions) are first
// rescaled onto their common max and summed with shuffles; lanes 0..7 then
// write the warp's (o, m, l) to comb[warp][h][0 .. D + 1]. NP = D / 16
// dimension pairs per lane, NV = D / 64 16-byte pieces.
template <int D, int G>
ATTN_DEVINL void warp_combine_write(f2 (&acc)[G][D / 16], float (&m_ref)[G], float (&l_run)[G],
                                    float* comb, int warp, int lane) {
  constexpr int NP = D / 16, NV = D / 64;
  const int grp = lane >> 3, sub = lane & 7;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float mw = fmaxf(m_ref[h], __shfl_xor_sync(0xffffffffu, m_ref[h], 8));
    mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, 16));
    const float wgt = (m_ref[h] == -INFINITY) ? 0.f : fast_exp2(m_ref[h] - mw);
    float l = l_run[h] * wgt;
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    l_run[h] = l;
    m_ref[h] = mw;
    const f2 w2{wgt, wgt};
#pragma unroll
    for (int e = 0; e < NP; ++e) {
      f2 a = mul2(acc[h][e], w2);
      a.x += __shfl_xor_sync(0xffffffffu, a.x, 8);
      a.y += __shfl_xor_sync(0xffffffffu, a.y, 8);
      a.x += __shfl_xor_sync(0xffffffffu, a.x, 16);
      a.y += __shfl_xor_sync(0xffffffffu, a.y, 16);
      acc[h][e] = a;
    }
  }
  if (grp == 0) {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float* row = comb + (warp * G + h) * (D + 2);
      if (sub == 0) {
        row[D] = m_ref[h];
        row[D + 1] = l_run[h];
      }
#pragma unroll
      for (int vv = 0; vv < NV; ++vv)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          row[64 * vv + 8 * sub + 2 * e] = acc[h][vv * 4 + e].x;
          row[64 * vv + 8 * sub + 2 * e + 1] = acc[h][vv * 4 + e].y;
        }
    }
  }
}

// The four warps' (o, m, l) of each query row onto their common max: the
// chunk's partial o (un-normalised), m (natural units) and l, written for
// rows row0 .. row0 + G - 1 at split s. Threads tid, tid + nthr, ...
template <int D, int G>
ATTN_DEVINL void final_combine(const float* comb, int tid, int nthr, size_t row0, int S, int s,
                               float* o_part, float* m_part, float* l_part) {
  for (int idx = tid; idx < G * D; idx += nthr) {
    const int h = idx / D, c = idx % D;
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) mx = fmaxf(mx, comb[(w * G + h) * (D + 2) + D]);
    float o = 0.f, l = 0.f;
    if (mx != -INFINITY) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float* row = comb + (w * G + h) * (D + 2);
        const float wt = (row[D] == -INFINITY) ? 0.f : fast_exp2(row[D] - mx);
        o = fmaf(wt, row[c], o);
        l = fmaf(wt, row[D + 1], l);
      }
    }
    const size_t qrow = row0 + h;
    o_part[(qrow * S + s) * D + c] = o;
    if (c == 0) {
      m_part[qrow * S + s] = (mx == -INFINITY) ? -INFINITY : mx * kLn2;   // natural units
      l_part[qrow * S + s] = l;
    }
  }
}

template <int D, int G>
constexpr size_t decode_smem_bytes() {
  // K and V ring; the final cross-warp combine (4 warps × G heads of
  // (o[D], m, l) in float32) reuses it.
  constexpr size_t ring = size_t(2) * kStages * kStageKeys * D * 2;
  constexpr size_t merge = size_t(4) * G * (D + 2) * 4;
  return ring > merge ? ring : merge;
}

// Gathered keys. Paged cache: pages [num_pages][Hkv][page_size][D];
// block_table [B][max_pages]; seq_lens [B]. Sparse index list (rows = 1):
// the cache stays [B][Hkv][L][D], block_table holds each request's listed
// rows [B][max_pages], seq_lens the list lengths, page_size = 1 and
// num_pages = L (every listed row is its own one-row page).
struct PagedKV {
  const int* block_table;
  const int* seq_lens;
  int num_pages, page_size, max_pages;
  int rows;   // 1: sparse index list into the per-request cache
};

// Where a chunk's keys come from: a contiguous cache, pages of a paged
// cache (bulk copies by one thread), or a list of rows (tile::gather4 copies
// of four rows each, issued by the lanes of warp 0).
enum KeySource : int { kContiguous = 0, kPages = 1, kListedRows = 2 };

// Four rows of a 2-D tensor map (box: one row of `cols` elements), given by
// their row coordinates, into consecutive rows at smem_dst (tile::gather4).
ATTN_DEVINL void tma_gather4(void* smem_dst, const CUtensorMap* map, int r0, int r1, int r2,
                             int r3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
      ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(r0), "r"(r1),
        "r"(r2), "r"(r3), "r"(smem_u32(bar))
      : "memory");
}

template <int D, int G, int kSource>
__global__ void __launch_bounds__(kThreads, 3)
decode_split_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                    const __nv_bfloat16* __restrict__ v, float* __restrict__ o_part,
                    float* __restrict__ m_part, float* __restrict__ l_part, int Hq, int Hkv,
                    int L, int S, int chunk, float scale, PagedKV pg, int rgroups,
                    const __grid_constant__ CUtensorMap map_k_rows,
                    const __grid_constant__ CUtensorMap map_v_rows) {
  constexpr bool kPaged = kSource != kContiguous;   // keys reached through a table
  constexpr int NV = D / 64;                       // 16-byte pieces per lane per row
  constexpr int kRowBytes = D * 2;
  constexpr int kStageBytes = kStageKeys * kRowBytes;
  // the merge kernel may launch (and wait for this grid) as the last wave runs
  pdl_launch_dependents();
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* sK = smem;
  uint8_t* sV = smem + kStages * kStageBytes;
  __shared__ uint64_t full_bar[kStages];
  __shared__ int abort_flag;
  __shared__ int chunk_pages[kPaged ? kChunkPagesCached : 1];
  constexpr int kPreStages = kSource == kPages ? 64 : 1;
  __shared__ size_t stage_src[kPreStages][2];   // element offsets of a stage's one or two segments
  __shared__ int stage_rows[kPreStages][2];

  // blockIdx.y = (KV head, group of G query rows); query row r of this CTA
  // is row b·Hq + blockIdx.y·G + r (Hq counts query rows: heads x tokens)
  const int s = blockIdx.x, gy = blockIdx.y, b = blockIdx.z;
  const int g = gy / rgroups;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grp = lane >> 3, sub = lane & 7;

  // one arrival per stage barrier (the expected-bytes arrival of the
  // thread that issues the stage's copies)
  if (tid == 0) {
    abort_flag = 0;
    for (int i = 0; i < kStages; ++i) mbar_init(&full_bar[i], 1);
    fence_barrier_init();
  }
  // Launched as a programmatic dependent: every global access of this grid
  // (q, the KV cache, the partials a previous merge may still be reading)
  // comes after the preceding grid has completed.
  pdl_wait_primary();

  // This CTA's keys [key_begin, key_end): chunk s of its request.
  const int max_len = kPaged ? pg.max_pages * pg.page_size : L;
  const int* table_row = kPaged ? pg.block_table + size_t(b) * pg.max_pages : nullptr;
  int Lb = L;
  bool bad = false;
  int p_first = 0;
  if (kPaged) {
    // The length and every table entry the chunk can touch, as independent
    // loads; entries are checked once the length says which ones are used.
    Lb = pg.seq_lens[b];
    const int nominal = s * chunk;
    p_first = nominal / pg.page_size;
    const int p_cap = min(pg.max_pages, (min(max_len, nominal + chunk) + pg.page_size - 1) /
                                            pg.page_size);
    int ent[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int p = p_first + tid + i * kThreads;
      ent[i] = p < p_cap ? table_row[p] : 0;
    }
    if (Lb < 0 || Lb > max_len) {
      if (s == 0 && g == 0 && tid == 0) attn_flag_error(kErrBadIndex);
      Lb = 0;
    }
    const int p_used = (min(Lb, nominal + chunk) + pg.page_size - 1) / pg.page_size;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int p = p_first + tid + i * kThreads;
      if (p < p_used) bad |= ent[i] < 0 || ent[i] >= pg.num_pages;
      if (tid + i * kThreads < kChunkPagesCached) chunk_pages[tid + i * kThreads] = ent[i];
    }
    // chunks of more than 4 x kThreads pages (pages far smaller than the
    // chunk): the rest checked straight from the table
    for (int p = p_first + 4 * kThreads + tid; p < p_used; p += kThreads) {
      const int e = table_row[p];
      bad |= e < 0 || e >= pg.num_pages;
    }
  }
  const int key_begin = min(Lb, s * chunk);
  const int key_end = min(Lb, key_begin + chunk);
  // (also orders the barrier initialisation and the cached entries before use)
  bad = __syncthreads_or(bad);
  if (bad) {
    // a page index out of range: the chunk reads nothing and leaves no mass
    if (tid == 0) attn_flag_error(kErrBadIndex);
    if (tid < G) {
      const size_t row = size_t(b) * Hq + gy * G + tid;
      m_part[row * S + s] = -INFINITY;
      l_part[row * S + s] = 0.f;
    }
    return;
  }
  const int nkeys = key_end - key_begin;
  // past the request's end: the merge never reads this chunk
  if (nkeys <= 0) return;
  const int nstages = (nkeys + kStageKeys - 1) / kStageKeys;

  // Element offset of key t of (b, g) in the K and V arrays.
  constexpr bool sparse = kSource == kListedRows;
  const size_t head_off = kPaged && !sparse ? size_t(g) * pg.page_size * D
                                            : (size_t(b) * Hkv + g) * size_t(L) * D;
  const size_t page_elems = sparse ? size_t(D) : size_t(Hkv) * pg.page_size * D;
  auto page_of = [&](int t) {
    const int i = t / pg.page_size - p_first;
    return i < kChunkPagesCached ? chunk_pages[i] : table_row[t / pg.page_size];
  };
  // Paged bulk copies: with pages of a multiple of 16 keys a 32-key stage
  // touches at most two pages, and the source offsets of the first
  // kPreStages stages are worked out here by all threads at once, so the
  // copying thread spends a few instructions per stage (the per-stage
  // barrier waits for it) instead of dividing by the page size.
  const bool pre = kSource == kPages && pg.page_size % 16 == 0;
  if (pre) {
    for (int st = tid; st < min(nstages, kPreStages); st += kThreads) {
      const int t0 = key_begin + st * kStageKeys;
      const int rows = min(kStageKeys, nkeys - st * kStageKeys);
      const int in_page = t0 % pg.page_size;
      const int seg = min(rows, pg.page_size - in_page);
      stage_src[st][0] = head_off + size_t(page_of(t0)) * page_elems + size_t(in_page) * D;
      stage_src[st][1] = seg < rows ? head_off + size_t(page_of(t0 + seg)) * page_elems : 0;
      stage_rows[st][0] = seg;
      stage_rows[st][1] = rows - seg;
    }
    __syncthreads();
  }
  auto issue = [&](int st) {
    const int buf = st % kStages;
    if (kSource == kListedRows) {
      // listed rows (every lane of warp 0): four rows per gather4 copy, lane
      // o < 8 copies K rows 4o .. 4o + 3 of the stage and lane 8 + o the same
      // V rows; a last copy of fewer rows repeats the stage's last row into
      // slots nobody reads
      const int e0 = st * kStageKeys;
      const int rows = min(kStageKeys, nkeys - e0);
      const int nops = (rows + 3) / 4;
      if (lane == 0) mbar_arrive_expect_tx(&full_bar[buf], 2 * uint32_t(nops) * 4 * kRowBytes);
      __syncwarp();
      const int o = lane & 7;
      if (lane < 16 && o < nops) {
        const int rbase = (b * Hkv + g) * L;   // row of key 0 of (request, KV head)
        int r[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          r[i] = rbase + page_of(key_begin + min(e0 + 4 * o + i, nkeys - 1));
        const uint32_t dst = buf * kStageBytes + 4 * o * kRowBytes;
        if (lane < 8)
          tma_gather4(sK + dst, &map_k_rows, r[0], r[1], r[2], r[3], &full_bar[buf]);
        else
          tma_gather4(sV + dst, &map_v_rows, r[0], r[1], r[2], r[3], &full_bar[buf]);
      }
    } else if (kPaged && pre && st < kPreStages) {
      // (every lane of warp 0) one copy per lane: lane 2·seg + tensor copies
      // segment seg of K (tensor 0) or V (tensor 1)
      const int r0 = stage_rows[st][0], r1 = stage_rows[st][1];
      if (lane == 0) mbar_arrive_expect_tx(&full_bar[buf], 2 * uint32_t(r0 + r1) * kRowBytes);
      __syncwarp();
      if (lane < (r1 > 0 ? 4 : 2)) {
        const int seg = lane >> 1;
        const size_t o = stage_src[st][seg];
        const uint32_t dst = buf * kStageBytes + (seg ? r0 : 0) * kRowBytes;
        const uint32_t bytes = uint32_t(seg ? r1 : r0) * kRowBytes;
        bulk_g2s(((lane & 1) ? sV : sK) + dst, ((lane & 1) ? v : k) + o, bytes, &full_bar[buf]);
      }
    } else if (kPaged) {
      // other page sizes, later stages: lane 0 alone, one copy per page the
      // stage touches
      if (lane == 0) {
        const int t0 = key_begin + st * kStageKeys;
        const int rows = min(kStageKeys, nkeys - st * kStageKeys);
        mbar_arrive_expect_tx(&full_bar[buf], 2 * uint32_t(rows) * kRowBytes);
        for (int t = t0, r = 0; r < rows;) {
          const int in_page = t % pg.page_size;
          const int seg = min(rows - r, pg.page_size - in_page);
          const size_t off = head_off + size_t(page_of(t)) * page_elems + size_t(in_page) * D;
          const uint32_t dst = buf * kStageBytes + r * kRowBytes;
          bulk_g2s(sK + dst, k + off, uint32_t(seg) * kRowBytes, &full_bar[buf]);
          bulk_g2s(sV + dst, v + off, uint32_t(seg) * kRowBytes, &full_bar[buf]);
          t += seg;
          r += seg;
        }
      }
    } else {
      // contiguous cache: thread 0 alone (the only issuer)
      const int t0 = key_begin + st * kStageKeys;
      const int rows = min(kStageKeys, nkeys - st * kStageKeys);
      mbar_arrive_expect_tx(&full_bar[buf], 2 * uint32_t(rows) * kRowBytes);
      const size_t off = head_off + size_t(t0) * D;
      bulk_g2s(sK + buf * kStageBytes, k + off, uint32_t(rows) * kRowBytes, &full_bar[buf]);
      bulk_g2s(sV + buf * kStageBytes, v + off, uint32_t(rows) * kRowBytes, &full_bar[buf]);
    }
  };
  int issued = 0;  // meaningful in the issuing thread (warp) only
  // Thread 0 issues the copies of a contiguous cache; for pages and listed
  // rows the lanes of warp 0 share them.
  const bool issuer = kSource == kContiguous ? tid == 0 : warp == 0;
  if (issuer)
    for (; issued < min(kStages, nstages); ++issued) issue(issued);

  // Query slice of this lane for all G heads, pre-scaled into log2 units,
  // as pairs of consecutive dimensions (packed f32x2 arithmetic).
  constexpr int NP = NV * 4;                       // dimension pairs per lane
  f2 qf[G][NP];
  const float qs = scale * kLog2e;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const __nv_bfloat16* qh = q + (size_t(b) * Hq + gy * G + h) * D;
#pragma unroll
    for (int vv = 0; vv < NV; ++vv) {
      const uint4 w = *reinterpret_cast<const uint4*>(qh + 64 * vv + 8 * sub);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) qf[h][vv * 4 + e] = f2{bf16lo(ws[e]) * qs, bf16hi(ws[e]) * qs};
    }
  }

  // Per group: reference max (log2 units; moved lazily), denominator, and
  // un-normalised output, all relative to the reference.
  f2 acc[G][NP];
  float m_ref[G], l_run[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m_ref[h] = -INFINITY;
    l_run[h] = 0.f;
#pragma unroll
    for (int e = 0; e < NP; ++e) acc[h][e] = f2{0.f, 0.f};
  }

  bool ok = true;
  for (int st = 0; st < nstages; ++st) {
    const int buf = st % kStages;
    const bool fail = !mbar_wait_bounded(&full_bar[buf], (st / kStages) & 1, &abort_flag);
    if (fail) abort_flag = 1;
    // One barrier per stage: all threads agree on failure, and the buffer of
    // stage st-1 is free once every thread has arrived here.
    if (__syncthreads_or(fail)) {
      // Let copies already issued land before shared memory goes away.
      if (tid == 0) {
        attn_flag_error(kErrTimeout);
        for (int t = st; t < issued; ++t)
          mbar_wait_bounded(&full_bar[t % kStages], (t / kStages) & 1, nullptr);
      }
      ok = false;
      break;
    }
    if (issuer && issued < nstages && st >= 1) issue(issued++);
    const int rows = min(kStageKeys, nkeys - st * kStageKeys);
    const uint8_t* kb = sK + buf * kStageBytes;
    const uint8_t* vb = sV + buf * kStageBytes;

    // This group's two keys of the stage: warp*8 + grp and warp*8 + grp + 4.
    float sc[2][G];
    int krow[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int kk = warp * 8 + grp + 4 * r;
      const bool valid = kk < rows;
      const int kr = valid ? kk : 0;
      krow[r] = kr;
      f2 part[G];
#pragma unroll
      for (int h = 0; h < G; ++h) part[h] = f2{0.f, 0.f};
#pragma unroll
      for (int vv = 0; vv < NV; ++vv) {
        const uint4 w = *reinterpret_cast<const uint4*>(kb + kr * kRowBytes + (64 * vv + 8 * sub) * 2);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const f2 kv{bf16lo(ws[e]), bf16hi(ws[e])};
#pragma unroll
          for (int h = 0; h < G; ++h) part[h] = fma2(qf[h][vv * 4 + e], kv, part[h]);
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float xsum = part[h].x + part[h].y;
        xsum += __shfl_xor_sync(0xffffffffu, xsum, 1);
        xsum += __shfl_xor_sync(0xffffffffu, xsum, 2);
        xsum += __shfl_xor_sync(0xffffffffu, xsum, 4);
        sc[r][h] = valid ? xsum : -INFINITY;
      }
    }

    // Online update of (m, l, o) for this group's two keys. The reference max
    // moves only when a score exceeds it by more than 2^8 (exact either way,
    // since l and o share the reference).
    bool need[G];
    bool any_need = false;
#pragma unroll
    for (int h = 0; h < G; ++h) {
      need[h] = max3(m_ref[h], sc[0][h], sc[1][h]) > m_ref[h] + 8.f;   // true from -inf too
      any_need |= need[h];
    }
    if (__any_sync(0xffffffffu, any_need)) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float m_new = need[h] ? max3(m_ref[h], sc[0][h], sc[1][h]) : m_ref[h];
        const float alpha = need[h] ? fast_exp2(m_ref[h] - m_new) : 1.f;   // 0 from -inf
        m_ref[h] = m_new;
        l_run[h] *= alpha;
        const f2 a2{alpha, alpha};
#pragma unroll
        for (int e = 0; e < NP; ++e) acc[h][e] = mul2(acc[h][e], a2);
      }
    }
    f2 p2[2][G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float nm = (m_ref[h] == -INFINITY) ? 0.f : -m_ref[h];
      const float p0 = fast_exp2(sc[0][h] + nm);
      const float p1 = fast_exp2(sc[1][h] + nm);
      l_run[h] += p0 + p1;
      p2[0][h] = f2{p0, p0};
      p2[1][h] = f2{p1, p1};
    }
#pragma unroll
    for (int r = 0; r < 2; ++r)
#pragma unroll
      for (int vv = 0; vv < NV; ++vv) {
        const uint4 x = *reinterpret_cast<const uint4*>(vb + krow[r] * kRowBytes + (64 * vv + 8 * sub) * 2);
        const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const f2 v2{bf16lo(xs[e]), bf16hi(xs[e])};
#pragma unroll
          for (int h = 0; h < G; ++h) acc[h][vv * 4 + e] = fma2(v2, p2[r][h], acc[h][vv * 4 + e]);
        }
      }
  }
  if (!ok) return;

  // Cross-group merge: exact rescale onto the common max, first the four
  // groups of each warp, then the four warps.
  __syncthreads();   // every warp is done with the ring, which the combine reuses
  float* comb = reinterpret_cast<float*>(smem);
  warp_combine_write<D, G>(acc, m_ref, l_run, comb, warp, lane);
  __syncthreads();
  final_combine<D, G>(comb, tid, kThreads, size_t(b) * Hq + gy * G, S, s, o_part, m_part, l_part);
}

// One warp per output row; lane owns float4 column groups lane, lane+32, ...
// A row merges its first nv partials: all S for a plain merge, else the
// chunks that hold keys of its request (ceil(n / chunk), n its length; a
// length outside [0, max_len] counts as 0). The partials are fetched eight
// at a time with independent loads (their weights exp(m_t - m) computed
// once per lane first), so a row costs about nv/8 memory round trips.
template <typename TOut>
__global__ void __launch_bounds__(256)
merge_kernel(const float* __restrict__ o_part, const float* __restrict__ m_part,
             const float* __restrict__ l_part, TOut* __restrict__ o, float* __restrict__ lse,
             int rows, int S, int d, const int* __restrict__ seq_lens, int Hq, int len,
             int max_len, int chunk) {
  constexpr int kBatch = 8;
  // Launched as a programmatic dependent: the partials are read only after
  // the preceding (split) grid has completed. Whatever follows may launch
  // early and wait for this grid the same way.
  pdl_wait_primary();
  pdl_launch_dependents();
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  int nv = S;
  if (chunk > 0) {
    int n = seq_lens != nullptr ? seq_lens[row / Hq] : len;
    if (n < 0 || n > max_len) n = 0;
    nv = min(S, (n + chunk - 1) / chunk);
  }
  const float* mr = m_part + size_t(row) * S;
  const float* lr = l_part + size_t(row) * S;
  float mx = -INFINITY;
  for (int t = lane; t < nv; t += 32) mx = fmaxf(mx, mr[t]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  float l = 0.f;
  if (mx != -INFINITY)
    for (int t = lane; t < nv; t += 32) {
      const float mt = mr[t];
      if (mt != -INFINITY) l = fmaf(expf(mt - mx), lr[t], l);
    }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
  const bool empty = !(l > 0.f);
  const float inv = empty ? 0.f : 1.f / l;
  const float4* prow = reinterpret_cast<const float4*>(o_part + size_t(row) * S * d);
  const int d4 = d / 4;
  for (int c4 = lane; c4 < d4; c4 += 32) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!empty)
      for (int t0 = 0; t0 < nv; t0 += kBatch) {
        float4 x[kBatch];
        float w[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int t = t0 + u;
          const float mt = t < nv ? mr[t] : -INFINITY;
          w[u] = mt == -INFINITY ? 0.f : expf(mt - mx);
          x[u] = w[u] != 0.f ? prow[size_t(t) * d4 + c4] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          acc.x = fmaf(w[u], x[u].x, acc.x);
          acc.y = fmaf(w[u], x[u].y, acc.y);
          acc.z = fmaf(w[u], x[u].z, acc.z);
          acc.w = fmaf(w[u], x[u].w, acc.w);
        }
      }
    TOut* orow = o + size_t(row) * d + 4 * c4;
    orow[0] = from_f32<TOut>(acc.x * inv);
    orow[1] = from_f32<TOut>(acc.y * inv);
    orow[2] = from_f32<TOut>(acc.z * inv);
    orow[3] = from_f32<TOut>(acc.w * inv);
  }
  if (lse != nullptr && lane == 0) lse[row] = empty ? -INFINITY : mx + logf(l);
}

template <int D, int G, int kSource>
cudaError_t launch_split_t(const DecodeArgs& a, int rgroups) {
  const size_t smem = decode_smem_bytes<D, G>();
  cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<D, G, kSource>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(decode_grid_splits(a), a.Hkv * rgroups, a.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const PagedKV pg{a.block_table, a.seq_lens, a.num_pages, a.page_size, a.max_pages,
                   a.sparse ? 1 : 0};
  // listed rows: the caches as [B·Hkv·L rows][d] for row gathers
  CUtensorMap mk{}, mv{};
  if (kSource == kListedRows) {
    const uint64_t rows = uint64_t(a.B) * a.Hkv * a.L;
    if (!make_map_bf16_rows(&mk, a.k, D, rows) || !make_map_bf16_rows(&mv, a.v, D, rows))
      return cudaErrorInvalidValue;
  }
  return cudaLaunchKernelEx(&cfg, decode_split_kernel<D, G, kSource>,
                            static_cast<const __nv_bfloat16*>(a.q),
                            static_cast<const __nv_bfloat16*>(a.k),
                            static_cast<const __nv_bfloat16*>(a.v), a.o_part, a.m_part, a.l_part,
                            a.Hq * a.T, a.Hkv, a.L, a.num_splits, decode_chunk(a), a.scale, pg,
                            rgroups, mk, mv);
}

// Query rows per KV head: (Hq / Hkv) x T. One CTA takes G of them, at most
// 4, and the rest go to further CTAs over the same keys. Eight rows per CTA
// need 200-255 registers a thread (spilling at d = 128) and leave one or two
// CTAs per SM: two CTAs of four rows each read the keys twice and still run
// 1.6x (d = 128) and 1.1x (d = 64) faster than one CTA of eight.
template <int D, int kSource>
cudaError_t launch_split_d(const DecodeArgs& a) {
  const int rows = (a.Hq / a.Hkv) * a.T;
  int G = 1;
  while (G * 2 <= 4 && rows % (G * 2) == 0) G *= 2;
  const int rgroups = rows / G;
  switch (G) {
    case 1: return launch_split_t<D, 1, kSource>(a, rgroups);
    case 2: return launch_split_t<D, 2, kSource>(a, rgroups);
    case 4: return launch_split_t<D, 4, kSource>(a, rgroups);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_decode_split(const DecodeArgs& a) {
  if (a.block_table != nullptr && a.sparse)
    return a.d == 64 ? launch_split_d<64, kListedRows>(a) : launch_split_d<128, kListedRows>(a);
  if (a.block_table != nullptr)
    return a.d == 64 ? launch_split_d<64, kPages>(a) : launch_split_d<128, kPages>(a);
  return a.d == 64 ? launch_split_d<64, kContiguous>(a) : launch_split_d<128, kContiguous>(a);
}

cudaError_t launch_merge(const MergeArgs& a) {
  // Programmatic dependent launch: the merge's launch overlaps the tail of
  // the kernel before it; the kernel waits for that grid before reading.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((a.rows + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.out_dt == ATTN_F32)
    return cudaLaunchKernelEx(&cfg, merge_kernel<float>, a.o_part, a.m_part, a.l_part,
                              static_cast<float*>(a.o), a.lse, a.rows, a.num_splits, a.d,
                              a.seq_lens, a.Hq, a.len, a.max_len, a.chunk);
  return cudaLaunchKernelEx(&cfg, merge_kernel<__nv_bfloat16>, a.o_part, a.m_part, a.l_part,
                            static_cast<__nv_bfloat16*>(a.o), a.lse, a.rows, a.num_splits, a.d,
                            a.seq_lens, a.Hq, a.len, a.max_len, a.chunk);
}

}  // namespace attn

// ----------------------------------------------------------------------------
// attn_decode_splitkv_noalloc: the same decode, with the split partials kept
// in a fixed array inside the library instead of a caller workspace, for
// callers that cannot allocate device memory when they decode.
// ----------------------------------------------------------------------------
namespace attn {
namespace {

constexpr size_t kNoAllocScratchBytes = ATTN_DECODE_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_decode_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};  // device address of the array, per device

}  // namespace

extern "C" ATTN_API attn_status attn_decode_splitkv_noalloc(const void* q, const void* k_cache,
                                                            const void* v_cache, void* o,
                                                            float* lse, int B, int Hq, int Hkv,
                                                            int L, int d, float scale,
                                                            int num_splits, void* stream) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    // Once per device, with that device current: the host-side name of the
    // array is not a device address, so ask the runtime for this device's.
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_decode_noalloc_scratch) != cudaSuccess || p == nullptr)
        return ATTN_ERR_CUDA;
      g_noalloc_addr[dev] = p;
    }
    scratch = g_noalloc_addr[dev];
  }
  // The workspace path validates every argument, rejects a call whose
  // partials exceed the array (ATTN_ERR_WORKSPACE) and launches nothing then.
  return attn_decode_splitkv(q, k_cache, v_cache, o, lse, B, Hq, Hkv, L, d, scale, num_splits,
                             scratch, kNoAllocScratchBytes, stream);
}

}  // namespace attn

// ----------------------------------------------------------------------------
// attn_selftest_bounded_wait: one warp waits, through the bounded wait that
// every kernel of the library uses, on an mbarrier that nothing will ever
// arrive on. When the limit runs out it records the timeout in the error word
// and returns, as a kernel does when a real wait runs out. Nothing
// asynchronous (bulk copy, tensor-core op) is in flight at any time.
// ----------------------------------------------------------------------------
namespace attn {
namespace {

__global__ void __launch_bounds__(32) bounded_wait_selftest_kernel(uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0 && !mbar_wait_bounded(&bar, 0, nullptr, limit_ns))
    attn_flag_error(kErrTimeout);
}

}  // namespace

extern "C" ATTN_API attn_status attn_selftest_bounded_wait(unsigned int limit_us, void* stream) {
  if (limit_us == 0 || limit_us > 1000000u) return ATTN_ERR_INVALID_ARG;
  bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      uint64_t(limit_us) * 1000ull);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attn

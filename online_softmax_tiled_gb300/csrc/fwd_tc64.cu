// bf16 tiled attention forward at head dimension 64 on the sm_103a tensor
// cores (tcgen05 + TMEM + TMA): a persistent kernel.
//
// Algorithm: the inner loop of the "Flash Attention 2" post
// (ahmadsaeedzaidi.github.io feed), section "Flash Attention 2": for a query
// tile Q_i and each key/value tile K_j, V_j: S_ij = scale·Q_i K_jᵀ, running
// row max m, P̃ = exp(S - m), running denominator l, Õ rescaled by
// exp(m_old - m_new) and accumulated with P̃ V_j; after the last tile
// O_i = Õ_i / l_i and LSE = m + ln l. Masks per the post's section "Causal
// masking", option A (mask.cuh). The two halves of a query tile's keys meet
// by the exact partition merge of the attention-residuals kernel lab
// (manishklach.github.io, "Phase 2") and the split-K notes of the ML notes
// (haolingpu.github.io): each partial result is rescaled onto the larger
// max and the sums are added.
//
// GB300 mapping at d = 64 (fwd_tc.cu keeps d = 128):
//  * At d = 64 a 128 x 128 step is short (about 1.2 us), so a one-tile CTA
//    spends a large share of its life starting up (barriers, TMEM, the
//    first Q and K loads) and draining (the last P̃V, the store). One CTA per
//    SM instead loops over 128-row query tiles (static round robin over the
//    grid), and its producer and MMA warps run into the next tile while the
//    softmax warps finish the current one. Warp 0 writes each tile's work
//    (coordinates and key-tile plan) into a shared slot and loads its Q and
//    K tiles; warp 3 loads the V tiles.
//  * The CTA's two softmax warpgroups split the key tiles of a query tile:
//    warpgroup t takes plan indices t, t + 2, ... with its own S_t, P̃_t and
//    Õ_t in tensor memory, its own (m, l) in registers, and its own MMA
//    issuing warp. At the end of a tile the two partial results of each row
//    merge exactly (weights 2^(m_t - m) onto the common max).
//  * TMEM: S0, S1 (128 columns each), Õ0, Õ1 (64 each), P̃0, P̃1 (64 each,
//    bf16 pairs): the next S_t is computed as soon as the softmax has read
//    the current one.
//  * Shared memory: two Q buffers (the next tile's Q loads early), K and V
//    rings of 6 and 4 stages indexed by load counters that run across tiles
//    (a K stage frees after its QKᵀ, a V stage only after its P̃V), and an O
//    staging tile for the TMA store.
//  * Every mbarrier wait is bounded; a timeout sets the error word, raises a
//    CTA abort flag and every role drains its in-flight work before exit.

#include "common.cuh"
#include "launchers.h"
#include "mask.cuh"
#include "tc_ptx.cuh"
#include "tma_host.h"

namespace attn {

ATTN_DEFINE_ERROR_WORD(take_error_fwd_tc64)

namespace {

constexpr int D = 64;
constexpr int kBM = 128;            // query rows per tile (TMEM lanes)
constexpr int kBN = 128;            // keys per K/V tile
constexpr int kThreads = 384;       // 12 warps
constexpr int kKStages = 6;         // K ring (a stage is released by the QKᵀ that reads it)
constexpr int kVStages = 4;         // V ring (released later, by the P̃V)
constexpr int kTileBytes = kBM * D * 2;                  // Q, K, V or O tile (16 KB)
constexpr int kQOff = 0;                                 // Q buffers 0, 1
constexpr int kKOff = 2 * kTileBytes;
constexpr int kVOff = kKOff + kKStages * kTileBytes;
constexpr int kOOff = kVOff + kVStages * kTileBytes;     // O staging
constexpr int kSmemBytes = kOOff + kTileBytes;
constexpr int kDynSmem = kSmemBytes + 1024;              // slack for 1024-byte alignment
// TMEM columns of warpgroup t: S_t, Õ_t, P̃_t
ATTN_DEVINL uint32_t col_s(int t) { return t == 0 ? 0u : 128u; }
ATTN_DEVINL uint32_t col_o(int t) { return t == 0 ? 256u : 320u; }
ATTN_DEVINL uint32_t col_p(int t) { return t == 0 ? 384u : 448u; }
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: Õ is rescaled when m grows > 2^8

// One query tile of the work list and the key tiles it visits.
struct TileWork {
  int bh, kvh, row0;
  int n;                 // key tiles visited (plan indices 0 .. n-1)
  KeyTilePlan plan;      // plan index -> key tile (general masks)
};

struct Bars {
  uint64_t q_full[2], q_empty[2];
  uint64_t w_free[2];    // the softmax warpgroups have read work slot 0 / 1
  uint64_t k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2], s_free[2], p_full[2], o_done[2];
  uint64_t o_free;
  uint64_t mma_drain[2];
  uint32_t tmem_base;
  int abort;
  int stop;         // the softmax warpgroups' joint decision to leave the tile loop
  PlanSlots plan;   // keys the tile's rows see (general masks with row ranges)
  // Tile k's work, written by the Q/K producer with its Q load into slot
  // k % 2 (the index arithmetic is done once per tile, off the softmax path)
  TileWork work[2];
};

ATTN_DEVINL void tma_store_3d(const CUtensorMap* map, const void* smem_src, int c0, int c1,
                              int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
      ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
ATTN_DEVINL void tma_store_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the source shared memory of every committed store has been read
ATTN_DEVINL void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// every committed store has completed
ATTN_DEVINL void tma_store_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
ATTN_DEVINL void named_bar_sync(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
ATTN_DEVINL void tmem_st32(uint32_t ta, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(ta), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
        "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]),
        "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]),
        "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

ATTN_DEVINL TileWork read_work(const TileWork* slot) {
  const volatile TileWork* v = slot;
  TileWork tw;
  tw.bh = v->bh;
  tw.kvh = v->kvh;
  tw.row0 = v->row0;
  tw.n = v->n;
  tw.plan.s0 = v->plan.s0;
  tw.plan.n0 = v->plan.n0;
  tw.plan.s1 = v->plan.s1;
  tw.plan.n1 = v->plan.n1;
  return tw;
}

// Key-tile steps of softmax warpgroup t (plan indices t, t + 2, ...).
ATTN_DEVINL int steps_of(int n, int t) { return (n - t + 1) / 2; }

// kGeneral = false: no mask or causal only (key tiles 0 .. n-1, masked past a
// single per-row limit); true: any MaskSpec. With per-row key ranges the
// launch has one tile per CTA and the plan is reduced over the rows before
// the roles start (held in Bars::plan).
template <bool kGeneral>
__global__ void __launch_bounds__(kThreads, 1)
fwd_tc64_kernel(const __grid_constant__ CUtensorMap map_q,
                const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_v,
                const __grid_constant__ CUtensorMap map_o, float* __restrict__ lse, int Hq,
                int Hkv, int Nq, int Nk, float scale, MaskSpec mask, int n_qblk, int n_tiles,
                int order_grp) {
  // Launched as a programmatic dependent of whatever precedes it in the
  // stream: the prologue overlaps that kernel's tail and every global access
  // follows the producer's (or the row-range reduction's) wait for it.
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ Bars bars;
  __shared__ int4 keys_of_row[kBM];        // row ranges: each row's visible key intervals
  __shared__ float part_m[2][kBM], part_l[2][kBM];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_heads = n_tiles / n_qblk;                 // B * Hq
  const bool row_ranges = kGeneral && mask.row_kv_start != nullptr;

  auto tile_work = [&](int w) {
    TileWork tw;
    int rank;
    grouped_tile_order(w, n_qblk, n_heads, order_grp, tw.bh, rank);
    const int qblk = n_qblk - 1 - rank;
    const int b = tw.bh / Hq, h = tw.bh % Hq;
    tw.kvh = b * Hkv + h / (Hq / Hkv);
    tw.row0 = qblk * kBM;
    if (!kGeneral) {
      tw.plan = KeyTilePlan{0, 0, 0, 0};
      if (tw.row0 >= Nq) {
        tw.n = 0;
      } else {
        const int nk_tiles = (Nk + kBN - 1) / kBN;
        const int row_last = min(tw.row0 + kBM - 1, Nq - 1);
        tw.n = mask.window_right == 0   // causal, bottom-right aligned
                   ? min(nk_tiles, (row_last + (Nk - Nq)) / kBN + 1)
                   : nk_tiles;
        tw.n = max(tw.n, 0);
      }
    } else {
      PlanSlots slots;
      if (row_ranges) {
        const volatile PlanSlots* v = &bars.plan;
        slots.lo1 = v->lo1;
        slots.hi1 = v->hi1;
        slots.lo2 = v->lo2;
        slots.hi2 = v->hi2;
        slots.last[0] = v->last[0];
      } else {
        slots = plan_slots_direct(mask, tw.row0, kBM, 1, Nq, Nk);
      }
      tw.plan = make_plan(slots, kBN);
      tw.n = slots.last[0] >= 0 ? tw.plan.count_upto(slots.last[0] / kBN) : 0;
    }
    return tw;
  };

  if (tid == 0) {
    bars.abort = 0;
    bars.stop = 0;
    bars.plan.init();
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.q_full[i], 1);
      mbar_init(&bars.q_empty[i], 2);          // both issuers, after their last QKᵀ of the tile
      mbar_init(&bars.w_free[i], 2 * kBM);     // every softmax thread, once it has read the slot
    }
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&bars.k_full[i], 1);
      mbar_init(&bars.k_empty[i], 1);          // each stage is read by one issuer's MMAs
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars.s_full[t], 1);
      mbar_init(&bars.s_free[t], kBM);
      mbar_init(&bars.p_full[t], kBM);
      mbar_init(&bars.o_done[t], 1);
      mbar_init(&bars.mma_drain[t], 1);
    }
    mbar_init(&bars.o_free, 2 * kBM);          // every softmax thread, once Õ0 and Õ1 are read
    fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&bars.tmem_base, 512);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars.tmem_base;
  volatile int* abort_flag = &bars.abort;

  if (row_ranges) {
    // One tile per CTA: its rows' key intervals and the plan they imply.
    if (warp >= 4 && warp < 8) {
      pdl_wait_primary();                                    // the ranges are inputs
      const TileWork tw0 = tile_work(int(blockIdx.x));       // (its plan is not read here)
      const int b = tw0.bh / Hq;
      const RowKeys rk = row_keys(mask, b, tw0.row0 + (tid - 128), Nq, Nk);
      store_row_keys(&keys_of_row[tid - 128], rk);
      plan_add_rows(&bars.plan, rk, 0);
    }
    __syncthreads();
  }

  // Register split, set inside each role: 128 x 80 (the TMA and MMA warps) +
  // 256 x 208 (softmax) <= 384 x 168 registers the CTA is launched with.

  if (warp == 0 || warp == 3) {
    // ------------------------------------------------------------ TMA producers
    // Warp 0: the tile's work description and Q, then its K tiles; warp 3:
    // its V tiles. Apart, a V stage still held by an unfinished P̃V does not
    // hold up the next K load.
    regs_dec<80>();
    if (lane == 0) {
      pdl_wait_primary();
      const bool qk = warp == 0;
      if (qk) {
        tc::tma_prefetch_desc(&map_q);
        tc::tma_prefetch_desc(&map_k);
      } else {
        tc::tma_prefetch_desc(&map_v);
      }
      int g = 0, issued_q = 0, issued = 0, k = 0;
      bool ok = true;
      for (int w = int(blockIdx.x); w < n_tiles && ok; w += int(gridDim.x), ++k) {
        const TileWork tw = tile_work(w);
        if (qk) {
          // Q of tile k into buffer k % 2 once both issuers' QKᵀ of tile k - 2
          // have read it, its work into slot k % 2 once the softmax
          // warpgroups have read tile k - 2's
          const int qs = k & 1;
          ok = mbar_wait_bounded(&bars.q_empty[qs], ((k >> 1) & 1) ^ 1, abort_flag);
          if (ok) ok = mbar_wait_bounded(&bars.w_free[qs], ((k >> 1) & 1) ^ 1, abort_flag);
          if (!ok) break;
          bars.work[qs] = tw;
          mbar_arrive_expect_tx(&bars.q_full[qs], kTileBytes);   // (releases the slot write)
          tc::tma_load_3d(smem + kQOff + qs * kTileBytes, &map_q, 0, tw.row0, tw.bh,
                          &bars.q_full[qs]);
          ++issued_q;
        }
        const int stages = qk ? kKStages : kVStages;
        uint64_t* full = qk ? bars.k_full : bars.v_full;
        uint64_t* empty = qk ? bars.k_empty : bars.v_empty;
        uint8_t* ring = smem + (qk ? kKOff : kVOff);
        const CUtensorMap* map = qk ? &map_k : &map_v;
        for (int j = 0; j < tw.n; ++j, ++g) {
          const int st = g % stages;
          const uint32_t ph = (g / stages) & 1;
          const int key_tile = kGeneral ? tw.plan.tile(j) : j;
          ok = mbar_wait_bounded(&empty[st], ph ^ 1, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&full[st], kTileBytes);
          tc::tma_load_3d(ring + st * kTileBytes, map, 0, key_tile * kBN, tw.kvh, &full[st]);
          ++issued;
        }
      }
      if (!ok) {
        attn_flag_error(kErrTimeout);
        bars.abort = 1;
        // Drain: wait for the loads this thread issued that may still be in
        // flight (the last two Q loads, the last ring's worth of K or V
        // loads) so no copy lands after the CTA exits.
        for (int kq = max(0, issued_q - 2); kq < issued_q; ++kq)
          mbar_wait_bounded(&bars.q_full[kq & 1], (kq >> 1) & 1, nullptr);
        const int stages = qk ? kKStages : kVStages;
        uint64_t* full = qk ? bars.k_full : bars.v_full;
        for (int j = max(0, issued - stages); j < issued; ++j)
          mbar_wait_bounded(&full[j % stages], (j / stages) & 1, nullptr);
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // One issuing warp per softmax warpgroup (the loop runs converged; one
    // elected lane issues). tcgen05.mma issue only returns as the tensor pipe
    // accepts the instruction, so a single issuer waiting on one
    // warpgroup's barrier would starve the pipe when the other's work is
    // ready.
    regs_dec<80>();
    const int t = warp - 1;
    constexpr uint32_t idesc_s = tc::idesc_bf16_f32(kBM, kBN, false, false);
    constexpr uint32_t idesc_o = tc::idesc_bf16_f32(kBM, D, false, true);
    const uint32_t q_base = smem_u32(smem + kQOff);
    const uint32_t k_base = smem_u32(smem + kKOff);
    const uint32_t v_base = smem_u32(smem + kVOff);
    bool ok = true;
    int g0 = 0;   // load-counter value of the tile's plan index 0
    int cs = 0;   // this warpgroup's key-tile steps before the tile
    int k = 0;
    bool any = false;
    for (int w = int(blockIdx.x); w < n_tiles && ok; w += int(gridDim.x), ++k) {
      const int qs = k & 1;
      const uint32_t qa = q_base + qs * kTileBytes;
      // Q of the tile and its work slot (both written before q_full)
      ok = mbar_wait_warp(&bars.q_full[qs], (k >> 1) & 1, abort_flag);
      if (!ok) break;
      const TileWork tw = read_work(&bars.work[qs]);
      const int n = steps_of(tw.n, t);
      // step i reads load g0 + t + 2i of each ring; S_t(i) follows the
      // softmax's read of this warpgroup's previous S
      auto issue_s = [&](int i) {
        const int g = g0 + t + 2 * i;
        const uint32_t ka = k_base + (g % kKStages) * kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc::mma_ss_warp(tmem + col_s(t), tc::smem_desc(qa + kk * 32, 16, 1024, tc::kLayoutSW128),
                          tc::smem_desc(ka + kk * 32, 16, 1024, tc::kLayoutSW128), idesc_s, kk > 0);
        tc::mma_commit_warp(&bars.s_full[t]);
        tc::mma_commit_warp(&bars.k_empty[g % kKStages]);
        if (i == n - 1) tc::mma_commit_warp(&bars.q_empty[qs]);   // the tile's last read of Q
      };
      auto wait_s_inputs = [&](int i) {
        const int g = g0 + t + 2 * i;
        bool r = true;
        if (cs + i > 0) r = mbar_wait_warp(&bars.s_free[t], (cs + i - 1) & 1, abort_flag);
        if (r) r = mbar_wait_warp(&bars.k_full[g % kKStages], (g / kKStages) & 1, abort_flag);
        return r;
      };
      if (n == 0) {
        // nothing of this tile: release its Q buffer (each load completes
        // one phase of q_full, each pair of releases one of q_empty)
        if (lane == 0) mbar_arrive(&bars.q_empty[qs]);
        __syncwarp();
      } else {
        ok = wait_s_inputs(0);
        if (ok) {
          tc::fence_after_sync();
          issue_s(0);
          any = true;
        }
        for (int i = 0; i < n && ok; ++i) {
          if (i + 1 < n) {
            ok = wait_s_inputs(i + 1);
            if (!ok) break;
            tc::fence_after_sync();
            issue_s(i + 1);
          }
          const int g = g0 + t + 2 * i;
          ok = mbar_wait_warp(&bars.v_full[g % kVStages], (g / kVStages) & 1, abort_flag);
          if (ok) ok = mbar_wait_warp(&bars.p_full[t], (cs + i) & 1, abort_flag);
          // the first P̃V of a tile overwrites Õ_t: the previous tile's merge
          // has read it
          if (ok && i == 0) ok = mbar_wait_warp(&bars.o_free, (k & 1) ^ 1, abort_flag);
          if (!ok) break;
          tc::fence_after_sync();
          const uint32_t va = v_base + (g % kVStages) * kTileBytes;
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk)
            tc::mma_ts_warp(tmem + col_o(t), tmem + col_p(t) + kk * 8,
                            tc::smem_desc(va + kk * 2048, kBN * 128, 1024, tc::kLayoutSW128),
                            idesc_o, (i > 0 || kk > 0) ? 1u : 0u);
          tc::mma_commit_warp(&bars.o_done[t]);
          tc::mma_commit_warp(&bars.v_empty[g % kVStages]);
        }
      }
      g0 += tw.n;
      cs += n;
    }
    if (!ok && lane == 0) {
      attn_flag_error(kErrTimeout);
      bars.abort = 1;
    }
    __syncwarp();
    // Drain: every MMA this warp issued has completed before TMEM is freed.
    if (any) {
      tc::mma_commit_warp(&bars.mma_drain[t]);
      mbar_wait_warp(&bars.mma_drain[t], 0, nullptr);
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    regs_inc<208>();
    const int t = (warp - 4) / 4;                  // key tiles t, t + 2, ... of each query tile
    const int quarter = warp % 4;                  // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;             // row within the tile (TMEM lane)
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + col_s(t);
    const uint32_t p_addr = tmem + lane_base + col_p(t);
    const uint32_t o_addr = tmem + lane_base + col_o(t);
    const float c = scale * kLog2e;               // scores in log2 units
    const bool storer = warp == 4 && lane == 0;    // issues the tile's TMA store
    int cs = 0;                                    // this warpgroup's steps before the tile
    bool ok = true;
    // An mbarrier probe takes ~150 cycles to answer even when the phase is
    // long complete, so the next step's S-full and this step's P̃V-done are
    // probed early without blocking (test_wait) and the answers used later;
    // a phase not yet complete then is waited for as usual.
    bool s_ready = false;                          // S of the next step known complete

    for (int w = int(blockIdx.x), k = 0; w < n_tiles; w += int(gridDim.x), ++k) {
      // the tile's work (written with its Q load into slot k % 2)
      const int qs = k & 1;
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars.q_full[qs], (k >> 1) & 1, abort_flag));
      const TileWork tw = read_work(&bars.work[qs]);
      mbar_arrive(&bars.w_free[qs]);
      const int nt = steps_of(tw.n, t);
      const int row = tw.row0 + r;                 // query row
      const int b = tw.bh / Hq;
      // general mask: this row's key intervals; otherwise its last key
      const RowKeys rk = !kGeneral    ? RowKeys{1, 0, 1, 0}
                         : row_ranges ? load_row_keys(&keys_of_row[r])
                                      : row_keys(mask, b, row, Nq, Nk);
      const int limit = mask.window_right == 0 ? min(Nk - 1, row + (Nk - Nq)) : Nk - 1;

      float m_ref = -INFINITY;                     // reference max (log2 units)
      float l_run = 0.f;
      for (int i = 0; i < nt && ok; ++i) {
        const int ci = cs + i;
        // Waits are made warp-uniform: tcgen05.ld/st below are warp-collective.
        if (!__all_sync(0xffffffffu,
                        s_ready || mbar_wait_bounded(&bars.s_full[t], ci & 1, abort_flag))) {
          ok = false;
          break;
        }
        s_ready = false;
        tc::fence_after_sync();
        uint32_t sr[128];
        tc::tmem_ld32(s_addr + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tc::tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tc::tmem_ld32(s_addr + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
        tc::tmem_ld32(s_addr + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
        tc::tmem_ld_wait();
        float* s = reinterpret_cast<float*>(sr);
        tc::fence_before_sync();
        mbar_arrive(&bars.s_free[t]);              // S_t may be recomputed now

        // Mask the keys this row does not see (past the end included) in a
        // tile that straddles one of its bounds.
        const int jj = t + 2 * i;
        const int key0 = (kGeneral ? tw.plan.tile(jj) : jj) * kBN;
        if (kGeneral) {
          if (!rk.covers(key0, key0 + kBN - 1)) {
#pragma unroll
            for (int wd = 0; wd < kBN / 32; ++wd) {
              const uint32_t vis = rk.bits(key0, wd);
#pragma unroll
              for (int cc = 0; cc < 32; ++cc)
                if (!(vis & (1u << cc))) s[32 * wd + cc] = -INFINITY;
            }
          }
        } else if (key0 + kBN - 1 > limit) {
#pragma unroll
          for (int cc = 0; cc < kBN; ++cc)
            if (key0 + cc > limit) s[cc] = -INFINITY;
        }
        // Row max as 8 independent chains (short dependency chains, more ILP).
        float m8[8];
#pragma unroll
        for (int kq = 0; kq < 8; ++kq) m8[kq] = fmaxf(s[kq], s[kq + 8]);
#pragma unroll
        for (int ii = 16; ii < kBN; ii += 16)
#pragma unroll
          for (int kq = 0; kq < 8; ++kq) m8[kq] = max3(m8[kq], s[ii + kq], s[ii + 8 + kq]);
        const float mx = fmaxf(max3(m8[0], m8[1], m8[2]),
                               fmaxf(max3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7])));
        const float m_cand = fmaxf(m_ref, mx * c);
        const bool need = m_cand - m_ref > kRescaleThreshold;   // also true while m_ref = -inf
        float alpha = 1.f;
        if (need) {
          alpha = fast_exp2(m_ref - m_cand);                   // 0 when m_ref = -inf
          m_ref = m_cand;
        }
        const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
        const bool pv_ready = i > 0 && mbar_test_wait(&bars.o_done[t], (ci - 1) & 1);

        // P̃ = exp2(s·c - m_ref) -> bf16 pairs, all 128 first: P̃_t may only
        // be written once the previous P̃V of this warpgroup has read it, and
        // the wait then overlaps the special-function work.
        const f2 cc2{c, c}, nm2{neg_m, neg_m};
        f2 rs2[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};   // 4 independent sums
        uint32_t pk[64];
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          f2 x = fma2(f2{s[2 * e], s[2 * e + 1]}, cc2, nm2);
          x.x = fast_exp2(x.x);
          x.y = fast_exp2(x.y);
          rs2[e & 3] = add2(rs2[e & 3], x);
          pk[e] = pack_bf16x2(x.x, x.y);
        }
        // the next step's scores (the following tile's first, after the last)
        const bool s_next = mbar_test_wait(&bars.s_full[t], (ci + 1) & 1);
        // (the previous P̃V of this warpgroup in an earlier tile was waited
        // for by that tile's merge)
        if (i > 0) {
          ok = __all_sync(0xffffffffu, pv_ready ||
                                       mbar_wait_bounded(&bars.o_done[t], (ci - 1) & 1, abort_flag));
          if (!ok) break;
          tc::fence_after_sync();
        }
        tmem_st32(p_addr, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        tmem_st32(p_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
        const f2 rsa = add2(add2(rs2[0], rs2[1]), add2(rs2[2], rs2[3]));
        l_run = fmaf(alpha, l_run, rsa.x + rsa.y);

        // Rescale Õ (the previous P̃V has landed) when the reference moved.
        if (i > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t orr[32];
            tc::tmem_ld32(o_addr + ch * 32, orr);
            tc::tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) orr[e] = __float_as_uint(__uint_as_float(orr[e]) * alpha);
            tmem_st32(o_addr + ch * 32, orr);
          }
        }
        tc::tmem_st_wait();
        tc::fence_before_sync();
        mbar_arrive(&bars.p_full[t]);
        s_ready = __all_sync(0xffffffffu, s_next);
      }
      cs += nt;

      // Merge and store. Õ_t is final once this warpgroup's last P̃V of the
      // tile has completed.
      if (ok && nt > 0)
        ok = mbar_wait_bounded(&bars.o_done[t], (cs - 1) & 1, abort_flag);
      ok = __all_sync(0xffffffffu, ok);
      part_m[t][r] = m_ref;
      part_l[t][r] = l_run;
      if (!ok) {
        if (lane == 0) attn_flag_error(kErrTimeout);
        bars.abort = 1;
      }
      // the previous tile's store has read the staging tile
      if (storer) tma_store_wait_read();
      named_bar_sync(1, 2 * kBM);                  // both warpgroups' Õ and (m, l) final
      const bool tile_rows = tw.row0 < Nq;
      if (tid == 128) bars.stop = bars.abort;      // one decision for both warpgroups
      // The two partial results of a row, each relative to its own
      // reference max, merge exactly: weights 2^(m_t - m) onto the common
      // max; a warpgroup that saw no key of the row carries no mass (and its
      // Õ columns, possibly never written this tile, are not summed).
      tc::fence_after_sync();
      const float m0 = part_m[0][r], m1 = part_m[1][r];
      const float l0 = part_l[0][r], l1 = part_l[1][r];
      // this warpgroup writes columns [32t, 32t + 32) of the row
      uint32_t o0[32], o1[32];
      tc::tmem_ld32(tmem + lane_base + col_o(0) + 32 * t, o0);
      tc::tmem_ld32(tmem + lane_base + col_o(1) + 32 * t, o1);
      tc::tmem_ld_wait();
      tc::fence_before_sync();
      mbar_arrive(&bars.o_free);                   // the next tile's P̃V may overwrite Õ
      if (tile_rows && !bars.abort) {
        const float mm = fmaxf(l0 > 0.f ? m0 : -INFINITY, l1 > 0.f ? m1 : -INFINITY);
        const float w0 = l0 > 0.f ? fast_exp2(m0 - mm) : 0.f;
        const float w1 = l1 > 0.f ? fast_exp2(m1 - mm) : 0.f;
        const float l = w0 * l0 + w1 * l1;
        const float inv_l = l > 0.f ? __frcp_rn(l) : 0.f;
        const float a0 = w0 * inv_l, a1 = w1 * inv_l;
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float x0 = (l0 > 0.f ? __uint_as_float(o0[2 * e]) * a0 : 0.f) +
                           (l1 > 0.f ? __uint_as_float(o1[2 * e]) * a1 : 0.f);
          const float x1 = (l0 > 0.f ? __uint_as_float(o0[2 * e + 1]) * a0 : 0.f) +
                           (l1 > 0.f ? __uint_as_float(o1[2 * e + 1]) * a1 : 0.f);
          pk[e] = pack_bf16x2(x0, x1);
        }
        // one 128-byte swizzle atom per row; 16-byte chunks 4t .. 4t + 3
        uint8_t* atom = smem + kOOff + r * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          *reinterpret_cast<uint4*>(atom + (((4 * t + u) ^ (r & 7)) * 16)) =
              make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        if (t == 0 && lse != nullptr && row < Nq)
          lse[size_t(tw.bh) * Nq + row] = l > 0.f ? (mm + __log2f(l)) * kLn2 : -INFINITY;
        fence_proxy_async_smem();
      }
      named_bar_sync(1, 2 * kBM);
      const bool stop = bars.stop != 0;
      if (storer && tile_rows && !stop) {
        tma_store_3d(&map_o, smem + kOOff, 0, tw.row0, tw.bh);
        tma_store_commit();
      }
      if (stop) break;
    }
    if (storer) tma_store_wait_all();
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

template <bool kGeneral>
cudaError_t launch_t(const FwdArgs& a) {
  CUtensorMap mq, mk, mv, mo;
  if (!make_map_bf16_3d(&mq, a.q, D, a.Nq, uint64_t(a.B) * a.Hq, kBM) ||
      !make_map_bf16_3d(&mk, a.k, D, a.Nk, uint64_t(a.B) * a.Hkv, kBN) ||
      !make_map_bf16_3d(&mv, a.v, D, a.Nk, uint64_t(a.B) * a.Hkv, kBN) ||
      !make_map_bf16_3d(&mo, a.o, D, a.Nq, uint64_t(a.B) * a.Hq, kBM))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(fwd_tc64_kernel<kGeneral>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem);
  if (e != cudaSuccess) return e;
  const int n_qblk = (a.Nq + kBM - 1) / kBM;
  const long tiles = long(n_qblk) * a.B * a.Hq;
  if (tiles > 0x7fffffffL) return cudaErrorInvalidValue;
  // one CTA per SM; with per-row key ranges one CTA per tile (the plan is
  // reduced over the tile's rows before the roles start)
  const int sms = device_sm_count();
  if (sms <= 0) return cudaErrorInvalidValue;
  const bool row_ranges = a.mask.row_kv_start != nullptr;
  const long grid = row_ranges ? tiles : (tiles < sms ? tiles : sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kDynSmem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fwd_tc64_kernel<kGeneral>, mq, mk, mv, mo, a.lse, a.Hq, a.Hkv,
                            a.Nq, a.Nk, a.scale, a.mask, n_qblk, int(tiles),
                            order_group(a.mask.varies(), 4LL * a.Nk * D));
}

}  // namespace

cudaError_t launch_fwd_tc64(const FwdArgs& a) {
  const MaskSpec& m = a.mask;
  const bool plain = m.window_left < 0 && m.window_right <= 0 && m.n_global == 0 &&
                     m.row_kv_start == nullptr;   // no mask, or causal
  return plain ? launch_t<false>(a) : launch_t<true>(a);
}

}  // namespace attn

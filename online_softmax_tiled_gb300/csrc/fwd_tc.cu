// bf16 tiled attention forward at head dimension 128 on the sm_103a tensor
// cores (tcgen05 + TMEM + TMA); d = 64 runs the persistent kernel of
// fwd_tc64.cu.
//
// Algorithm: the inner loop of the "Flash Attention 2" post
// (ahmadsaeedzaidi.github.io feed), section "Flash Attention 2": for a query
// tile Q_i and each key/value tile K_j, V_j: S_ij = scale·Q_i K_jᵀ, running
// row max m, P̃ = exp(S - m), running denominator l, Õ rescaled by
// exp(m_old - m_new) and accumulated with P̃ V_j; after the last tile
// O_i = Õ_i / l_i and LSE = m + ln l. Masks per the post's section "Causal
// masking", option A, which covers arbitrary masks: the CTA visits only the
// key tiles some row of it can see (mask.cuh: at most two ranges) and the
// tiles that straddle a row's boundary are masked element by element.
//
// GB300 mapping (differs from the post's SRAM-only picture):
//  * One CTA owns two 128-row query tiles and streams 128-key K/V tiles
//    through a shared-memory ring filled by TMA (128-byte swizzle, zero fill
//    past the end of the sequence). Without grouped-query sharing the two
//    tiles are consecutive rows of one head (256 rows); when two query heads
//    share a KV head (Hq / Hkv even) they are the same 128 rows of two heads
//    of the group, so every K/V tile loaded feeds both heads (the grouped
//    heads of the KV-compression post's SnapKV code read one KV head).
//  * S = Q Kᵀ and Õ += P̃ V run on tcgen05.mma (bf16 in, fp32 out) with both
//    accumulators in tensor memory: S0, S1 (128 columns each) and Õ0, Õ1
//    (d columns each).
//  * One warpgroup per query tile owns the softmax: each thread owns one row
//    (TMEM lane), reads its 128 scores with tcgen05.ld, keeps m and l in
//    fp32 registers, and writes P̃ (bf16) back into the first 64 columns of
//    its S buffer, where the P̃ V MMA reads it as the A operand.
//  * The issue order S0(j), S1(j), PV0(j), S0(j+1), PV1(j), S1(j+1), ...
//    lets each warpgroup's softmax overlap the other tile's MMAs.
//  * Rescaling is lazy: the reference max only moves when the row max grows
//    by more than 8 (log2 units), so Õ in TMEM is rarely re-read. Any
//    reference value gives the exact result as long as Õ and l share it.
//  * Every mbarrier wait is bounded; a timeout sets the error word, raises a
//    CTA abort flag and every role drains its in-flight work before exit.

#include "common.cuh"
#include "launchers.h"
#include "mask.cuh"
#include "tc_ptx.cuh"
#include "tma_host.h"

namespace attn {

ATTN_DEFINE_ERROR_WORD(take_error_fwd_tc)

namespace {

constexpr int kBM = 128;            // query rows per tile (TMEM lanes)
constexpr int kBN = 128;            // keys per K/V tile
constexpr int kThreads = 384;       // 12 warps
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: Õ is rescaled when m grows > 2^8

template <int D>
struct FwdCfg {
  static_assert(D == 128, "d = 64 runs fwd_tc64_kernel");
  static constexpr int kStages = 2;
  static constexpr int kAtoms = D / 64;                   // 128-byte swizzle atoms per row
  static constexpr int kTileBytes = kBM * D * 2;          // Q, K or V tile
  static constexpr int kQOff = 0;                         // Q0, Q1
  static constexpr int kKOff = 2 * kTileBytes;
  static constexpr int kVOff = kKOff + kStages * kTileBytes;
  static constexpr int kSmemBytes = kVOff + kStages * kTileBytes;
  static constexpr int kDynSmem = kSmemBytes + 1024;      // slack for 1024-byte alignment
  // TMEM columns: S0, S1, O0, O1 fill all 512 columns and P̃ is written over
  // the scores it came from.
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO0 = 256, kColO1 = 256 + D;
  static constexpr uint32_t kColP0 = kColS0, kColP1 = kColS1;
};

struct Bars {
  uint64_t q_full;
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t mma_drain;
  uint32_t tmem_base;
  int abort;
  PlanSlots plan;   // keys the CTA's rows see (general masks)
};

ATTN_DEVINL void tma_store_3d(const CUtensorMap* map, const void* smem_src, int c0, int c1,
                              int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
      ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
ATTN_DEVINL void tma_store_commit_and_wait() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
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

// Number of K/V tiles a query tile starting at row_first visits without a
// general mask (0 if the tile has no valid row): all of them, or up to the
// causal diagonal.
ATTN_DEVINL int kv_tiles_for(int row_first, int Nq, int Nk, bool causal) {
  if (row_first >= Nq) return 0;
  const int nk_tiles = (Nk + kBN - 1) / kBN;
  if (!causal) return nk_tiles;
  const int row_last = min(row_first + kBM - 1, Nq - 1);
  return min(nk_tiles, (row_last + (Nk - Nq)) / kBN + 1);   // bottom-right alignment
}

// kGeneral = false: no mask or causal only (the CTA visits key tiles 0, 1, ...
// and masks past a single per-row limit); true: any MaskSpec.
template <int D, bool kGeneral>
__global__ void __launch_bounds__(kThreads, 1)
fwd_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
              const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_o,
              float* __restrict__ lse, int Hq, int Hkv, int Nq, int Nk, float scale,
              MaskSpec mask, int n_qblk, int order_grp, int head_pairs) {
  using C = FwdCfg<D>;
  // Launched as a programmatic dependent of whatever precedes it in the
  // stream: the prologue (barriers, TMEM) overlaps that kernel's tail and
  // the TMA producer waits for it before the first load. Every global access
  // of this kernel follows those loads.
  pdl_launch_dependents();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ Bars bars;
  __shared__ int4 keys_of_row[2 * kBM];   // each row's visible key intervals

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Heads (or head pairs) in groups whose K/V fit in L2 together (causal;
  // head-major otherwise); in a group the heaviest (latest) query blocks
  // first. head_pairs: the CTA's tiles t = 0, 1 are rows [row0, row0 + 128)
  // of query heads 2p and 2p + 1, which read the same KV head; otherwise
  // rows row0 + 128·t of one head.
  int hp, rank;
  grouped_tile_order(int(blockIdx.x), n_qblk, int(gridDim.x) / n_qblk, order_grp, hp, rank);
  const int qblk = n_qblk - 1 - rank;
  const int bh = head_pairs ? 2 * hp : hp;            // b·Hq + h of tile 0
  const int b = bh / Hq, h = bh % Hq;
  const int kvh = b * Hkv + h / (Hq / Hkv);
  const int row0 = qblk * (head_pairs ? kBM : 2 * kBM);
  auto tile_row0 = [&](int t) { return head_pairs ? row0 : row0 + t * kBM; };
  auto tile_bh = [&](int t) { return head_pairs ? bh + t : bh; };

  if (tid == 0) {
    bars.abort = 0;
    bars.plan.init();
    mbar_init(&bars.q_full, 1);
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&bars.k_full[i], 1);
      mbar_init(&bars.k_empty[i], 1);
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars.s_full[t], 1);
      mbar_init(&bars.p_full[t], kBM);
      mbar_init(&bars.o_done[t], 1);
    }
    mbar_init(&bars.mma_drain, 1);
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

  // The Q tiles do not depend on the mask: their loads start first.
  if (warp == 0 && lane == 0) {
    pdl_wait_primary();
    tc::tma_prefetch_desc(&map_q);
    tc::tma_prefetch_desc(&map_k);
    tc::tma_prefetch_desc(&map_v);
    mbar_arrive_expect_tx(&bars.q_full, 2 * C::kTileBytes);
    for (int t = 0; t < 2; ++t)
      for (int a = 0; a < C::kAtoms; ++a)
        tc::tma_load_3d(smem + C::kQOff + t * C::kTileBytes + a * (kBM * 128), &map_q, 64 * a,
                        tile_row0(t), tile_bh(t), &bars.q_full);
  }
  // The key tiles to visit. Without row ranges the plan follows from the
  // mask directly (no barrier: the loads start at once); with them every
  // softmax thread (one query row) adds the keys its row sees and all roles
  // wait for the sum. Query tile t visits the prefix of the plan that ends
  // with its last visible key.
  PlanSlots slots;
  if (!kGeneral) {
    // tiles 0 .. n-1; the plan is only read by the general path
    const bool causal = mask.window_right == 0;
    slots.init();
    slots.lo1 = 0;
    slots.hi1 = Nk - 1;
    slots.last[0] = kv_tiles_for(tile_row0(0), Nq, Nk, causal) * kBN - 1;
    slots.last[1] = kv_tiles_for(tile_row0(1), Nq, Nk, causal) * kBN - 1;
  } else if (mask.row_kv_start == nullptr) {
    slots = plan_slots_direct(mask, row0, kBM, head_pairs ? 1 : 2, Nq, Nk);
    if (head_pairs) slots.last[1] = slots.last[0];   // the same rows
    if (tid == 0) bars.plan = slots;   // the producer thread reads it back below
  } else {
    if (warp >= 4) {
      const int t = (warp - 4) / 4;
      pdl_wait_primary();                                    // the ranges are inputs
      const RowKeys rk = row_keys(mask, b, tile_row0(t) + (warp % 4) * 32 + lane, Nq, Nk);
      store_row_keys(&keys_of_row[tid - 128], rk);
      plan_add_rows(&bars.plan, rk, t);
    }
    __syncthreads();
    slots = bars.plan;
  }
  const KeyTilePlan plan = make_plan(slots, kBN);
  const int n_t[2] = {slots.last[0] >= 0 ? plan.count_upto(slots.last[0] / kBN) : 0,
                      slots.last[1] >= 0 ? plan.count_upto(slots.last[1] / kBN) : 0};
  auto key_tile = [&](int j) {
    return kGeneral ? make_plan_volatile(&bars.plan, kBN).tile(j) : j;
  };
  const int nj = max(n_t[0], n_t[1]);

  // Register split, set inside each role: 128 x 80 (TMA, MMA, idle warps) +
  // 256 x 208 (softmax) <= 384 x 168 registers the CTA is launched with.

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    regs_dec<80>();
    if (lane == 0 && nj > 0) {
      int issued_k = 0, issued_v = 0;
      bool ok = true;
      for (int j = 0; j < nj && ok; ++j) {
        const int st = j % C::kStages;
        const uint32_t ph = (j / C::kStages) & 1;
        if (j >= C::kStages) ok = mbar_wait_bounded(&bars.k_empty[st], ph ^ 1, abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars.k_full[st], C::kTileBytes);
        for (int a = 0; a < C::kAtoms; ++a)
          tc::tma_load_3d(smem + C::kKOff + st * C::kTileBytes + a * (kBN * 128), &map_k, 64 * a,
                          key_tile(j) * kBN, kvh, &bars.k_full[st]);
        ++issued_k;
        if (j >= C::kStages) ok = mbar_wait_bounded(&bars.v_empty[st], ph ^ 1, abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars.v_full[st], C::kTileBytes);
        for (int a = 0; a < C::kAtoms; ++a)
          tc::tma_load_3d(smem + C::kVOff + st * C::kTileBytes + a * (kBN * 128), &map_v, 64 * a,
                          key_tile(j) * kBN, kvh, &bars.v_full[st]);
        ++issued_v;
      }
      if (!ok) {
        attn_flag_error(kErrTimeout);
        bars.abort = 1;
        // Drain: wait for the loads this thread issued (each at most once
        // unconsumed per stage) so no copy lands after the CTA exits.
        mbar_wait_bounded(&bars.q_full, 0, nullptr);
        for (int j = max(0, issued_k - C::kStages); j < issued_k; ++j)
          mbar_wait_bounded(&bars.k_full[j % C::kStages], (j / C::kStages) & 1, nullptr);
        for (int j = max(0, issued_v - C::kStages); j < issued_v; ++j)
          mbar_wait_bounded(&bars.v_full[j % C::kStages], (j / C::kStages) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop; one elected lane issues each MMA, in the
    // order S0, S1, PV0, S0', PV1, S1', ... (P̃ lives in the S columns, so
    // S_t(j+1) follows PV_t(j)).
    regs_dec<80>();
    if (nj > 0) {
      constexpr uint32_t idesc_s = tc::idesc_bf16_f32(kBM, kBN, false, false);
      constexpr uint32_t idesc_o = tc::idesc_bf16_f32(kBM, D, false, true);
      const uint32_t s_col[2] = {C::kColS0, C::kColS1};
      const uint32_t o_col[2] = {C::kColO0, C::kColO1};
      const uint32_t q_base = smem_u32(smem + C::kQOff);
      const uint32_t k_base = smem_u32(smem + C::kKOff);
      const uint32_t v_base = smem_u32(smem + C::kVOff);

      auto issue_s = [&](int t, int j) {
        const uint32_t qa = q_base + t * C::kTileBytes;
        const uint32_t ka = k_base + (j % C::kStages) * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk / 4) * (kBM * 128) + (kk % 4) * 32;
          tc::mma_ss_warp(tmem + s_col[t], tc::smem_desc(qa + off, 16, 1024, tc::kLayoutSW128),
                          tc::smem_desc(ka + off, 16, 1024, tc::kLayoutSW128), idesc_s, kk > 0);
        }
        tc::mma_commit_warp(&bars.s_full[t]);
      };
      auto issue_pv = [&](int t, int j) {
        const uint32_t va = v_base + (j % C::kStages) * C::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          tc::mma_ts_warp(tmem + o_col[t], tmem + s_col[t] + kk * 8,
                          tc::smem_desc(va + kk * 2048, kBN * 128, 1024, tc::kLayoutSW128), idesc_o,
                          (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc::mma_commit_warp(&bars.o_done[t]);
      };

      bool ok = mbar_wait_warp(&bars.q_full, 0, abort_flag);
      if (ok) ok = mbar_wait_warp(&bars.k_full[0], 0, abort_flag);
      if (ok) {
        tc::fence_after_sync();
        for (int t = 0; t < 2; ++t)
          if (n_t[t] > 0) issue_s(t, 0);
        tc::mma_commit_warp(&bars.k_empty[0]);
      }
      for (int j = 0; j < nj && ok; ++j) {
        const bool has_next = j + 1 < nj;
        ok = mbar_wait_warp(&bars.v_full[j % C::kStages], (j / C::kStages) & 1, abort_flag);
        if (ok && has_next)
          ok = mbar_wait_warp(&bars.k_full[(j + 1) % C::kStages], ((j + 1) / C::kStages) & 1,
                              abort_flag);
        for (int t = 0; t < 2 && ok; ++t) {
          if (j < n_t[t]) {
            ok = mbar_wait_warp(&bars.p_full[t], j & 1, abort_flag);
            if (!ok) break;
            tc::fence_after_sync();
            issue_pv(t, j);
          }
          if (has_next && j + 1 < n_t[t]) issue_s(t, j + 1);
        }
        if (!ok) break;
        tc::mma_commit_warp(&bars.v_empty[j % C::kStages]);
        if (has_next) tc::mma_commit_warp(&bars.k_empty[(j + 1) % C::kStages]);
      }
      if (!ok && lane == 0) {
        attn_flag_error(kErrTimeout);
        bars.abort = 1;
      }
      __syncwarp();
      // Drain: every MMA this warp issued has completed before TMEM is freed.
      tc::mma_commit_warp(&bars.mma_drain);
      mbar_wait_warp(&bars.mma_drain, 0, nullptr);
    }
  } else if (warp < 4) {
    regs_dec<80>();                                // idle warp of the first warpgroup
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    regs_inc<208>();
    const int t = (warp - 4) / 4;                  // query tile of this warpgroup
    const int quarter = warp % 4;                  // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;             // row within the tile (TMEM lane)
    const int row = tile_row0(t) + r;              // query row
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + (t == 0 ? C::kColS0 : C::kColS1);
    const uint32_t p_addr = tmem + lane_base + (t == 0 ? C::kColP0 : C::kColP1);
    const uint32_t o_addr = tmem + lane_base + (t == 0 ? C::kColO0 : C::kColO1);
    const float c = scale * kLog2e;               // scores in log2 units
    const int nt = n_t[t];
    // general mask: this row's key intervals; otherwise its last key
    const RowKeys rk = !kGeneral ? RowKeys{1, 0, 1, 0}
                       : mask.row_kv_start == nullptr ? row_keys(mask, b, row, Nq, Nk)
                                                      : load_row_keys(&keys_of_row[tid - 128]);
    const int limit = mask.window_right == 0 ? min(Nk - 1, row + (Nk - Nq)) : Nk - 1;

    float m_ref = -INFINITY;                       // reference max (log2 units)
    float l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      // Waits are made warp-uniform: tcgen05.ld/st below are warp-collective.
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&bars.s_full[t], j & 1, abort_flag))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      uint32_t sr[128];
      tc::tmem_ld32(s_addr + 0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tc::tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tc::tmem_ld32(s_addr + 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[64]));
      tc::tmem_ld32(s_addr + 96, *reinterpret_cast<uint32_t(*)[32]>(&sr[96]));
      tc::tmem_ld_wait();
      float* s = reinterpret_cast<float*>(sr);

      // Mask the keys this row does not see (past the end included) in a
      // tile that straddles one of its bounds.
      const int key0 = (kGeneral ? plan.tile(j) : j) * kBN;
      if (kGeneral) {
        if (!rk.covers(key0, key0 + kBN - 1)) {
#pragma unroll
          for (int w = 0; w < kBN / 32; ++w) {
            const uint32_t vis = rk.bits(key0, w);
#pragma unroll
            for (int cc = 0; cc < 32; ++cc)
              if (!(vis & (1u << cc))) s[32 * w + cc] = -INFINITY;
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
      for (int k = 0; k < 8; ++k) m8[k] = fmaxf(s[k], s[k + 8]);
#pragma unroll
      for (int i = 16; i < kBN; i += 16)
#pragma unroll
        for (int k = 0; k < 8; ++k) m8[k] = max3(m8[k], s[i + k], s[i + 8 + k]);
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

      // P̃ = exp2(s·c - m_ref) -> bf16 pairs over the first 64 score columns
      const f2 cc2{c, c}, nm2{neg_m, neg_m};
      f2 rs2[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};   // 4 independent sums
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint32_t pk[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          f2 x = fma2(f2{s[half * 64 + 2 * e], s[half * 64 + 2 * e + 1]}, cc2, nm2);
          x.x = fast_exp2(x.x);
          x.y = fast_exp2(x.y);
          rs2[e & 3] = add2(rs2[e & 3], x);
          pk[e] = pack_bf16x2(x.x, x.y);
        }
        tmem_st32(p_addr + half * 32, pk);
      }
      const f2 rsa = add2(add2(rs2[0], rs2[1]), add2(rs2[2], rs2[3]));
      const float rs = rsa.x + rsa.y;
      l_run = fmaf(alpha, l_run, rs);

      // Rescale Õ (once the previous P̃V has landed) when the reference moved.
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars.o_done[t], (j - 1) & 1, abort_flag));
        if (!ok) break;
        tc::fence_after_sync();
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
    }

    // Epilogue: O = Õ / l -> bf16 -> swizzled smem (the dead Q tile) -> TMA
    // store. A tile that visited no key stores zeros (and LSE = -inf) once
    // its Q tile, the staging area, has landed.
    const bool tile_rows = tile_row0(t) < Nq;
    if (ok && nt > 0)
      ok = mbar_wait_bounded(&bars.o_done[t], (nt - 1) & 1, abort_flag);
    else if (ok)
      ok = mbar_wait_bounded(&bars.q_full, 0, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    if (ok && tile_rows) {
      tc::fence_after_sync();
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
      uint8_t* stage = smem + C::kQOff + t * C::kTileBytes;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        // (a tile that visited no key never wrote its Õ columns: zeros)
        uint32_t orr[32];
        tc::tmem_ld32(o_addr + ch * 32, orr);
        tc::tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = nt > 0 ? pack_bf16x2(__uint_as_float(orr[2 * e]) * inv_l,
                                       __uint_as_float(orr[2 * e + 1]) * inv_l)
                         : 0u;
        // 32 columns = 4 chunks of 16 bytes; atom = ch / 2, chunk index in row = (ch % 2) * 4 + u
        uint8_t* atom = stage + (ch / 2) * (kBM * 128) + r * 128;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int chunk = (ch % 2) * 4 + u;
          *reinterpret_cast<uint4*>(atom + ((chunk ^ (r & 7)) * 16)) =
              make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
      if (lse != nullptr && row < Nq)
        lse[size_t(tile_bh(t)) * Nq + row] = l_run > 0.f ? (m_ref + __log2f(l_run)) * kLn2 : -INFINITY;
      fence_proxy_async_smem();
    } else if (!ok) {
      if (lane == 0) attn_flag_error(kErrTimeout);
      bars.abort = 1;
    }
    // Every warp of the warpgroup reaches this barrier, failed or not.
    named_bar_sync(1 + t, kBM);
    if (tile_rows && quarter == 0 && lane == 0 && !bars.abort) {
      uint8_t* stage = smem + C::kQOff + t * C::kTileBytes;
      for (int a = 0; a < C::kAtoms; ++a)
        tma_store_3d(&map_o, stage + a * (kBM * 128), 64 * a, tile_row0(t), tile_bh(t));
      tma_store_commit_and_wait();
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

template <int D, bool kGeneral>
cudaError_t launch_fwd_tc_d(const FwdArgs& a) {
  using C = FwdCfg<D>;
  CUtensorMap mq, mk, mv, mo;
  if (!make_map_bf16_3d(&mq, a.q, D, a.Nq, uint64_t(a.B) * a.Hq, kBM) ||
      !make_map_bf16_3d(&mk, a.k, D, a.Nk, uint64_t(a.B) * a.Hkv, kBN) ||
      !make_map_bf16_3d(&mv, a.v, D, a.Nk, uint64_t(a.B) * a.Hkv, kBN) ||
      !make_map_bf16_3d(&mo, a.o, D, a.Nq, uint64_t(a.B) * a.Hq, kBM))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(fwd_tc_kernel<D, kGeneral>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kDynSmem);
  if (e != cudaSuccess) return e;
  // Two query heads per CTA when they share a KV head (Hq / Hkv even),
  // else two row tiles of one head.
  const int head_pairs = (a.Hq / a.Hkv) % 2 == 0 ? 1 : 0;
  const int rows_per_cta = head_pairs ? kBM : 2 * kBM;
  const int n_qblk = (a.Nq + rows_per_cta - 1) / rows_per_cta;
  const long blocks = long(n_qblk) * a.B * (head_pairs ? a.Hq / 2 : a.Hq);
  if (blocks > 0x7fffffffL) return cudaErrorInvalidValue;
  // K/V re-read per head (pair) within an L2 group: a pair shares one KV head
  const long long kv_bytes = 4LL * a.Nk * D;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(blocks));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kDynSmem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fwd_tc_kernel<D, kGeneral>, mq, mk, mv, mo, a.lse, a.Hq, a.Hkv, a.Nq,
                            a.Nk, a.scale, a.mask, n_qblk,
                            order_group(a.mask.varies(), kv_bytes), head_pairs);
}

}  // namespace

cudaError_t launch_fwd_tc(const FwdArgs& a) {
  if (a.d == 64) return launch_fwd_tc64(a);   // persistent kernel (fwd_tc64.cu)
  const MaskSpec& m = a.mask;
  const bool plain = m.window_left < 0 && m.window_right <= 0 && m.n_global == 0 &&
                     m.row_kv_start == nullptr;   // no mask, or causal
  return plain ? launch_fwd_tc_d<128, false>(a) : launch_fwd_tc_d<128, true>(a);
}

}  // namespace attn

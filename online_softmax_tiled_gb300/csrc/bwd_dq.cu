// bf16 attention backward, the dQ pass, on the sm_103a tensor cores
// (tcgen05 + TMEM + TMA), d = 128.
//
// Recomputation backward of the "Flash Attention 2" post (ahmadsaeedzaidi.github.io
// feed), section "Flash Attention 2", "Recomputation in backward pass": S and
// P are rebuilt tile by tile from the saved row LSE, P = exp(scale·S - LSE).
// With dP = dO Vᵀ and the row term D = rowsum(dO ∘ O) (preprocess kernel),
// the Jacobian-vector product of the softmax-backward note
// (shreyansh26.github.io feed), section "Backpropagating Through Softmax",
// gives dS = P ∘ (dP - D), and dQ = scale·dS K.
//
// This pass owns one 128-row query tile (Q_i, dO_i resident in shared
// memory) and streams the key/value tiles that the tile sees, so dQ_i is
// accumulated in tensor memory and written once, in bf16: no float32
// accumulator, no atomics, no conversion pass. dK and dV come from the
// key-tile pass (bwd_tc.cu), which then needs no dQ work at all; the two
// passes recompute S and dP each (two of the five GEMMs twice) in exchange
// for full-width (N = 128) MMAs here and a short dependency chain there.
//
// GB300 mapping (rows = queries on the 128 TMEM lanes):
//  * S_j = Q_i K_jᵀ into S0/S1 (two buffers), dP_j = dO_i V_jᵀ into dP,
//    dQ += dS_j K_j into dQ (A = dS_j from tensor memory, bf16 pairs written
//    over the consumed S_j columns).
//  * Two softmax warpgroups split the 128 key columns of a step in halves;
//    thread = query row, so LSE and D are per-thread scalars.
//  * One converged MMA warp issues dP(j+1) as soon as dP(j) has been read,
//    then dQ(j) and S(j+2) once the softmax of step j has written dS(j).
//  * Every mbarrier wait is bounded (error word + abort flag + drain).

#include "common.cuh"
#include "launchers.h"
#include "mask.cuh"
#include "tc_ptx.cuh"
#include "tma_host.h"

namespace attn {

ATTN_DEFINE_ERROR_WORD(take_error_bwd_dq)

namespace {

constexpr int kBM = 128;            // query rows per CTA (TMEM lanes)
constexpr int kBN = 128;            // keys per step
constexpr int kD = 128;             // head dimension of this pass
constexpr int kThreads = 384;       // 12 warps
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr float kLog2e = 1.4426950408889634f;

struct DqCfg {
  static constexpr int kTile = kBM * kD * 2;               // 32 KB bf16 tile (Q, dO, K_j, V_j)
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kOffQ + kTile;
  static constexpr int kOffK = kOffDO + kTile;             // [kKStages]
  static constexpr int kOffV = kOffK + kKStages * kTile;   // [kVStages]
  static constexpr int kSmemBytes = kOffV + kVStages * kTile;
  static constexpr int kDynSmem = kSmemBytes + 1024;
  // tensor memory columns
  static constexpr uint32_t kColS0 = 0, kColS1 = 128, kColDP = 256, kColDQ = 384;
  static_assert(kDynSmem + 256 <= 232448, "shared-memory budget");
};

struct DqBars {
  uint64_t q_full;
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2], p_full[2];
  uint64_t dp_full, dp_free;
  uint64_t dq_done, mma_drain;
  uint32_t tmem_base;
  int abort;
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

// D = X Yᵀ over the head dimension into tensor memory at d_tmem: X and Y
// are 128 x d tiles (K-major, 128-byte swizzle, 64-column atoms of 128 rows)
// at shared addresses xa and ya. Called by every lane of the issuing warp.
ATTN_DEVINL void mma_xyt(uint32_t d_tmem, uint32_t xa, uint32_t ya) {
  constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, kBN, false, false);
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk) {
    const uint32_t off = (kk / 4) * (kBM * 128) + (kk % 4) * 32;
    tc::mma_ss_warp(d_tmem, tc::smem_desc(xa + off, 16, 1024, tc::kLayoutSW128),
                    tc::smem_desc(ya + off, 16, 1024, tc::kLayoutSW128), idesc, kk > 0);
  }
}

// dQ (+)= dS_j K_j into d_tmem: A = dS_j as bf16 pairs over the S_j columns
// at s_tmem (keys 64h .. 64h+63 of softmax warpgroup h at columns 64h ..
// 64h+31), B = K_j at shared address ka read MN-major. `first`: overwrite.
ATTN_DEVINL void mma_dsk(uint32_t d_tmem, uint32_t s_tmem, uint32_t ka, bool first) {
  constexpr uint32_t idesc = tc::idesc_bf16_f32(kBM, kD, false, true);
#pragma unroll
  for (int kk = 0; kk < kBN / 16; ++kk) {
    const uint32_t a_col = (kk / 4) * 64 + (kk % 4) * 8;
    tc::mma_ts_warp(d_tmem, s_tmem + a_col,
                    tc::smem_desc(ka + kk * 2048, kBN * 128, 1024, tc::kLayoutSW128), idesc,
                    (!first || kk > 0) ? 1u : 0u);
  }
}

// dS = P ∘ (dP - D) over one thread's 64 key columns of a step, as bf16
// pairs: P = exp2(S·scale·log2e - LSE·log2e) (c = scale·log2e, nl =
// -LSE·log2e, nd = -D), zero on keys the row does not see. Without a
// general mask (kGeneral = false) those are the keys past `limit` (and, with
// kLo, before `lo`: a window's left edge); with one,
// the clear bits of the 32-bit visibility masks vis0 (first 32 columns) and
// vis1. `masked` = false: every column is visible.
template <bool kGeneral, bool kLo = false>
ATTN_DEVINL void ds_pairs(const uint32_t (&sr)[64], const uint32_t (&dr)[64], float c, float nl,
                          float nd, bool masked, int key0, int limit, uint32_t vis0,
                          uint32_t vis1, uint32_t (&pk)[32], int lo = 0) {
  const f2 c2{c, c}, nl2{nl, nl}, nd2{nd, nd};
#pragma unroll
  for (int e = 0; e < 32; ++e) {
    const f2 x = fma2(f2{__uint_as_float(sr[2 * e]), __uint_as_float(sr[2 * e + 1])}, c2, nl2);
    f2 p{fast_exp2(x.x), fast_exp2(x.y)};
    if (masked) {
      if (kGeneral) {
        const uint32_t vis = e < 16 ? vis0 : vis1;
        if (!(vis & (1u << ((2 * e) & 31)))) p.x = 0.f;
        if (!(vis & (1u << ((2 * e + 1) & 31)))) p.y = 0.f;
      } else {
        if (key0 + 2 * e > limit || (kLo && key0 + 2 * e < lo)) p.x = 0.f;
        if (key0 + 2 * e + 1 > limit || (kLo && key0 + 2 * e + 1 < lo)) p.y = 0.f;
      }
    }
    const f2 dpd = add2(f2{__uint_as_float(dr[2 * e]), __uint_as_float(dr[2 * e + 1])}, nd2);
    const f2 ds = mul2(p, dpd);
    pk[e] = pack_bf16x2(ds.x, ds.y);
  }
}

// Key tiles a 128-row query tile starting at row_first visits (0 if the tile
// has no valid row); causal alignment is bottom-right.
ATTN_DEVINL int key_tiles_for(int row_first, int Nq, int Nk, int causal) {
  if (row_first >= Nq) return 0;
  const int nk_tiles = (Nk + kBN - 1) / kBN;
  if (!causal) return nk_tiles;
  const int row_last = min(row_first + kBM - 1, Nq - 1);
  return min(nk_tiles, (row_last + (Nk - Nq)) / kBN + 1);
}

// kGeneral = false: no mask or causal only; true: any MaskSpec (the key
// tiles of the plan, per-element visibility as 32-bit masks).
template <bool kGeneral>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dq_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
              const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
              const __grid_constant__ CUtensorMap map_dq, const float* __restrict__ lse,
              const float* __restrict__ row_term, int Hq, int Hkv, int Nq, int Nk, float scale,
              MaskSpec mask, int n_qt, int order_grp) {
  using C = DqCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ DqBars bars;
  __shared__ PlanSlots plan_slots;   // (no per-row slots: the dynamic buffers leave no room)

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Causal: heads in groups whose K/V fit in L2 together, and in a group the
  // query tiles with the most key steps first, so each group (and the grid)
  // ends with its shortest tiles. Otherwise head-major order.
  int bh, rank;
  grouped_tile_order(int(blockIdx.x), n_qt, int(gridDim.x) / n_qt, order_grp, bh, rank);
  const int qt = n_qt - 1 - rank;
  const int b = bh / Hq, h = bh % Hq;
  const int kvh = b * Hkv + h / (Hq / Hkv);
  const int row0 = qt * kBM;
  if (tid == 0) {
    plan_slots.init();
    bars.abort = 0;
    mbar_init(&bars.q_full, 1);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&bars.k_full[i], 1);
      mbar_init(&bars.k_empty[i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], 256);     // both softmax warpgroups
    }
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.dp_free, 256);
    mbar_init(&bars.dq_done, 1);
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

  // Key tiles to visit: 0 .. n-1 (no mask, causal), or the plan of the
  // mask (direct without row ranges; a reduction over the rows with them).
  int n;
  if (!kGeneral) {
    n = key_tiles_for(row0, Nq, Nk, mask.window_right == 0);
  } else {
    PlanSlots slots;
    if (mask.row_kv_start == nullptr) {
      slots = plan_slots_direct(mask, row0, kBM, 1, Nq, Nk);
      if (tid == 0) plan_slots = slots;   // the producer thread reads it back
    } else {
      if (warp >= 4 && warp < 8) {
        // (the ranges are inputs, complete before the plainly launched
        // preprocess started, and this grid starts after that)
        plan_add_rows(&plan_slots, row_keys(mask, b, row0 + (warp - 4) * 32 + lane, Nq, Nk), 0);
      }
      __syncthreads();
      slots = plan_slots;
    }
    n = slots.last[0] >= 0 ? make_plan(slots, kBN).count_upto(slots.last[0] / kBN) : 0;
  }
  auto key_tile = [&](int j) {
    return kGeneral ? make_plan_volatile(&plan_slots, kBN).tile(j) : j;
  };

  // Register split, set inside each role: 128 x 80 (TMA, MMA, idle warps) +
  // 256 x 208 (softmax) <= 384 x 168 registers the CTA is launched with.
  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    regs_dec<80>();
    if (lane == 0 && n > 0) {
      tc::tma_prefetch_desc(&map_k);
      tc::tma_prefetch_desc(&map_v);
      mbar_arrive_expect_tx(&bars.q_full, 2 * C::kTile);
      for (int a = 0; a < kD / 64; ++a) {
        tc::tma_load_3d(smem + C::kOffQ + a * (kBM * 128), &map_q, 64 * a, row0, bh, &bars.q_full);
        tc::tma_load_3d(smem + C::kOffDO + a * (kBM * 128), &map_do, 64 * a, row0, bh,
                        &bars.q_full);
      }
      int issued_k = 0, issued_v = 0;
      bool ok = true;
      for (int j = 0; j < n && ok; ++j) {
        const int sk = j % kKStages, sv = j % kVStages;
        if (j >= kKStages) ok = mbar_wait_bounded(&bars.k_empty[sk], ((j / kKStages) - 1) & 1, abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars.k_full[sk], C::kTile);
        for (int a = 0; a < kD / 64; ++a)
          tc::tma_load_3d(smem + C::kOffK + sk * C::kTile + a * (kBN * 128), &map_k, 64 * a,
                          key_tile(j) * kBN, kvh, &bars.k_full[sk]);
        ++issued_k;
        if (j >= kVStages) ok = mbar_wait_bounded(&bars.v_empty[sv], ((j / kVStages) - 1) & 1, abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars.v_full[sv], C::kTile);
        for (int a = 0; a < kD / 64; ++a)
          tc::tma_load_3d(smem + C::kOffV + sv * C::kTile + a * (kBN * 128), &map_v, 64 * a,
                          key_tile(j) * kBN, kvh, &bars.v_full[sv]);
        ++issued_v;
      }
      if (!ok) {
        attn_flag_error(kErrTimeout);
        bars.abort = 1;
        // Drain: every load this thread issued has landed before the CTA exits.
        mbar_wait_bounded(&bars.q_full, 0, nullptr);
        for (int j = max(0, issued_k - kKStages); j < issued_k; ++j)
          mbar_wait_bounded(&bars.k_full[j % kKStages], (j / kKStages) & 1, nullptr);
        for (int j = max(0, issued_v - kVStages); j < issued_v; ++j)
          mbar_wait_bounded(&bars.v_full[j % kVStages], (j / kVStages) & 1, nullptr);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop; one elected lane issues each MMA.
    regs_dec<80>();
    if (n > 0) {
      const uint32_t q_base = smem_u32(smem + C::kOffQ);
      const uint32_t do_base = smem_u32(smem + C::kOffDO);
      const uint32_t k_base = smem_u32(smem + C::kOffK);
      const uint32_t v_base = smem_u32(smem + C::kOffV);
      auto issue_qk = [&](uint32_t col, uint32_t xa, uint32_t ya) { mma_xyt(tmem + col, xa, ya); };
      auto s_col = [](int j) { return (j & 1) ? C::kColS1 : C::kColS0; };
      auto issue_s = [&](int j) {
        issue_qk(s_col(j), q_base, k_base + (j % kKStages) * C::kTile);
        tc::mma_commit_warp(&bars.s_full[j & 1]);
      };
      auto issue_dp = [&](int j) {
        issue_qk(C::kColDP, do_base, v_base + (j % kVStages) * C::kTile);
        tc::mma_commit_warp(&bars.dp_full);
        tc::mma_commit_warp(&bars.v_empty[j % kVStages]);   // V_j's only use
      };
      auto issue_dq = [&](int j) {
        mma_dsk(tmem + C::kColDQ, tmem + s_col(j), k_base + (j % kKStages) * C::kTile, j == 0);
        tc::mma_commit_warp(&bars.k_empty[j % kKStages]);   // K_j's last use
      };

      bool ok = mbar_wait_warp(&bars.q_full, 0, abort_flag);
      if (ok) ok = mbar_wait_warp(&bars.k_full[0], 0, abort_flag);
      if (ok) {
        tc::fence_after_sync();
        issue_s(0);
      }
      if (ok) ok = mbar_wait_warp(&bars.v_full[0], 0, abort_flag);
      if (ok) {
        tc::fence_after_sync();
        issue_dp(0);
      }
      if (ok && n > 1) {
        ok = mbar_wait_warp(&bars.k_full[1 % kKStages], 0, abort_flag);
        if (ok) {
          tc::fence_after_sync();
          issue_s(1);
        }
      }
      for (int j = 0; j < n && ok; ++j) {
        const int j1 = j + 1, j2 = j + 2;
        if (j1 < n) {
          // dP(j+1) as soon as the softmax has read dP(j) and V_{j+1} is in
          ok = mbar_wait2_warp(&bars.dp_free, j & 1, &bars.v_full[j1 % kVStages],
                               (j1 / kVStages) & 1, abort_flag);
          if (!ok) break;
          tc::fence_after_sync();
          issue_dp(j1);
        }
        // K_{j+2} has normally landed long before: probe it with p_full(j)
        const int ks = (j2 < n ? j2 : j) % kKStages;
        const uint32_t kp = j2 < n ? (j2 / kKStages) & 1 : (j / kKStages) & 1;
        ok = mbar_wait2_warp(&bars.p_full[j & 1], (j >> 1) & 1, &bars.k_full[ks], kp, abort_flag);
        if (!ok) break;
        tc::fence_after_sync();
        issue_dq(j);
        if (j2 < n) issue_s(j2);   // over the S_j columns, after dQ(j) has read dS_j (issue order)
      }
      if (!ok && lane == 0) {
        attn_flag_error(kErrTimeout);
        bars.abort = 1;
      }
      __syncwarp();
      tc::mma_commit_warp(&bars.dq_done);
      // Drain: every MMA this warp issued has completed before TMEM is freed.
      tc::mma_commit_warp(&bars.mma_drain);
      mbar_wait_warp(&bars.mma_drain, 0, nullptr);
    }
  } else if (warp < 4) {
    regs_dec<80>();                                // idle
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    regs_inc<208>();
    const int half = (warp - 4) >> 2;              // key columns [64·half, 64·half + 64)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;             // query row in the tile (TMEM lane)
    const int row = row0 + r;
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    const float c = scale * kLog2e;
    const bool row_in = row < Nq;
    const size_t ri = size_t(bh) * Nq + (row_in ? row : 0);
    // rows past Nq and rows that see no key (LSE = -inf): P = 0
    const float lse_r = row_in ? lse[ri] : -INFINITY;
    const float nl = lse_r == -INFINITY ? -INFINITY : -lse_r * kLog2e;   // -LSE·log2e
    const float nd = row_in ? -row_term[ri] : 0.f;                       // -D
    const int limit = mask.window_right == 0 ? min(Nk - 1, row + (Nk - Nq)) : Nk - 1;
    const RowKeys rk = kGeneral ? row_keys(mask, b, row, Nq, Nk) : RowKeys{1, 0, 1, 0};
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      if (!mbar_wait2_warp(&bars.s_full[j & 1], (j >> 1) & 1, &bars.dp_full, j & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const uint32_t s_addr = tmem + lane_base + ((j & 1) ? C::kColS1 : C::kColS0) + half * 64;
      uint32_t sr[64], dr[64];
      tc::tmem_ld32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tc::tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tc::tmem_ld32(tmem + lane_base + C::kColDP + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
      tc::tmem_ld32(tmem + lane_base + C::kColDP + half * 64 + 32,
                    *reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
      tc::tmem_ld_wait();
      tc::fence_before_sync();
      mbar_arrive(&bars.dp_free);                  // dP(j+1) may overwrite dP now

      // Keys this row does not see (past the end included) contribute
      // nothing: a single limit without a general mask, 32-bit visibility
      // masks with one.
      const int key0 = (kGeneral ? make_plan_volatile(&plan_slots, kBN).tile(j) : j) * kBN +
                       half * 64;
      const bool masked = kGeneral ? !rk.covers(key0, key0 + 63) : key0 + 63 > limit;
      const uint32_t vis0 = kGeneral && masked ? rk.bits(key0, 0) : 0xffffffffu;
      const uint32_t vis1 = kGeneral && masked ? rk.bits(key0, 1) : 0xffffffffu;
      uint32_t pk[32];                             // dS_j as bf16 pairs
      ds_pairs<kGeneral>(sr, dr, c, nl, nd, masked, key0, limit, vis0, vis1, pk);
      // over the S_j columns this warpgroup has just read
      tmem_st32(s_addr, pk);
      tc::tmem_st_wait();
      tc::fence_before_sync();
      mbar_arrive(&bars.p_full[j & 1]);
    }

    // Epilogue: dQ = scale·(Σ dS K) -> bf16 -> swizzled smem (the Q tile,
    // read by no MMA any more) -> TMA store; warpgroup `half` owns the
    // 64-dimension atom `half`.
    if (ok && n > 0) ok = mbar_wait_bounded(&bars.dq_done, 0, abort_flag);
    ok = __all_sync(0xffffffffu, ok);
    uint8_t* atom = smem + C::kOffQ + half * (kBM * 128) + r * 128;
    if (ok) {
      tc::fence_after_sync();
#pragma unroll
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t v[32];
        if (n > 0) {
          tc::tmem_ld32(tmem + lane_base + C::kColDQ + half * 64 + ch * 32, v);
          tc::tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) v[e] = 0u;  // no key is visible: dQ = 0
        }
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e)
          pk[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * scale, __uint_as_float(v[2 * e + 1]) * scale);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int chunk = ch * 4 + u;
          *reinterpret_cast<uint4*>(atom + ((chunk ^ (r & 7)) * 16)) =
              make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
      }
      fence_proxy_async_smem();
    } else {
      if (lane == 0) attn_flag_error(kErrTimeout);
      bars.abort = 1;
    }
    // Every warp of the warpgroup reaches this barrier, failed or not.
    named_bar_sync(1 + half, kBM);
    if (quarter == 0 && lane == 0 && !bars.abort && row0 < Nq) {
      tma_store_3d(&map_dq, smem + C::kOffQ + half * (kBM * 128), 64 * half, row0, bh);
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

// ----------------------------------------------------------------------------
// Persistent form (no mask, causal, or a window): one CTA per SM takes 128-row query
// tiles in turn, the first from its CTA index and the others from a device
// counter (dynamic scheduling: a CTA that finishes early takes the next
// tile, so the causal mix of long and short tiles balances). Tiles are
// numbered heaviest first within L2-sized head groups, as in the per-tile
// grid. The roles keep one global step count across tiles: the K/V rings
// (their own producer warp), the two S buffers and their barriers run on
// without a break, the next tile's Q is loaded as soon as the current
// tile's last S has read it and its dO once the last dP has (both
// prefetched into L2 well before), and the softmax warpgroups store the
// finished dQ rows straight to global memory while the tensor core starts
// the next tile.
// ----------------------------------------------------------------------------
struct PqBars {
  uint64_t q_full, q_empty, do_full, do_empty;
  uint64_t k_full[kKStages], k_empty[kKStages];
  uint64_t v_full[kVStages], v_empty[kVStages];
  uint64_t s_full[2], p_full[2];
  uint64_t dp_full, dp_free;
  uint64_t dq_done, mma_drain;
  uint64_t item_full[2], item_empty[2];
  int item[2];
  uint32_t tmem_base;
  int abort;
};

// Work item w (heaviest first within head groups) -> (b·Hq + h, query tile).
ATTN_DEVINL void dq_item(int w, int n_qt, int n_heads, int order_grp, int& bh, int& qt) {
  int rank;
  grouped_tile_order(w, n_qt, n_heads, order_grp, bh, rank);
  qt = n_qt - 1 - rank;
}

ATTN_DEVINL void tma_prefetch_l2_3d(const CUtensorMap* map, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
               ::"l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2) : "memory");
}

template <bool kWin>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dq_persistent_kernel(const __grid_constant__ CUtensorMap map_q,
                         const __grid_constant__ CUtensorMap map_k,
                         const __grid_constant__ CUtensorMap map_v,
                         const __grid_constant__ CUtensorMap map_do,
                         __nv_bfloat16* __restrict__ dq, const float* __restrict__ lse,
                         const float* __restrict__ row_term, int* __restrict__ counter, int Hq,
                         int Hkv, int Nq, int Nk, float scale, int causal, int win_left,
                         int win_right, int n_qt, int n_items, int order_grp) {
  using C = DqCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ PqBars bars;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_heads = int(n_items / n_qt);
  if (tid == 0) {
    bars.abort = 0;
    mbar_init(&bars.q_full, 1);
    mbar_init(&bars.q_empty, 1);
    mbar_init(&bars.do_full, 1);
    mbar_init(&bars.do_empty, 1);
    for (int i = 0; i < kKStages; ++i) {
      mbar_init(&bars.k_full[i], 1);
      mbar_init(&bars.k_empty[i], 1);
    }
    for (int i = 0; i < kVStages; ++i) {
      mbar_init(&bars.v_full[i], 1);
      mbar_init(&bars.v_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.s_full[i], 1);
      mbar_init(&bars.p_full[i], 256);     // both softmax warpgroups
      mbar_init(&bars.item_full[i], 1);    // the producer
      mbar_init(&bars.item_empty[i], 10);  // lane 0 of the K/V, MMA and 8 softmax warps
    }
    mbar_init(&bars.dp_full, 1);
    mbar_init(&bars.dp_free, 256);
    mbar_init(&bars.dq_done, 1);
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

  // The k-th work item of this CTA, published by the scheduler in slot k & 1;
  // w < 0 ends the loop. Consumers (K/V producer, MMA warp, softmax warps)
  // free the slot.
  auto read_item = [&](int k, bool& ok) {
    const int slot = k & 1;
    ok = mbar_wait_warp(&bars.item_full[slot], (k >> 1) & 1, abort_flag);
    const int w = ok ? *reinterpret_cast<volatile int*>(&bars.item[slot]) : -1;
    __syncwarp();
    if (lane == 0 && ok) mbar_arrive(&bars.item_empty[slot]);
    return w;
  };
  // Key tiles first .. first + n - 1 of query tile qt: from 0 (no mask,
  // causal), or (window: row i sees keys i' - win_left .. i' + win_right,
  // i' = i + Nk - Nq, a negative bound open) the tiles of the keys its rows
  // see; the launch guarantees at least one.
  auto tiles_of = [&](int qt, int& first) -> int {
    first = 0;
    if (!kWin) return key_tiles_for(qt * kBM, Nq, Nk, causal);
    const int q0 = qt * kBM;
    if (q0 >= Nq) return 0;
    const long long shift = (long long)Nk - Nq;
    const long long q1 = min(q0 + kBM - 1, Nq - 1);
    const long long lo = win_left >= 0 ? max(0LL, q0 + shift - win_left) : 0LL;
    const long long hi =
        win_right >= 0 ? min((long long)Nk - 1, q1 + shift + win_right) : (long long)Nk - 1;
    if (lo > hi) return 0;
    first = int(lo / kBN);
    return int(hi / kBN) - first + 1;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ scheduler, Q / dO producer
    // Takes the items, publishes them, and loads each item's Q and dO as
    // soon as the previous item's last S (for Q) and last dP (for dO) have
    // read theirs. The K/V ring has its own producer (warp 2), so those
    // loads never wait behind a Q or dO buffer.
    regs_dec<80>();
    if (lane == 0) {
      tc::tma_prefetch_desc(&map_q);
      tc::tma_prefetch_desc(&map_do);
      bool ok = true;
      int issued_q = 0, issued_do = 0;
      int next = int(blockIdx.x) < n_items ? int(blockIdx.x) : -1;
      for (int k = 0; ok; ++k) {
        const int w = next;
        const int slot = k & 1;
        if (k >= 2) ok = mbar_wait_bounded(&bars.item_empty[slot], ((k >> 1) - 1) & 1, abort_flag);
        if (!ok) break;
        bars.item[slot] = w;
        mbar_arrive(&bars.item_full[slot]);
        if (w < 0) break;
        int bh, qt;
        dq_item(w, n_qt, n_heads, order_grp, bh, qt);
        if (k >= 1) ok = mbar_wait_bounded(&bars.q_empty, (k - 1) & 1, abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars.q_full, C::kTile);
        for (int a = 0; a < kD / 64; ++a)
          tc::tma_load_3d(smem + C::kOffQ + a * (kBM * 128), &map_q, 64 * a, qt * kBM, bh,
                          &bars.q_full);
        ++issued_q;
        if (k >= 1) ok = mbar_wait_bounded(&bars.do_empty, (k - 1) & 1, abort_flag);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars.do_full, C::kTile);
        for (int a = 0; a < kD / 64; ++a)
          tc::tma_load_3d(smem + C::kOffDO + a * (kBM * 128), &map_do, 64 * a, qt * kBM, bh,
                          &bars.do_full);
        ++issued_do;
        // The next item, taken now so its Q and dO can be prefetched into L2
        // well before their load. The counter is zeroed by the preprocess,
        // complete before the key-tile pass let this grid start.
        next = int(gridDim.x) + atomicAdd(counter, 1);
        if (next >= n_items) next = -1;
        if (next >= 0) {
          int nbh, nqt;
          dq_item(next, n_qt, n_heads, order_grp, nbh, nqt);
          for (int a = 0; a < kD / 64; ++a) {
            tma_prefetch_l2_3d(&map_q, 64 * a, nqt * kBM, nbh);
            tma_prefetch_l2_3d(&map_do, 64 * a, nqt * kBM, nbh);
          }
        }
      }
      if (!ok) {
        attn_flag_error(kErrTimeout);
        bars.abort = 1;
        // Drain: every load this thread issued has landed before the CTA exits.
        if (issued_q > 0) mbar_wait_bounded(&bars.q_full, (issued_q - 1) & 1, nullptr);
        if (issued_do > 0) mbar_wait_bounded(&bars.do_full, (issued_do - 1) & 1, nullptr);
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ K/V producer
    regs_dec<80>();
    if (lane == 0) {
      tc::tma_prefetch_desc(&map_k);
      tc::tma_prefetch_desc(&map_v);
    }
    bool ok = true;
    int g = 0, issued_k = 0, issued_v = 0;
    for (int k = 0; ok; ++k) {
      const int w = read_item(k, ok);
      if (!ok || w < 0) break;
      if (lane == 0) {
        int bh, qt;
        dq_item(w, n_qt, n_heads, order_grp, bh, qt);
        const int kvh = (bh / Hq) * Hkv + (bh % Hq) / (Hq / Hkv);
        int first;
        const int n = tiles_of(qt, first);
        for (int j = 0; j < n && ok; ++j, ++g) {
          const int sk = g % kKStages, sv = g % kVStages;
          if (g >= kKStages) ok = mbar_wait_bounded(&bars.k_empty[sk], ((g / kKStages) - 1) & 1, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&bars.k_full[sk], C::kTile);
          for (int a = 0; a < kD / 64; ++a)
            tc::tma_load_3d(smem + C::kOffK + sk * C::kTile + a * (kBN * 128), &map_k, 64 * a,
                            (first + j) * kBN, kvh, &bars.k_full[sk]);
          ++issued_k;
          if (g >= kVStages) ok = mbar_wait_bounded(&bars.v_empty[sv], ((g / kVStages) - 1) & 1, abort_flag);
          if (!ok) break;
          mbar_arrive_expect_tx(&bars.v_full[sv], C::kTile);
          for (int a = 0; a < kD / 64; ++a)
            tc::tma_load_3d(smem + C::kOffV + sv * C::kTile + a * (kBN * 128), &map_v, 64 * a,
                            (first + j) * kBN, kvh, &bars.v_full[sv]);
          ++issued_v;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (!ok && lane == 0) {
      attn_flag_error(kErrTimeout);
      bars.abort = 1;
      // Drain: every load this thread issued has landed before the CTA exits.
      for (int t = max(0, issued_k - kKStages); t < issued_k; ++t)
        mbar_wait_bounded(&bars.k_full[t % kKStages], (t / kKStages) & 1, nullptr);
      for (int t = max(0, issued_v - kVStages); t < issued_v; ++t)
        mbar_wait_bounded(&bars.v_full[t % kVStages], (t / kVStages) & 1, nullptr);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs this loop; one elected lane issues each MMA.
    regs_dec<80>();
    const uint32_t q_base = smem_u32(smem + C::kOffQ);
    const uint32_t do_base = smem_u32(smem + C::kOffDO);
    const uint32_t k_base = smem_u32(smem + C::kOffK);
    const uint32_t v_base = smem_u32(smem + C::kOffV);
    auto s_col = [](int g) { return (g & 1) ? C::kColS1 : C::kColS0; };
    // `last`: the item's last step, whose S (dP) reads Q (dO) for the last time
    auto issue_s = [&](int g, bool last) {
      mma_xyt(tmem + s_col(g), q_base, k_base + (g % kKStages) * C::kTile);
      tc::mma_commit_warp(&bars.s_full[g & 1]);
      if (last) tc::mma_commit_warp(&bars.q_empty);
    };
    auto issue_dp = [&](int g, bool last) {
      mma_xyt(tmem + C::kColDP, do_base, v_base + (g % kVStages) * C::kTile);
      tc::mma_commit_warp(&bars.dp_full);
      tc::mma_commit_warp(&bars.v_empty[g % kVStages]);   // V's only use
      if (last) tc::mma_commit_warp(&bars.do_empty);
    };
    bool ok = true;
    int g0 = 0;                                   // global index of the item's first step
    for (int k = 0; ok; ++k) {
      const int w = read_item(k, ok);
      if (!ok || w < 0) break;
      int bh, qt;
      dq_item(w, n_qt, n_heads, order_grp, bh, qt);
      int first;
      const int n = tiles_of(qt, first);
      // Item start: S and dP of its first step, S of its second. The tensor
      // pipe runs this warp's MMAs in order: S(g0) overwrites the S buffer
      // only after the previous item's dQ has read dS from it, dP(g0) the dP
      // buffer only after the softmax has read the previous dP (its p_full
      // preceded that dQ), and dQ(g0) (overwrite) comes after the softmax
      // warpgroups have read the previous item's dQ out (before their p_full).
      ok = mbar_wait2_warp(&bars.q_full, k & 1, &bars.k_full[g0 % kKStages],
                           (g0 / kKStages) & 1, abort_flag);
      if (!ok) break;
      tc::fence_after_sync();
      issue_s(g0, n == 1);
      ok = mbar_wait2_warp(&bars.do_full, k & 1, &bars.v_full[g0 % kVStages],
                           (g0 / kVStages) & 1, abort_flag);
      if (!ok) break;
      tc::fence_after_sync();
      issue_dp(g0, n == 1);
      if (n > 1) {
        const int g1 = g0 + 1;
        ok = mbar_wait_warp(&bars.k_full[g1 % kKStages], (g1 / kKStages) & 1, abort_flag);
        if (!ok) break;
        tc::fence_after_sync();
        issue_s(g1, n == 2);
      }
      for (int j = 0; j < n && ok; ++j) {
        const int g = g0 + j;
        if (j + 1 < n) {
          // dP(g+1) as soon as the softmax has read dP(g) and V_{g+1} is in
          ok = mbar_wait2_warp(&bars.dp_free, g & 1, &bars.v_full[(g + 1) % kVStages],
                               ((g + 1) / kVStages) & 1, abort_flag);
          if (!ok) break;
          tc::fence_after_sync();
          issue_dp(g + 1, j + 1 == n - 1);
        }
        const int gk = j + 2 < n ? g + 2 : g;
        ok = mbar_wait2_warp(&bars.p_full[g & 1], (g >> 1) & 1, &bars.k_full[gk % kKStages],
                             (gk / kKStages) & 1, abort_flag);
        if (!ok) break;
        tc::fence_after_sync();
        mma_dsk(tmem + C::kColDQ, tmem + s_col(g), k_base + (g % kKStages) * C::kTile, j == 0);
        tc::mma_commit_warp(&bars.k_empty[g % kKStages]);   // K's last use
        if (j == n - 1) tc::mma_commit_warp(&bars.dq_done);
        if (j + 2 < n) issue_s(g + 2, j + 2 == n - 1);
      }
      g0 += n;
    }
    if (!ok && lane == 0) {
      attn_flag_error(kErrTimeout);
      bars.abort = 1;
    }
    __syncwarp();
    // Drain: every MMA this warp issued has completed before TMEM is freed.
    tc::mma_commit_warp(&bars.mma_drain);
    mbar_wait_warp(&bars.mma_drain, 0, nullptr);
  } else if (warp == 3) {
    regs_dec<80>();                                // idle
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    regs_inc<208>();
    const int half = (warp - 4) >> 2;              // key columns [64·half, 64·half + 64)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;             // query row in the tile (TMEM lane)
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    const float c = scale * kLog2e;
    bool ok = true;
    int g = 0;
    for (int k = 0; ok; ++k) {
      const int w = read_item(k, ok);
      if (!ok || w < 0) break;
      int bh, qt;
      dq_item(w, n_qt, n_heads, order_grp, bh, qt);
      int first;
      const int n = tiles_of(qt, first);
      const int row = qt * kBM + r;
      const bool row_in = row < Nq;
      const size_t ri = size_t(bh) * Nq + (row_in ? row : 0);
      // rows past Nq and rows that see no key (LSE = -inf): P = 0
      const float lse_r = row_in ? lse[ri] : -INFINITY;
      const float nl = lse_r == -INFINITY ? -INFINITY : -lse_r * kLog2e;   // -LSE·log2e
      const float nd = row_in ? -row_term[ri] : 0.f;                       // -D
      // keys this row sees: lo .. limit
      int limit = causal ? min(Nk - 1, row + (Nk - Nq)) : Nk - 1;
      int lo = 0;
      if (kWin) {
        const long long ip = (long long)row + Nk - Nq;
        limit = win_right >= 0 ? int(min((long long)Nk - 1, ip + win_right)) : Nk - 1;
        lo = win_left >= 0 ? int(max(0LL, min((long long)Nk, ip - win_left))) : 0;
      }
      for (int j = 0; j < n; ++j, ++g) {
        if (!mbar_wait2_warp(&bars.s_full[g & 1], (g >> 1) & 1, &bars.dp_full, g & 1,
                             abort_flag)) {
          ok = false;
          break;
        }
        tc::fence_after_sync();
        const uint32_t s_addr = tmem + lane_base + ((g & 1) ? C::kColS1 : C::kColS0) + half * 64;
        uint32_t sr[64], dr[64];
        tc::tmem_ld32(s_addr, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tc::tmem_ld32(s_addr + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tc::tmem_ld32(tmem + lane_base + C::kColDP + half * 64,
                      *reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
        tc::tmem_ld32(tmem + lane_base + C::kColDP + half * 64 + 32,
                      *reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
        tc::tmem_ld_wait();
        tc::fence_before_sync();
        mbar_arrive(&bars.dp_free);                  // dP(g+1) may overwrite dP now
        const int key0 = (first + j) * kBN + half * 64;
        uint32_t pk[32];                             // dS as bf16 pairs
        ds_pairs<false, kWin>(sr, dr, c, nl, nd, key0 + 63 > limit || (kWin && key0 < lo), key0,
                              limit, 0u, 0u, pk, lo);
        tmem_st32(s_addr, pk);                       // over the S columns just read
        tc::tmem_st_wait();
        tc::fence_before_sync();
        mbar_arrive(&bars.p_full[g & 1]);
      }
      if (!ok) break;
      // Epilogue: dQ = scale·(Σ dS K), warpgroup `half` owns dimensions
      // [64·half, 64·half + 64) of its row, stored as bf16 straight to
      // global memory (128 contiguous bytes per row).
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars.dq_done, k & 1, abort_flag));
      if (!ok) break;
      tc::fence_after_sync();
      uint32_t v[64];
      tc::tmem_ld32(tmem + lane_base + C::kColDQ + half * 64, *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      tc::tmem_ld32(tmem + lane_base + C::kColDQ + half * 64 + 32,
                    *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      tc::tmem_ld_wait();
      tc::fence_before_sync();   // the next item's first dQ overwrites these columns
      if (row_in) {
        uint4* dst = reinterpret_cast<uint4*>(dq + (size_t(bh) * Nq + row) * kD + half * 64);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            pk[e] = pack_bf16x2(__uint_as_float(v[8 * u + 2 * e]) * scale,
                                __uint_as_float(v[8 * u + 2 * e + 1]) * scale);
          dst[u] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
    }
    if (!ok) {
      if (lane == 0) attn_flag_error(kErrTimeout);
      bars.abort = 1;
    }
  }

  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_bwd_dq(const BwdArgs& a) {
  using C = DqCfg;
  if (a.d != kD) return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv, mdo, mdq;
  const uint64_t bhq = uint64_t(a.B) * a.Hq, bhk = uint64_t(a.B) * a.Hkv;
  if (!make_map_bf16_3d(&mq, a.q, kD, a.Nq, bhq, kBM) ||
      !make_map_bf16_3d(&mdo, a.dO, kD, a.Nq, bhq, kBM) ||
      !make_map_bf16_3d(&mk, a.k, kD, a.Nk, bhk, kBN) ||
      !make_map_bf16_3d(&mv, a.v, kD, a.Nk, bhk, kBN) ||
      !make_map_bf16_3d(&mdq, a.dq, kD, a.Nq, bhq, kBM))
    return cudaErrorInvalidValue;
  const MaskSpec& m = a.mask;
  const int n_qt = (a.Nq + kBM - 1) / kBM;
  const long items = long(n_qt) * a.B * a.Hq;
  if (items > 0x7fffffffL) return cudaErrorInvalidValue;
  const int order_grp = order_group(m.varies(), 4LL * a.Nk * kD);
  if (a.sched != nullptr && bwd_persistent(a.d, a.dt, m, a.Nq, a.Nk)) {
    // one CTA per SM, work from the counter; a programmatic dependent of the
    // key-tile pass, which lets it start once the preprocess (row term,
    // counter) is complete
    const bool win = bwd_dq_window(m);
    const auto kern = win ? bwd_dq_persistent_kernel<true> : bwd_dq_persistent_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         C::kDynSmem);
    if (e != cudaSuccess) return e;
    const int sms = device_sm_count();
    if (sms <= 0) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(unsigned(items < sms ? items : sms));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kDynSmem;
    cfg.stream = a.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mdo, static_cast<__nv_bfloat16*>(a.dq),
                              a.lse, static_cast<const float*>(a.row_term), a.sched, a.Hq, a.Hkv,
                              a.Nq, a.Nk, a.scale, a.causal, m.window_left, m.window_right, n_qt,
                              int(items), order_grp);
  }
  const bool general = !(m.window_left < 0 && m.window_right <= 0 && m.n_global == 0 &&
                         m.row_kv_start == nullptr);
  const auto kern = general ? bwd_dq_kernel<true> : bwd_dq_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::kDynSmem);
  if (e != cudaSuccess) return e;
  const long blocks = items;
  // Launched as a programmatic dependent of the key-tile pass: it reads only
  // the inputs and the preprocess's row term (the key-tile pass lets it
  // start only once every one of its CTAs has seen the preprocess
  // complete), so it needs no grid-dependency wait and fills the SMs that
  // the key-tile pass's last wave leaves idle.
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
  return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, mdo, mdq, a.lse,
                            static_cast<const float*>(a.row_term), a.Hq, a.Hkv, a.Nq, a.Nk,
                            a.scale, a.mask, n_qt, order_grp);
}

}  // namespace attn

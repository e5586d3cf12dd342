// bf16 attention backward on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Recomputation backward of the "Flash Attention 2" post
// (ahmadsaeedzaidi.github.io feed), section "Flash Attention 2",
// "Recomputation in backward pass": nothing N×N is stored by the forward; S
// and P are rebuilt tile by tile, P = exp(scale·S - LSE) from the saved row
// LSE. The softmax step is the Jacobian-vector product of the
// softmax-backward note (shreyansh26.github.io feed), section
// "Backpropagating Through Softmax": dS = P ∘ (dP - D) with dP = dO Vᵀ and
// the row term D = rowsum(dO ∘ O) (preprocess kernel). Then dV = Pᵀ dO,
// dK = scale·dSᵀ Q, dQ = scale·dS K.
//
// GB300 mapping:
//  * One CTA owns a 128-key tile K_j, V_j of one KV head (K-major in shared
//    memory, loaded once by TMA) and loops over every query head of its GQA
//    group and every query tile Q_i, dO_i (BQ rows) that sees those keys.
//  * Per step, with keys on the 128 TMEM lanes:
//      Sᵀ = K_j Q_iᵀ and dPᵀ = V_j dO_iᵀ          (tcgen05.mma, fp32 in TMEM)
//      Pᵀ = exp2(Sᵀ·scale·log2e - LSE·log2e), dSᵀ = Pᵀ ∘ (dPᵀ - D)
//                                     (two warpgroups, one key row per thread;
//                                      bf16 pairs back into TMEM)
//      dV_j += Pᵀ dO_i, dK_j += dSᵀ Q_i           (A from TMEM, accumulators in
//                                                  TMEM, d columns each)
//  * d = 128: that is all this pass does; dQ comes from the query-tile pass
//    (bwd_dq.cu). Two (Sᵀ, dPᵀ) buffers let one converged MMA warp issue
//    dV(s), dK(s) and then Sᵀ/dPᵀ(s+2) back to back while the softmax works
//    on step s+1: the tensor pipe runs the warp's MMAs in order, so step
//    s+2 overwrites Pᵀ/dSᵀ(s) only after dV(s), dK(s) have read them.
//  * d = 64 (BQ = 128, one buffer): dQ = dS K_j is computed here too, from a
//    dSᵀ copy in shared memory, and a third warpgroup adds it into a float32
//    accumulator with coalesced reductions; the attention-residuals lab
//    (manishklach.github.io) reduces multi-writer gradients the same way.
//  * dK and dV have one writer: the CTA stores them once, by TMA.
//  * Every mbarrier wait is bounded (error word + abort flag + drain).

#include "common.cuh"
#include "launchers.h"
#include "mask.cuh"
#include "tc_ptx.cuh"
#include "tma_host.h"

namespace attn {

ATTN_DEFINE_ERROR_WORD(take_error_bwd_tc)

namespace {

constexpr int kBK = 128;            // keys per CTA (TMEM lanes)
constexpr int kThreads = 512;       // 16 warps
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdCfg {
  static constexpr int BQ = (D == 128) ? 64 : 128;        // query rows per step
  // d = 64: dQ = dS K_j (M = BQ) is computed here and added into the float32
  // accumulator; d = 128: dQ comes from the query-tile pass.
  static constexpr bool kFusedDq = (D == 64);
  static constexpr int kPsBufs = kFusedDq ? 1 : 0;        // dSᵀ shared-memory buffers
  static constexpr int kQStages = kFusedDq ? 3 : 4;       // Q_i, dO_i, LSE, D ring
  // shared memory (bytes; every tile 1024-aligned)
  static constexpr int kKVTile = kBK * D * 2;             // K_j or V_j
  static constexpr int kQTile = BQ * D * 2;               // Q_i or dO_i
  static constexpr int kPsTile = kBK * BQ * 2;            // dSᵀ (bf16, the A operand of dQ)
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kOffK + kKVTile;
  static constexpr int kOffQ = kOffV + kKVTile;                      // [stage] Q, dO
  static constexpr int kOffP = kOffQ + kQStages * 2 * kQTile;       // [buf] dSᵀ
  // d = 128: the per-query terms enter the scores through the tensor core
  // (see bwd_issue_sdp): a ones tile A (128 x 16) and per stage a tile B
  // (BQ x 32: the bf16 parts of -LSE/scale, then of -D), both K-major
  // without swizzle. d = 64: the softmax reads -LSE·log2e and -D from
  // per-stage float vectors.
  static constexpr bool kAugTerms = !kFusedDq;
  static constexpr int kAugTile = 2 * BQ * 16 * 2;                  // B: 2·BQ rows x 16
  static constexpr int kOffOnes = kOffP + kPsBufs * kPsTile;        // A: 128 x 16 ones
  static constexpr int kOffAug = kOffOnes + (kAugTerms ? kBK * 16 * 2 : 0);   // [stage] B
  static constexpr int kOffVec = kOffAug + (kAugTerms ? kQStages * kAugTile : 0);
  static constexpr int kSmemBytes = kOffVec + (kAugTerms ? 0 : kQStages * 2 * BQ * 4);
  static constexpr int kDynSmem = kSmemBytes + 1024;
  // tensor memory columns. d = 128: two (Sᵀ, dPᵀ) buffers of 64 + 64
  // columns, dV, dK 128 each (2·128 + 2·128 = 512). d = 64: one (Sᵀ, dPᵀ)
  // buffer of 128 + 128, two dQ buffers of 64, dV, dK 64 each.
  static constexpr int kSdpBufs = kFusedDq ? 1 : 2;
  static constexpr uint32_t kSdpCols = 2 * BQ;
  static constexpr uint32_t kColDQ = kSdpBufs * kSdpCols;            // d = 64 only
  static constexpr uint32_t kDqCols = D;
  static constexpr uint32_t kColDV = kFusedDq ? kColDQ + 2 * kDqCols : kSdpBufs * kSdpCols;
  static constexpr uint32_t kColDK = kColDV + D;
  static_assert(kColDK + D <= 512, "TMEM budget");
  __host__ __device__ static constexpr uint32_t col_s(int b) { return b * kSdpCols; }
  __host__ __device__ static constexpr uint32_t col_dp(int b) { return b * kSdpCols + BQ; }
  // Pᵀ and dSᵀ (bf16 pairs) are written over the consumed Sᵀ / dPᵀ columns:
  // the warpgroup owning query columns [CW·h, CW·h + CW) stores its pairs at
  // columns [CW·h, CW·h + CW/2) of the buffer. Column of query q0 (multiple of 16):
  static constexpr int CW = BQ / 2;
  __host__ __device__ static constexpr uint32_t col_pair(int q0) {
    return (q0 / CW) * CW + (q0 % CW) / 2;
  }
  static_assert(kDynSmem + 256 <= 232448, "shared-memory budget (dynamic + static)");
};

struct BwdBars {
  uint64_t kv_full;
  uint64_t q_full[4], q_empty[4];
  uint64_t sdp_full[2], p_full[2];
  uint64_t ps_free[2];
  uint64_t dq_full[2], dq_free[2];
  uint64_t dkv_full, mma_drain;
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
ATTN_DEVINL void red_add_v4(float* addr, float a, float b, float c, float d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(addr), "f"(a), "f"(b),
               "f"(c), "f"(d) : "memory");
}

// Byte offset of element (row, col) of a bf16 tile stored as 64-column,
// 128-byte-swizzled atoms of `rows` rows each (the TMA SWIZZLE_128B layout).
ATTN_DEVINL uint32_t sw128_offset(int row, int col, int rows) {
  const int atom = col >> 6, c = col & 63;
  const int chunk = c >> 3;
  return uint32_t(atom * rows * 128 + row * 128 + ((chunk ^ (row & 7)) << 4) + ((c & 7) << 1));
}

// Sᵀ = K_j Q_iᵀ and dPᵀ = V_j dO_iᵀ of step s into (Sᵀ, dPᵀ) buffer s % NB
// (all operands K-major, 128-byte swizzle), then commit to `done`. Called by
// all lanes of the issuing warp.
template <int D>
ATTN_DEVINL void bwd_issue_sdp(uint8_t* smem, uint32_t tmem, int s, uint64_t* done) {
  using C = BwdCfg<D>;
  constexpr int BQ = C::BQ;
  constexpr uint32_t idesc_sdp = tc::idesc_bf16_f32(kBK, BQ, false, false);
  const int st = s % C::kQStages;
  const int b = s % C::kSdpBufs;
  const uint64_t k_km = tc::smem_desc(smem_u32(smem + C::kOffK), 16, 1024, tc::kLayoutSW128);
  const uint64_t v_km = tc::smem_desc(smem_u32(smem + C::kOffV), 16, 1024, tc::kLayoutSW128);
  const uint64_t qd = tc::smem_desc(smem_u32(smem + C::kOffQ + (st * 2) * C::kQTile), 16, 1024,
                                    tc::kLayoutSW128);
  const uint64_t dd = tc::smem_desc(smem_u32(smem + C::kOffQ + (st * 2 + 1) * C::kQTile), 16,
                                    1024, tc::kLayoutSW128);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t ka = ((kk / 4) * (kBK * 128) + (kk % 4) * 32) >> 4;   // K_j / V_j
    const uint64_t qb = ((kk / 4) * (BQ * 128) + (kk % 4) * 32) >> 4;    // Q_i / dO_i
    tc::mma_ss_warp(tmem + C::col_s(b), k_km + ka, qd + qb, idesc_sdp, kk > 0);
    tc::mma_ss_warp(tmem + C::col_dp(b), v_km + ka, dd + qb, idesc_sdp, kk > 0);
  }
  if (C::kAugTerms) {
    // Sᵀ += 1 · (-LSE/scale parts) and dPᵀ += 1 · (-D parts) in one K = 16
    // step over both (dPᵀ's columns follow Sᵀ's), so Pᵀ = exp2(Sᵀ·scale·
    // log2e) and dSᵀ = Pᵀ ∘ dPᵀ need no per-column loads. Layout: core
    // matrices of 8 rows x 16 bytes, 2 along K (lbo 128), 8-row groups every
    // 256 bytes; A = 128 x 16 ones, B = 2·BQ rows (the -LSE parts of the BQ
    // query rows, then their -D parts) x 16.
    constexpr uint32_t idesc_aug = tc::idesc_bf16_f32(kBK, 2 * BQ, false, false);
    static_assert(C::col_dp(0) == C::col_s(0) + BQ, "dPᵀ columns follow Sᵀ's");
    const uint64_t ones = tc::smem_desc(smem_u32(smem + C::kOffOnes), 128, 256, tc::kLayoutNone);
    const uint64_t aug = tc::smem_desc(smem_u32(smem + C::kOffAug + st * C::kAugTile), 128, 256,
                                       tc::kLayoutNone);
    tc::mma_ss_warp(tmem + C::col_s(b), ones, aug, idesc_aug, 1u);
  }
  tc::mma_commit_warp(done);
}

// One thread's share of a step's softmax backward, keys on the TMEM lanes:
// its key row (lane r, key index `key`) and its warpgroup's CW query
// columns from cbase, in (Sᵀ, dPᵀ) buffer b and Q stage st. Pᵀ =
// exp2(Sᵀ·scale·log2e - LSE·log2e) and dSᵀ = Pᵀ ∘ (dPᵀ - D) (d = 128: the
// -LSE/scale and -D terms are already in the scores; d = 64: read per
// column from the stage's vectors), as bf16 pairs written back over the
// columns just read (the A operands of dV and dK); d = 64 also writes a dSᵀ
// copy to shared memory for dQ. masked_row: some column may be hidden, then
// (no general mask) columns before qmin and every column of a key past Nk
// get P = 0, or (general mask) the columns whose row interval in keys_st
// does not contain the key; a window mask also hides the columns past qmax.
template <int D, bool kGeneral, bool kWin>
ATTN_DEVINL void bwd_pds_step(uint8_t* smem, uint32_t tmem, uint32_t lane_base, int b, int st,
                              int r, int key, bool key_in, int cbase, int qmin, int qmax,
                              bool masked_row,
                              float c, const int4* keys_st) {
  using C = BwdCfg<D>;
  constexpr int BQ = C::BQ;
  constexpr int CW = BQ / 2;
  const float* vec = reinterpret_cast<const float*>(smem + C::kOffVec + st * 2 * BQ * 4);
  uint8_t* dst = smem + C::kOffP;
  const f2 c2{c, c};
#pragma unroll
  for (int chunk = 0; chunk < CW / 32; ++chunk) {
    uint32_t sr[32], dr[32];
    const int col0 = cbase + chunk * 32;
    tc::tmem_ld32(tmem + lane_base + C::col_s(b) + col0, sr);
    tc::tmem_ld32(tmem + lane_base + C::col_dp(b) + col0, dr);
    tc::tmem_ld_wait();
    uint32_t pk[16], dk[16];                  // bf16 pairs of the 32 columns
#pragma unroll
    for (int g8 = 0; g8 < 4; ++g8) {          // 8 columns = one 16-byte chunk of dSᵀ
#pragma unroll
      for (int h4 = 0; h4 < 2; ++h4) {
        const int cb = g8 * 8 + h4 * 4;         // column within the 32
        // -LSE·log2e and -D per column (d = 64); d = 128 has them in the scores
        const float4 nl = C::kAugTerms ? make_float4(0.f, 0.f, 0.f, 0.f)
                                       : *reinterpret_cast<const float4*>(vec + col0 + cb);
        const float4 nd = C::kAugTerms ? make_float4(0.f, 0.f, 0.f, 0.f)
                                       : *reinterpret_cast<const float4*>(vec + BQ + col0 + cb);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int e = cb + 2 * u;
          f2 x = fma2(f2{__uint_as_float(sr[e]), __uint_as_float(sr[e + 1])}, c2,
                      u == 0 ? f2{nl.x, nl.y} : f2{nl.z, nl.w});
          f2 p{fast_exp2(x.x), fast_exp2(x.y)};
          if (masked_row) {
            const int col = col0 + e;
            if (kGeneral) {
              if (!load_row_keys(&keys_st[col]).visible(key)) p.x = 0.f;
              if (!load_row_keys(&keys_st[col + 1]).visible(key)) p.y = 0.f;
            } else {
              if (!key_in || col < qmin || (kWin && col > qmax)) p.x = 0.f;
              if (!key_in || col + 1 < qmin || (kWin && col + 1 > qmax)) p.y = 0.f;
            }
          }
          const f2 dpd = add2(f2{__uint_as_float(dr[e]), __uint_as_float(dr[e + 1])},
                              u == 0 ? f2{nd.x, nd.y} : f2{nd.z, nd.w});
          const f2 ds = mul2(p, dpd);
          pk[e >> 1] = pack_bf16x2(p.x, p.y);
          dk[e >> 1] = pack_bf16x2(ds.x, ds.y);
        }
      }
      const uint32_t off = sw128_offset(r, col0 + g8 * 8, kBK);
      if (C::kFusedDq)             // dSᵀ copy for dQ = dS K_j
        *reinterpret_cast<uint4*>(dst + off) =
          make_uint4(dk[4 * g8], dk[4 * g8 + 1], dk[4 * g8 + 2], dk[4 * g8 + 3]);
    }
    // Pᵀ and dSᵀ pairs over the columns just read (A operands of dV, dK)
    tc::tmem_st16(tmem + lane_base + C::col_s(b) + C::col_pair(col0), pk);
    tc::tmem_st16(tmem + lane_base + C::col_dp(b) + C::col_pair(col0), dk);
  }
}

// The (head, query tile) steps of one CTA: every query head of the group,
// and per head the query tiles from the first one that sees key k0 (causal)
// to the last, or (general masks) the query tiles listed in shared memory.
constexpr int kMaxListedQTiles = 1024;
struct StepPlan {
  int first_tile, tiles_per_head, group, n;
  const unsigned short* list;   // general masks: query tiles, ascending
  ATTN_DEVINL void init(int k0, int Nq, int Nk, int causal, int group_, int BQ) {
    group = group_;
    list = nullptr;
    const int nq_tiles = (Nq + BQ - 1) / BQ;
    first_tile = 0;
    if (causal) first_tile = max(0, k0 - (Nk - Nq)) / BQ;
    tiles_per_head = max(0, nq_tiles - first_tile);
    n = (k0 < Nk) ? tiles_per_head * group : 0;
  }
  // Keys [k0, k1] and a window mask (row i sees keys i' - wl .. i' + wr,
  // i' = i + Nk - Nq; a negative bound is open): the rows that see one of
  // the keys are i in [k0 - wr - shift, k1 + wl - shift], one run of tiles.
  ATTN_DEVINL void init_window(int k0, int k1, int Nq, int Nk, int wl, int wr, int group_,
                               int BQ) {
    group = group_;
    list = nullptr;
    const long long shift = (long long)Nk - Nq;
    long long lo = 0, hi = (long long)Nq - 1;
    if (wr >= 0) lo = max(lo, (long long)k0 - wr - shift);
    if (wl >= 0) hi = min(hi, (long long)k1 + wl - shift);
    first_tile = lo <= hi ? int(lo / BQ) : 0;
    tiles_per_head = lo <= hi ? int(hi / BQ) - first_tile + 1 : 0;
    n = (k0 < Nk) ? tiles_per_head * group : 0;
  }
  ATTN_DEVINL void init_listed(const unsigned short* list_, int count, int group_, int k0, int Nk) {
    group = group_;
    list = list_;
    first_tile = 0;
    tiles_per_head = count;
    n = (k0 < Nk) ? count * group : 0;
  }
  ATTN_DEVINL void at(int s, int& hh, int& qt) const {
    hh = s / tiles_per_head;
    qt = list != nullptr ? int(list[s % tiles_per_head]) : first_tile + s % tiles_per_head;
  }
};

// General masks: the query tiles (of BQ rows) with a row that sees a key of
// [k0, k1], listed ascending in `list`; returns their number. All threads of
// the CTA call this (it has two barriers).
template <int kThreadsT>
ATTN_DEVINL int list_query_tiles(const MaskSpec& m, int b, int k0, int k1, int Nq, int Nk, int BQ,
                                 uint32_t* bits, unsigned short* list, int* count) {
  const int tid = threadIdx.x;
  const int nq_tiles = (Nq + BQ - 1) / BQ;
  const int words = (nq_tiles + 31) / 32;
  for (int w = tid; w < words; w += kThreadsT) bits[w] = 0u;
  __syncthreads();
  for (int i = tid; i < Nq; i += kThreadsT) {
    const RowKeys r = row_keys(m, b, i, Nq, Nk);
    const bool sees = (r.lo1 <= r.hi1 && r.lo1 <= k1 && r.hi1 >= k0) ||
                      (r.lo2 <= r.hi2 && r.lo2 <= k1 && r.hi2 >= k0);
    if (sees) atomicOr(&bits[(i / BQ) >> 5], 1u << ((i / BQ) & 31));
  }
  __syncthreads();
  if (tid < 32) {
    // words <= kMaxListedQTiles / 32 = 32: one word per lane
    const uint32_t wbits = tid < words ? bits[tid] : 0u;
    const int cnt = __popc(wbits);
    int before = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, before, off);
      if (tid >= off) before += t;
    }
    before -= cnt;
    uint32_t x = wbits;
    for (int k = 0; x != 0u; ++k) {
      const int bit = __ffs(x) - 1;
      list[before + k] = (unsigned short)(tid * 32 + bit);
      x &= x - 1u;
    }
    if (tid == 31) *count = before + cnt;
  }
  __syncthreads();
  return *count;
}

// kGeneral = false: no mask, causal, or a window (query tiles and masked
// columns from the window's bounds); true: any MaskSpec (listed query tiles,
// per-step row key intervals, per-element masking of straddling steps).
template <int D, bool kGeneral, bool kWin>
__global__ void __launch_bounds__(kThreads, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
              const __grid_constant__ CUtensorMap map_v, const __grid_constant__ CUtensorMap map_do,
              const __grid_constant__ CUtensorMap map_dk, const __grid_constant__ CUtensorMap map_dv,
              const float* __restrict__ lse, const float* __restrict__ row_term,
              float* __restrict__ dq_acc, int Hq, int Hkv, int Nq, int Nk, float scale,
              MaskSpec mask, int n_ktiles, int order_grp) {
  using C = BwdCfg<D>;
  constexpr int BQ = C::BQ;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  __shared__ BwdBars bars;
  // general masks: the listed query tiles, and per stage the key intervals of
  // its rows plus whether every (row, key) pair of the step is visible
  __shared__ uint32_t qtile_bits[kGeneral ? kMaxListedQTiles / 32 : 1];
  __shared__ unsigned short qtile_list[kGeneral ? kMaxListedQTiles : 1];
  __shared__ int qtile_count;
  __shared__ int4 stage_keys[kGeneral ? C::kQStages : 1][kGeneral ? BQ : 1];
  __shared__ int stage_clean[kGeneral ? C::kQStages : 1];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Causal: KV heads in groups whose Q/dO fit in L2 together, and in a group
  // the key tiles with the most query steps (the first ones) first.
  // Otherwise head-major order.
  int bhkv, ktile;
  grouped_tile_order(int(blockIdx.x), n_ktiles, int(gridDim.x) / n_ktiles, order_grp, bhkv,
                     ktile);
  const int b = bhkv / Hkv, g = bhkv % Hkv;
  const int group = Hq / Hkv;
  const int k0 = ktile * kBK;
  StepPlan plan;
  if (kWin)
    plan.init_window(k0, min(k0 + kBK - 1, Nk - 1), Nq, Nk, mask.window_left, mask.window_right,
                     group, BQ);
  else if (!kGeneral)
    plan.init(k0, Nq, Nk, mask.window_right == 0, group, BQ);

  if (tid == 0) {
    bars.abort = 0;
    mbar_init(&bars.kv_full, 1);
    for (int i = 0; i < C::kQStages; ++i) {
      mbar_init(&bars.q_full[i], 1 + 32);   // TMA producer + 32 LSE/D loader lanes
      mbar_init(&bars.q_empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars.ps_free[i], 1);
      mbar_init(&bars.dq_full[i], 1);
      mbar_init(&bars.dq_free[i], 128);
    }
    mbar_init(&bars.sdp_full[0], 1);
    mbar_init(&bars.sdp_full[1], 1);
    // two p_full barriers (step parity): the softmax of step s+1 may finish
    // before the MMA thread has observed step s, which a single barrier would
    // alias; step s+2 cannot (its Sᵀ/dPᵀ are issued after step s is consumed)
    mbar_init(&bars.p_full[0], 256);     // both Pᵀ/dSᵀ warpgroups
    mbar_init(&bars.p_full[1], 256);
    mbar_init(&bars.dkv_full, 1);
    mbar_init(&bars.mma_drain, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&bars.tmem_base, 512);
    tc::tmem_relinquish();
  }
  if (C::kAugTerms) {
    // the ones tile (bf16 1.0 everywhere) and all-zero per-query tiles; the
    // loader later rewrites only the parts' 16-byte chunks
    uint32_t* ones = reinterpret_cast<uint32_t*>(smem + C::kOffOnes);
    for (int i = tid; i < kBK * 16 / 2; i += kThreads) ones[i] = 0x3F803F80u;
    uint32_t* aug = reinterpret_cast<uint32_t*>(smem + C::kOffAug);
    for (int i = tid; i < C::kQStages * C::kAugTile / 4; i += kThreads) aug[i] = 0u;
    fence_proxy_async_smem();   // read by the tensor core (async proxy)
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = bars.tmem_base;
  volatile int* abort_flag = &bars.abort;
  if (kGeneral) {
    // (the row ranges are inputs: complete before the plainly launched
    // preprocess started, and this grid starts after that)
    const int cnt = list_query_tiles<kThreads>(mask, b, k0, min(k0 + kBK - 1, Nk - 1), Nq, Nk,
                                               BQ, qtile_bits, qtile_list, &qtile_count);
    plan.init_listed(qtile_list, cnt, group, k0, Nk);
  }
  const int n = plan.n;

  // Register split, set inside each role (launch: 512 x 128): warps 0-3
  // (TMA, MMA, LSE/D loader, idle) 120; the two Pᵀ/dSᵀ warpgroups 136 each;
  // the dQ/epilogue warpgroup 120. 128 x (120 + 136 + 136 + 120) = 512 x 128.
  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer
    regs_dec<120>();
    if (lane == 0 && n > 0) {
      tc::tma_prefetch_desc(&map_q);
      tc::tma_prefetch_desc(&map_do);
      mbar_arrive_expect_tx(&bars.kv_full, 2 * C::kKVTile);
      for (int a = 0; a < D / 64; ++a) {
        tc::tma_load_3d(smem + C::kOffK + a * kBK * 128, &map_k, 64 * a, k0, bhkv, &bars.kv_full);
        tc::tma_load_3d(smem + C::kOffV + a * kBK * 128, &map_v, 64 * a, k0, bhkv, &bars.kv_full);
      }
      int issued = 0;
      bool ok = true;
      for (int s = 0; s < n && ok; ++s) {
        const int st = s % C::kQStages;
        if (s >= C::kQStages)
          ok = mbar_wait_bounded(&bars.q_empty[st], ((s / C::kQStages) - 1) & 1, abort_flag);
        if (!ok) break;
        int hh, qt;
        plan.at(s, hh, qt);
        const int bh = b * Hq + g * group + hh;
        mbar_arrive_expect_tx(&bars.q_full[st], 2 * C::kQTile);
        uint8_t* qs = smem + C::kOffQ + st * 2 * C::kQTile;
        for (int a = 0; a < D / 64; ++a) {
          tc::tma_load_3d(qs + a * BQ * 128, &map_q, 64 * a, qt * BQ, bh, &bars.q_full[st]);
          tc::tma_load_3d(qs + C::kQTile + a * BQ * 128, &map_do, 64 * a, qt * BQ, bh,
                          &bars.q_full[st]);
        }
        ++issued;
      }
      if (!ok) {
        attn_flag_error(kErrTimeout);
        bars.abort = 1;
        mbar_wait_bounded(&bars.kv_full, 0, nullptr);
        for (int s = max(0, issued - C::kQStages); s < issued; ++s)
          mbar_wait_bounded(&bars.q_full[s % C::kQStages], (s / C::kQStages) & 1, nullptr);
      }
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------- LSE / D loader
    regs_dec<120>();
    // Per step: -LSE·log2e and -D of the BQ query rows into the stage's
    // vectors; rows past Nq get -LSE·log2e = -inf (P = 0) and -D = 0.
    // The global loads of a step are issued before waiting for its stage to
    // free up, so their latency overlaps the wait.
    constexpr int kPer = BQ / 32;
    float nl[kPer], nd[kPer];
    // d = 128 launches as a programmatic dependent of the preprocess: the row
    // term D is read only once that grid has completed (a no-op otherwise).
    pdl_wait_primary();
    // The dQ pass that follows (d = 128) reads none of this kernel's outputs,
    // only the row term and its work counter, both written by the
    // preprocess: let it start on the SMs this grid's last wave leaves idle
    // once every CTA here has seen the preprocess complete.
    pdl_launch_dependents();
    auto fetch = [&](int s) {
      int hh, qt;
      plan.at(s, hh, qt);
      const size_t bh = size_t(b) * Hq + g * group + hh;
#pragma unroll
      for (int u = 0; u < kPer; ++u) {
        const int q = qt * BQ + u * 32 + lane;
        const bool in = q < Nq;
        const float l = in ? lse[bh * Nq + q] : -INFINITY;   // -inf: the row sees no key
        nl[u] = l == -INFINITY ? -INFINITY : -l * kLog2e;
        nd[u] = in ? -row_term[bh * Nq + q] : 0.f;
      }
    };
    bool ok = true;
    if (n > 0) fetch(0);
    for (int s = 0; s < n && ok; ++s) {
      const int st = s % C::kQStages;
      if (s >= C::kQStages)
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars.q_empty[st],
                                                       ((s / C::kQStages) - 1) & 1, abort_flag));
      if (!ok) break;
      if (C::kAugTerms) {
        // B row n (8-row group n/8 at 256 bytes, row n%8 at 16 bytes, first
        // K chunk) = three bf16 parts of -LSE/scale of query row n (exact
        // sum); B row BQ + n (2048 bytes further: BQ/8 groups) = three parts
        // of its -D; the second K chunk of every row stays zero
        uint8_t* aug = smem + C::kOffAug + st * C::kAugTile;
        const float inv_c = 1.f / (scale * kLog2e);
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int nrow = u * 32 + lane;
          uint8_t* rowp = aug + (nrow >> 3) * 256 + (nrow & 7) * 16;
          float vals[2] = {nl[u] * inv_c, nd[u]};
#pragma unroll
          for (int w = 0; w < 2; ++w) {
            const float v = vals[w];
            const __nv_bfloat16 h1 = __float2bfloat16_rn(v);
            // -inf (a row past Nq): -inf, 0, 0 (P = 0 without a NaN)
            const float r1 = isinf(v) ? 0.f : v - __bfloat162float(h1);
            const __nv_bfloat16 h2 = __float2bfloat16_rn(r1);
            const __nv_bfloat16 h3 = __float2bfloat16_rn(r1 - __bfloat162float(h2));
            const uint32_t w0 = uint32_t(__bfloat16_as_ushort(h1)) |
                                (uint32_t(__bfloat16_as_ushort(h2)) << 16);
            const uint32_t w1 = uint32_t(__bfloat16_as_ushort(h3));
            *reinterpret_cast<uint4*>(rowp + w * (BQ / 8) * 256) = make_uint4(w0, w1, 0u, 0u);
          }
        }
        fence_proxy_async_smem();   // read by the tensor core (async proxy)
      } else {
        float* vec = reinterpret_cast<float*>(smem + C::kOffVec + st * 2 * BQ * 4);
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          vec[u * 32 + lane] = nl[u];
          vec[BQ + u * 32 + lane] = nd[u];
        }
      }
      if (kGeneral) {
        // the key intervals of the step's rows; the step is clean if every
        // row sees every key of the tile (rows past Nq have P = 0 anyway)
        int hh, qt;
        plan.at(s, hh, qt);
        bool clean = k0 + kBK - 1 < Nk;
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
          const int q = qt * BQ + u * 32 + lane;
          const RowKeys rq = row_keys(mask, b, q, Nq, Nk);
          store_row_keys(&stage_keys[st][u * 32 + lane], rq);
          clean &= q >= Nq || rq.covers(k0, k0 + kBK - 1);
        }
        clean = __all_sync(0xffffffffu, clean);
        if (lane == 0) stage_clean[st] = clean ? 1 : 0;
        __syncwarp();
      }
      mbar_arrive(&bars.q_full[st]);
      if (s + 1 < n) fetch(s + 1);
    }
    if (!ok && lane == 0) {
      attn_flag_error(kErrTimeout);
      bars.abort = 1;
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp runs this loop; one elected lane issues each MMA.
    regs_dec<120>();
    {
      constexpr uint32_t idesc_kv = tc::idesc_bf16_f32(kBK, D, false, true);
      constexpr uint32_t idesc_dq = tc::idesc_bf16_f32(BQ, D, true, true);    // d = 64 only
      // Base descriptors; a descriptor's start-address field is (bytes >> 4),
      // so moving inside a tile adds (offset >> 4) to the 64-bit value.
      const uint64_t k_mn = tc::smem_desc(smem_u32(smem + C::kOffK), kBK * 128, 1024, tc::kLayoutSW128);
      auto q_mn = [&](int st, int which) {   // Q (0) or dO (1) of a stage, MN-major
        return tc::smem_desc(smem_u32(smem + C::kOffQ + (st * 2 + which) * C::kQTile), BQ * 128,
                             1024, tc::kLayoutSW128);
      };
      auto ps_mn = [&](int pb) {              // dSᵀ as an MN-major operand
        return tc::smem_desc(smem_u32(smem + C::kOffP + pb * C::kPsTile), kBK * 128, 1024,
                             tc::kLayoutSW128);
      };
      auto issue_sdp = [&](int s) { bwd_issue_sdp<D>(smem, tmem, s, &bars.sdp_full[s % C::kSdpBufs]); };

      // dV += Pᵀ dO ; dK += dSᵀ Q (; d = 64: dQ = dS K_j)   for step s (after its p_full)
      auto issue_grads = [&](int s) {
        const int st = s % C::kQStages;
        const int b = s % C::kSdpBufs;
        {
          // A = Pᵀ / dSᵀ from tensor memory (bf16 pairs), B = dO / Q MN-major
          const uint64_t dob = q_mn(st, 1), qb = q_mn(st, 0);
#pragma unroll
          for (int kk = 0; kk < BQ / 16; ++kk) {
            const uint32_t ac = C::col_pair(kk * 16);
            const uint64_t step = uint64_t(kk * 2048) >> 4;                      // 16 query rows
            const uint32_t acc = (s > 0 || kk > 0) ? 1u : 0u;
            tc::mma_ts_warp(tmem + C::kColDV, tmem + C::col_s(b) + ac, dob + step, idesc_kv, acc);
            tc::mma_ts_warp(tmem + C::kColDK, tmem + C::col_dp(b) + ac, qb + step, idesc_kv, acc);
          }
        }
        tc::mma_commit_warp(&bars.q_empty[st]);      // Q_i, dO_i, LSE, D of the stage consumed
        if (C::kFusedDq) {
          // dQ = dS K_j (A = dSᵀ MN-major over query atoms, B = K_j) into dQ buffer s & 1
          const int db = s & 1;
          const uint64_t a0 = ps_mn(0), b0 = k_mn;
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint64_t step = uint64_t(kk * 2048) >> 4;   // 16 keys down both operands
            tc::mma_ss_warp(tmem + C::kColDQ + db * C::kDqCols, a0 + step, b0 + step, idesc_dq,
                            kk > 0);
          }
          tc::mma_commit_warp(&bars.dq_full[db]);
          tc::mma_commit_warp(&bars.ps_free[0]);
        }
      };

      // Issue order: Sᵀ/dPᵀ of the first kSdpBufs steps, then per step s the
      // gradients of s followed by Sᵀ/dPᵀ(s + kSdpBufs) into the buffer step s
      // used. The tensor pipe runs this warp's MMAs in order, so the new
      // scores overwrite Pᵀ/dSᵀ(s) only after the gradients of s have read them.
      bool ok = true;
      if (n > 0) ok = mbar_wait_warp(&bars.kv_full, 0, abort_flag);
      for (int t = 0; t < min(n, C::kSdpBufs) && ok; ++t) {
        ok = mbar_wait_warp(&bars.q_full[t % C::kQStages], (t / C::kQStages) & 1, abort_flag);
        if (!ok) break;
        tc::fence_after_sync();
        issue_sdp(t);
      }
      for (int s = 0; s < n && ok; ++s) {
        // Q/dO of step s + kSdpBufs have normally landed long before: probe
        // them together with p_full(s)
        const int tq = s + C::kSdpBufs < n ? s + C::kSdpBufs : s;
        ok = mbar_wait2_warp(&bars.p_full[s & 1], (s >> 1) & 1, &bars.q_full[tq % C::kQStages],
                             (tq / C::kQStages) & 1, abort_flag);
        if (!ok) break;
        tc::fence_after_sync();
        if (C::kFusedDq && s >= 2) {   // dQ TMEM buffer s & 1 drained (step s-2)
          ok = mbar_wait_warp(&bars.dq_free[s & 1], ((s >> 1) - 1) & 1, abort_flag);
          if (!ok) break;
          tc::fence_after_sync();
        }
        issue_grads(s);
        const int t = s + C::kSdpBufs;
        if (t < n) issue_sdp(t);
      }
      if (!ok && lane == 0) {
        attn_flag_error(kErrTimeout);
        bars.abort = 1;
      }
      __syncwarp();
      tc::mma_commit_warp(&bars.dkv_full);
      tc::mma_commit_warp(&bars.mma_drain);
      mbar_wait_warp(&bars.mma_drain, 0, nullptr);
    }
  } else if (warp == 3) {
    regs_dec<120>();                                 // idle
  } else if (warp >= 4 && warp < 12) {
    // ---------------------------------------------------------- Pᵀ, dSᵀ warpgroups
    // Two warpgroups share the key rows (TMEM lanes) and split the BQ query
    // columns of each step in halves.
    regs_inc<136>();
    constexpr int CW = BQ / 2;                         // columns per warpgroup
    const int half = (warp - 4) >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;                 // key row in the tile (TMEM lane)
    const int key = k0 + r;
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    const float c = scale * kLog2e;
    const int shift = Nk - Nq;
    const int cbase = half * CW;
    bool ok = true;
    for (int s = 0; s < n; ++s) {
      const int st = s % C::kQStages;
      int hh, qt;
      plan.at(s, hh, qt);
      const int q0 = qt * BQ;
      const int b = s % C::kSdpBufs;
      bool w = mbar_wait2_warp(&bars.sdp_full[b], (s / C::kSdpBufs) & 1, &bars.q_full[st],
                               (s / C::kQStages) & 1, abort_flag);
      if (C::kFusedDq && s >= 1)   // the dSᵀ copy of step s-1 has been read by dQ(s-1)
        w = w && mbar_wait_bounded(&bars.ps_free[0], (s - 1) & 1, abort_flag);
      if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
      tc::fence_after_sync();
      const bool key_in = key < Nk;
      // first and last query columns (relative to q0) that see this key row
      // under a window mask (causal: the first only); general masks: the
      // step is masked unless every pair is visible
      int qmin = (!kGeneral && mask.window_right == 0) ? key - shift - q0 : -1;
      int qmax = INT_MAX;
      if (kWin) {
        qmin = mask.window_right >= 0
                   ? int(clampll((long long)key - mask.window_right - shift - q0, INT_MIN, INT_MAX))
                   : INT_MIN;
        qmax = mask.window_left >= 0
                   ? int(clampll((long long)key + mask.window_left - shift - q0, INT_MIN, INT_MAX))
                   : INT_MAX;
      }
      const bool masked_row = kGeneral ? stage_clean[st] == 0
                              : (!key_in || qmin > cbase || (kWin && qmax < cbase + CW - 1));
      bwd_pds_step<D, kGeneral, kWin>(smem, tmem, lane_base, b, st, r, key, key_in, cbase, qmin,
                                      qmax, masked_row, c,
                                      kGeneral ? &stage_keys[st][0] : nullptr);
      tc::tmem_st_wait();
      // generic-proxy writes of the dSᵀ copy -> tensor-core (async proxy) reads
      if (C::kFusedDq) fence_proxy_async_smem();
      tc::fence_before_sync();
      mbar_arrive(&bars.p_full[s & 1]);
    }
    if (!ok) {
      if (lane == 0) attn_flag_error(kErrTimeout);
      bars.abort = 1;
    }
  } else {
    // ---------------------------------------------------------- dQ drain, dK/dV epilogue
    regs_dec<120>();
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;                 // TMEM lane
    const uint32_t lane_base = uint32_t(quarter * 32) << 16;
    // d = 64: lane = query row, 64 columns = the dimensions; 16-byte
    // reductions into the float32 accumulator. d = 128 has no dQ here.
    bool ok = true;
    for (int s = 0; s < (C::kFusedDq ? n : 0); ++s) {
      const int db = s & 1;
      int hh, qt;
      plan.at(s, hh, qt);
      const size_t bh = size_t(b) * Hq + g * group + hh;
      const int q0 = qt * BQ;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&bars.dq_full[db], (s >> 1) & 1, abort_flag))) {
        ok = false;
        break;
      }
      tc::fence_after_sync();
      const uint32_t col0 = C::kColDQ + db * C::kDqCols;
      uint32_t v0[32], v1[32];
      tc::tmem_ld32(tmem + lane_base + col0, v0);
      tc::tmem_ld32(tmem + lane_base + col0 + 32, v1);
      tc::tmem_ld_wait();
      tc::fence_before_sync();
      mbar_arrive(&bars.dq_free[db]);
      if (q0 + r < Nq) {
        float* row = dq_acc + (bh * Nq + q0 + r) * D;
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          red_add_v4(row + e, __uint_as_float(v0[e]) * scale, __uint_as_float(v0[e + 1]) * scale,
                     __uint_as_float(v0[e + 2]) * scale, __uint_as_float(v0[e + 3]) * scale);
          red_add_v4(row + 32 + e, __uint_as_float(v1[e]) * scale,
                     __uint_as_float(v1[e + 1]) * scale, __uint_as_float(v1[e + 2]) * scale,
                     __uint_as_float(v1[e + 3]) * scale);
        }
      }
    }
    // dK = scale·(dSᵀ Q summed), dV = Pᵀ dO summed -> bf16 -> K_j / V_j tiles -> TMA store.
    if (ok && n > 0)
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars.dkv_full, 0, abort_flag));
    if (ok) {
      tc::fence_after_sync();
      uint8_t* kst = smem + C::kOffK;
      uint8_t* vst = smem + C::kOffV;
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t kr[32], vr[32];
        if (n > 0) {
          tc::tmem_ld32(tmem + lane_base + C::kColDK + ch * 32, kr);
          tc::tmem_ld32(tmem + lane_base + C::kColDV + ch * 32, vr);
          tc::tmem_ld_wait();
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) kr[e] = vr[e] = 0u;   // no query sees these keys
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t kp[4], vp[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int i = u * 8 + 2 * e;
            kp[e] = pack_bf16x2(__uint_as_float(kr[i]) * scale, __uint_as_float(kr[i + 1]) * scale);
            vp[e] = pack_bf16x2(__uint_as_float(vr[i]), __uint_as_float(vr[i + 1]));
          }
          const uint32_t off = sw128_offset(r, ch * 32 + u * 8, kBK);
          *reinterpret_cast<uint4*>(kst + off) = make_uint4(kp[0], kp[1], kp[2], kp[3]);
          *reinterpret_cast<uint4*>(vst + off) = make_uint4(vp[0], vp[1], vp[2], vp[3]);
        }
      }
      fence_proxy_async_smem();
    } else {
      if (lane == 0) attn_flag_error(kErrTimeout);
      bars.abort = 1;
    }
    // Every warp of the warpgroup reaches this barrier, failed or not.
    named_bar_sync(1, 128);
    if (quarter == 0 && lane == 0 && !bars.abort) {
      uint8_t* kst = smem + C::kOffK;
      uint8_t* vst = smem + C::kOffV;
      for (int a = 0; a < D / 64; ++a) {
        tma_store_3d(&map_dk, kst + a * kBK * 128, 64 * a, k0, bhkv);
        tma_store_3d(&map_dv, vst + a * kBK * 128, 64 * a, k0, bhkv);
      }
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

template <int D, bool kGeneral, bool kWin>
cudaError_t launch_bwd_tc_d(const BwdArgs& a) {
  using C = BwdCfg<D>;
  CUtensorMap mq, mk, mv, mdo, mdk, mdv;
  const uint64_t bhq = uint64_t(a.B) * a.Hq, bhk = uint64_t(a.B) * a.Hkv;
  if (!make_map_bf16_3d(&mq, a.q, D, a.Nq, bhq, C::BQ) ||
      !make_map_bf16_3d(&mdo, a.dO, D, a.Nq, bhq, C::BQ) ||
      !make_map_bf16_3d(&mk, a.k, D, a.Nk, bhk, kBK) ||
      !make_map_bf16_3d(&mv, a.v, D, a.Nk, bhk, kBK) ||
      !make_map_bf16_3d(&mdk, a.dk, D, a.Nk, bhk, kBK) ||
      !make_map_bf16_3d(&mdv, a.dv, D, a.Nk, bhk, kBK))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(bwd_tc_kernel<D, kGeneral, kWin>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kDynSmem);
  if (e != cudaSuccess) return e;
  const int n_ktiles = (a.Nk + kBK - 1) / kBK;
  // Q and dO of every query head of a KV head are re-read by all its key
  // tiles; groups of up to 64 MiB of them (measured: one group of 32 heads
  // of 2 MB ran 2 % faster than two groups of 16)
  const int order_grp = order_group(a.mask.varies(), 4LL * a.Nq * D * (a.Hq / a.Hkv), 64LL << 20);
  const long blocks = long(n_ktiles) * a.B * a.Hkv;
  if (blocks > 0x7fffffffL) return cudaErrorInvalidValue;
  if (C::kFusedDq) {
    // d = 64 adds into the accumulator the preprocess zeroes: plain launch
    bwd_tc_kernel<D, kGeneral, kWin><<<unsigned(blocks), kThreads, C::kDynSmem, a.stream>>>(
        mq, mk, mv, mdo, mdk, mdv, a.lse, a.row_term, a.dq_acc, a.Hq, a.Hkv, a.Nq, a.Nk,
        a.scale, a.mask, n_ktiles, order_grp);
    return cudaGetLastError();
  }
  // d = 128: programmatic dependent of the preprocess; only the LSE/D loader
  // waits for it (it reads the row term), the prologue (TMEM, K/V, Q/dO
  // loads) overlaps the preprocess's tail.
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
  return cudaLaunchKernelEx(&cfg, bwd_tc_kernel<D, kGeneral, kWin>, mq, mk, mv, mdo, mdk, mdv, a.lse,
                            static_cast<const float*>(a.row_term), a.dq_acc, a.Hq, a.Hkv, a.Nq,
                            a.Nk, a.scale, a.mask, n_ktiles, order_grp);
}

}  // namespace

cudaError_t launch_bwd_tc(const BwdArgs& a) {
  const MaskSpec& m = a.mask;
  // no mask or causal; a window (query tiles and masks from its bounds);
  // anything else through the listed query tiles and row intervals
  const bool causal_only = m.window_left < 0 && m.window_right <= 0 && m.n_global == 0 &&
                           m.row_kv_start == nullptr;
  const bool window = m.n_global == 0 && m.row_kv_start == nullptr;
  if (causal_only)
    return a.d == 64 ? launch_bwd_tc_d<64, false, false>(a) : launch_bwd_tc_d<128, false, false>(a);
  if (window)
    return a.d == 64 ? launch_bwd_tc_d<64, false, true>(a) : launch_bwd_tc_d<128, false, true>(a);
  return a.d == 64 ? launch_bwd_tc_d<64, true, false>(a) : launch_bwd_tc_d<128, true, false>(a);
}

}  // namespace attn

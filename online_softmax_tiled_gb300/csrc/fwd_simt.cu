// Float32-FFMA tiled attention forward (no tensor cores, no TF32).
//
// Serves float32 inputs, where the accuracy bar (1e-5 absolute against a
// float64 reference) rules out TF32 tensor-core products. The schedule is the
// inner loop of the "Flash Attention 2" post (ahmadsaeedzaidi.github.io feed),
// section "Flash Attention 2": one CTA owns a 64-row query tile Q_i and
// streams 64-row K_j, V_j tiles through shared memory, keeping the running
// row max m, denominator l and un-normalised output Õ on chip; Õ is divided
// by l once after the last tile. The probabilities of a tile are taken
// relative to the new running max directly, P̃ = exp(S - m_new), which equals
// the page's e^(m_ij - m_new)·exp(S - m_ij) with one exponential fewer.
// Masks (the post's section "Causal masking", option A): the CTA visits only
// the key tiles some of its rows see (mask.cuh) and masks the rest per
// element.

#include "common.cuh"
#include "launchers.h"
#include "mask.cuh"

namespace attn {
namespace {

constexpr int kBR = 64;     // query rows per CTA
constexpr int kBC = 64;     // keys per inner step
constexpr int kThreads = 128;

template <int D>
constexpr size_t simt_fwd_smem_bytes() {
  return sizeof(float) * (size_t(kBR) * (D + 1) + size_t(kBC) * (D + 1) + size_t(kBC) * D +
                          size_t(kBR) * (kBC + 1));
}

// Thread (ty, tx): ty = tid / 8 owns query rows 4*ty .. 4*ty+3 of the tile;
// tx = tid % 8 owns key columns tx + 8*c (c < 8) of S and output columns
// tx + 8*c (c < D/8) of Õ. The 8 threads of one row group are 8 consecutive
// lanes, so row reductions are 3 xor-shuffles.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
fwd_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                T* __restrict__ o, float* __restrict__ lse, int Hq, int Hkv, int Nq, int Nk,
                float scale, MaskSpec mask) {
  extern __shared__ float smem[];
  float* sQ = smem;                         // [kBR][D+1]
  float* sK = sQ + kBR * (D + 1);           // [kBC][D+1]
  float* sV = sK + kBC * (D + 1);           // [kBC][D]
  float* sP = sV + kBC * D;                 // [kBR][kBC+1]

  const int tid = threadIdx.x;
  const int ty = tid >> 3, tx = tid & 7;
  const int bh = blockIdx.y;
  const int b = bh / Hq, h = bh % Hq;
  const int g = h / (Hq / Hkv);
  const int row0 = blockIdx.x * kBR;

  const T* qh = q + (size_t(bh) * Nq) * D;
  const T* kh = k + (size_t(b * Hkv + g) * Nk) * D;
  const T* vh = v + (size_t(b * Hkv + g) * Nk) * D;

  for (int idx = tid; idx < kBR * D; idx += kThreads) {
    const int r = idx / D, c = idx % D;
    sQ[r * (D + 1) + c] = (row0 + r < Nq) ? to_f32(qh[size_t(row0 + r) * D + c]) : 0.f;
  }

  constexpr int DC = D / 8;
  float acc[4][DC];
  float m_run[4], l_run[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    m_run[i] = -INFINITY;
    l_run[i] = 0.f;
#pragma unroll
    for (int c = 0; c < DC; ++c) acc[i][c] = 0.f;
  }

  // Keys of this thread's four rows, and the key tiles any row of the CTA sees.
  __shared__ PlanSlots slots;
  if (tid == 0) slots.init();
  __syncthreads();
  RowKeys rk[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    rk[i] = row_keys(mask, b, row0 + 4 * ty + i, Nq, Nk);
    plan_add_rows(&slots, rk[i], 0);
  }
  __syncthreads();
  const KeyTilePlan plan = make_plan(slots, kBC);

  for (int jt = 0; jt < plan.total(); ++jt) {
    const int kv0 = plan.tile(jt) * kBC;
    __syncthreads();
    for (int idx = tid; idx < kBC * D; idx += kThreads) {
      const int r = idx / D, c = idx % D;
      const bool in = kv0 + r < Nk;
      sK[r * (D + 1) + c] = in ? to_f32(kh[size_t(kv0 + r) * D + c]) : 0.f;
      sV[r * D + c] = in ? to_f32(vh[size_t(kv0 + r) * D + c]) : 0.f;
    }
    __syncthreads();

    // Step 1: S_ij = scale · Q_i K_jᵀ (4 rows × 8 keys per thread)
    float s[4][8];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < 8; ++c) s[i][c] = 0.f;
#pragma unroll 4
    for (int t = 0; t < D; ++t) {
      float qv[4], kv[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) qv[i] = sQ[(4 * ty + i) * (D + 1) + t];
#pragma unroll
      for (int c = 0; c < 8; ++c) kv[c] = sK[(tx + 8 * c) * (D + 1) + t];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 8; ++c) s[i][c] = fmaf(qv[i], kv[c], s[i][c]);
    }

    // Steps 2-4: masked row max, probabilities, running statistics
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float mx = -INFINITY;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int col = kv0 + tx + 8 * c;
        const bool vis = rk[i].visible(col);   // also false past Nk
        s[i][c] = vis ? s[i][c] * scale : -INFINITY;
        mx = fmaxf(mx, s[i][c]);
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      const float m_new = fmaxf(m_run[i], mx);
      // alpha = exp(m_old - m_new); both -inf means nothing seen yet
      const float alpha = (m_run[i] == -INFINITY) ? 0.f : expf(m_run[i] - m_new);
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const float p = (s[i][c] == -INFINITY) ? 0.f : expf(s[i][c] - m_new);
        rs += p;
        sP[(4 * ty + i) * (kBC + 1) + tx + 8 * c] = p;
      }
      rs += __shfl_xor_sync(0xffffffffu, rs, 1);
      rs += __shfl_xor_sync(0xffffffffu, rs, 2);
      rs += __shfl_xor_sync(0xffffffffu, rs, 4);
      l_run[i] = alpha * l_run[i] + rs;
      m_run[i] = m_new;
#pragma unroll
      for (int c = 0; c < DC; ++c) acc[i][c] *= alpha;
    }
    __syncthreads();

    // Step 5: Õ += P̃ V_j
#pragma unroll 4
    for (int j = 0; j < kBC; ++j) {
      float pv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) pv[i] = sP[(4 * ty + i) * (kBC + 1) + j];
#pragma unroll
      for (int c = 0; c < DC; ++c) {
        const float vv = sV[j * D + tx + 8 * c];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[i][c] = fmaf(pv[i], vv, acc[i][c]);
      }
    }
  }

  // Safe normalisation O_i = Õ_i ⊘ l_i; LSE = m + ln l
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int row = row0 + 4 * ty + i;
    if (row >= Nq) continue;
    const bool empty = !(l_run[i] > 0.f);
    const float inv = empty ? 0.f : 1.f / l_run[i];
    T* orow = o + (size_t(bh) * Nq + row) * D;
#pragma unroll
    for (int c = 0; c < DC; ++c) orow[tx + 8 * c] = from_f32<T>(acc[i][c] * inv);
    if (lse != nullptr && tx == 0)
      lse[size_t(bh) * Nq + row] = empty ? -INFINITY : m_run[i] + logf(l_run[i]);
  }
}

template <typename T, int D>
cudaError_t launch_fwd_simt_t(const FwdArgs& a) {
  const size_t smem = simt_fwd_smem_bytes<D>();
  cudaError_t e = cudaFuncSetAttribute(fwd_simt_kernel<T, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  dim3 grid((a.Nq + kBR - 1) / kBR, a.B * a.Hq);
  fwd_simt_kernel<T, D><<<grid, kThreads, smem, a.stream>>>(
      static_cast<const T*>(a.q), static_cast<const T*>(a.k), static_cast<const T*>(a.v),
      static_cast<T*>(a.o), a.lse, a.Hq, a.Hkv, a.Nq, a.Nk, a.scale, a.mask);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_fwd_simt(const FwdArgs& a) {
  if (a.dt == ATTN_F32) {
    return a.d == 64 ? launch_fwd_simt_t<float, 64>(a) : launch_fwd_simt_t<float, 128>(a);
  }
  return a.d == 64 ? launch_fwd_simt_t<__nv_bfloat16, 64>(a)
                   : launch_fwd_simt_t<__nv_bfloat16, 128>(a);
}

}  // namespace attn

// Float32-FFMA tiled attention backward (no tensor cores).
//
// Recomputation backward of the "Flash Attention 2" post
// (ahmadsaeedzaidi.github.io feed), section "Flash Attention 2",
// "Recomputation in backward pass": S and P are rebuilt tile by tile from Q,
// K and the saved LSE (P = exp(scale·Q Kᵀ - LSE)) instead of being stored.
// The softmax step is the Jacobian-vector product of the softmax-backward
// note (shreyansh26.github.io feed), section "Backpropagating Through
// Softmax": dS = P ∘ (dP - D), with the row term D = rowsum(dO ∘ O) from the
// preprocess kernel.
//
// Schedule: one CTA owns a 32-key tile K_j, V_j of one KV head and loops over
// every query head of its GQA group and every 32-row query tile that can see
// those keys, accumulating dK_j and dV_j in registers (single writer, so no
// atomics for them); dQ_i += scale·dS K_j goes to the float32 accumulator
// with atomic adds (several key tiles write the same dQ rows).

#include "common.cuh"
#include "launchers.h"
#include "mask.cuh"

namespace attn {
namespace {

constexpr int kB = 32;        // keys per CTA and query rows per inner step
constexpr int kThreads = 128;

template <int D>
constexpr size_t simt_bwd_smem_bytes() {
  return sizeof(float) * (4 * size_t(kB) * (D + 1) + 2 * size_t(kB) * (kB + 1) + 2 * kB);
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
bwd_simt_kernel(const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
                const T* __restrict__ dO, const float* __restrict__ lse,
                const float* __restrict__ row_term, float* __restrict__ dq_acc,
                T* __restrict__ dk, T* __restrict__ dv, int Hq, int Hkv, int Nq, int Nk,
                float scale, MaskSpec mask) {
  extern __shared__ float smem[];
  float* sK = smem;                      // [kB][D+1]
  float* sV = sK + kB * (D + 1);         // [kB][D+1]
  float* sQ = sV + kB * (D + 1);         // [kB][D+1]
  float* sG = sQ + kB * (D + 1);         // dO tile [kB][D+1]
  float* sP = sG + kB * (D + 1);         // [kB][kB+1]   P[i][j]
  float* sS = sP + kB * (kB + 1);        // [kB][kB+1]   dS[i][j]
  float* sL = sS + kB * (kB + 1);        // LSE of the query tile
  float* sD = sL + kB;                   // row term of the query tile

  const int tid = threadIdx.x;
  const int bg = blockIdx.y;
  const int b = bg / Hkv, g = bg % Hkv;
  const int group = Hq / Hkv;
  const int kv0 = blockIdx.x * kB;
  const int shift = Nk - Nq;

  const T* kh = k + (size_t(bg) * Nk) * D;
  const T* vh = v + (size_t(bg) * Nk) * D;
  for (int idx = tid; idx < kB * D; idx += kThreads) {
    const int r = idx / D, c = idx % D;
    const bool in = kv0 + r < Nk;
    sK[r * (D + 1) + c] = in ? to_f32(kh[size_t(kv0 + r) * D + c]) : 0.f;
    sV[r * (D + 1) + c] = in ? to_f32(vh[size_t(kv0 + r) * D + c]) : 0.f;
  }

  constexpr int DC = D / 4;
  const int ti = tid >> 2;        // row index (query row for S/dQ, key row for dK/dV)
  const int tc = tid & 3;         // column phase
  float dk_acc[DC], dv_acc[DC];
#pragma unroll
  for (int c = 0; c < DC; ++c) dk_acc[c] = dv_acc[c] = 0.f;

  // First query row that can see key kv0: with a plain causal mask
  // (bottom-right alignment) the earlier tiles are skipped; other masks
  // visit every query tile and mask per pair.
  const bool plain_causal = mask.window_left < 0 && mask.window_right == 0 &&
                            mask.n_global == 0 && mask.row_kv_start == nullptr;
  int q_begin = 0;
  if (plain_causal) q_begin = max(0, kv0 - shift) / kB * kB;

  for (int hh = 0; hh < group; ++hh) {
    const int h = g * group + hh;
    const size_t bh = size_t(b) * Hq + h;
    const T* qh = q + bh * Nq * D;
    const T* gh = dO + bh * Nq * D;
    for (int q0 = q_begin; q0 < Nq; q0 += kB) {
      __syncthreads();
      for (int idx = tid; idx < kB * D; idx += kThreads) {
        const int r = idx / D, c = idx % D;
        const bool in = q0 + r < Nq;
        sQ[r * (D + 1) + c] = in ? to_f32(qh[size_t(q0 + r) * D + c]) : 0.f;
        sG[r * (D + 1) + c] = in ? to_f32(gh[size_t(q0 + r) * D + c]) : 0.f;
      }
      if (tid < kB) {
        const bool in = q0 + tid < Nq;
        sL[tid] = in ? lse[bh * Nq + q0 + tid] : 0.f;
        sD[tid] = in ? row_term[bh * Nq + q0 + tid] : 0.f;
      }
      __syncthreads();

      // S = scale·Q Kᵀ and dP = dO Vᵀ for row ti, keys tc + 4c
      float s[8], dp[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) s[c] = dp[c] = 0.f;
#pragma unroll 4
      for (int t = 0; t < D; ++t) {
        const float qv = sQ[ti * (D + 1) + t];
        const float gv = sG[ti * (D + 1) + t];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const int j = tc + 4 * c;
          s[c] = fmaf(qv, sK[j * (D + 1) + t], s[c]);
          dp[c] = fmaf(gv, sV[j * (D + 1) + t], dp[c]);
        }
      }
      const int row = q0 + ti;
      const float l_i = sL[ti], d_i = sD[ti];
      const RowKeys rk = row_keys(mask, b, row, Nq, Nk);   // nothing for rows past Nq
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const int j = tc + 4 * c;
        const int col = kv0 + j;
        const bool vis = rk.visible(col) && l_i != -INFINITY;
        const float p = vis ? expf(s[c] * scale - l_i) : 0.f;
        sP[ti * (kB + 1) + j] = p;
        sS[ti * (kB + 1) + j] = p * (dp[c] - d_i);
      }
      __syncthreads();

      // dV_j += Pᵀ dO_i ; dK_j += dSᵀ Q_i   (key row ti, columns tc + 4c)
#pragma unroll 2
      for (int i = 0; i < kB; ++i) {
        const float p = sP[i * (kB + 1) + ti];
        const float ds = sS[i * (kB + 1) + ti];
#pragma unroll
        for (int c = 0; c < DC; ++c) {
          dv_acc[c] = fmaf(p, sG[i * (D + 1) + tc + 4 * c], dv_acc[c]);
          dk_acc[c] = fmaf(ds, sQ[i * (D + 1) + tc + 4 * c], dk_acc[c]);
        }
      }
      // dQ_i += scale·dS K_j   (query row ti, columns tc + 4c)
      if (q0 + ti < Nq) {
        float* qrow = dq_acc + (bh * Nq + q0 + ti) * D;
#pragma unroll 4
        for (int c = 0; c < DC; ++c) {
          const int col = tc + 4 * c;
          float acc = 0.f;
#pragma unroll 8
          for (int j = 0; j < kB; ++j) acc = fmaf(sS[ti * (kB + 1) + j], sK[j * (D + 1) + col], acc);
          atomicAdd(qrow + col, acc * scale);
        }
      }
    }
  }

  if (kv0 + ti < Nk) {
    T* dkrow = dk + (size_t(bg) * Nk + kv0 + ti) * D;
    T* dvrow = dv + (size_t(bg) * Nk + kv0 + ti) * D;
#pragma unroll
    for (int c = 0; c < DC; ++c) {
      dkrow[tc + 4 * c] = from_f32<T>(dk_acc[c] * scale);
      dvrow[tc + 4 * c] = from_f32<T>(dv_acc[c]);
    }
  }
}

template <typename T, int D>
cudaError_t launch_bwd_simt_t(const BwdArgs& a) {
  const size_t smem = simt_bwd_smem_bytes<D>();
  cudaError_t e = cudaFuncSetAttribute(bwd_simt_kernel<T, D>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
  if (e != cudaSuccess) return e;
  dim3 grid((a.Nk + kB - 1) / kB, a.B * a.Hkv);
  bwd_simt_kernel<T, D><<<grid, kThreads, smem, a.stream>>>(
      static_cast<const T*>(a.q), static_cast<const T*>(a.k), static_cast<const T*>(a.v),
      static_cast<const T*>(a.dO), a.lse, a.row_term, a.dq_acc, static_cast<T*>(a.dk),
      static_cast<T*>(a.dv), a.Hq, a.Hkv, a.Nq, a.Nk, a.scale, a.mask);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_simt(const BwdArgs& a) {
  if (a.dt == ATTN_F32)
    return a.d == 64 ? launch_bwd_simt_t<float, 64>(a) : launch_bwd_simt_t<float, 128>(a);
  return a.d == 64 ? launch_bwd_simt_t<__nv_bfloat16, 64>(a)
                   : launch_bwd_simt_t<__nv_bfloat16, 128>(a);
}

}  // namespace attn

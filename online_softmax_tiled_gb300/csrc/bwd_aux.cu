// Backward helpers: the row-term preprocess and the dQ conversion.
//
// Row term. The softmax-backward note (shreyansh26.github.io feed), section
// "Backpropagating Through Softmax", writes the softmax Jacobian-vector
// product as P ∘ (dP - rowsum(P ∘ dP)). With O = P V and dP = dO Vᵀ,
// rowsum(P ∘ dP) = Σ_j P_ij Σ_c dO_ic V_jc = Σ_c dO_ic O_ic, so the row term
// D_i = rowsum(dO ∘ O) is computed here from O and dO in one streaming pass,
// before the main backward kernels run. When a pass adds dQ into the float32
// accumulator (d = 64, float32 inputs), the same pass zeroes it first; when
// the dQ pass is persistent, it zeroes its work counter.
//
// dQ conversion. After the main kernel, dQ = dtype(dQ_acc) (round to nearest
// even for bf16); the bf16 d = 128 path writes dQ directly and skips it.

#include "common.cuh"
#include "launchers.h"

namespace attn {
namespace {

// bf16 rows are read 16 bytes (8 values) per lane: D / 8 lanes cover a row,
// so a warp handles 32·8 / D rows at once. float32 rows: one warp per row,
// lane l handles columns l, l+32, ... (coalesced).
template <typename T, int D>
__global__ void __launch_bounds__(256)
bwd_preprocess_kernel(const T* __restrict__ o, const T* __restrict__ dO,
                      float* __restrict__ row_term, float* __restrict__ dq_acc,
                      int* __restrict__ sched, long rows) {
  // the key-tile pass (d = 128) may launch while this grid's last blocks run;
  // it waits for this grid before reading the row term, and lets the dQ
  // pass (which reads the row term and the work counter) start only after
  pdl_launch_dependents();
  if (sched != nullptr && blockIdx.x == 0 && threadIdx.x == 0) *sched = 0;
  const int lane = threadIdx.x & 31;
  if constexpr (sizeof(T) == 2) {
    constexpr int kLanesPerRow = D / 8;
    constexpr int kRowsPerWarp = 32 / kLanesPerRow;
    const long row = (long(blockIdx.x) * 8 + (threadIdx.x >> 5)) * kRowsPerWarp + lane / kLanesPerRow;
    const int c8 = (lane % kLanesPerRow) * 8;
    float acc = 0.f;
    if (row < rows) {
      const uint4 ov = *reinterpret_cast<const uint4*>(o + row * D + c8);
      const uint4 gv = *reinterpret_cast<const uint4*>(dO + row * D + c8);
      const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc = fmaf(bf16lo(ow[i]), bf16lo(gw[i]), acc);
        acc = fmaf(bf16hi(ow[i]), bf16hi(gw[i]), acc);
      }
    }
#pragma unroll
    for (int off = kLanesPerRow / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (row >= rows) return;
    if (lane % kLanesPerRow == 0) row_term[row] = acc;
    if (dq_acc == nullptr) return;     // no pass adds into the accumulator
    float4* qrow = reinterpret_cast<float4*>(dq_acc + row * D + c8);
    qrow[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    qrow[1] = make_float4(0.f, 0.f, 0.f, 0.f);
  } else {
    const long row = long(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (row >= rows) return;
    const T* orow = o + row * D;
    const T* grow = dO + row * D;
    float acc = 0.f;
#pragma unroll
    for (int c = lane; c < D; c += 32) acc = fmaf(to_f32(orow[c]), to_f32(grow[c]), acc);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) row_term[row] = acc;
    if (dq_acc == nullptr) return;     // no pass adds into the accumulator
    float* qrow = dq_acc + row * D;
#pragma unroll
    for (int c = lane; c < D; c += 32) qrow[c] = 0.f;
  }
}

template <typename T>
__global__ void __launch_bounds__(256)
bwd_convert_kernel(const float4* __restrict__ src, T* __restrict__ dst, long n4) {
  for (long i = long(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += long(gridDim.x) * blockDim.x) {
    const float4 x = src[i];
    T* d = dst + 4 * i;
    d[0] = from_f32<T>(x.x);
    d[1] = from_f32<T>(x.y);
    d[2] = from_f32<T>(x.z);
    d[3] = from_f32<T>(x.w);
  }
}

template <typename T>
cudaError_t launch_pre_t(const BwdArgs& a) {
  const long rows = long(a.B) * a.Hq * a.Nq;
  // 8 warps per block; a bf16 warp covers 256 / d rows, a float32 warp one row
  const long rows_per_block = sizeof(T) == 2 ? 8L * (256 / a.d) : 8L;
  const unsigned blocks = unsigned((rows + rows_per_block - 1) / rows_per_block);
  float* acc = a.zero_dq_acc ? a.dq_acc : nullptr;
  if (a.d == 64)
    bwd_preprocess_kernel<T, 64><<<blocks, 256, 0, a.stream>>>(
        static_cast<const T*>(a.o), static_cast<const T*>(a.dO), a.row_term, acc, a.sched, rows);
  else
    bwd_preprocess_kernel<T, 128><<<blocks, 256, 0, a.stream>>>(
        static_cast<const T*>(a.o), static_cast<const T*>(a.dO), a.row_term, acc, a.sched, rows);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_convert_t(const BwdArgs& a) {
  const long n4 = long(a.B) * a.Hq * a.Nq * a.d / 4;
  long blocks = (n4 + 255) / 256;
  if (blocks > 152L * 16) blocks = 152L * 16;
  bwd_convert_kernel<T><<<unsigned(blocks), 256, 0, a.stream>>>(
      reinterpret_cast<const float4*>(a.dq_acc), static_cast<T*>(a.dq), n4);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_preprocess(const BwdArgs& a) {
  return a.dt == ATTN_F32 ? launch_pre_t<float>(a) : launch_pre_t<__nv_bfloat16>(a);
}

cudaError_t launch_bwd_convert(const BwdArgs& a) {
  return a.dt == ATTN_F32 ? launch_convert_t<float>(a) : launch_convert_t<__nv_bfloat16>(a);
}

}  // namespace attn

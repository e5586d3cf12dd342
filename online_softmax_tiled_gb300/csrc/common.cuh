// Shared device/host helpers for the sm_103a attention kernels.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "attn.h"

#define ATTN_DEVINL __device__ __forceinline__

namespace attn {

// ----------------------------------------------------------------------------
// Error word. Each translation unit owns one (kernels in different units are
// compiled without relocatable device code, so a single shared __device__
// variable is not possible); the host polls all of them in attn_sync_status.
// Bits: 1 = a bounded wait ran out; 2 = an index read from device memory (a
// paged-decode length or block-table entry) was out of range.
// ----------------------------------------------------------------------------
enum : uint32_t { kErrTimeout = 1u, kErrBadIndex = 2u };

#define ATTN_DEFINE_ERROR_WORD(fn_name)                                          \
  static __device__ uint32_t g_attn_err_word;                                  \
  ATTN_DEVINL void attn_flag_error(uint32_t bits) {                            \
    atomicOr(&g_attn_err_word, bits);                                          \
  }                                                                            \
  uint32_t fn_name() {                                                         \
    uint32_t v = 0, zero = 0;                                                  \
    if (cudaMemcpyFromSymbol(&v, g_attn_err_word, sizeof(v)) != cudaSuccess)   \
      return 0xffffffffu;                                                      \
    if (v) cudaMemcpyToSymbol(g_attn_err_word, &zero, sizeof(zero));           \
    return v;                                                                  \
  }

// ----------------------------------------------------------------------------
// Small numeric helpers
// ----------------------------------------------------------------------------
ATTN_DEVINL float to_f32(float x) { return x; }
ATTN_DEVINL float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> ATTN_DEVINL T from_f32(float x);
template <> ATTN_DEVINL float from_f32<float>(float x) { return x; }
template <> ATTN_DEVINL __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// 2^x on the special-function unit (ex2.approx, relative error ~2^-22).
ATTN_DEVINL float fast_exp2(float x) {
  float y;
  asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Pack two floats into a bf16x2 word, round-to-nearest-even; `lo` goes to the
// low half (the lower-addressed element).
ATTN_DEVINL uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// Packed float32 pairs (sm_100 family FFMA2 / FADD2) and the 3-input max.
struct f2 {
  float x, y;
};
ATTN_DEVINL f2 fma2(f2 a, f2 b, f2 c) {
  uint64_t ra, rb, rc, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rc) : "f"(c.x), "f"(c.y));
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(rd) : "l"(ra), "l"(rb), "l"(rc));
  f2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}
ATTN_DEVINL f2 add2(f2 a, f2 b) {
  uint64_t ra, rb, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  f2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}
ATTN_DEVINL f2 mul2(f2 a, f2 b) {
  uint64_t ra, rb, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  f2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}
ATTN_DEVINL float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start once every CTA of the preceding kernel has executed
// launch_dependents (or exited); wait_primary blocks until that kernel has
// completed and its memory is visible. A kernel that does not read what the
// preceding kernel writes need not wait.
ATTN_DEVINL void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
ATTN_DEVINL void pdl_wait_primary() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Register re-split between warpgroups (all warps of a warpgroup execute it).
template <int N> ATTN_DEVINL void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N> ATTN_DEVINL void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

ATTN_DEVINL float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
ATTN_DEVINL float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

ATTN_DEVINL uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Upper bound on any single device-side wait. Legitimate waits in these
// kernels last microseconds; anything near this limit is a bug or a hang.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

// ----------------------------------------------------------------------------
// mbarrier helpers (shared::cta addresses as 32-bit)
// ----------------------------------------------------------------------------
ATTN_DEVINL uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

ATTN_DEVINL void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

ATTN_DEVINL void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

ATTN_DEVINL void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

ATTN_DEVINL void mbar_arrive(uint64_t* bar) {
  asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}"
               ::"r"(smem_u32(bar)) : "memory");
}

ATTN_DEVINL void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}"
      ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

ATTN_DEVINL bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Non-blocking probe of phase `parity` (for loops that poll several barriers).
ATTN_DEVINL bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Bounded wait for phase `parity` of `bar`. Returns false if it ran out (or if
// `*abort` was raised by another thread of the CTA while waiting). The clock
// is first read after 256 unsuccessful probes: reading %globaltimer costs
// about 100 cycles, which a wait that succeeds at once must not pay (measured
// on GB300: 119 vs 17 cycles per completed-phase wait).
ATTN_DEVINL bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort,
                                   uint64_t limit_ns = kWaitLimitNs) {
  uint64_t t0 = 0;
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0) {
      if (abort != nullptr && *abort) return false;
      const uint64_t now = global_timer_ns();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > limit_ns) {
        return false;
      }
    }
  }
}

// The same wait made by every lane of a converged warp; the result is the
// AND over the lanes, so the warp stays converged after it.
ATTN_DEVINL bool mbar_wait_warp(uint64_t* bar, uint32_t parity, volatile int* abort) {
  return __all_sync(0xffffffffu, mbar_wait_bounded(bar, parity, abort));
}

// Two waits made together by every lane of a converged warp. A probe of an
// mbarrier takes ~120 cycles to answer (measured on GB300) but probes that do
// not depend on each other overlap, so issuing both before using either
// makes a pair of completed phases cost one probe latency.
ATTN_DEVINL bool mbar_wait2_warp(uint64_t* b1, uint32_t p1, uint64_t* b2, uint32_t p2,
                                 volatile int* abort) {
  const bool r1 = mbar_try_wait(b1, p1);
  const bool r2 = mbar_try_wait(b2, p2);
  if (__all_sync(0xffffffffu, r1 && r2)) return true;
  return mbar_wait_warp(b1, p1, abort) && mbar_wait_warp(b2, p2, abort);
}

// ----------------------------------------------------------------------------
// Bulk (non-tensor) async copy global -> shared, completing on an mbarrier.
// Both addresses 16-byte aligned, size a multiple of 16.
// ----------------------------------------------------------------------------
// Order of the CTAs of a grid of n_tiles work tiles per head over n_heads
// heads: heads in groups of `group` (the last group may be smaller), and
// inside a group the tiles by rank, all heads of the group at rank 0, then
// at rank 1, ... A kernel maps rank 0 to its heaviest tile, so that within
// a group (sized on the host so that the group's re-read operands stay in
// L2) the longest CTAs start first and the group ends with the shortest;
// group = 1 is plain head-major order.
ATTN_DEVINL void grouped_tile_order(int block, int n_tiles, int n_heads, int group, int& head,
                                    int& rank) {
  const int g0 = (block / (n_tiles * group)) * group;
  const int hcount = min(group, n_heads - g0);
  const int idx = block - g0 * n_tiles;
  head = g0 + idx % hcount;
  rank = idx / hcount;
}

// 16-byte asynchronous copy global -> shared (cp.async, 16-byte aligned
// addresses), and an arrival on an mbarrier once every cp.async this thread
// issued before it has landed (the barrier's expected count includes it).
ATTN_DEVINL void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)),
               "l"(gmem_src) : "memory");
}
ATTN_DEVINL void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
ATTN_DEVINL void cp_async_mbar_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

ATTN_DEVINL void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

}  // namespace attn

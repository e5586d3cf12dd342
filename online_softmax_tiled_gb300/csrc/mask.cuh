// Attention masks on the device: which keys each query row sees, and which
// key tiles a group of rows must visit.
//
// Flash Attention 2 post (ahmadsaeedzaidi.github.io feed), section "Causal
// masking", option A and its "Why": an arbitrary mask (sliding window,
// document boundaries, prefix LM, ...) is a 0 / -inf term added to the scores
// before the online softmax; key tiles no row can see are skipped and the
// tiles that straddle a boundary are masked element by element.
//
// A MaskSpec (launchers.h) gives every row at most two visible key
// intervals: its window around position i' = i + Nk - Nq (bottom-right
// alignment, as for causal) clipped to the row's key range, and the global
// keys [0, n_global) clipped to the same range.
#pragma once

#include <climits>

#include "common.cuh"
#include "launchers.h"

namespace attn {

// Visible keys of one row: [lo1, hi1] ∪ [lo2, hi2], inclusive; an interval
// with lo > hi is empty. All bounds lie in [-1, Nk].
struct RowKeys {
  int lo1, hi1, lo2, hi2;
  ATTN_DEVINL bool visible(int j) const {
    return (j >= lo1 && j <= hi1) || (j >= lo2 && j <= hi2);
  }
  // every key of [j0, j1] visible
  ATTN_DEVINL bool covers(int j0, int j1) const {
    return (j0 >= lo1 && j1 <= hi1) || (j0 >= lo2 && j1 <= hi2);
  }
  ATTN_DEVINL bool empty() const { return lo1 > hi1 && lo2 > hi2; }
  // visibility of keys key0 + 32w .. key0 + 32w + 31 as a bit mask
  ATTN_DEVINL uint32_t bits(int key0, int w) const {
    const int base = key0 + 32 * w;
    return range_bits(lo1 - base, hi1 - base) | range_bits(lo2 - base, hi2 - base);
  }
  ATTN_DEVINL static uint32_t range_bits(int a, int b) {   // bits a..b of 0..31
    a = max(a, 0);
    b = min(b, 31);
    if (a > b) return 0u;
    const uint32_t ones = (b - a == 31) ? 0xffffffffu : ((1u << (b - a + 1)) - 1u);
    return ones << a;
  }
  // last visible key, -1 if none
  ATTN_DEVINL int last() const { return max(lo1 <= hi1 ? hi1 : -1, lo2 <= hi2 ? hi2 : -1); }
};

ATTN_DEVINL long long clampll(long long x, long long lo, long long hi) {
  return x < lo ? lo : (x > hi ? hi : x);
}

// Keys of query row i of batch entry b (rows past Nq see nothing). Reads the
// row's key range from global memory when the spec has one.
ATTN_DEVINL RowKeys row_keys(const MaskSpec& m, int b, int i, int Nq, int Nk) {
  RowKeys r{1, 0, 1, 0};
  if (i < 0 || i >= Nq) return r;
  long long s = 0, e = Nk;
  if (m.row_kv_start != nullptr) {
    s = clampll(m.row_kv_start[size_t(b) * Nq + i], 0, Nk);
    e = clampll(m.row_kv_end[size_t(b) * Nq + i], 0, Nk);
  }
  const long long ip = (long long)i + Nk - Nq;
  const long long wlo = m.window_left >= 0 ? ip - m.window_left : 0;
  const long long whi = m.window_right >= 0 ? ip + m.window_right : (long long)Nk - 1;
  r.lo1 = int(clampll(wlo > s ? wlo : s, 0, Nk));
  r.hi1 = int(clampll((whi < e - 1 ? whi : e - 1), -1, (long long)Nk - 1));
  r.lo2 = int(s);
  r.hi2 = int(clampll(((long long)m.n_global < e ? (long long)m.n_global : e) - 1, -1,
                      (long long)Nk - 1));
  return r;
}

// Per-CTA reduction of its rows' keys: the union of the window parts, of the
// global parts, and the last visible key of each query tile.
struct PlanSlots {
  int lo1, hi1, lo2, hi2;
  int last[2];
  ATTN_DEVINL void init() {
    lo1 = lo2 = INT_MAX;
    hi1 = hi2 = -1;
    last[0] = last[1] = -1;
  }
};

// The same slots computed directly, for a spec without row ranges: a row's
// window bounds grow with the row, so the rows whose window meets the keys
// are contiguous and their windows tile one interval; the global keys are
// the same for every row. `ntiles` query tiles of `tile_rows` rows from
// row_first.
ATTN_DEVINL PlanSlots plan_slots_direct(const MaskSpec& m, int row_first, int tile_rows,
                                        int ntiles, int Nq, int Nk) {
  PlanSlots ps;
  ps.init();
  const long long shift = (long long)Nk - Nq;
  const long long g_hi = ((long long)m.n_global < Nk ? (long long)m.n_global : Nk) - 1;
  for (int t = 0; t < ntiles; ++t) {
    const long long r0 = (long long)row_first + (long long)t * tile_rows;
    const long long r1 = min(r0 + tile_rows - 1, (long long)Nq - 1);
    if (r0 > r1) continue;
    long long a = r0 + shift, z = r1 + shift;                   // positions i'
    if (m.window_right >= 0) a = a > -(long long)m.window_right ? a : -(long long)m.window_right;
    if (m.window_left >= 0) {
      const long long top = (long long)Nk - 1 + m.window_left;
      z = z < top ? z : top;
    }
    long long last = -1;
    if (g_hi >= 0) {
      ps.lo2 = 0;
      ps.hi2 = max(ps.hi2, int(g_hi));
      last = g_hi;
    }
    if (a <= z) {
      const long long lo = m.window_left >= 0 ? clampll(a - m.window_left, 0, Nk) : 0;
      const long long hi = m.window_right >= 0 ? clampll(z + m.window_right, -1, (long long)Nk - 1)
                                               : (long long)Nk - 1;
      ps.lo1 = min(ps.lo1, int(lo));
      ps.hi1 = max(ps.hi1, int(hi));
      last = last > hi ? last : hi;
    }
    ps.last[t] = int(last);
  }
  return ps;
}

// All 32 lanes of a warp call this, each with the keys of one row of query
// tile t (the warp's rows all belong to tile t).
ATTN_DEVINL void plan_add_rows(PlanSlots* ps, const RowKeys& r, int t) {
  const bool e1 = r.lo1 <= r.hi1, e2 = r.lo2 <= r.hi2;
  const int lo1 = __reduce_min_sync(0xffffffffu, e1 ? r.lo1 : INT_MAX);
  const int hi1 = __reduce_max_sync(0xffffffffu, e1 ? r.hi1 : -1);
  const int lo2 = __reduce_min_sync(0xffffffffu, e2 ? r.lo2 : INT_MAX);
  const int hi2 = __reduce_max_sync(0xffffffffu, e2 ? r.hi2 : -1);
  const int lst = __reduce_max_sync(0xffffffffu, r.last());
  if ((threadIdx.x & 31) == 0) {
    atomicMin(&ps->lo1, lo1);
    atomicMax(&ps->hi1, hi1);
    atomicMin(&ps->lo2, lo2);
    atomicMax(&ps->hi2, hi2);
    atomicMax(&ps->last[t], lst);
  }
}

// The key tiles a CTA visits, in ascending order: [s0, s0 + n0) then
// [s1, s1 + n1). Each query tile visits a prefix of this sequence.
struct KeyTilePlan {
  int s0, n0, s1, n1;
  ATTN_DEVINL int tile(int j) const { return j < n0 ? s0 + j : s1 + (j - n0); }
  ATTN_DEVINL int total() const { return n0 + n1; }
  // length of the prefix that ends at the last tile with index <= last_tile
  ATTN_DEVINL int count_upto(int last_tile) const {
    const int c0 = min(n0, max(0, last_tile - s0 + 1));
    const int c1 = min(n1, max(0, last_tile - s1 + 1));
    return c0 + c1;
  }
};

ATTN_DEVINL KeyTilePlan make_plan(const PlanSlots& ps, int tile_keys) {
  int a0 = 0, a1 = -1, b0 = 0, b1 = -1;          // inclusive tile ranges
  if (ps.lo2 <= ps.hi2) { a0 = ps.lo2 / tile_keys; a1 = ps.hi2 / tile_keys; }
  if (ps.lo1 <= ps.hi1) { b0 = ps.lo1 / tile_keys; b1 = ps.hi1 / tile_keys; }
  KeyTilePlan p{0, 0, 0, 0};
  const bool ha = a0 <= a1, hb = b0 <= b1;
  if (ha && hb && b0 <= a1 + 1 && a0 <= b1 + 1) {   // overlapping or adjacent: one range
    p.s0 = min(a0, b0);
    p.n0 = max(a1, b1) - p.s0 + 1;
  } else if (ha && hb) {
    const bool a_first = a0 < b0;
    p.s0 = a_first ? a0 : b0;
    p.n0 = a_first ? a1 - a0 + 1 : b1 - b0 + 1;
    p.s1 = a_first ? b0 : a0;
    p.n1 = a_first ? b1 - b0 + 1 : a1 - a0 + 1;
  } else if (ha) {
    p.s0 = a0;
    p.n0 = a1 - a0 + 1;
  } else if (hb) {
    p.s0 = b0;
    p.n0 = b1 - b0 + 1;
  }
  return p;
}

// The same, read from shared slots at the point of use (volatile: nothing
// is kept in registers across a loop that is short of them).
ATTN_DEVINL KeyTilePlan make_plan_volatile(const PlanSlots* ps, int tile_keys) {
  const volatile PlanSlots* v = ps;
  PlanSlots c;
  c.lo1 = v->lo1;
  c.hi1 = v->hi1;
  c.lo2 = v->lo2;
  c.hi2 = v->hi2;
  return make_plan(c, tile_keys);
}

ATTN_DEVINL void store_row_keys(int4* slot, const RowKeys& r) {
  *slot = make_int4(r.lo1, r.hi1, r.lo2, r.hi2);
}
ATTN_DEVINL RowKeys load_row_keys(const int4* slot) {
  int4 x;
  asm volatile("ld.shared.v4.s32 {%0, %1, %2, %3}, [%4];"
               : "=r"(x.x), "=r"(x.y), "=r"(x.z), "=r"(x.w) : "r"(smem_u32(slot)));
  return RowKeys{x.x, x.y, x.z, x.w};
}

}  // namespace attn

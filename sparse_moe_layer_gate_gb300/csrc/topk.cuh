// Warp-level top-k helpers shared by the routing and planning kernels.
//
// Order of every selection: logit descending, lower expert id first on equal
// logits. Lane l of a warp owns the EPL consecutive experts [l*EPL, l*EPL+EPL).
#pragma once

#include <climits>

#include "common.cuh"

namespace epoch {

// Unsigned key with the order of the float value: positive values get the
// sign bit set, negative values are inverted. -0 is folded into +0 and NaN into
// -inf first, so equal values share a key and NaN ranks with -inf.
__device__ __forceinline__ unsigned order_key(float v) {
  const float c = v != v ? -INFINITY : v + 0.0f;
  const unsigned b = __float_as_uint(c);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(unsigned k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// The EPL consecutive logits [lane*EPL, lane*EPL + EPL) of one row of G
// (E floats); experts >= E get -inf. Vector loads when the row is 16-byte
// aligned. The row was written by an earlier kernel (read-only path).
template <int EPL>
__device__ __forceinline__ void lane_logits(const float *__restrict__ row, int E, float (&v)[EPL]) {
  const int e0 = lane_id() * EPL;
  if constexpr (EPL % 4 == 0) {
    if ((E & 3) == 0 && e0 + EPL <= E) {
      const float4 *src = reinterpret_cast<const float4 *>(row + e0);
#pragma unroll
      for (int q = 0; q < EPL / 4; ++q) {
        const float4 a = __ldg(src + q);
        v[4 * q] = a.x;
        v[4 * q + 1] = a.y;
        v[4 * q + 2] = a.z;
        v[4 * q + 3] = a.w;
      }
      return;
    }
  }
#pragma unroll
  for (int c = 0; c < EPL; ++c) v[c] = e0 + c < E ? __ldg(row + e0 + c) : -INFINITY;
}

// The general case of warp_topk, out of line (rare: more than 32 entries at or
// above the threshold, or k > 16): k rounds, each taking the best remaining
// lane best (a warp max, then the lowest lane holding it: lanes own ascending
// id ranges, so that is the lowest id). key: this lane's EPL keys (0:
// ineligible).
template <int EPL>
__device__ __noinline__ void warp_topk_rounds(const unsigned *key_in, int k, int *my_sel, float *my_val) {
  constexpr unsigned kAll = 0xffffffffu;
  const int lane = lane_id();
  unsigned key[EPL];
#pragma unroll
  for (int c = 0; c < EPL; ++c) key[c] = key_in[c];
  unsigned bk = key[0];
  int bc = 0;
#pragma unroll
  for (int c = 1; c < EPL; ++c)
    if (key[c] > bk) {
      bk = key[c];
      bc = c;
    }
  for (int j = 0; j < k; ++j) {
    const unsigned best = __reduce_max_sync(kAll, bk);
    const unsigned hold = __ballot_sync(kAll, bk == best && bk != 0u);
    const int win = __ffs(hold) - 1;  // -1: nothing eligible is left
    const int wsel = __shfl_sync(kAll, lane * EPL + bc, win < 0 ? 0 : win);
    if (lane == j && win >= 0) {
      *my_sel = wsel;
      *my_val = key_value(best);
    }
    if (lane == win) {  // take the entry, then this lane's next best
#pragma unroll
      for (int c = 0; c < EPL; ++c)
        if (c == bc) key[c] = 0u;
      bk = key[0];
      bc = 0;
#pragma unroll
      for (int c = 1; c < EPL; ++c)
        if (key[c] > bk) {
          bk = key[c];
          bc = c;
        }
    }
  }
}

// Top-k of one position by one warp. Lane l owns the EPL experts
// [l*EPL, l*EPL + EPL) with logits v; entries with ok false never win. Every
// comparison is on (order key desc, id asc). `scratch` is 32 entries of
// shared memory owned by the calling warp.
//
// Each lane finds its best entry, and the warp ranks the 32 lane bests. The
// k-th best lane best is a threshold: the k lanes ranked before it each hold
// an entry at or above it, so every one of the k best entries is at or above
// it too. Usually only a few entries pass; they are compacted into `scratch`,
// each is ranked against the others, and the entry of rank j lands in slot j.
// When more than 32 pass (values clustered in a few lanes) or k > 16, k rounds
// take the best remaining lane best instead (a warp max, then the lowest lane
// holding it: lanes own ascending id ranges, so that is the lowest id).
// On return, lane j < k holds selection j: *my_sel (expert; -1 if fewer than
// j + 1 entries are eligible) and *my_val (its logit, -0 read as +0 and NaN as
// -inf).
template <int EPL>
__device__ __forceinline__ void warp_topk(const float (&v)[EPL], const bool (&ok)[EPL], int k, int *my_sel,
                                          float *my_val, uint2 *scratch) {
  constexpr unsigned kAll = 0xffffffffu;
  const int lane = lane_id();
  unsigned key[EPL];  // 0: ineligible or taken (every real key, -inf's included, is above it)
#pragma unroll
  for (int c = 0; c < EPL; ++c) key[c] = ok[c] ? order_key(v[c]) : 0u;
  unsigned bk = key[0];  // this lane's best: highest key, lowest index on equal keys
  int bc = 0;
#pragma unroll
  for (int c = 1; c < EPL; ++c)
    if (key[c] > bk) {
      bk = key[c];
      bc = c;
    }
  *my_sel = -1;
  *my_val = -INFINITY;
  if (k <= 16) {
    int r = 0;  // rank of this lane's best among the lane bests
    // (a partly rolled loop: this code runs once per position and iteration,
    // usually from a cold instruction cache, where its size costs more than
    // the loop overhead)
#pragma unroll 4
    for (int i = 0; i < 32; ++i) {
      const unsigned o = __shfl_sync(kAll, bk, i);
      r += (o > bk) || (o == bk && i < lane);
    }
    const unsigned tb = __ballot_sync(kAll, r == k - 1 && bk != 0u);
    unsigned tkey = 0u;  // no threshold (fewer than k lanes hold an eligible entry): every eligible entry passes
    int tid = INT_MAX;
    if (tb) {
      const int tl = __ffs(tb) - 1;
      tkey = __shfl_sync(kAll, bk, tl);
      tid = __shfl_sync(kAll, lane * EPL + bc, tl);
    }
    unsigned cm = 0u;
#pragma unroll
    for (int c = 0; c < EPL; ++c)
      if (key[c] != 0u && (key[c] > tkey || (key[c] == tkey && lane * EPL + c <= tid))) cm |= 1u << c;
    const int cnt = __popc(cm);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(kAll, incl, o);
      if (lane >= o) incl += y;
    }
    const int total = __shfl_sync(kAll, incl, 31);
    if (total <= 32) {
      int pos = incl - cnt;
#pragma unroll
      for (int c = 0; c < EPL; ++c)
        if ((cm >> c) & 1u) scratch[pos++] = make_uint2(key[c], static_cast<unsigned>(lane * EPL + c));
      __syncwarp();
      const uint2 mine = lane < total ? scratch[lane] : make_uint2(0u, 0u);
      int rk = 0;
      for (int i = 0; i < total; ++i) {
        const uint2 o = scratch[i];
        rk += (o.x > mine.x) || (o.x == mine.x && o.y < mine.y);
      }
      __syncwarp();
      if (lane < total && rk < k) scratch[rk] = mine;
      __syncwarp();
      if (lane < k && lane < total) {
        const uint2 sel = scratch[lane];
        *my_sel = static_cast<int>(sel.y);
        *my_val = key_value(sel.x);
      }
      __syncwarp();
      return;
    }
  }
  warp_topk_rounds<EPL>(key, k, my_sel, my_val);
}

// Group-limited eligibility (the group rule of sigmoid routers): the E experts
// form n_group groups of gs = E / n_group consecutive ids. Lane l owns the
// EPL experts [l*EPL, l*EPL + EPL) with selection scores c (eligible where ok).
// A group's score is the sum of its two largest eligible c (one eligible: that
// c); groups with an eligible expert are ranked by score desc, lower group id
// first; the first topk_group are chosen, and further ones in rank order while
// the chosen groups hold fewer than k eligible experts. Clears ok[] outside
// the chosen groups. n_group <= 32.
template <int EPL>
__device__ __forceinline__ void warp_group_limit(const float (&c)[EPL], bool (&ok)[EPL], int E, int n_group,
                                                 int topk_group, int k) {
  constexpr unsigned kAll = 0xffffffffu;
  const int lane = lane_id(), gs = E / n_group;
  float my_score = -INFINITY;  // lane g < n_group: group g's score and eligible count
  int my_cnt = 0;
  for (int g = 0; g < n_group; ++g) {
    unsigned k1 = 0u, k2 = 0u;  // this lane's two best keys in group g (0: none)
    int cnt = 0;
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
      const int e = lane * EPL + q;
      if (ok[q] && e / gs == g) {
        const unsigned key = order_key(c[q]);
        ++cnt;
        if (key > k1) {
          k2 = k1;
          k1 = key;
        } else if (key > k2) {
          k2 = key;
        }
      }
    }
    const unsigned m1 = __reduce_max_sync(kAll, k1);
    const unsigned hold = __ballot_sync(kAll, k1 == m1 && k1 != 0u);
    const int wl = hold ? __ffs(hold) - 1 : -1;
    const unsigned m2 = __reduce_max_sync(kAll, lane == wl ? k2 : k1);  // the best key left
    const int n = static_cast<int>(__reduce_add_sync(kAll, static_cast<unsigned>(cnt)));
    if (lane == g) {
      my_cnt = n;
      my_score = m1 == 0u ? -INFINITY : (m2 == 0u ? key_value(m1) : key_value(m1) + key_value(m2));
    }
  }
  int r = 0;  // rank among the groups holding an eligible expert
#pragma unroll 4
  for (int i = 0; i < 32; ++i) {
    const float os = __shfl_sync(kAll, my_score, i);
    const int oc = __shfl_sync(kAll, my_cnt, i);
    r += (i < n_group && oc > 0) && (os > my_score || (os == my_score && i < lane));
  }
  int before = 0;  // eligible experts of the groups ranked before
#pragma unroll 4
  for (int i = 0; i < 32; ++i) {
    const int orr = __shfl_sync(kAll, r, i);
    const int oc = __shfl_sync(kAll, my_cnt, i);
    before += (i < n_group && oc > 0 && orr < r) ? oc : 0;
  }
  const unsigned chosen = __ballot_sync(kAll, lane < n_group && my_cnt > 0 && (r < topk_group || before < k));
#pragma unroll
  for (int q = 0; q < EPL; ++q) {
    const int e = lane * EPL + q;
    if (ok[q] && !((chosen >> (e / gs)) & 1u)) ok[q] = false;
  }
}

}  // namespace epoch

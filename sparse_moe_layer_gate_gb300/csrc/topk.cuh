// Warp-level top-k helpers shared by the routing and planning kernels.
//
// Order of every selection: logit descending, lower expert id first on equal
// logits. Lane l of a warp owns the EPL consecutive experts [l*EPL, l*EPL+EPL).
#pragma once

#include <climits>

#include "common.cuh"

namespace epoch {

// (value desc, id asc) order used for every top-k: true if (va, ia) ranks first.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Unsigned key with the order of the float value: positive values get the
// sign bit set, negative values are inverted. -0 is folded into +0 and NaN into
// -inf first, so keys compare exactly like ranks_before's values.
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

// Top-k of one position by one warp. Lane l owns the EPL experts
// [l*EPL, l*EPL + EPL) with logits v (ineligible ones must not win). Each lane
// sorts its own entries (value desc, id asc) with a bitonic network; then k
// rounds pick the best list head across the warp and pop it from its lane.
// On return, lane j < k holds selection j: *my_sel (expert) and *my_val (logit).
template <int EPL>
__device__ __forceinline__ void warp_topk(float (&v)[EPL], const bool (&ok)[EPL], int k, int *my_sel,
                                          float *my_val) {
  const int lane = lane_id();
  int id[EPL];
#pragma unroll
  for (int c = 0; c < EPL; ++c) {
    id[c] = ok[c] ? lane * EPL + c : INT_MAX;
    if (!ok[c]) v[c] = -INFINITY;
  }
  // bitonic sort, descending in (value, then lower id first)
#pragma unroll
  for (int size = 2; size <= EPL; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int j = i ^ stride;
        if (j > i) {
          const bool desc = (i & size) == 0;
          const bool swap = desc ? ranks_before(v[j], id[j], v[i], id[i]) : ranks_before(v[i], id[i], v[j], id[j]);
          if (swap) {
            const float tv = v[i];
            v[i] = v[j];
            v[j] = tv;
            const int ti = id[i];
            id[i] = id[j];
            id[j] = ti;
          }
        }
      }
    }
  }
  // k rounds over the lanes' list heads. A head's value is mapped to an
  // unsigned key whose order is the float order (-0 folded into +0 and NaN
  // into -inf, so equal values share a key); one warp max-reduction finds the
  // best value, a min-reduction the lowest id among the lanes holding it, and
  // the winning lane pops its head.
  *my_sel = -1;
  *my_val = -INFINITY;
  for (int j = 0; j < k; ++j) {
    const unsigned key = order_key(v[0]);
    const unsigned best = __reduce_max_sync(0xffffffffu, key);
    const int bi = __reduce_min_sync(0xffffffffu, key == best ? id[0] : INT_MAX);
    if (lane == j) {
      *my_sel = bi;
      *my_val = key_value(best);
    }
    if (id[0] == bi) {
#pragma unroll
      for (int c = 0; c + 1 < EPL; ++c) {
        v[c] = v[c + 1];
        id[c] = id[c + 1];
      }
      v[EPL - 1] = -INFINITY;
      id[EPL - 1] = INT_MAX;
    }
  }
}

}  // namespace epoch

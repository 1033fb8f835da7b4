// Per-position classification and support-restricted top-k of one iteration,
// shared by the tcgen05 gate's epilogue (bf16 layers) and the select kernel
// that follows the FFMA gate (fp32 layers).
//
// Walk-through page "Epoch 完全拆解:把扩散块编译成稀疏 MoE 服务单元":
//  - section "Liveness-Shard Parallelism": Z_i (stable decoded positions whose
//    cached routed row is reused), N_i = D_i \ D_{i-1} (newly decoded), and the
//    fresh set F_i = everything else (still-live Mask positions, new commits,
//    decoded rows without a cached row or with one at least R iterations old);
//  - section "Expert Atlas", step three: top-k of G[t, .] restricted to the
//    block's support, weights from the selected logits;
//  - sections "Two Clocks" and "cold、hot-update、hot-skip": any liveness
//    anomaly (a decoded position turning live) sends the iteration back to
//    the full fresh path with every expert eligible.
#pragma once

#include <climits>

#include "common.cuh"
#include "layer.h"
#include "topk.cuh"

namespace epoch {

// Position categories; a code packs the category with three flag bits.
enum Category { C_LIVE = 0, C_NEW, C_MISS, C_STALE, C_REUSE };
constexpr int kCodeLive = 16;  // treated as live (live flag set, or decoded flag clear)
constexpr int kCodeBad = 32;   // contradictory flags (both or neither set)
constexpr int kCodeAnom = 64;  // decoded at the previous iteration, live now

// Category of a position from its flags and the previous iteration's state:
// live (still Mask, or not decoded), newly decoded, decoded without a row,
// decoded with a row at least R iterations old, or stable decoded (reuses its
// cached row).
__device__ __forceinline__ int classify_code(const Dims &d, bool lv, bool dc, bool prev, int stamp) {
  const bool il = lv || !dc;
  const int flags = (il ? kCodeLive : 0) | (lv == dc ? kCodeBad : 0) | (il && prev ? kCodeAnom : 0);
  if (il) return C_LIVE | flags;
  if (!prev) return C_NEW | flags;
  if (stamp < 0) return C_MISS | flags;
  if (d.R != INT_MAX && d.iter - stamp >= d.R) return C_STALE | flags;
  return C_REUSE | flags;
}

// 0x80 in every byte of x that is zero, 0 elsewhere.
__device__ __forceinline__ uint32_t zero_bytes(uint32_t x) {
  const uint32_t t = (x & 0x7F7F7F7Fu) + 0x7F7F7F7Fu;
  return ~(t | x | 0x7F7F7F7Fu);
}

// True if any position turned from decoded to live (decoded at the previous
// iteration, now live or not decoded), over this thread's share of the
// positions: thread `part` of `parts` takes 4-position words part, part +
// parts, ... (the caller ORs the answers of all its threads). The flags are
// read four at a time, with no branch between the loads.
__device__ __forceinline__ bool any_anomaly(const Dims &d, const uint8_t *__restrict__ live,
                                            const uint8_t *__restrict__ decoded,
                                            const uint8_t *__restrict__ prev_old, int part, int parts) {
  const bool vec = ((reinterpret_cast<uintptr_t>(live) | reinterpret_cast<uintptr_t>(decoded) |
                     reinterpret_cast<uintptr_t>(prev_old)) & 3u) == 0;
  const int n4 = vec ? d.n_pos / 4 : 0;
  uint32_t any = 0;
  const uint32_t *l4 = reinterpret_cast<const uint32_t *>(live);
  const uint32_t *d4 = reinterpret_cast<const uint32_t *>(decoded);
  const uint32_t *p4 = reinterpret_cast<const uint32_t *>(prev_old);
#pragma unroll 4
  for (int q = part; q < n4; q += parts) {
    const uint32_t lv = l4[q], dc = d4[q], pv = p4[q];
    any |= ((~zero_bytes(lv)) | zero_bytes(dc)) & ~zero_bytes(pv) & 0x80808080u;
  }
  for (int t = 4 * n4 + part; t < d.n_pos; t += parts)
    any |= static_cast<uint32_t>((live[t] != 0) | (decoded[t] == 0)) & static_cast<uint32_t>(prev_old[t] != 0);
  return any != 0;
}

// Records position t's code and this iteration's state: its stamp (this
// iteration if fresh, else the previous one) and decoded flag.
__device__ __forceinline__ void record_position(const Dims &d, const Work &ws, int t, int code, int32_t stamp) {
  const int wr = (d.state_rd & 1) ^ 1;
  ws.cat[t] = static_cast<uint8_t>(code);
  ws.stamp[static_cast<size_t>(wr) * d.Nmax + t] = stamp;
  ws.prev_dec[static_cast<size_t>(wr) * d.Nmax + t] = (code & kCodeLive) ? 0 : 1;
}

// Classification of position t by one thread: writes its code and this
// iteration's state and returns whether t is fresh.
__device__ __forceinline__ bool classify_and_update(const Dims &d, const Work &ws, const uint8_t *__restrict__ live,
                                                    const uint8_t *__restrict__ decoded, int t, bool force) {
  const int rd = d.state_rd & 1;
  const int32_t st = ws.stamp[static_cast<size_t>(rd) * d.Nmax + t];
  const int code = classify_code(d, live[t] != 0, decoded[t] != 0, ws.prev_dec[static_cast<size_t>(rd) * d.Nmax + t] != 0, st);
  const bool fresh = force || (code & 15) != C_REUSE;
  record_position(d, ws, t, code, fresh ? d.iter : st);
  return fresh;
}

// The previous iteration's coverage shortfall makes this one full fresh
// (unless a host fallback already does): 2, else 0.
__device__ __forceinline__ int shortfall_flag(const Dims &d, const Work &ws) {
  return (d.cov_check && !d.host_fallback && !d.plan_mode && ws.ctrl->short_next) ? 2 : 0;
}

// Top-k of fresh position t by one warp over the eligible experts (every
// expert when `force`, else the support mask), ordered by logit desc, lower id
// first; weights = softmax over the k selected logits, summed in selection
// order. Lane l holds the logits v of experts [l*EPL, l*EPL + EPL); `scratch`
// is the warp's 32 entries of shared memory for the top-k. Writes sel/selw of
// t and sets bit t of the selected experts' words in `words`; sel_out
// (nullable, shared memory) gets the k selected experts as well.
//
// Group-limited sigmoid router (d.router == 1; v holds x W_r^T without the
// bias): scores s = sigmoid(v), selection scores c = s + bias, the group rule
// of warp_group_limit, the top-k of c, weights = the selected s divided by
// their sum in selection order. With d.raw_weights the weights are not
// renormalised: the selected s, or (softmax router) the dense router
// probabilities -- the softmax of v over every expert, eligible or not.
// With d.cov_check the position's support coverage is checked as well (see
// the coverage fields of epoch_layer_config) against support_mask, the block
// support, and an under-covered position is counted in cov_under.
// Top-k of the group-limited sigmoid router (see select_position), out of
// line so that the default router's path stays short: lane l passes its EPL
// logits v (without the bias) and eligibility; *sel and *wgt get lane l's
// selection (l < k).
template <int EPL>
__device__ __noinline__ void select_sigmoid_group(const Dims &d, const float *v_in, const bool *ok_in,
                                                  const float *bias, uint2 *scratch, int *sel_out, float *wgt_out) {
  const int lane = lane_id(), e0 = lane * EPL, k = d.k;
  float v[EPL], cs[EPL];
  bool ok[EPL];
#pragma unroll
  for (int c = 0; c < EPL; ++c) {
    v[c] = v_in[c];
    ok[c] = ok_in[c];
    const int e = e0 + c;
    cs[c] = e < d.E ? 1.f / (1.f + expf(-v[c])) + bias[e] : -INFINITY;
  }
  warp_group_limit<EPL>(cs, ok, d.E, d.n_group, d.topk_group, k);
  int sel;
  float val;
  warp_topk<EPL>(cs, ok, k, &sel, &val, scratch);
  // the selected expert's logit, from the lane that owns it
  const int owner = sel >= 0 ? sel / EPL : 0, idx = sel >= 0 ? sel - owner * EPL : 0;
  float z = 0.f;
#pragma unroll
  for (int c = 0; c < EPL; ++c) {
    const float o = __shfl_sync(0xffffffffu, v[c], owner);
    if (c == idx) z = o;
  }
  const float sg = lane < k ? 1.f / (1.f + expf(-z)) : 0.f;
  float denom = 0.f;
  for (int j = 0; j < k; ++j) denom += __shfl_sync(0xffffffffu, sg, j);
  *sel_out = sel;
  *wgt_out = d.raw_weights ? sg : sg / denom;
}

// Support coverage of one fresh position (see select_position), out of line:
// its dense selection (every expert eligible) and the share of that
// selection's raw score mass on the experts of support_mask. Returns whether
// the position is under the coverage floor (on every lane).
template <int EPL>
__device__ __noinline__ bool coverage_under(const Dims &d, const float *v_in, const uint8_t *support_mask,
                                            const float *bias, uint2 *scratch) {
  const int lane = lane_id(), e0 = lane * EPL, k = d.k;
  float v[EPL];
  bool all[EPL];
#pragma unroll
  for (int c = 0; c < EPL; ++c) {
    v[c] = v_in[c];
    all[c] = e0 + c < d.E;
  }
  int dsel;
  float dval, score;
  if (d.router == 0) {
    warp_topk<EPL>(v, all, k, &dsel, &dval, scratch);
    float m = -INFINITY;
#pragma unroll
    for (int c = 0; c < EPL; ++c) m = fmaxf(m, v[c]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float sum = 0.f;
#pragma unroll
    for (int c = 0; c < EPL; ++c) sum += e0 + c < d.E ? expf(v[c] - m) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    score = lane < k ? expf(dval - m) / sum : 0.f;
  } else {
    float cs[EPL];
#pragma unroll
    for (int c = 0; c < EPL; ++c) cs[c] = e0 + c < d.E ? 1.f / (1.f + expf(-v[c])) + bias[e0 + c] : -INFINITY;
    warp_group_limit<EPL>(cs, all, d.E, d.n_group, d.topk_group, k);
    warp_topk<EPL>(cs, all, k, &dsel, &dval, scratch);
    const int owner = dsel >= 0 ? dsel / EPL : 0, idx = dsel >= 0 ? dsel - owner * EPL : 0;
    float z = 0.f;
#pragma unroll
    for (int c = 0; c < EPL; ++c) {
      const float o = __shfl_sync(0xffffffffu, v[c], owner);
      if (c == idx) z = o;
    }
    score = lane < k ? 1.f / (1.f + expf(-z)) : 0.f;
  }
  float mass = 0.f, covered = 0.f;
  for (int j = 0; j < k; ++j) {  // in selection order
    const float sj = __shfl_sync(0xffffffffu, score, j);
    const int ej = __shfl_sync(0xffffffffu, dsel, j);
    mass += sj;
    if (ej >= 0 && support_mask[ej]) covered += sj;
  }
  return covered < d.cov_alpha * mass;
}

// Weight without renormalisation for the softmax router, out of line: the
// dense router probability of the lane's selected logit val (softmax of the
// row over every expert, eligible or not; lanes >= k get 0).
template <int EPL>
__device__ __noinline__ float dense_probability(const Dims &d, const float *v_in, float val) {
  const int lane = lane_id(), e0 = lane * EPL;
  float m = -INFINITY;
#pragma unroll
  for (int c = 0; c < EPL; ++c) m = fmaxf(m, v_in[c]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float sum = 0.f;
#pragma unroll
  for (int c = 0; c < EPL; ++c) sum += e0 + c < d.E ? expf(v_in[c] - m) : 0.f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  return lane < d.k ? expf(val - m) / sum : 0.f;
}

template <int EPL>
__device__ __forceinline__ void select_position(const Dims &d, const Work &ws, int t, const float (&v)[EPL],
                                                const uint8_t *support_mask, bool force, uint32_t *words,
                                                uint2 *scratch, const float *bias, int16_t *sel_out = nullptr) {
  const int lane = lane_id(), e0 = lane * EPL, k = d.k;
  bool ok[EPL];
#pragma unroll
  for (int c = 0; c < EPL; ++c) {
    const int e = e0 + c;
    ok[c] = e < d.E && (force || support_mask[e] != 0);
  }
  int sel;
  float val, wgt;
  if (d.router == 0) {
    warp_topk<EPL>(v, ok, k, &sel, &val, scratch);
    if (d.raw_weights) {
      wgt = dense_probability<EPL>(d, v, val);
    } else {
      const float top = __shfl_sync(0xffffffffu, val, 0);
      const float ex = lane < k ? expf(val - top) : 0.f;
      float denom = 0.f;
      for (int j = 0; j < k; ++j) denom += __shfl_sync(0xffffffffu, ex, j);
      wgt = ex / denom;
    }
  } else {
    select_sigmoid_group<EPL>(d, v, ok, bias, scratch, &sel, &wgt);
  }
  if (lane < k) {
    if (sel < 0 || sel >= d.E) {
      set_error(ws.err, EPOCH_DEVERR_BOUNDS);
    } else {
      ws.sel[static_cast<size_t>(t) * k + lane] = sel;
      ws.selw[static_cast<size_t>(t) * k + lane] = wgt;
      if (sel_out) sel_out[lane] = static_cast<int16_t>(sel);
      atomicOr(&words[static_cast<size_t>(sel) * d.cmax + (t >> 5)], 1u << (t & 31));
    }
  }
  if (d.cov_check && coverage_under<EPL>(d, v, support_mask, bias, scratch) && lane == 0)
    atomicAdd(ws.cov_under, 1);
}

// Per-iteration handshake state, set by block 0 of the kernel that classifies
// the positions (the gate, or the select kernel) while no later kernel of the
// iteration reads it yet: the anomaly flag, and the counters the expert kernel
// advances on the routed tiles (tiles drawn, up tiles done per group); it
// reads them only once this call's worklist is complete. (The shared-expert
// tile counters, which the expert kernel uses from its launch, are zeroed by
// the combine kernel of the call before, and by a block plan.)
// flags: bit 0 a decoded -> live anomaly, bit 1 the previous iteration's
// coverage shortfall (both make the iteration full fresh).
__device__ __forceinline__ void reset_iteration_state(const Dims &d, const Work &ws, int flags) {
  for (int g = threadIdx.x; g < d.E * (d.I / 128); g += blockDim.x) ws.done_up[g] = 0;
  if (threadIdx.x == 0) {
    ws.ctrl->anom = flags;
    ws.tile_ctr[0] = 0;
  }
}

// Selection words this iteration writes (the other half is cleared for the next one).
__device__ __forceinline__ uint32_t *words_written(const Dims &d, const Work &ws) {
  return ws.sel_words + static_cast<size_t>((d.state_rd & 1) ^ 1) * d.E * d.cmax;
}

}  // namespace epoch

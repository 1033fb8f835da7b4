// Routing side of the Epoch MoE-layer iteration (sm_103a): block plan (hit-
// count prefix and Expert Atlas planners), liveness classification and
// compaction, support-restricted top-k (fp32 layers; bf16 layers take it in
// the gate's epilogue), the worklist kernel (worklist.cuh), and the weighted
// combine with the routed-output cache.
//
// Source: walk-through page "Epoch 完全拆解:把扩散块编译成稀疏 MoE 服务单元" ([W]):
//   section "Expert Atlas" (G in R^{N x E}; the hot path keeps the support as a
//   mask and re-runs the top-k rule over it every iteration), section
//   "Liveness-Shard Parallelism" (Z_i, N_i, F_i; B_i = Compact(H, F_i);
//   Y[F_i] = Y_F, Y[not F_i] = C_l[not F_i]), section "FreshLane Dispatch"
//   (pack, count exchange -> offsets, light-traffic expert kernel, combine by
//   compact offset, scatter/merge), section "cold、hot-update、hot-skip"
//   (cold path clears the per-block cache and builds the support).
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "layer.h"
#include "select.cuh"
#include "topk.cuh"
#include "worklist.cuh"
#include "gate_tail.cuh"

namespace epoch {

const char *const kKindName[K_NUM] = {"gate",        "plan_topk", "plan_support", "routing", "experts",
                                      "expert_down", "combine",   "wait_test",    "select"};

// ---------------------------------------------------------------- helpers

// A block plan's reset of the iteration state (all threads of one CTA): both
// halves of the stamps, decoded flags and selection words, and the arrival
// count of the gate's grid barrier, the gate tail's tallies and the shared-
// expert tile counters (left over only by a timed-out call). Every iteration
// of the block that follows starts from this state, whatever calls ran before
// it.
__device__ void clear_block_state(const Dims &d, const Work &ws) {
  for (int t = threadIdx.x; t < 2 * d.Nmax; t += blockDim.x) {
    ws.stamp[t] = -1;
    ws.prev_dec[t] = 0;
  }
  for (int q = threadIdx.x; q < 2 * d.E * d.cmax; q += blockDim.x) ws.sel_words[q] = 0u;
  if (threadIdx.x == 0) {
    ws.gate_arrive[0] = 0;
    ws.gate_arrive[1] = 0;
    *ws.cov_under = 0;
  }
  if (threadIdx.x < 8) ws.tally[threadIdx.x] = 0;
  for (int q = threadIdx.x; q < sh_stride(d); q += blockDim.x) ws.sh_ctr[q] = 0;
}

// ---------------------------------------------------------------- gate (SIMT)
// G = x W_r^T + b for fp32 layers: one warp per (position, expert), lanes
// split H, fixed-order reduction (deterministic).
template <typename T>
__global__ void k_gate_simt(Dims d, const T *__restrict__ x, const T *__restrict__ wr, const float *__restrict__ bias,
                            float *__restrict__ g, Work ws) {
  (void)ws;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int lane = lane_id();
  for (int o = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; o < d.n_pos * d.E; o += warps) {
    const int t = o / d.E, e = o % d.E;
    const T *xr = x + static_cast<size_t>(t) * d.H;
    const T *wrow = wr + static_cast<size_t>(e) * d.H;
    float acc = 0.f;
    for (int h = lane; h < d.H; h += 32) acc = fmaf(to_f32(xr[h]), to_f32(wrow[h]), acc);
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (lane == 0) g[static_cast<size_t>(t) * d.E + e] = d.router ? acc : acc + bias[e];
  }
}

// ---------------------------------------------------------------- block plan
// Dense top-k of every position over all experts -> hit counts (integer atomics).
template <int EPL>
__global__ void k_plan_topk(Dims d, const float *__restrict__ logits, const float *__restrict__ bias,
                            int32_t *__restrict__ counts) {
  __shared__ uint2 s_scr[8][32];  // top-k scratch of each warp (256 threads)
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int lane = lane_id();
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < d.n_pos; t += warps) {
    float v[EPL];
    bool ok[EPL];
    lane_logits<EPL>(logits + static_cast<size_t>(t) * d.E, d.E, v);
#pragma unroll
    for (int c = 0; c < EPL; ++c) ok[c] = lane * EPL + c < d.E;
    int sel;
    float val;
    if (d.router != 0) {  // the group-limited sigmoid rule, every expert eligible
#pragma unroll
      for (int c = 0; c < EPL; ++c) {
        const int e = lane * EPL + c;
        v[c] = e < d.E ? 1.f / (1.f + expf(-v[c])) + bias[e] : -INFINITY;
      }
      warp_group_limit<EPL>(v, ok, d.E, d.n_group, d.topk_group, d.k);
    }
    warp_topk<EPL>(v, ok, d.k, &sel, &val, s_scr[warp_id()]);
    const size_t row = d.req_size > 0 ? static_cast<size_t>(t / d.req_size) * d.E : 0;
    if (lane < d.k && sel >= 0) atomicAdd(&counts[row + sel], 1);
  }
}

// One CTA per support (the block's, or request r's with per-request
// supports): rank experts by (count desc, id asc), take the smallest prefix
// whose counts reach the threshold (at least k; every expert when
// all_experts) -- for a request, ceil(tau * n_r * k) over its own n_r
// positions, formed on the device exactly as the host forms the block's --
// and, for a block plan (cold path), clear the block's stamps, previous-decoded
// flags and coverage state; a hot update keeps them.
__global__ void __launch_bounds__(1024) k_plan_support(Dims d, Work ws, int32_t threshold, int all_experts,
                                                       int clear_state, int32_t *ids_out, int32_t *len_out,
                                                       double tau) {
  const KernelMark mark_(d, ws, K_PLAN_SUPPORT);
  __shared__ int32_t cnt[1024];
  __shared__ int32_t sorted_cnt[1024];
  __shared__ int32_t len_s;
  const int tid = threadIdx.x;
  const int E = d.E, r = blockIdx.x;
  const bool per_req = d.req_size > 0;
  if (per_req) {
    const int n_r = min(d.req_size, d.n_pos - r * d.req_size);
    threshold = static_cast<int32_t>(ceil(tau * static_cast<double>(n_r * d.k)));
  }
  int32_t *ranked = per_req ? ws.req_ids + static_cast<size_t>(r) * E : ws.support_ids;
  uint8_t *mask = ws.support_mask + static_cast<size_t>(r) * E;
  if (tid < E) cnt[tid] = ws.plan_counts[static_cast<size_t>(r) * E + tid];
  if (tid == 0) len_s = E;
  __syncthreads();
  if (tid < E) {
    const int c = cnt[tid];
    int rank = 0;
    for (int e = 0; e < E; ++e) {
      const int ce = cnt[e];
      rank += (ce > c) || (ce == c && e < tid);
    }
    ranked[rank] = tid;
    if (ids_out && !per_req) ids_out[rank] = tid;
    sorted_cnt[rank] = c;
  }
  __syncthreads();
  // inclusive prefix of the ranked counts (E <= 1024, simple Hillis-Steele)
  for (int off = 1; off < E; off <<= 1) {
    int add = 0;
    if (tid < E && tid >= off) add = sorted_cnt[tid - off];
    __syncthreads();
    if (tid < E) sorted_cnt[tid] += add;
    __syncthreads();
  }
  if (!all_experts && tid < E) {
    const bool reach = sorted_cnt[tid] >= threshold;
    const bool before = tid > 0 && sorted_cnt[tid - 1] >= threshold;
    if (reach && !before) len_s = tid + 1;
  }
  __syncthreads();
  int len = len_s;
  if (len < d.k) len = d.k;
  if (len > E) len = E;
  if (tid < E) {
    int rank = 0;
    const int c = cnt[tid];
    for (int e = 0; e < E; ++e) {
      const int ce = cnt[e];
      rank += (ce > c) || (ce == c && e < tid);
    }
    mask[tid] = rank < len ? 1 : 0;
  }
  if (tid == 0) {
    if (per_req) {
      ws.req_len[r] = len;
    } else {
      ws.ctrl->support_len = len;
      if (len_out) *len_out = len;
    }
    if (clear_state && r == 0) ws.ctrl->short_next = 0;  // a new block starts without a coverage shortfall
  }
  if (clear_state && r == 0) clear_block_state(d, ws);
}

// Per-request supports: the union of the requests' supports (their masks,
// rows [0, n_req)) is the layer's candidate set, in ascending expert order;
// one CTA.
__global__ void __launch_bounds__(1024) k_plan_union(Dims d, Work ws, int32_t *ids_out, int32_t *len_out) {
  __shared__ int32_t tmp[33];
  const int tid = threadIdx.x, E = d.E;
  const int n_req = (d.n_pos + d.req_size - 1) / d.req_size;
  int in = 0;
  if (tid < E)
    for (int r = 0; r < n_req && !in; ++r) in = ws.support_mask[static_cast<size_t>(r) * E + tid];
  // exclusive scan of the membership flags over the expert ids
  const int lane = lane_id(), wid = warp_id();
  int incl = in;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) tmp[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int x = lane < static_cast<int>(blockDim.x >> 5) ? tmp[lane] : 0;
    int xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, xi, o);
      if (lane >= o) xi += u;
    }
    tmp[lane] = xi - x;
    if (lane == 31) tmp[32] = xi;
  }
  __syncthreads();
  const int pos = tmp[wid] + incl - in, total = tmp[32];
  if (tid < E && in) {
    ws.support_ids[pos] = tid;
    if (ids_out) ids_out[pos] = tid;
  }
  if (tid < E && tid >= total) ws.support_ids[tid] = -1;  // beyond the union
  if (tid == 0) {
    ws.ctrl->support_len = total;
    if (len_out) *len_out = total;
  }
}

// ---------------------------------------------------------------- Expert Atlas planner
// The planner of [W] section "Expert Atlas" (softmax router, one support per
// call): extended candidates, popularity, greedy repair of under-covered
// tokens. Float sums that decide an ordering (popularity, the repair gain G_e)
// are accumulated as 64-bit fixed point (2^40 per unit of routing mass), so
// that the order of the atomic additions cannot change them; per-token sums
// run in candidate order in float.
constexpr int kAtlasK = 32;  // candidates per token at most (k + m)
constexpr double kAtlasFix = 1099511627776.0;  // 2^40

// One warp per position: its K = min(k + m, E) best experts by logit (lower id
// first), their dense router probabilities W (softmax over all experts), the
// coverage floor r = alpha * (mass of the first k), and the popularity sums
// p_e += W over the candidate edges.
template <int EPL>
__global__ void k_atlas_cand(Dims d, Work ws, int K, float alpha) {
  __shared__ uint2 s_scr[8][32];
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int lane = lane_id();
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < d.n_pos; t += warps) {
    float v[EPL];
    bool ok[EPL];
    lane_logits<EPL>(ws.logits + static_cast<size_t>(t) * d.E, d.E, v);
#pragma unroll
    for (int c = 0; c < EPL; ++c) ok[c] = lane * EPL + c < d.E;
    int sel;
    float val;
    warp_topk<EPL>(v, ok, K, &sel, &val, s_scr[warp_id()]);
    float m = -INFINITY;
#pragma unroll
    for (int c = 0; c < EPL; ++c) m = fmaxf(m, v[c]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float sum = 0.f;
#pragma unroll
    for (int c = 0; c < EPL; ++c) sum += lane * EPL + c < d.E ? expf(v[c] - m) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    const float w = (lane < K && sel >= 0) ? expf(val - m) / sum : 0.f;
    float topk = 0.f;
    for (int j = 0; j < d.k; ++j) topk += __shfl_sync(0xffffffffu, w, j);
    if (lane < K) {
      ws.atlas_cand[static_cast<size_t>(t) * kAtlasK + lane] = sel;
      ws.atlas_w[static_cast<size_t>(t) * kAtlasK + lane] = w;
      if (sel >= 0) atomicAdd(ws.atlas_pop + sel, static_cast<unsigned long long>(llrint(static_cast<double>(w) * kAtlasFix)));
    }
    if (lane == 0) ws.atlas_r[t] = alpha * topk;
  }
}

// One CTA: the initial support (the max(B, k) most popular experts, lower id
// first on equal popularity), then repair rounds while more than (1 - q) N
// tokens are under-covered (C_t < r_t): for every expert outside the support,
// G_e = sum over under-covered t and their candidate edges to e of
// min(W, r_t - C_t) and H_e = the under-covered t with C_t + W >= r_t; the at
// most c experts of largest positive H_e + beta G_e (lower id first) join; a
// round with no positive score ends the search. support_ids gets the support
// in entry order, then the other experts in id order.
__global__ void __launch_bounds__(1024) k_atlas_plan(Dims d, Work ws, int K, int B, int c, double q, double beta,
                                                     int clear_state, int32_t *ids_out, int32_t *len_out) {
  const KernelMark mark_(d, ws, K_PLAN_SUPPORT);
  __shared__ unsigned long long s_fix[1024];  // popularity, then G_e of a round
  __shared__ int32_t s_h[1024];
  __shared__ uint8_t s_in[1024];
  __shared__ double s_score[1024];            // repair scores of a round (-1: not a candidate)
  __shared__ int32_t s_len, s_rounds;
  const int tid = threadIdx.x, E = d.E, N = d.n_pos;
  if (tid < E) s_fix[tid] = ws.atlas_pop[tid];
  if (tid == 0) {
    s_len = min(max(B, d.k), E);
    s_rounds = 0;
  }
  __syncthreads();
  const int n_init = s_len;
  if (tid < E) {
    const unsigned long long p = s_fix[tid];
    int rank = 0;
    for (int e = 0; e < E; ++e) rank += (s_fix[e] > p) || (s_fix[e] == p && e < tid);
    s_in[tid] = rank < n_init ? 1 : 0;
    if (rank < n_init) ws.support_ids[rank] = tid;
  }
  __syncthreads();
  __shared__ int32_t s_warp[32];
  // per-block sum of one int per thread
  auto block_sum = [&](int v) {
    v = __reduce_add_sync(0xffffffffu, v);
    if (lane_id() == 0) s_warp[warp_id()] = v;
    __syncthreads();
    int tot = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) tot += s_warp[w];
    __syncthreads();
    return tot;
  };
  auto coverage = [&](int t) {
    const int32_t *ct = ws.atlas_cand + static_cast<size_t>(t) * kAtlasK;
    const float *wt = ws.atlas_w + static_cast<size_t>(t) * kAtlasK;
    float cov = 0.f;
    for (int j = 0; j < K; ++j) {  // candidate order
      const int e = ct[j];
      if (e >= 0 && e < E && s_in[e]) cov += wt[j];
    }
    return cov;
  };
  int n_under = 0;
  for (int round = 0; round <= E; ++round) {
    int under = 0;
    for (int t = tid; t < N; t += blockDim.x) under += coverage(t) < ws.atlas_r[t] ? 1 : 0;
    n_under = block_sum(under);
    if (!(static_cast<double>(n_under) > (1.0 - q) * N)) break;
    // gains of the experts outside the support over the under-covered tokens
    if (tid < E) {
      s_fix[tid] = 0ull;
      s_h[tid] = 0;
    }
    __syncthreads();
    for (int t = tid; t < N; t += blockDim.x) {
      const float cov = coverage(t), r = ws.atlas_r[t];
      if (!(cov < r)) continue;
      const int32_t *ct = ws.atlas_cand + static_cast<size_t>(t) * kAtlasK;
      const float *wt = ws.atlas_w + static_cast<size_t>(t) * kAtlasK;
      for (int j = 0; j < K; ++j) {
        const int e = ct[j];
        if (e < 0 || e >= E || s_in[e]) continue;
        const float w = wt[j];
        atomicAdd(s_fix + e, static_cast<unsigned long long>(llrint(static_cast<double>(fminf(w, r - cov)) * kAtlasFix)));
        if (cov + w >= r) atomicAdd(s_h + e, 1);
      }
    }
    __syncthreads();
    // the at most c experts of largest positive score join (lower id first on equal scores)
    double score = 0.0;
    bool posv = false;
    if (tid < E && !s_in[tid]) {
      score = static_cast<double>(s_h[tid]) + beta * (static_cast<double>(s_fix[tid]) / kAtlasFix);
      posv = score > 0.0;
    }
    const int n_pos_scores = block_sum(posv ? 1 : 0);
    if (n_pos_scores == 0) break;
    if (tid < E) s_score[tid] = posv ? score : -1.0;
    __syncthreads();
    const int base = s_len;
    if (posv) {
      int rank = 0;
      for (int e = 0; e < E; ++e) rank += (s_score[e] > score) || (s_score[e] == score && e < tid);
      if (rank < c) ws.support_ids[base + rank] = tid;
    }
    __syncthreads();
    const int n_add = min(c, n_pos_scores);
    if (tid < n_add) s_in[ws.support_ids[base + tid]] = 1;
    if (tid == 0) {
      s_len = base + n_add;
      s_rounds = round + 1;
    }
    __syncthreads();
  }
  // support in entry order, then the other experts in id order; the mask
  const int len = s_len;
  if (tid < E) {
    ws.support_mask[tid] = s_in[tid];
    if (!s_in[tid]) {
      int before = 0;
      for (int e = 0; e < tid; ++e) before += s_in[e] ? 0 : 1;
      ws.support_ids[len + before] = tid;
    }
  }
  __syncthreads();
  if (ids_out)
    for (int e = tid; e < E; e += blockDim.x) ids_out[e] = ws.support_ids[e];
  if (tid == 0) {
    ws.ctrl->support_len = len;
    if (len_out) *len_out = len;
    ws.atlas_out[0] = static_cast<double>(n_under) > (1.0 - q) * N ? 0 : 1;  // covered_ok
    ws.atlas_out[1] = n_under;
    ws.atlas_out[2] = s_rounds;
    if (clear_state) ws.ctrl->short_next = 0;
  }
  if (clear_state) clear_block_state(d, ws);
}

// ---------------------------------------------------------------- select (fp32 layers)
// Classification and support-restricted top-k of every position from the
// logits of the FFMA gate (the tcgen05 gate of bf16 layers does the same in its
// epilogue): one warp per position. Every CTA first scans all positions for a
// decoded -> live transition, which makes every position fresh with every
// expert eligible.
template <int EPL>
__global__ void __launch_bounds__(256) k_select(Dims d, Work ws, const uint8_t *__restrict__ live,
                                                const uint8_t *__restrict__ decoded, const float *__restrict__ bias) {
  const KernelMark mark_(d, ws, K_SELECT);
  __shared__ uint2 s_scr[8][32];  // top-k scratch of each warp
  pdl_wait();
  const int rd = d.state_rd & 1;
  const bool anom = __syncthreads_or(
      any_anomaly(d, live, decoded, ws.prev_dec + static_cast<size_t>(rd) * d.Nmax, threadIdx.x, blockDim.x) ? 1 : 0);
  const int flags = (anom ? 1 : 0) | shortfall_flag(d, ws);
  const bool force = d.host_fallback != 0 || flags != 0;
  if (blockIdx.x == 0) reset_iteration_state(d, ws, flags);
  uint32_t *words = words_written(d, ws);
  const int lane = lane_id(), warps = gridDim.x * (blockDim.x >> 5);
  for (int t = blockIdx.x * (blockDim.x >> 5) + warp_id(); t < d.n_pos; t += warps) {
    int fresh = 0;
    if (lane == 0) fresh = classify_and_update(d, ws, live, decoded, t, force) ? 1 : 0;
    fresh = __shfl_sync(0xffffffffu, fresh, 0);
    if (!fresh) continue;
    float v[EPL];
    lane_logits<EPL>(ws.logits + static_cast<size_t>(t) * d.E, d.E, v);
    const uint8_t *mask = ws.support_mask + (d.req_size > 0 ? static_cast<size_t>(t / d.req_size) * d.E : 0);
    select_position<EPL>(d, ws, t, v, mask, force, words, s_scr[warp_id()], bias);
  }
}

// ---------------------------------------------------------------- worklist
// The worklist kernel, where the gate does not build the worklist in its own
// tail (fp32 layers, gates of more than one wave, the hot-update path): every
// CTA runs the phases of worklist.cuh with all its threads. xv: x as 16-byte
// vectors, whose worklist rows the CTAs copy into xp for the tcgen05 expert
// kernel (bf16 layers); null for fp32 layers, whose FFMA experts read x
// through wl_pos.
__global__ void __launch_bounds__(kRouteThreads) k_route(Dims d, Work ws, const uint4 *xv) {
  const KernelMark mark_(d, ws, K_ROUTING);
  pdl_trigger();
  __shared__ WlSmem sm;
  __shared__ int32_t s_off[1025];
  const Group g{static_cast<int>(threadIdx.x), kRouteThreads, 0};
  wl_prepare(d, ws, sm, s_off, g);
  pdl_wait();  // the kernel before has finished: selection words, selections, codes, anomaly flag
  const WlPlan pl = wl_phase_a(d, ws, sm, s_off, nullptr, blockIdx.x == 0, g);
  wl_rows(d, ws, sm, s_off, pl, xv, xv ? d.H * 2 / 16 : 0, blockIdx.x, gridDim.x, g);
  wl_bookkeeping(d, ws, sm, s_off, pl, blockIdx.x, gridDim.x, g, nullptr);
}

// ---------------------------------------------------------------- combine + cache
// Eight consecutive elements of a row, stored as one or two 16-byte vectors.
__device__ __forceinline__ void store8(float *p, const float (&v)[8]) {
  *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4 *>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}
__device__ __forceinline__ void store8(__nv_bfloat16 *p, const float (&v)[8]) {
  uint4 u;
  __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&u);
#pragma unroll
  for (int q = 0; q < 4; ++q) h[q] = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
  *reinterpret_cast<uint4 *>(p) = u;
}

constexpr int kTraceRowCombine = 7;

// Eight consecutive elements of a row as loaded (converted after every load of
// a run has been issued).
template <typename T> struct Row8;
template <> struct Row8<__nv_bfloat16> {
  uint4 u;
  __device__ __forceinline__ void load(const __nv_bfloat16 *p) { u = *reinterpret_cast<const uint4 *>(p); }
  __device__ __forceinline__ void get(float (&v)[8]) const {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __bfloat1622float2(h[q]);
      v[2 * q] = f.x;
      v[2 * q + 1] = f.y;
    }
  }
};
template <> struct Row8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float *p) {
    a = *reinterpret_cast<const float4 *>(p);
    b = *reinterpret_cast<const float4 *>(p + 4);
  }
  __device__ __forceinline__ void get(float (&v)[8]) const {
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
};

// One CTA per position, 8 elements per thread per pass. Expert outputs O are
// stored in the layer dtype. Fresh t:
// r = sum_j w_j O[slot(t, j)] (j ascending, fp32) and the cache row is refilled
// ([W] section "Liveness-Shard Parallelism": Y[F_i] = Y_F); reused t: r = the
// cached row (Y[not F_i] = C_l[not F_i]). Then y = r + shared outputs (+ x when
// residual), rounded once: the dense shard is restored at the layer boundary.
// The fresh index, slots and weights come from the worklist bookkeeping; each
// pass requests every row it needs (the k expert-output rows or the cached
// row, the shared outputs, x) before using any of them.
template <typename T>
__global__ void __launch_bounds__(128, 7) k_combine(Dims d, Work ws, const T *__restrict__ x, T *__restrict__ y) {
  const KernelMark mark_(d, ws, K_COMBINE);
  int64_t *trace = (d.trace && blockIdx.x < kTraceCtas && threadIdx.x == 0)
                       ? ws.trace + (static_cast<size_t>(kTraceRowCombine) * kTraceCtas + blockIdx.x) * kTraceFields
                       : nullptr;
  if (trace) {
    trace[0] = static_cast<int64_t>(globaltimer_ns());
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    trace[7] = smid;
  }
  const int t = blockIdx.x;
  const int H = d.H, k = d.k;
  __shared__ int32_t slot_s[16];
  __shared__ float w_s[16];
  __shared__ int f_s;
  // Every kernel of the iteration before this one has completed: the expert
  // outputs, and the worklist bookkeeping (the gate's tail or the worklist
  // kernel, both before the experts). A hardware wait: no thread of this grid
  // polls memory while the experts stream.
  pdl_wait();
  if (blockIdx.x == 0) {
    // the next call's expert kernel takes shared-expert tiles from its launch
    for (int q = threadIdx.x; q < sh_stride(d); q += blockDim.x) ws.sh_ctr[q] = 0;
    if (d.wl_in_gate && threadIdx.x == 0) gate_tail_stats(d, ws);
  }
  if (t < d.n_pos) {
    if (threadIdx.x < k) {
      slot_s[threadIdx.x] = ws.slot[static_cast<size_t>(t) * k + threadIdx.x];
      w_s[threadIdx.x] = ws.selw[static_cast<size_t>(t) * k + threadIdx.x];
    }
    if (threadIdx.x == 0) f_s = ws.fidx[t];
  }
  if (trace) trace[1] = static_cast<int64_t>(globaltimer_ns());
  if (t >= d.n_pos) return;
  __syncthreads();
  const int f = f_s;
  if (f >= 0 && threadIdx.x < k && (slot_s[threadIdx.x] < 0 || slot_s[threadIdx.x] >= d.Nmax * k)) {
    set_error(ws.err, EPOCH_DEVERR_BOUNDS);
    slot_s[threadIdx.x] = 0;
  }
  __syncthreads();
  if (trace) trace[2] = static_cast<int64_t>(globaltimer_ns());
  T *cache = reinterpret_cast<T *>(ws.cache) + static_cast<size_t>(t) * H;
  const T *o_int = static_cast<const T *>(ws.o_int);
  const T *o_sh = static_cast<const T *>(ws.o_sh) + static_cast<size_t>(t) * H;
  constexpr int kU = sizeof(T) == 2 ? 4 : 2;  // expert rows requested together (at most 72 registers)
  constexpr int kS = 2;                       // shared-expert rows requested with them
#pragma unroll 1
  for (int h0 = threadIdx.x * 8; h0 < H; h0 += blockDim.x * 8) {
    Row8<T> ro[kU], rs[kS], rx;
    if (f >= 0) {
#pragma unroll
      for (int j = 0; j < kU; ++j)
        if (j < k) ro[j].load(o_int + static_cast<size_t>(slot_s[j]) * H + h0);
    } else {
      ro[0].load(cache + h0);
    }
#pragma unroll
    for (int s = 0; s < kS; ++s)
      if (s < d.n_sh) rs[s].load(o_sh + static_cast<size_t>(s) * d.Nmax * H + h0);
    if (d.residual) rx.load(x + static_cast<size_t>(t) * H + h0);
    // shared outputs (+ x) in expert order
    float base[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) base[q] = 0.f;
#pragma unroll
    for (int s = 0; s < kS; ++s)
      if (s < d.n_sh) {
        float o[8];
        rs[s].get(o);
#pragma unroll
        for (int q = 0; q < 8; ++q) base[q] += o[q];
      }
#pragma unroll 1
    for (int s = kS; s < d.n_sh; ++s) {
      Row8<T> r2;
      r2.load(o_sh + static_cast<size_t>(s) * d.Nmax * H + h0);
      float o[8];
      r2.get(o);
#pragma unroll
      for (int q = 0; q < 8; ++q) base[q] += o[q];
    }
    if (d.residual) {
      float xv[8];
      rx.get(xv);
#pragma unroll
      for (int q = 0; q < 8; ++q) base[q] += xv[q];
    }
    // routed part: weighted expert outputs (refilling the cache row), or the cached row
    float r[8];
    if (f >= 0) {
#pragma unroll
      for (int q = 0; q < 8; ++q) r[q] = 0.f;
#pragma unroll
      for (int j = 0; j < kU; ++j)
        if (j < k) {
          float o[8];
          ro[j].get(o);
          const float wj = w_s[j];
#pragma unroll
          for (int q = 0; q < 8; ++q) r[q] = fmaf(wj, o[q], r[q]);
        }
#pragma unroll 1
      for (int j0 = kU; j0 < k; j0 += kU) {  // further rows, kU at a time
#pragma unroll
        for (int j = 0; j < kU; ++j)
          if (j0 + j < k) ro[j].load(o_int + static_cast<size_t>(slot_s[j0 + j]) * H + h0);
#pragma unroll
        for (int j = 0; j < kU; ++j)
          if (j0 + j < k) {
            float o[8];
            ro[j].get(o);
            const float wj = w_s[j0 + j];
#pragma unroll
            for (int q = 0; q < 8; ++q) r[q] = fmaf(wj, o[q], r[q]);
          }
      }
      store8(cache + h0, r);
    } else {
      ro[0].get(r);
    }
#pragma unroll
    for (int q = 0; q < 8; ++q) r[q] += base[q];
    store8(y + static_cast<size_t>(t) * H + h0, r);
  }
  if (trace) trace[3] = static_cast<int64_t>(globaltimer_ns());
}

// ---------------------------------------------------------------- bounded-wait test
// Waits on an mbarrier that nothing ever completes; the bounded wait must give
// up after timeout_ns, set the timeout bit and return.
__global__ void k_wait_test(uint32_t *err, int64_t timeout_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(smem_u32(&bar), 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    (void)mbar_wait_bounded(smem_u32(&bar), 0, &abort_flag, err, static_cast<uint64_t>(timeout_ns));
  }
  __syncthreads();
}

// ---------------------------------------------------------------- launchers

static int epl_for(int E) {
  const int epl = (E + 31) / 32;
  return epl <= 1 ? 1 : epl <= 2 ? 2 : epl <= 4 ? 4 : epl <= 8 ? 8 : epl <= 16 ? 16 : 32;
}

int num_sms() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

cudaError_t launch_kernel(const void *fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void **args,
                          bool programmatic, int cluster) {
  static bool pdl_ok = true;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (cluster > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  const bool pdl = programmatic && pdl_ok;
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  cudaError_t e = cudaLaunchKernelExC(&cfg, fn, args);
  if (e != cudaSuccess && pdl && (e == cudaErrorInvalidValue || e == cudaErrorNotSupported)) {
    (void)cudaGetLastError();
    pdl_ok = false;
    cfg.numAttrs = n - 1;
    e = cudaLaunchKernelExC(&cfg, fn, args);
  }
  return e;
}

cudaError_t launch_gate_simt(const Dims &d, const Weights &w, const Work &ws, const void *x, int bf16,
                             cudaStream_t s) {
  const int outputs = d.n_pos * d.E;
  int blocks = (outputs + 7) / 8;
  if (blocks > 8 * num_sms()) blocks = 8 * num_sms();
  if (bf16) {
    static bool carve_ = (prefer_max_shared(k_gate_simt<__nv_bfloat16>) == cudaSuccess);
    (void)carve_;
    k_gate_simt<__nv_bfloat16><<<blocks, 256, 0, s>>>(d, static_cast<const __nv_bfloat16 *>(x),
                                                      static_cast<const __nv_bfloat16 *>(w.w_router), w.b_router,
                                                      ws.logits, ws);
  } else {
    static bool carve_ = (prefer_max_shared(k_gate_simt<float>) == cudaSuccess);
    (void)carve_;
    k_gate_simt<float><<<blocks, 256, 0, s>>>(d, static_cast<const float *>(x),
                                              static_cast<const float *>(w.w_router), w.b_router, ws.logits, ws);
  }
  return cudaGetLastError();
}

cudaError_t launch_plan_topk(const Dims &d, const Weights &w, const Work &ws, cudaStream_t s) {
  int blocks = (d.n_pos + 7) / 8;
  switch (epl_for(d.E)) {
#define EPOCH_CASE(N)                                                                  \
  case N: {                                                                            \
    static bool c_ = (prefer_max_shared(k_plan_topk<N>) == cudaSuccess);               \
    (void)c_;                                                                          \
    k_plan_topk<N><<<blocks, 256, 0, s>>>(d, ws.logits, w.b_router, ws.plan_counts);              \
    break;                                                                             \
  }
    EPOCH_CASE(1) EPOCH_CASE(2) EPOCH_CASE(4) EPOCH_CASE(8) EPOCH_CASE(16) EPOCH_CASE(32)
#undef EPOCH_CASE
  }
  return cudaGetLastError();
}

cudaError_t launch_plan_support(const Dims &d, const Work &ws, int32_t threshold, int all_experts,
                                int clear_state, int32_t *ids_out, int32_t *len_out, double tau, cudaStream_t s) {
  static bool carve_ = (prefer_max_shared(k_plan_support) == cudaSuccess && prefer_max_shared(k_plan_union) == cudaSuccess);
  (void)carve_;
  const int n_req = d.req_size > 0 ? (d.n_pos + d.req_size - 1) / d.req_size : 1;
  k_plan_support<<<n_req, 1024, 0, s>>>(d, ws, threshold, all_experts, clear_state, ids_out, len_out, tau);
  if (d.req_size > 0) {
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    k_plan_union<<<1, 1024, 0, s>>>(d, ws, ids_out, len_out);
  }
  return cudaGetLastError();
}

cudaError_t launch_atlas(const Dims &d, const Work &ws, const AtlasParams &a, int clear_state, int32_t *ids_out,
                         int32_t *len_out, cudaStream_t s) {
  const int K = min(d.k + a.m, d.E);
  if (K > kAtlasK) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(ws.atlas_pop, 0, sizeof(unsigned long long) * d.E, s);
  if (e != cudaSuccess) return e;
  const int blocks = (d.n_pos + 7) / 8;
  const float alpha = static_cast<float>(a.alpha);
  switch (epl_for(d.E)) {
#define EPOCH_CASE(N)                                                   \
  case N:                                                               \
    k_atlas_cand<N><<<blocks, 256, 0, s>>>(d, ws, K, alpha);            \
    break;
    EPOCH_CASE(1) EPOCH_CASE(2) EPOCH_CASE(4) EPOCH_CASE(8) EPOCH_CASE(16) EPOCH_CASE(32)
#undef EPOCH_CASE
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  static bool carve_ = (prefer_max_shared(k_atlas_plan) == cudaSuccess);
  (void)carve_;
  k_atlas_plan<<<1, 1024, 0, s>>>(d, ws, K, a.B, a.c, a.q, a.beta, clear_state, ids_out, len_out);
  return cudaGetLastError();
}

cudaError_t launch_select(const Dims &d, const Work &ws, const uint8_t *live, const uint8_t *decoded,
                          const float *bias, cudaStream_t s) {
  int blocks = (d.n_pos + 7) / 8;
  if (blocks > 2 * num_sms()) blocks = 2 * num_sms();
  switch (epl_for(d.E)) {
#define EPOCH_CASE(N)                                                                  \
  case N: {                                                                            \
    static bool c_ = (prefer_max_shared(k_select<N>) == cudaSuccess);                  \
    (void)c_;                                                                          \
    k_select<N><<<blocks, 256, 0, s>>>(d, ws, live, decoded, bias);                          \
    break;                                                                             \
  }
    EPOCH_CASE(1) EPOCH_CASE(2) EPOCH_CASE(4) EPOCH_CASE(8) EPOCH_CASE(16) EPOCH_CASE(32)
#undef EPOCH_CASE
  }
  return cudaGetLastError();
}

int route_ctas() { return num_sms(); }

// One CTA per SM, launched programmatically: the CTAs become resident while
// the kernel before runs and wait for it (pdl_wait) before reading.
cudaError_t launch_route(const Dims &d, const Work &ws, const void *x, cudaStream_t s) {
  if (d.E > 8 * kRouteThreads) return cudaErrorInvalidConfiguration;
  static bool c_ = (prefer_max_shared(k_route) == cudaSuccess);
  if (!c_) return cudaErrorInvalidConfiguration;
  Dims dd = d;
  Work ww = ws;
  const uint4 *xv = static_cast<const uint4 *>(x);
  void *args[] = {&dd, &ww, &xv};
  return launch_kernel(reinterpret_cast<void *>(k_route), dim3(route_ctas()), dim3(kRouteThreads), 0, s, args,
                       true);
}

cudaError_t launch_combine(const Dims &d, const Work &ws, const void *x, void *y, int bf16, cudaStream_t s) {
  if (bf16) {
    static bool carve_ = (prefer_max_shared(k_combine<__nv_bfloat16>) == cudaSuccess);
    (void)carve_;
    const __nv_bfloat16 *xb = static_cast<const __nv_bfloat16 *>(x);
    __nv_bfloat16 *yb = static_cast<__nv_bfloat16 *>(y);
    Dims dd = d;
    Work ww = ws;
    void *args[] = {&dd, &ww, &xb, &yb};
    return launch_kernel(reinterpret_cast<void *>(k_combine<__nv_bfloat16>), dim3(d.n_pos), dim3(128), 0, s, args,
                         true);
  }
  static bool carve_ = (prefer_max_shared(k_combine<float>) == cudaSuccess);
  (void)carve_;
  k_combine<float><<<d.n_pos, 128, 0, s>>>(d, ws, static_cast<const float *>(x), static_cast<float *>(y));
  return cudaGetLastError();
}

cudaError_t launch_wait_test(uint32_t *err, int64_t timeout_ns, cudaStream_t s) {
  static bool carve_ = (prefer_max_shared(k_wait_test) == cudaSuccess);
  (void)carve_;
  k_wait_test<<<1, 32, 0, s>>>(err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace epoch

// Routing side of the Epoch MoE-layer iteration (sm_103a): block plan,
// liveness classification and compaction, support-restricted top-k, the
// expert-sorted worklist, the permute into compact rows, and the weighted
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

namespace epoch {

const char *const kKindName[K_NUM] = {"gate",     "plan_topk", "plan_support", "classify",
                                      "route",    "worklist",  "permute",      "expert_up",
                                      "expert_down", "combine", "wait_test",   "memset"};

// ---------------------------------------------------------------- helpers

// (value desc, id asc) order used for every top-k: true if (va, ia) ranks first.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Warp-wide arg-best of (v, id) pairs; every lane returns the winner.
__device__ __forceinline__ void warp_best(float &v, int &id) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, id, o);
    if (ranks_before(ov, oi, v, id)) {
      v = ov;
      id = oi;
    }
  }
}

// Logits of the EPL consecutive experts [lane*EPL, lane*EPL + EPL) of position
// t: split-K partial sums in a fixed order, then the bias. Experts >= E get
// -inf. Vector loads when the row is 16-byte aligned.
template <int EPL>
__device__ __forceinline__ void lane_logits(const float *__restrict__ gparts, int SK, int Nmax, int E, int t,
                                            const float *__restrict__ bias, float (&v)[EPL]) {
  const int e0 = lane_id() * EPL;
#pragma unroll
  for (int c = 0; c < EPL; ++c) v[c] = 0.f;
  if constexpr (EPL % 4 == 0) {
    if ((E & 3) == 0 && e0 + EPL <= E) {
#pragma unroll 4
      for (int s = 0; s < SK; ++s) {
        const float4 *src = reinterpret_cast<const float4 *>(gparts + (static_cast<size_t>(s) * Nmax + t) * E + e0);
#pragma unroll
        for (int q = 0; q < EPL / 4; ++q) {
          const float4 a = __ldg(src + q);
          v[4 * q] += a.x;
          v[4 * q + 1] += a.y;
          v[4 * q + 2] += a.z;
          v[4 * q + 3] += a.w;
        }
      }
      const float4 *bs = reinterpret_cast<const float4 *>(bias + e0);
#pragma unroll
      for (int q = 0; q < EPL / 4; ++q) {
        const float4 b = __ldg(bs + q);
        v[4 * q] += b.x;
        v[4 * q + 1] += b.y;
        v[4 * q + 2] += b.z;
        v[4 * q + 3] += b.w;
      }
      return;
    }
  }
#pragma unroll
  for (int c = 0; c < EPL; ++c) {
    const int e = e0 + c;
    if (e < E) {
      float g = 0.f;
      for (int s = 0; s < SK; ++s) g += __ldg(gparts + (static_cast<size_t>(s) * Nmax + t) * E + e);
      v[c] = g + __ldg(bias + e);
    } else {
      v[c] = -INFINITY;
    }
  }
}

// Top-k of one position by one warp over lane-owned experts lane*EPL + c;
// ineligible experts never win. Every lane gets the selection (order: value
// desc, id asc) in sel/val.
template <int EPL>
__device__ __forceinline__ void warp_topk(const float (&v)[EPL], const bool (&ok)[EPL], int k, int (&sel)[16],
                                          float (&val)[16]) {
  bool taken[EPL];
#pragma unroll
  for (int c = 0; c < EPL; ++c) taken[c] = !ok[c];
  const int e0 = lane_id() * EPL;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j < k) {
      float bv = -INFINITY;
      int bi = INT_MAX;
#pragma unroll
      for (int c = 0; c < EPL; ++c) {
        if (!taken[c] && ranks_before(v[c], e0 + c, bv, bi)) {
          bv = v[c];
          bi = e0 + c;
        }
      }
      warp_best(bv, bi);
      sel[j] = bi;
      val[j] = bv;
#pragma unroll
      for (int c = 0; c < EPL; ++c)
        if (e0 + c == bi) taken[c] = true;
    }
  }
}

// Exclusive scan over a CTA of up to 1024 threads; *total gets the sum.
__device__ __forceinline__ int block_excl_scan(int v, int *warp_tmp, int *total) {
  const int lane = lane_id(), wid = warp_id(), nw = (blockDim.x + 31) >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_tmp[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int x = lane < nw ? warp_tmp[lane] : 0;
    int xi = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, xi, o);
      if (lane >= o) xi += u;
    }
    warp_tmp[lane] = xi - x;
    if (lane == 31) warp_tmp[32] = xi;
  }
  __syncthreads();
  const int r = warp_tmp[wid] + incl - v;
  *total = warp_tmp[32];
  __syncthreads();
  return r;
}

// ---------------------------------------------------------------- gate (SIMT)
// G part 0 = x W_r^T for fp32 layers: one warp per (position, expert), lanes
// split H, fixed-order reduction (deterministic).
template <typename T>
__global__ void k_gate_simt(Dims d, const T *__restrict__ x, const T *__restrict__ wr, float *__restrict__ g) {
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
    if (lane == 0) g[static_cast<size_t>(t) * d.E + e] = acc;
  }
}

// ---------------------------------------------------------------- block plan
// Dense top-k of every position over all experts -> hit counts (integer atomics).
template <int EPL>
__global__ void k_plan_topk(Dims d, const float *__restrict__ gparts, const float *__restrict__ bias,
                            int32_t *__restrict__ counts) {
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int lane = lane_id();
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < d.n_pos; t += warps) {
    float v[EPL];
    bool ok[EPL];
    lane_logits<EPL>(gparts, d.SK, d.Nmax, d.E, t, bias, v);
#pragma unroll
    for (int c = 0; c < EPL; ++c) ok[c] = lane * EPL + c < d.E;
    int sel[16];
    float val[16];
    warp_topk<EPL>(v, ok, d.k, sel, val);
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < d.k && j == lane) atomicAdd(&counts[sel[j]], 1);
  }
}

// One CTA: rank experts by (count desc, id asc), take the smallest prefix whose
// counts reach `threshold` (at least k; every expert when all_experts), and
// clear the block's stamps and previous-decoded flags (cold path).
__global__ void __launch_bounds__(1024) k_plan_support(Dims d, Work ws, int32_t threshold, int all_experts) {
  const KernelMark mark_(d, ws, K_PLAN_SUPPORT);
  __shared__ int32_t cnt[1024];
  __shared__ int32_t sorted_cnt[1024];
  __shared__ int32_t len_s;
  const int tid = threadIdx.x;
  const int E = d.E;
  if (tid < E) cnt[tid] = ws.plan_counts[tid];
  if (tid == 0) len_s = E;
  __syncthreads();
  if (tid < E) {
    const int c = cnt[tid];
    int rank = 0;
    for (int e = 0; e < E; ++e) {
      const int ce = cnt[e];
      rank += (ce > c) || (ce == c && e < tid);
    }
    ws.support_ids[rank] = tid;
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
    ws.support_mask[tid] = rank < len ? 1 : 0;
  }
  if (tid == 0) ws.ctrl->support_len = len;
  for (int t = tid; t < d.Nmax; t += blockDim.x) {
    ws.stamp[t] = -1;
    ws.prev_dec[t] = 0;
  }
}

// ---------------------------------------------------------------- classify + compact
// One CTA of 1024 threads; thread j owns the consecutive positions
// [j*c, (j+1)*c), so a block-wide exclusive scan keeps the fresh list ascending.
__global__ void __launch_bounds__(1024) k_classify(Dims d, Work ws, const uint8_t *__restrict__ live,
                                                   const uint8_t *__restrict__ decoded) {
  const KernelMark mark_(d, ws, K_CLASSIFY);
  constexpr int kThreads = 1024;
  __shared__ int32_t warp_sum[32];
  __shared__ int32_t cat[8];
  const int tid = threadIdx.x;
  if (tid < 8) cat[tid] = 0;
  if (tid < d.E) ws.expert_cnt[tid] = 0;  // the route kernel counts each expert's rows
  const int n = d.n_pos;
  const int per = (n + kThreads - 1) / kThreads;
  const int lo = min(tid * per, n), hi = min(lo + per, n);

  // pass 1: liveness anomalies (decoded -> live) and malformed flags
  int anomaly = 0, bad = 0;
  for (int t = lo; t < hi; ++t) {
    const bool lv = live[t] != 0, dc = decoded[t] != 0;
    const bool is_live = lv || !dc;
    bad += (lv == dc);
    anomaly |= (is_live && ws.prev_dec[t]);
  }
  const int any_anomaly = __syncthreads_or(anomaly);
  const bool force = d.host_fallback || any_anomaly;

  // pass 2: categories and fresh flags
  int nf = 0;
  int c_live = 0, c_new = 0, c_miss = 0, c_stale = 0, c_forced = 0, c_reuse = 0;
  for (int t = lo; t < hi; ++t) {
    const bool lv = live[t] != 0, dc = decoded[t] != 0;
    const bool is_live = lv || !dc;
    const int st = ws.stamp[t];
    bool fresh = true;
    if (is_live) {
      ++c_live;
    } else if (!ws.prev_dec[t]) {
      ++c_new;
    } else if (st < 0) {
      ++c_miss;
    } else if (d.R != INT_MAX && d.iter - st >= d.R) {
      ++c_stale;
    } else if (force) {
      ++c_forced;
    } else {
      ++c_reuse;
      fresh = false;
    }
    nf += fresh;
  }
  // block exclusive scan of nf
  const int lane = lane_id(), wid = warp_id();
  int incl = nf;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sum[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int ws_v = warp_sum[lane];
    int wi = ws_v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += v;
    }
    warp_sum[lane] = wi - ws_v;  // exclusive warp offsets
  }
  __syncthreads();
  int f = warp_sum[wid] + incl - nf;

  // pass 3: write the compact list, stamps and the new previous-decoded flags
  for (int t = lo; t < hi; ++t) {
    const bool lv = live[t] != 0, dc = decoded[t] != 0;
    const bool is_live = lv || !dc;
    const int st = ws.stamp[t];
    const bool reuse = !is_live && ws.prev_dec[t] && st >= 0 && !(d.R != INT_MAX && d.iter - st >= d.R) && !force;
    if (!reuse) {
      ws.fresh_pos[f] = t;
      ws.fidx[t] = f;
      ws.stamp[t] = d.iter;
      ++f;
    } else {
      ws.fidx[t] = -1;
    }
    ws.prev_dec[t] = is_live ? 0 : 1;
  }
  atomicAdd(&cat[0], c_live);
  atomicAdd(&cat[1], c_new);
  atomicAdd(&cat[2], c_miss);
  atomicAdd(&cat[3], c_stale);
  atomicAdd(&cat[4], c_forced);
  atomicAdd(&cat[5], c_reuse);
  atomicAdd(&cat[6], bad);
  __syncthreads();
  if (tid == 0) {
    const int n_fresh = n - cat[5];
    const int fb = (d.host_fallback ? 1 : 0) | (any_anomaly ? 2 : 0);
    ws.ctrl->n_fresh = n_fresh;
    ws.ctrl->fallback = fb;
    ws.ctrl->n_edges = n_fresh * d.k;
    epoch_iter_stats *st = ws.stats;
    st->iteration = d.iter;
    st->n_pos = n;
    st->n_live = cat[0];
    st->n_new = cat[1];
    st->n_miss = cat[2];
    st->n_stale = cat[3];
    st->n_forced = cat[4];
    st->n_reuse = cat[5];
    st->n_fresh = n_fresh;
    st->n_edges = n_fresh * d.k;
    st->support_len = fb ? d.E : ws.ctrl->support_len;
    st->fallback = fb;
    st->bad_flags = cat[6];
    if (cat[6]) set_error(ws.err, EPOCH_DEVERR_FLAGS);
  }
}

// ---------------------------------------------------------------- restricted top-k
// One CTA of 32 warps per chunk of 32 fresh positions, one warp per position.
// Each fresh position takes its top-k over the support (every expert on a
// fallback) and softmax weights over the selected logits, and sets bit p of the
// chunk's per-expert mask; mask popcounts give the worklist its offsets with
// no sort ("count exchange" of [W] section "FreshLane Dispatch", on chip).
template <int EPL>
__global__ void __launch_bounds__(1024) k_route(Dims d, Work ws, const float *__restrict__ bias) {
  const KernelMark mark_(d, ws, K_ROUTE);
  __shared__ uint32_t mask[1024];
  const int chunk = blockIdx.x;
  const int n_fresh = ws.ctrl->n_fresh;
  if (chunk * 32 >= n_fresh) return;
  for (int e = threadIdx.x; e < d.E; e += blockDim.x) mask[e] = 0;
  __syncthreads();
  const int lane = lane_id(), p = warp_id();
  const int f = chunk * 32 + p;
  if (f < n_fresh) {
    const int t = ws.fresh_pos[f];
    const bool all = ws.ctrl->fallback != 0;
    float v[EPL];
    bool ok[EPL];
    lane_logits<EPL>(ws.gparts, d.SK, d.Nmax, d.E, t, bias, v);
#pragma unroll
    for (int c = 0; c < EPL; ++c) {
      const int e = lane * EPL + c;
      ok[c] = e < d.E && (all || ws.support_mask[e]);
    }
    int sel[16];
    float val[16];
    warp_topk<EPL>(v, ok, d.k, sel, val);
    float denom = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j)
      if (j < d.k) denom += expf(val[j] - val[0]);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (j < d.k && j == lane) {
        const int e = sel[j];
        ws.sel[f * d.k + j] = e;
        ws.selw[f * d.k + j] = expf(val[j] - val[0]) / denom;
        if (e >= 0 && e < d.E) atomicOr(&mask[e], 1u << p);
        else set_error(ws.err, EPOCH_DEVERR_BOUNDS);
      }
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < d.E; e += blockDim.x) {
    const uint32_t m = mask[e];
    ws.chunk_mask[static_cast<size_t>(e) * d.cmax + chunk] = m;
    if (m) atomicAdd(&ws.expert_cnt[e], __popc(m));
  }
}

// ---------------------------------------------------------------- worklist
// CTA e < E places expert e's rows: row offsets[e] + (rows of expert e in
// earlier chunks) + (bits of its chunk mask below p), so rows are grouped by
// expert with positions ascending, with no sort and no atomics; warp w of the
// CTA takes chunk w of each 32-chunk pass. The last CTA writes the expert
// offsets and the grouped-GEMM tile lists: routed experts with at least one
// row, then the shared experts over every position; experts with no rows get
// no tile, so their weights are never read ([W] section "FreshLane Dispatch":
// invalid slots load no expert weights).
__global__ void __launch_bounds__(1024) k_worklist(Dims d, Work ws) {
  const KernelMark mark_(d, ws, K_WORKLIST);
  __shared__ int32_t tmp[33];
  __shared__ int32_t wsum[32];
  const int E = d.E, k = d.k;
  const int tid = threadIdx.x, lane = lane_id(), wid = warp_id();
  const int n_fresh = ws.ctrl->n_fresh;
  const int n_chunks = (n_fresh + 31) / 32;
  if (static_cast<int>(blockIdx.x) < E) {
    const int e = blockIdx.x;
    if (ws.expert_cnt[e] == 0) return;
    int part = 0;
    for (int q = tid; q < e; q += blockDim.x) part += ws.expert_cnt[q];
    int off;
    (void)block_excl_scan(part, tmp, &off);
    int run = 0;
    for (int c0 = 0; c0 < n_chunks; c0 += 32) {
      const int c = c0 + wid;
      const uint32_t m = c < n_chunks ? ws.chunk_mask[static_cast<size_t>(e) * d.cmax + c] : 0u;
      if (lane == 0) wsum[wid] = __popc(m);
      __syncthreads();
      if (wid == 0) {
        const int x = wsum[lane];
        int xi = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int u = __shfl_up_sync(0xffffffffu, xi, o);
          if (lane >= o) xi += u;
        }
        wsum[lane] = xi - x;
        if (lane == 31) tmp[32] = xi;
      }
      __syncthreads();
      if ((m >> lane) & 1u) {
        const int f = c * 32 + lane;
        const int dst = off + run + wsum[wid] + __popc(m & ((1u << lane) - 1u));
        if (dst < 0 || dst >= d.Nmax * k || f >= n_fresh) {
          set_error(ws.err, EPOCH_DEVERR_BOUNDS);
        } else {
          ws.wl_pos[dst] = ws.fresh_pos[f];
          for (int j = 0; j < k; ++j)
            if (ws.sel[f * k + j] == e) ws.slot[f * k + j] = dst;
        }
      }
      run += tmp[32];
      __syncthreads();
    }
    return;
  }
  // ---- last CTA: offsets and tile lists
  const int cnt = tid < E ? ws.expert_cnt[tid] : 0;
  int total;
  const int off = block_excl_scan(cnt, tmp, &total);
  if (tid < E) ws.offsets[tid] = off;
  if (tid == 0) ws.offsets[E] = total;
  const int G = E + d.n_sh;
  const bool routed = tid < E;
  const bool grp = tid < G;
  const int rows = routed ? cnt : (grp ? d.n_pos : 0);
  const int r0 = routed ? off : 0;
  int tu = 0, td = 0;
  if (grp && rows > 0 && d.tn_up > 0) {
    tu = ((rows + d.tn_up - 1) / d.tn_up) * ((routed ? d.I : d.I_s) / 128);
    td = ((rows + d.tn_dn - 1) / d.tn_dn) * (d.H / 128);
  }
  int n_up, n_dn, n_hit;
  const int bu = block_excl_scan(tu, tmp, &n_up);
  const int bd = block_excl_scan(td, tmp, &n_dn);
  (void)block_excl_scan(routed && cnt > 0 ? 1 : 0, tmp, &n_hit);
  if (tu > 0) {
    const int nt = (rows + d.tn_up - 1) / d.tn_up;
    const int mt = (routed ? d.I : d.I_s) / 128;
    for (int q = 0; q < tu; ++q) {
      const int m = q / nt, tt = q % nt;
      const int slot = bu + q;
      if (slot < d.max_tiles_up)
        ws.tiles_up[slot] = make_int4(tid, m, r0 + tt * d.tn_up, min(d.tn_up, rows - tt * d.tn_up));
      else
        set_error(ws.err, EPOCH_DEVERR_BOUNDS);
    }
    (void)mt;
  }
  if (td > 0) {
    const int nt = (rows + d.tn_dn - 1) / d.tn_dn;
    for (int q = 0; q < td; ++q) {
      const int m = q / nt, tt = q % nt;
      const int slot = bd + q;
      if (slot < d.max_tiles_dn)
        ws.tiles_dn[slot] = make_int4(tid, m, r0 + tt * d.tn_dn, min(d.tn_dn, rows - tt * d.tn_dn));
      else
        set_error(ws.err, EPOCH_DEVERR_BOUNDS);
    }
  }
  if (tid == 0) {
    const int up = min(n_up, d.max_tiles_up), dn = min(n_dn, d.max_tiles_dn);
    ws.ctrl->n_hit = n_hit;
    ws.ctrl->tiles_up = up;
    ws.ctrl->tiles_dn = dn;
    ws.stats->n_hit_experts = n_hit;
    ws.stats->tiles_up = up;
    ws.stats->tiles_down = dn;
  }
}

// ---------------------------------------------------------------- permute
// Xp[l] = x[wl_pos[l]]: one warp per worklist row, 16-byte vectors.
__global__ void k_permute(Dims d, Work ws, const uint4 *__restrict__ x, int vec_per_row) {
  const KernelMark mark_(d, ws, K_PERMUTE);
  const int n = ws.ctrl->n_edges;
  const int warps = (gridDim.x * blockDim.x) >> 5;
  uint4 *xp = reinterpret_cast<uint4 *>(ws.xp);
  for (int l = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; l < n; l += warps) {
    const int t = ws.wl_pos[l];
    if (t < 0 || t >= d.n_pos) {
      if (lane_id() == 0) set_error(ws.err, EPOCH_DEVERR_BOUNDS);
      continue;
    }
    const uint4 *src = x + static_cast<size_t>(t) * vec_per_row;
    uint4 *dst = xp + static_cast<size_t>(l) * vec_per_row;
    for (int v = lane_id(); v < vec_per_row; v += 32) dst[v] = src[v];
  }
}

// ---------------------------------------------------------------- combine + cache
// Eight consecutive elements of a row, loaded/stored as one or two 16-byte vectors.
__device__ __forceinline__ void load8(const float *p, float (&v)[8]) {
  const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&v)[8]) {
  const uint4 u = *reinterpret_cast<const uint4 *>(p);
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float2 f = __bfloat1622float2(h[q]);
    v[2 * q] = f.x;
    v[2 * q + 1] = f.y;
  }
}
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

// One CTA per position, 8 elements per thread per pass. Fresh t:
// r = sum_j w_j O[slot(t, j)] (j ascending, fp32) and the cache row is refilled
// ([W] section "Liveness-Shard Parallelism": Y[F_i] = Y_F); reused t: r = the
// cached row (Y[not F_i] = C_l[not F_i]). Then y = r + shared outputs (+ x when
// residual), rounded once: the dense shard is restored at the layer boundary.
template <typename T>
__global__ void __launch_bounds__(128) k_combine(Dims d, Work ws, const T *__restrict__ x, T *__restrict__ y) {
  const KernelMark mark_(d, ws, K_COMBINE);
  const int t = blockIdx.x;
  if (t >= d.n_pos) return;
  const int f = ws.fidx[t];
  const int H = d.H, k = d.k;
  T *cache = reinterpret_cast<T *>(ws.cache) + static_cast<size_t>(t) * H;
  __shared__ int32_t slot_s[16];
  __shared__ float w_s[16];
  if (f >= 0 && threadIdx.x < k) {
    int sl = ws.slot[f * k + threadIdx.x];
    if (sl < 0 || sl >= d.Nmax * k) {
      set_error(ws.err, EPOCH_DEVERR_BOUNDS);
      sl = 0;
    }
    slot_s[threadIdx.x] = sl;
    w_s[threadIdx.x] = ws.selw[f * k + threadIdx.x];
  }
  __syncthreads();
  for (int h0 = threadIdx.x * 8; h0 < H; h0 += blockDim.x * 8) {
    float r[8];
    if (f >= 0) {
#pragma unroll
      for (int q = 0; q < 8; ++q) r[q] = 0.f;
      for (int j = 0; j < k; ++j) {
        float o[8];
        load8(ws.o_int + static_cast<size_t>(slot_s[j]) * H + h0, o);
        const float wj = w_s[j];
#pragma unroll
        for (int q = 0; q < 8; ++q) r[q] = fmaf(wj, o[q], r[q]);
      }
      store8(cache + h0, r);
    } else {
      load8(cache + h0, r);
    }
    for (int s = 0; s < d.n_sh; ++s) {
      float o[8];
      load8(ws.o_sh + (static_cast<size_t>(s) * d.Nmax + t) * H + h0, o);
#pragma unroll
      for (int q = 0; q < 8; ++q) r[q] += o[q];
    }
    if (d.residual) {
      float xv[8];
      load8(x + static_cast<size_t>(t) * H + h0, xv);
#pragma unroll
      for (int q = 0; q < 8; ++q) r[q] += xv[q];
    }
    store8(y + static_cast<size_t>(t) * H + h0, r);
  }
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

cudaError_t launch_gate_simt(const Dims &d, const Weights &w, const Work &ws, const void *x, int bf16,
                             cudaStream_t s) {
  const int outputs = d.n_pos * d.E;
  int blocks = (outputs + 7) / 8;
  if (blocks > 8 * num_sms()) blocks = 8 * num_sms();
  if (bf16) {
    static bool carve_ = (prefer_max_shared(k_gate_simt<__nv_bfloat16>) == cudaSuccess);
    (void)carve_;
    k_gate_simt<__nv_bfloat16><<<blocks, 256, 0, s>>>(d, static_cast<const __nv_bfloat16 *>(x),
                                                      static_cast<const __nv_bfloat16 *>(w.w_router), ws.gparts);
  } else {
    static bool carve_ = (prefer_max_shared(k_gate_simt<float>) == cudaSuccess);
    (void)carve_;
    k_gate_simt<float><<<blocks, 256, 0, s>>>(d, static_cast<const float *>(x),
                                              static_cast<const float *>(w.w_router), ws.gparts);
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
    k_plan_topk<N><<<blocks, 256, 0, s>>>(d, ws.gparts, w.b_router, ws.plan_counts);  \
    break;                                                                             \
  }
    EPOCH_CASE(1) EPOCH_CASE(2) EPOCH_CASE(4) EPOCH_CASE(8) EPOCH_CASE(16) EPOCH_CASE(32)
#undef EPOCH_CASE
  }
  return cudaGetLastError();
}

cudaError_t launch_plan_support(const Dims &d, const Work &ws, int32_t threshold, int all_experts,
                                cudaStream_t s) {
  static bool carve_ = (prefer_max_shared(k_plan_support) == cudaSuccess);
  (void)carve_;
  k_plan_support<<<1, 1024, 0, s>>>(d, ws, threshold, all_experts);
  return cudaGetLastError();
}

cudaError_t launch_classify(const Dims &d, const Work &ws, const uint8_t *live, const uint8_t *decoded,
                            cudaStream_t s) {
  static bool carve_ = (prefer_max_shared(k_classify) == cudaSuccess);
  (void)carve_;
  k_classify<<<1, 1024, 0, s>>>(d, ws, live, decoded);
  return cudaGetLastError();
}

cudaError_t launch_route(const Dims &d, const Weights &w, const Work &ws, cudaStream_t s) {
  const int chunks = (d.Nmax + 31) / 32;
  switch (epl_for(d.E)) {
#define EPOCH_CASE(N)                                                    \
  case N: {                                                              \
    static bool c_ = (prefer_max_shared(k_route<N>) == cudaSuccess);     \
    (void)c_;                                                            \
    k_route<N><<<chunks, 1024, 0, s>>>(d, ws, w.b_router);               \
    break;                                                               \
  }
    EPOCH_CASE(1) EPOCH_CASE(2) EPOCH_CASE(4) EPOCH_CASE(8) EPOCH_CASE(16) EPOCH_CASE(32)
#undef EPOCH_CASE
  }
  return cudaGetLastError();
}

cudaError_t launch_worklist(const Dims &d, const Work &ws, cudaStream_t s) {
  static bool carve_ = (prefer_max_shared(k_worklist) == cudaSuccess);
  (void)carve_;
  k_worklist<<<d.E + 1, 1024, 0, s>>>(d, ws);
  return cudaGetLastError();
}

cudaError_t launch_permute(const Dims &d, const Work &ws, const void *x, int bf16, cudaStream_t s) {
  const int vec = d.H * (bf16 ? 2 : 4) / 16;
  int blocks = (d.Nmax * d.k + 7) / 8;
  if (blocks > 4 * num_sms()) blocks = 4 * num_sms();
  static bool carve_ = (prefer_max_shared(k_permute) == cudaSuccess);
  (void)carve_;
  k_permute<<<blocks, 256, 0, s>>>(d, ws, static_cast<const uint4 *>(x), vec);
  return cudaGetLastError();
}

cudaError_t launch_combine(const Dims &d, const Work &ws, const void *x, void *y, int bf16, cudaStream_t s) {
  if (bf16) {
    static bool carve_ = (prefer_max_shared(k_combine<__nv_bfloat16>) == cudaSuccess);
    (void)carve_;
    k_combine<__nv_bfloat16><<<d.n_pos, 128, 0, s>>>(d, ws, static_cast<const __nv_bfloat16 *>(x),
                                                     static_cast<__nv_bfloat16 *>(y));
  } else {
    static bool carve_ = (prefer_max_shared(k_combine<float>) == cudaSuccess);
    (void)carve_;
    k_combine<float><<<d.n_pos, 128, 0, s>>>(d, ws, static_cast<const float *>(x), static_cast<float *>(y));
  }
  return cudaGetLastError();
}

cudaError_t launch_wait_test(uint32_t *err, int64_t timeout_ns, cudaStream_t s) {
  static bool carve_ = (prefer_max_shared(k_wait_test) == cudaSuccess);
  (void)carve_;
  k_wait_test<<<1, 32, 0, s>>>(err, timeout_ns);
  return cudaGetLastError();
}

}  // namespace epoch

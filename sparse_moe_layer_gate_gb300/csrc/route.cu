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
#include "topk.cuh"

namespace epoch {

const char *const kKindName[K_NUM] = {"gate",    "plan_topk",   "plan_support", "routing",
                                      "experts", "expert_down", "combine",      "wait_test"};

// ---------------------------------------------------------------- helpers

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
// G = x W_r^T + b for fp32 layers: one warp per (position, expert), lanes
// split H, fixed-order reduction (deterministic).
template <typename T>
__global__ void k_gate_simt(Dims d, const T *__restrict__ x, const T *__restrict__ wr, const float *__restrict__ bias,
                            float *__restrict__ g, Work ws) {
  if (blockIdx.x == 0) {  // counters of the next routing and expert launches
    if (threadIdx.x == 0) {
      *ws.gbar = 0u;
      *ws.route_done = 0u;
    }
  }
  clear_selection_masks(d, ws);
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
    if (lane == 0) g[static_cast<size_t>(t) * d.E + e] = acc + bias[e];
  }
}

// ---------------------------------------------------------------- block plan
// Dense top-k of every position over all experts -> hit counts (integer atomics).
template <int EPL>
__global__ void k_plan_topk(Dims d, const float *__restrict__ logits, int32_t *__restrict__ counts) {
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
    warp_topk<EPL>(v, ok, d.k, &sel, &val);
    if (lane < d.k) atomicAdd(&counts[sel], 1);
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
  for (int t = tid; t < 2 * d.Nmax; t += blockDim.x) {  // both halves of the iteration state
    ws.stamp[t] = -1;
    ws.prev_dec[t] = 0;
  }
}

// ---------------------------------------------------------------- fused routing
// Grid-wide barrier of the cooperative routing kernel: every CTA arrives once
// per phase; a CTA whose wait expires sets the timeout bit and the whole grid
// unwinds (the others time out at this or the next barrier).
__device__ __forceinline__ bool grid_sync(unsigned int *bar, unsigned int target, uint32_t *err, uint64_t tmo,
                                          int *s_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(bar, 1u);
    const uint64_t t0 = globaltimer_ns();
    int ok = 1;
    for (;;) {
      unsigned int v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(bar) : "memory");
      if (v >= target) break;
      if (globaltimer_ns() - t0 > tmo) {
        set_error(err, EPOCH_DEVERR_TIMEOUT);
        ok = 0;
        break;
      }
      __nanosleep(40);
    }
    __threadfence();
    *s_ok = ok;
  }
  __syncthreads();
  return *s_ok != 0;
}

// Tile bookkeeping of the expert kernel, written by one CTA. The groups -- the
// shared experts (every position) and the routed experts -- are listed widest
// first, so that the expert kernel, which hands tiles out in list order, ends
// on narrow tiles whose epilogues are short: the shared experts, then routed
// experts with >= 96 rows, >= 32 rows, fewer (an expert with no row holds no
// tile and its weights are never read), by id within a class. The order comes
// from a stable counting sort: per-class counts packed two to an int, two
// block scans. grp_list[p] = (token tiles of the groups before p) <<
// kGrpIdBits | group of p, grp_list[E + n_sh] = all token tiles << kGrpIdBits.
// The expert kernel decodes its tile indices from this list and the expert
// offsets; tile totals and the number of hit experts go to the control block
// and the statistics.
__device__ void write_group_tiles(const Dims &d, const Work &ws, const int32_t *s_off, int32_t *tmp, int n) {
  const int tid = threadIdx.x;
  const int E = d.E, G2 = E + d.n_sh;
  // thread tid holds groups 2 tid, 2 tid + 1 (id order; G2 <= 2 * kRoutingThreads)
  int cls[2] = {-1, -1}, nt[2] = {0, 0}, hit = 0;
  int pk0 = 0, pk1 = 0;  // this thread's count of each class: 0, 1 in pk0, 2, 3 in pk1 (16-bit fields)
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int g = 2 * tid + h;
    if (g < G2) {
      const bool shared = g >= E;
      const int rows = shared ? n : s_off[g + 1] - s_off[g];
      nt[h] = d.tn > 0 ? (rows + d.tn - 1) / d.tn : 0;
      hit += !shared && rows > 0;
      const int c = shared ? 3 : rows >= 96 ? 2 : rows >= 32 ? 1 : 0;
      cls[h] = c;
      if (c < 2) pk0 += 1 << (16 * (c & 1));
      else pk1 += 1 << (16 * (c & 1));
    }
  }
  int tot0, tot1, n_hit;
  const int ex0 = block_excl_scan(pk0, tmp, &tot0);
  const int ex1 = block_excl_scan(pk1, tmp, &tot1);
  (void)block_excl_scan(hit, tmp, &n_hit);
  auto field = [](int packed, int c) { return (packed >> (16 * (c & 1))) & 0xffff; };
  const int count3 = field(tot1, 3), count2 = field(tot1, 2), count1 = field(tot0, 1);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int c = cls[h];
    if (c < 0) continue;
    const int base = c == 3 ? 0 : c == 2 ? count3 : c == 1 ? count3 + count2 : count3 + count2 + count1;
    const int pos = base + field(c < 2 ? ex0 : ex1, c) + (h == 1 && cls[0] == c ? 1 : 0);
    ws.grp_list[pos] = (nt[h] << kGrpIdBits) | (2 * tid + h);  // token tiles until the prefix below
  }
  __syncthreads();  // the list in sorted order is visible to the whole CTA
  int g_at[2] = {0, 0}, nt_at[2] = {0, 0};
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int p = 2 * tid + h;
    if (p < G2) {
      const int v = ws.grp_list[p];
      g_at[h] = v & ((1 << kGrpIdBits) - 1);
      nt_at[h] = v >> kGrpIdBits;
    }
  }
  int total;
  const int before = block_excl_scan(nt_at[0] + nt_at[1], tmp, &total);
  if (total >= (1 << (31 - kGrpIdBits))) {
    if (tid == 0) set_error(ws.err, EPOCH_DEVERR_BOUNDS);
    total = 0;
  }
  if (2 * tid < G2) ws.grp_list[2 * tid] = (before << kGrpIdBits) | g_at[0];
  if (2 * tid + 1 < G2) ws.grp_list[2 * tid + 1] = ((before + nt_at[0]) << kGrpIdBits) | g_at[1];
  if (tid == 0) {
    ws.grp_list[G2] = total << kGrpIdBits;
    const int t_sh = d.tn > 0 ? d.n_sh * ((n + d.tn - 1) / d.tn) : 0;
    const int up = d.tn > 0 && total > 0 ? (d.I_s / 128) * t_sh + (d.I / 128) * (total - t_sh) : 0;
    const int dn = d.tn > 0 && total > 0 ? (d.H / kBmDn) * total : 0;
    ws.ctrl->n_hit = n_hit;
    ws.ctrl->tiles_up = up;
    ws.ctrl->tiles_dn = dn;
    ws.stats->n_hit_experts = n_hit;
    ws.stats->tiles_up = up;
    ws.stats->tiles_down = dn;
  }
}

// Position categories of the routing kernel, and the per-CTA counters it sums.
enum Category { C_LIVE = 0, C_NEW, C_MISS, C_STALE, C_REUSE, C_BAD, C_ANOM, C_REUSE_BEFORE };
static_assert(C_REUSE_BEFORE < kBlkFields, "category counters");

// One cooperative launch (one CTA per SM, 16 warps) runs the whole routing
// side of an iteration in four phases separated by grid barriers:
//  A  classify ([W] section "Liveness-Shard Parallelism"): each CTA takes a
//     slice of positions -- live (still Mask), newly decoded (D_i \ D_{i-1}),
//     decoded without a row, decoded with a row at least R iterations old, or
//     stable decoded (Z_i, reuses its cached row). A decoded -> live transition
//     anywhere, or a host-detected mismatch, makes the iteration full fresh
//     ([W] sections "Two Clocks", "cold、hot-update、hot-skip").
//  A' compaction: slice offsets from the per-CTA counts, an ascending fresh
//     list, stamps of fresh rows, the new previous-decoded flags, statistics.
//  B  one warp per fresh position: top-k of its logits over the support mask
//     (every expert on a fallback), softmax weights over the selected logits
//     ([W] section "Expert Atlas", step three); bit (f mod 32) of word
//     (e, f / 32) marks that fresh position f selected expert e.
//  C  worklist ([W] section "FreshLane Dispatch": pack, count exchange,
//     compact dispatch -- here on chip): expert offsets from the counts; one
//     warp per (expert, 32-position chunk) places its rows at
//     offset(e) + rows of e in earlier chunks + bits below p, so rows are
//     grouped by expert with positions ascending, and copies each row of x
//     into the compact buffer. CTA 0 writes the grouped-GEMM tile lists.
template <int EPL>
__device__ __forceinline__ void routing_body(const Dims &d, const Work &ws,
                                             const uint8_t *__restrict__ live, const uint8_t *__restrict__ decoded,
                                             const uint4 *__restrict__ x, int vec_per_row) {
  const KernelMark mark_(d, ws, K_ROUTING);
  int64_t *trace_r = (d.trace && blockIdx.x < kTraceCtas)
                         ? ws.trace + (3ull * kTraceCtas + blockIdx.x) * kTraceFields
                         : nullptr;
  if (trace_r && threadIdx.x == 0) trace_r[0] = static_cast<int64_t>(globaltimer_ns());
  pdl_trigger();  // the expert kernel may start its launch; it waits on route_done
  __shared__ int32_t tmp[33];
  __shared__ int32_t s_cat[kBlkFields];
  __shared__ int32_t s_off[1025];
  __shared__ int16_t s_rank[kRoutingThreads];  // rank of each slice row in the slice's fresh rows, -1 reused
  __shared__ int s_ok;
  const int G = gridDim.x, b = blockIdx.x, tid = threadIdx.x;
  const int lane = lane_id(), wid = warp_id(), nwarps = kRoutingThreads / 32;
  const int n = d.n_pos, E = d.E, k = d.k;
  const uint64_t tmo = static_cast<uint64_t>(d.timeout_ns);

  // ---- phase 1a, while the gate kernel may still run: it reads only the
  // masks and the previous iteration's state and writes only this iteration's.
  // Every CTA classifies every position from the previous state
  // (double-buffered: read half rd, write half rd ^ 1, so no CTA can overwrite
  // what another still reads), which gives the anomaly flag, the fresh count
  // and this CTA's offset in the fresh list; then it writes the new state of
  // its own slice of positions.
  const int rd = d.state_rd & 1, wr = rd ^ 1;
  const int32_t *stamp_old = ws.stamp + static_cast<size_t>(rd) * d.Nmax;
  const uint8_t *prev_old = ws.prev_dec + static_cast<size_t>(rd) * d.Nmax;
  int32_t *stamp_new = ws.stamp + static_cast<size_t>(wr) * d.Nmax;
  uint8_t *prev_new = ws.prev_dec + static_cast<size_t>(wr) * d.Nmax;
  const int per = (n + G - 1) / G;  // <= kRoutingThreads (the launch checks the grid)
  const int lo = min(b * per, n), hi = min(lo + per, n);
  if (tid < kBlkFields) s_cat[tid] = 0;
  for (int g = b * kRoutingThreads + tid; g < E + d.n_sh; g += G * kRoutingThreads) ws.done_up[g] = 0;
  if (b == 0 && tid == 0) *ws.tile_ctr = 0;  // the expert kernel hands tiles out from this counter
  // positions beyond this call's n_pos keep their state
  for (int t = n + b * kRoutingThreads + tid; t < d.Nmax; t += G * kRoutingThreads) {
    stamp_new[t] = stamp_old[t];
    prev_new[t] = prev_old[t];
  }
  // category of position t: live (still Mask, or not decoded), newly decoded,
  // decoded without a row, decoded with a row at least R iterations old, or
  // stable decoded (reuses its cached row)
  // (packed: category | live << 4 | contradictory flags << 5 | decoded -> live << 6)
  auto classify = [&](int t) -> int {
    const bool lv = live[t] != 0, dc = decoded[t] != 0;
    const bool il = lv || !dc, prev = prev_old[t] != 0;
    const int st = stamp_old[t];
    const int flags = (il ? 16 : 0) | (lv == dc ? 32 : 0) | (il && prev ? 64 : 0);
    if (il) return C_LIVE | flags;
    if (!prev) return C_NEW | flags;
    if (st < 0) return C_MISS | flags;
    if (d.R != INT_MAX && d.iter - st >= d.R) return C_STALE | flags;
    return C_REUSE | flags;
  };
  {
    int cnt[kBlkFields];
#pragma unroll
    for (int c = 0; c < kBlkFields; ++c) cnt[c] = 0;
    for (int t = tid; t < n; t += kRoutingThreads) {
      const int code = classify(t), c = code & 15;
#pragma unroll
      for (int q = 0; q < C_BAD; ++q) cnt[q] += c == q;
      cnt[C_BAD] += (code >> 5) & 1;
      cnt[C_ANOM] |= (code >> 6) & 1;
      cnt[C_REUSE_BEFORE] += c == C_REUSE && t < lo;
    }
#pragma unroll
    for (int c = 0; c < kBlkFields; ++c) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) cnt[c] += __shfl_xor_sync(0xffffffffu, cnt[c], o);
    }
    __syncthreads();  // s_cat cleared
    if (lane == 0) {
#pragma unroll
      for (int c = 0; c < kBlkFields; ++c) atomicAdd(&s_cat[c], cnt[c]);
    }
    __syncthreads();
  }
  const bool any_anom = s_cat[C_ANOM] != 0;
  const bool force = d.host_fallback || any_anom;
  const int n_fresh = force ? n : n - s_cat[C_REUSE];
  const int fresh_before = force ? lo : lo - s_cat[C_REUSE_BEFORE];
  if (b == 0 && tid == 0) {
    const int fb = (d.host_fallback ? 1 : 0) | (any_anom ? 2 : 0);
    ws.ctrl->n_fresh = n_fresh;
    ws.ctrl->fallback = fb;
    ws.ctrl->n_edges = n_fresh * k;
    epoch_iter_stats *st = ws.stats;
    st->iteration = d.iter;
    st->n_pos = n;
    st->n_live = s_cat[C_LIVE];
    st->n_new = s_cat[C_NEW];
    st->n_miss = s_cat[C_MISS];
    st->n_stale = s_cat[C_STALE];
    st->n_forced = force ? s_cat[C_REUSE] : 0;
    st->n_reuse = force ? 0 : s_cat[C_REUSE];
    st->n_fresh = n_fresh;
    st->n_edges = n_fresh * k;
    st->support_len = fb ? E : ws.ctrl->support_len;
    st->fallback = fb;
    st->bad_flags = s_cat[C_BAD];
    if (s_cat[C_BAD]) set_error(ws.err, EPOCH_DEVERR_FLAGS);
  }
  {
    const int t = lo + tid;
    const bool mine = t < hi;
    bool il = false, fresh = false;
    if (mine) {
      const int code = classify(t);
      il = (code & 16) != 0;
      fresh = (code & 15) != C_REUSE || force;
    }
    int slice_fresh;
    const int rank = block_excl_scan(fresh ? 1 : 0, tmp, &slice_fresh);
    if (mine) {
      if (fresh) {
        const int f = fresh_before + rank;
        ws.fresh_pos[f] = t;
        ws.fidx[t] = f;
        stamp_new[t] = d.iter;
      } else {
        ws.fidx[t] = -1;
        stamp_new[t] = stamp_old[t];
      }
      prev_new[t] = il ? 0 : 1;
      s_rank[tid] = static_cast<int16_t>(fresh ? rank : -1);
    }
  }
  __syncthreads();  // s_rank
  if (trace_r && tid == 0) trace_r[1] = static_cast<int64_t>(globaltimer_ns());

  // ---- phase 1b, after the gate kernel: one warp per fresh row of the slice
  // takes the top-k of its logits over the support mask (every expert on a
  // fallback) and the softmax weights over the selected logits ([W] section
  // "Expert Atlas", step three); bit (f mod 32) of word (e, f / 32) marks that
  // fresh position f selected expert e (words zeroed by the gate kernel).
  pdl_wait();
  if (trace_r && tid == 0) trace_r[2] = static_cast<int64_t>(globaltimer_ns());
  for (int r = wid; r < hi - lo; r += nwarps) {
    const int rank = s_rank[r];
    if (rank < 0) continue;
    const int t = lo + r, f = fresh_before + rank, e0 = lane * EPL;
    float v[EPL];
    lane_logits<EPL>(ws.logits + static_cast<size_t>(t) * E, E, v);
    bool ok[EPL];
#pragma unroll
    for (int c = 0; c < EPL; ++c) {
      const int e = e0 + c;
      ok[c] = e < E && (force || ws.support_mask[e]);
    }
    int sel;
    float val;
    warp_topk<EPL>(v, ok, k, &sel, &val);
    const float top = __shfl_sync(0xffffffffu, val, 0);
    const float ex = lane < k ? expf(val - top) : 0.f;
    float denom = 0.f;  // summed in selection order j = 0..k-1 (deterministic)
    for (int j = 0; j < k; ++j) denom += __shfl_sync(0xffffffffu, ex, j);
    if (lane < k) {
      if (sel < 0 || sel >= E || f >= n_fresh) {
        set_error(ws.err, EPOCH_DEVERR_BOUNDS);
      } else {
        ws.sel[f * k + lane] = sel;
        ws.selw[f * k + lane] = ex / denom;
        atomicOr(&ws.chunk_mask[static_cast<size_t>(sel) * d.cmax + (f >> 5)], 1u << (f & 31));
      }
    }
  }
  if (!grid_sync(ws.gbar, 1u * G, ws.err, tmo, &s_ok)) return;
  if (trace_r && tid == 0) trace_r[3] = static_cast<int64_t>(globaltimer_ns());

  // ---- phase C: expert offsets, worklist rows, compact copies of x, tile lists
  const int fresh_chunks = (n_fresh + 31) / 32;
  {
    // rows of each expert = popcount of its selection masks (every CTA derives
    // the offsets itself; no global counters)
    int cnt2[2] = {0, 0};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int e = 2 * tid + h;
      if (e < E) {
        const uint32_t *row = ws.chunk_mask + static_cast<size_t>(e) * d.cmax;
        int a0 = 0, a1 = 0, a2 = 0, a3 = 0;
        int c = 0;
        for (; c + 4 <= fresh_chunks; c += 4) {
          a0 += __popc(row[c]);
          a1 += __popc(row[c + 1]);
          a2 += __popc(row[c + 2]);
          a3 += __popc(row[c + 3]);
        }
        for (; c < fresh_chunks; ++c) a0 += __popc(row[c]);
        cnt2[h] = a0 + a1 + a2 + a3;
      }
    }
    const int c0 = cnt2[0], c1 = cnt2[1];
    int tot;
    const int o = block_excl_scan(c0 + c1, tmp, &tot);
    if (2 * tid < E) s_off[2 * tid] = o;
    if (2 * tid + 1 < E) s_off[2 * tid + 1] = o + c0;
    if (tid == 0) s_off[E] = tot;
    __syncthreads();
  }
  // With more than one CTA, CTA 0 writes the expert offsets and the group list
  // while the others place the worklist rows, meet at a second barrier and copy
  // each worklist row of x into the compact buffer; the expert kernel starts
  // once every CTA has counted itself done.
  const bool split = G > 1;
  const int wb = split ? b - 1 : b, wg = split ? G - 1 : G;  // worker CTAs
  if (!(split && b == 0)) {
    for (int pair = wb * nwarps + wid; pair < E * fresh_chunks; pair += wg * nwarps) {
      const int e = pair / fresh_chunks, c = pair % fresh_chunks;
      const uint32_t *row = ws.chunk_mask + static_cast<size_t>(e) * d.cmax;
      const uint32_t m = row[c];
      if (m == 0u) continue;
      int before_c = 0;
      for (int c2 = lane; c2 < c; c2 += 32) before_c += __popc(row[c2]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) before_c += __shfl_xor_sync(0xffffffffu, before_c, o);
      if ((m >> lane) & 1u) {  // lane p places the edge of fresh position 32 c + p
        const int f = c * 32 + lane;
        const int dst = s_off[e] + before_c + __popc(m & ((1u << lane) - 1u));
        if (dst < 0 || dst >= d.Nmax * k || f >= n_fresh) {
          set_error(ws.err, EPOCH_DEVERR_BOUNDS);
        } else {
          ws.wl_pos[dst] = ws.fresh_pos[f];
          for (int j = 0; j < k; ++j)
            if (ws.sel[f * k + j] == e) ws.slot[f * k + j] = dst;
        }
      }
    }
    if (trace_r && tid == 0) trace_r[4] = static_cast<int64_t>(globaltimer_ns());
    if (split) {
      if (!grid_sync(ws.gbar, 1u * G + (G - 1), ws.err, tmo, &s_ok)) return;
    } else {
      __syncthreads();
    }
  } else if (trace_r && tid == 0) {
    trace_r[4] = static_cast<int64_t>(globaltimer_ns());
  }
  if (b == 0) {
    for (int e = tid; e <= E; e += kRoutingThreads) ws.offsets[e] = s_off[e];
    if (trace_r && tid == 0) trace_r[5] = static_cast<int64_t>(globaltimer_ns());
    write_group_tiles(d, ws, s_off, tmp, n);
    if (trace_r && tid == 0) trace_r[6] = static_cast<int64_t>(globaltimer_ns());
    if (split) return;
  }

  // ---- phase 3: copy each worklist row of x into the compact buffer
  const int n_edges = n_fresh * k;
  for (int l = wb * nwarps + wid; l < n_edges; l += wg * nwarps) {
    const int tp = ws.wl_pos[l];
    if (tp < 0 || tp >= n) {
      if (lane == 0) set_error(ws.err, EPOCH_DEVERR_BOUNDS);
      continue;
    }
    const uint4 *src = x + static_cast<size_t>(tp) * vec_per_row;
    uint4 *out = reinterpret_cast<uint4 *>(ws.xp) + static_cast<size_t>(l) * vec_per_row;
    // all loads of a batch are issued before its stores (the destination may
    // alias nothing the loads read, but the compiler cannot know that)
    for (int v0 = 0; v0 < vec_per_row; v0 += 32 * 8) {
      uint4 buf[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int v = v0 + q * 32 + lane;
        if (v < vec_per_row) buf[q] = __ldg(src + v);
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int v = v0 + q * 32 + lane;
        if (v < vec_per_row) out[v] = buf[q];
      }
    }
  }
  if (trace_r && tid == 0) trace_r[5] = static_cast<int64_t>(globaltimer_ns());
}

// The launch: after its last write every CTA counts itself into route_done
// (zeroed by the gate kernel) with release semantics; the expert kernel, which
// may already be running (programmatic dependent launch), acquires that count
// instead of waiting for this grid to retire.
template <int EPL>
__global__ void __launch_bounds__(kRoutingThreads) k_routing(Dims d, Work ws,
                                                             const uint8_t *__restrict__ live,
                                                             const uint8_t *__restrict__ decoded,
                                                             const uint4 *__restrict__ x, int vec_per_row) {
  routing_body<EPL>(d, ws, live, decoded, x, vec_per_row);
  __syncthreads();  // every return in the body is uniform over the CTA
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(ws.route_done, 1u);
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

// One CTA per position, 8 elements per thread per pass. Expert outputs O are
// stored in the layer dtype. Fresh t:
// r = sum_j w_j O[slot(t, j)] (j ascending, fp32) and the cache row is refilled
// ([W] section "Liveness-Shard Parallelism": Y[F_i] = Y_F); reused t: r = the
// cached row (Y[not F_i] = C_l[not F_i]). Then y = r + shared outputs (+ x when
// residual), rounded once: the dense shard is restored at the layer boundary.
template <typename T>
__global__ void __launch_bounds__(128) k_combine(Dims d, Work ws, const T *__restrict__ x, T *__restrict__ y) {
  const KernelMark mark_(d, ws, K_COMBINE);
  pdl_wait();
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
        load8(static_cast<const T *>(ws.o_int) + static_cast<size_t>(slot_s[j]) * H + h0, o);
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
      load8(static_cast<const T *>(ws.o_sh) + (static_cast<size_t>(s) * d.Nmax + t) * H + h0, o);
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

// One routing CTA per SM (at most kMaxRoutingGrid). The grid barriers need
// every CTA resident at once, which holds without a cooperative launch: the
// kernel is launched while the gate kernel (at most one CTA per SM, and never
// waiting on routing) may still run, so CTAs that do not fit yet start as gate
// CTAs retire, and the kernels after it are launched only once every routing
// CTA has started (programmatic launch trigger). Every wait is bounded anyway.
int routing_grid() { return num_sms() < kMaxRoutingGrid ? num_sms() : kMaxRoutingGrid; }

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
                          bool cooperative, bool programmatic) {
  static bool pdl_ok = true;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (cooperative) {
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = 1;
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
    k_plan_topk<N><<<blocks, 256, 0, s>>>(d, ws.logits, ws.plan_counts);              \
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

// Cooperative launch (the phases wait on one another through grid barriers,
// so every CTA must be resident): one CTA per SM, capped at what fits.
cudaError_t launch_routing(const Dims &d, const Weights &w, const Work &ws, const uint8_t *live,
                           const uint8_t *decoded, const void *x, int bf16, cudaStream_t s) {
  const int grid = routing_grid();
  // slices of at most kRoutingThreads positions per CTA
  const int min_grid = (d.n_pos + kRoutingThreads - 1) / kRoutingThreads;
  if (grid < min_grid) return cudaErrorInvalidConfiguration;
  Dims dd = d;
  Work ww = ws;
  const int vec = d.H * (bf16 ? 2 : 4) / 16;
  const uint4 *xv = static_cast<const uint4 *>(x);
  void *args[] = {&dd, &ww, const_cast<uint8_t **>(&live), const_cast<uint8_t **>(&decoded),
                  const_cast<uint4 **>(&xv), const_cast<int *>(&vec)};
  switch (epl_for(d.E)) {
#define EPOCH_CASE(N)                                                                                    \
  case N: {                                                                                              \
    static bool c_ = (prefer_max_shared(k_routing<N>) == cudaSuccess);                                   \
    (void)c_;                                                                                            \
    return launch_kernel(reinterpret_cast<void *>(k_routing<N>), dim3(grid), dim3(kRoutingThreads), 0, s, args, \
                         false, true);                                                                   \
  }
    EPOCH_CASE(1) EPOCH_CASE(2) EPOCH_CASE(4) EPOCH_CASE(8) EPOCH_CASE(16) EPOCH_CASE(32)
#undef EPOCH_CASE
  }
  return cudaErrorInvalidValue;
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
                         false, true);
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

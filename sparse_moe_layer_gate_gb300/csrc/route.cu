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
#include "select.cuh"
#include "topk.cuh"

namespace epoch {

const char *const kKindName[K_NUM] = {"gate",    "plan_topk",   "plan_support", "routing", "experts",
                                      "expert_down", "combine", "wait_test", "select", "permute"};

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

// Exclusive scan of four values at once over a CTA of up to 1024 threads
// (independent components, one pass); *total gets the sums.
__device__ __forceinline__ int4 block_excl_scan4(int4 v, int4 *warp_tmp, int4 *total) {
  const int lane = lane_id(), wid = warp_id(), nw = (blockDim.x + 31) >> 5;
  auto scan = [&](int4 a) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int ux = __shfl_up_sync(0xffffffffu, a.x, o), uy = __shfl_up_sync(0xffffffffu, a.y, o);
      const int uz = __shfl_up_sync(0xffffffffu, a.z, o), uw = __shfl_up_sync(0xffffffffu, a.w, o);
      if (lane >= o) {
        a.x += ux;
        a.y += uy;
        a.z += uz;
        a.w += uw;
      }
    }
    return a;
  };
  const int4 incl = scan(v);
  if (lane == 31) warp_tmp[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int4 x = lane < nw ? warp_tmp[lane] : make_int4(0, 0, 0, 0);
    const int4 xi = scan(x);
    warp_tmp[lane] = make_int4(xi.x - x.x, xi.y - x.y, xi.z - x.z, xi.w - x.w);
    if (lane == 31) warp_tmp[32] = xi;
  }
  __syncthreads();
  const int4 b = warp_tmp[wid];
  *total = warp_tmp[32];
  __syncthreads();
  return make_int4(b.x + incl.x - v.x, b.y + incl.y - v.y, b.z + incl.z - v.z, b.w + incl.w - v.w);
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
    if (lane < d.k && sel >= 0) atomicAdd(&counts[sel], 1);
  }
}

// One CTA: rank experts by (count desc, id asc), take the smallest prefix whose
// counts reach `threshold` (at least k; every expert when all_experts), and,
// for a block plan (cold path), clear the block's stamps and previous-decoded
// flags; a hot update keeps them.
__global__ void __launch_bounds__(1024) k_plan_support(Dims d, Work ws, int32_t threshold, int all_experts,
                                                       int clear_state, int32_t *ids_out, int32_t *len_out) {
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
    if (ids_out) ids_out[rank] = tid;
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
  if (tid == 0) {
    ws.ctrl->support_len = len;
    if (len_out) *len_out = len;
  }
  if (clear_state) {
    for (int t = tid; t < 2 * d.Nmax; t += blockDim.x) {  // both halves of the iteration state
      ws.stamp[t] = -1;
      ws.prev_dec[t] = 0;
    }
  }
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
  const bool force = d.host_fallback != 0 || anom;
  uint32_t *words = words_written(d, ws);
  const int lane = lane_id(), warps = gridDim.x * (blockDim.x >> 5);
  for (int t = blockIdx.x * (blockDim.x >> 5) + warp_id(); t < d.n_pos; t += warps) {
    int fresh = 0;
    if (lane == 0) fresh = classify_and_update(d, ws, live, decoded, t, force) ? 1 : 0;
    fresh = __shfl_sync(0xffffffffu, fresh, 0);
    if (!fresh) continue;
    float v[EPL];
    lane_logits<EPL>(ws.logits + static_cast<size_t>(t) * d.E, d.E, v);
    select_position<EPL>(d, ws, t, v, ws.support_mask, force, words, s_scr[warp_id()], bias);
  }
}

// ---------------------------------------------------------------- worklist
// One CTA builds the iteration's worklist from the selection words the gate
// (or select) kernel set ([W] section "FreshLane Dispatch": pack, count
// exchange -> offsets, compact dispatch -- here the count exchange is a
// popcount over per-expert bitmasks on one chip). Only experts that can hold a
// selection are visited: the support, or every expert on a fallback. Every
// step before the worklist is published reads shared memory only, after one
// batched load of the candidates' words (global memory round trips, not
// arithmetic, bound this kernel):
//  1 rows of each candidate expert and per-word prefixes (one warp per expert);
//  2 expert offsets (scan), the expert kernel's group list and tile counts;
//  3 worklist positions, expert-major, positions ascending: the row of fresh
//    position t for expert e is offset(e) + rows of e before t;
//  4 publish (route_done = this call's sequence number, release), so the
//    expert kernel, already running, starts on the routed tiles;
//  5 then, off the critical path: the ascending fresh list, the worklist row of
//    every selection (for the combine), statistics, the state of positions
//    beyond n_pos, the cleared selection words and shared-expert counters of
//    the next iteration.
constexpr int kRouteSmemWords = 12 * 1024;  // candidate words (and prefixes) kept in shared memory

__global__ void __launch_bounds__(kRouteThreads, 1) k_route(Dims d, Work ws) {
  const KernelMark mark_(d, ws, K_ROUTING);
  pdl_trigger();  // the expert kernel may start its launch; it waits on route_done for routed tiles
  extern __shared__ uint32_t s_dyn[];
  __shared__ int32_t tmp[33];
  __shared__ int4 tmp4[33];
  __shared__ int32_t s_off[1025];
  __shared__ int16_t s_cand[1024];  // candidate experts (support ranking, or every expert)
  __shared__ int16_t s_cidx[1024];  // candidate index of an expert, -1 if none
  __shared__ int32_t s_cat[8];
  __shared__ int s_force, s_anom, s_supp;
  const int tid = threadIdx.x, lane = lane_id(), wid = warp_id(), nw = kRouteThreads / 32;
  const int n = d.n_pos, E = d.E, k = d.k, cmax = d.cmax;
  const int nch = (n + 31) >> 5;
  const int rd = d.state_rd & 1, wr = rd ^ 1;
  int64_t *trace = (d.trace && blockIdx.x < kTraceCtas) ? ws.trace + (3ull * kTraceCtas + blockIdx.x) * kTraceFields
                                                         : nullptr;
  if (trace && tid == 0) {
    trace[0] = static_cast<int64_t>(globaltimer_ns());
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    trace[7] = smid;
  }
  // the block plan (written before this iteration began) can be read at once
  if (tid < 8) s_cat[tid] = 0;
  if (tid == 0) s_supp = min(E, ws.ctrl->support_len);
  for (int e = tid; e < E; e += kRouteThreads) s_cand[e] = static_cast<int16_t>(ws.support_ids[e]);
  for (int e = tid; e <= E; e += kRouteThreads) s_off[e] = 0;
  pdl_wait();  // the gate / select kernel has finished: selection words, selections, codes
  if (trace && tid == 0) trace[1] = static_cast<int64_t>(globaltimer_ns());
  const uint32_t *words = ws.sel_words + static_cast<size_t>(wr) * E * cmax;

  // Candidates: the support, or every expert on a host-detected fallback.
  // Their words are requested together with the decoded -> live scan of the
  // codes the gate wrote (one round trip); an anomaly found there turns the
  // iteration into a fallback and the words of every expert are loaded.
  uint32_t *sw = s_dyn;
  int32_t *sp = reinterpret_cast<int32_t *>(s_dyn + kRouteSmemWords);
  auto load_words = [&](int n_c) {
    for (int q0 = tid; q0 < n_c * nch; q0 += kRouteThreads * 8) {
      uint32_t v[8];
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const int q = q0 + b * kRouteThreads;
        v[b] = q < n_c * nch ? words[static_cast<size_t>(s_cand[q / nch]) * cmax + q % nch] : 0u;
      }
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const int q = q0 + b * kRouteThreads;
        if (q < n_c * nch) sw[q] = v[b];
      }
    }
  };
  if (d.host_fallback)
    for (int e = tid; e < E; e += kRouteThreads) s_cand[e] = static_cast<int16_t>(e);
  __syncthreads();
  int n_cand = d.host_fallback ? E : s_supp;
  bool in_smem = n_cand * nch <= kRouteSmemWords;
  {
    int anom = 0;
    for (int t = tid; t < n; t += kRouteThreads) anom |= ws.cat[t] & kCodeAnom;
    if (in_smem) load_words(n_cand);
    const int any = __syncthreads_or(anom);
    if (tid == 0) {
      s_anom = any != 0;
      s_force = (d.host_fallback != 0 || any != 0) ? 1 : 0;
    }
    __syncthreads();
  }
  const bool force = s_force != 0;
  if (force && !d.host_fallback) {  // anomaly: every expert is a candidate
    for (int e = tid; e < E; e += kRouteThreads) s_cand[e] = static_cast<int16_t>(e);
    __syncthreads();
    n_cand = E;
    in_smem = n_cand * nch <= kRouteSmemWords;
    if (in_smem) load_words(n_cand);
  }
  for (int e = tid; e < E; e += kRouteThreads) s_cidx[e] = -1;
  __syncthreads();
  for (int i = tid; i < n_cand; i += kRouteThreads) s_cidx[s_cand[i]] = static_cast<int16_t>(i);
  int64_t *trace2 = trace ? ws.trace + (5ull * kTraceCtas + blockIdx.x) * kTraceFields : nullptr;
  if (trace2 && tid == 0) trace2[0] = static_cast<int64_t>(globaltimer_ns());
  __syncthreads();
  auto word = [&](int ci, int c) -> uint32_t {
    return in_smem ? sw[ci * nch + c] : words[static_cast<size_t>(s_cand[ci]) * cmax + c];
  };
  auto pre = [&](int ci, int c) -> int32_t & {
    return in_smem ? sp[ci * nch + c] : ws.pre[static_cast<size_t>(s_cand[ci]) * cmax + c];
  };

  // ---- 1: rows of each candidate expert and the per-word prefixes
  {
    const int cpl = (nch + 31) / 32;
    for (int ci = wid; ci < n_cand; ci += nw) {
      const int c0 = min(nch, lane * cpl), c1 = min(nch, c0 + cpl);
      int sum = 0;
      for (int c = c0; c < c1; ++c) sum += __popc(word(ci, c));
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
      }
      int run = incl - sum;
      for (int c = c0; c < c1; ++c) {
        pre(ci, c) = run;
        run += __popc(word(ci, c));
      }
      if (lane == 31) s_off[s_cand[ci]] = incl;  // count, scanned below
    }
  }
  __syncthreads();
  if (trace && tid == 0) trace[2] = static_cast<int64_t>(globaltimer_ns());

  // ---- 2: one scan over the experts in id order (thread tid owns [tid * gpt,
  // tid * gpt + gpt)) gives the expert offsets and, per row-count class of the
  // group list (2: >= 96 rows, 1: >= 32, 0: fewer; listed in that order, by id
  // within a class), the list positions and token-tile prefixes: .x rows,
  // .y experts of class 0 | class 1 << 16, .z experts of class 2 | its tiles
  // << 16, .w tiles of class 0 | class 1 << 16.
  int n_edges, n_tiles;
  {
    const int gpt = (E + kRouteThreads - 1) / kRouteThreads;
    const int g0 = tid * gpt;
    auto cls_of = [](int r) { return r >= 96 ? 2 : r >= 32 ? 1 : 0; };
    int c[4] = {0, 0, 0, 0};
    int4 v = make_int4(0, 0, 0, 0);
#pragma unroll
    for (int h = 0; h < 4; ++h)
      if (h < gpt && g0 + h < E) {
        const int r = s_off[g0 + h], k2 = cls_of(r), nt = d.tn > 0 ? (r + d.tn - 1) / d.tn : 0;
        c[h] = r;
        v.x += r;
        if (k2 == 0) {
          v.y += 1;
          v.w += nt;
        } else if (k2 == 1) {
          v.y += 1 << 16;
          v.w += nt << 16;
        } else {
          v.z += 1 | (nt << 16);
        }
      }
    int4 tot;
    const int4 ex = block_excl_scan4(v, reinterpret_cast<int4 *>(tmp4), &tot);
    const int n2 = tot.z & 0xffff, n1 = tot.y >> 16;
    const int t2 = tot.z >> 16, t1 = tot.w >> 16, t0 = tot.w & 0xffff;
    const int pos_base[3] = {n2 + n1, n2, 0};
    const int tile_base[3] = {t2 + t1, t2, 0};
    int rank[3] = {ex.y & 0xffff, ex.y >> 16, ex.z & 0xffff};
    int tb[3] = {ex.w & 0xffff, ex.w >> 16, ex.z >> 16};
    int before = ex.x;
    n_edges = tot.x;
    n_tiles = t0 + t1 + t2;
#pragma unroll
    for (int h = 0; h < 4; ++h)
      if (h < gpt && g0 + h < E) {
        const int e = g0 + h, r = c[h], k2 = cls_of(r), nt = d.tn > 0 ? (r + d.tn - 1) / d.tn : 0;
        s_off[e] = before;
        ws.offsets[e] = before;
        before += r;
        ws.grp_list[pos_base[k2] + rank[k2]++] = ((tile_base[k2] + tb[k2]) << kGrpIdBits) | e;
        tb[k2] += nt;
      }
    if (tid == 0) {
      s_off[E] = n_edges;
      ws.offsets[E] = n_edges;
      ws.grp_list[E] = n_tiles << kGrpIdBits;
      ws.ctrl->tiles_up = d.tn > 0 ? (d.I / 128) * n_tiles : 0;
      ws.ctrl->tiles_dn = d.tn > 0 ? (d.H / kBmDn) * n_tiles : 0;
    }
  }
  __syncthreads();
  if (trace2 && tid == 0) trace2[1] = static_cast<int64_t>(globaltimer_ns());
  for (int g = tid; g < E; g += kRouteThreads) ws.done_up[g] = 0;
  if (tid == 0) {
    ws.tile_ctr[0] = 0;  // routed tiles drawn
    ws.tile_ctr[2] = 0;  // 16-byte vectors of worklist rows copied into xp
    ws.ctrl->n_edges = n_edges;
  }
  if (trace && tid == 0) trace[3] = static_cast<int64_t>(globaltimer_ns());

  // ---- 3: worklist positions, one thread per candidate word
  for (int q = tid; q < n_cand * nch; q += kRouteThreads) {
    const int ci = q / nch, c = q - ci * nch;
    uint32_t w = word(ci, c);
    if (w == 0u) continue;
    int dst = s_off[s_cand[ci]] + pre(ci, c);
    while (w) {
      const int b = __ffs(w) - 1;
      w &= w - 1u;
      if (dst < 0 || dst >= d.Nmax * k) {
        set_error(ws.err, EPOCH_DEVERR_BOUNDS);
        break;
      }
      ws.wl_pos[dst++] = 32 * c + b;
    }
  }
  // ---- 4: publish the worklist (every thread's writes, then one release)
  if (trace2 && tid == 0) trace2[2] = static_cast<int64_t>(globaltimer_ns());
  __syncthreads();
  if (tid == 0) {
    if (trace2) trace2[3] = static_cast<int64_t>(globaltimer_ns());
    __threadfence();
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(ws.route_done), "r"(d.seq) : "memory");
  }
  if (trace && tid == 0) trace[4] = static_cast<int64_t>(globaltimer_ns());

  // ---- 5: fresh list, selection slots, statistics; thread tid owns a
  // contiguous range of positions so the fresh list comes out ascending
  const int ppt = (n + kRouteThreads - 1) / kRouteThreads;
  const int p0 = min(n, tid * ppt), p1 = min(n, p0 + ppt);
  int cnt[5] = {0, 0, 0, 0, 0}, bad = 0;
  for (int t = p0; t < p1; ++t) {
    const int code = ws.cat[t];
    const int c = code & 15;
#pragma unroll
    for (int q = 0; q < 5; ++q) cnt[q] += c == q;
    bad += (code & kCodeBad) ? 1 : 0;
  }
  int n_fresh;
  int f = block_excl_scan((p1 - p0) - (force ? 0 : cnt[C_REUSE]), tmp, &n_fresh);
  for (int t = p0; t < p1; ++t) {
    const bool fresh = force || (ws.cat[t] & 15) != C_REUSE;
    if (!fresh) {
      ws.fidx[t] = -1;
      continue;
    }
    ws.fresh_pos[f] = t;
    ws.fidx[t] = f++;
    const int c = t >> 5;
    const uint32_t below = (1u << (t & 31)) - 1u;
    for (int j = 0; j < k; ++j) {
      const int e = ws.sel[static_cast<size_t>(t) * k + j];
      if (e < 0 || e >= E) {
        set_error(ws.err, EPOCH_DEVERR_BOUNDS);
        ws.slot[static_cast<size_t>(t) * k + j] = 0;
        continue;
      }
      const int ci = s_cidx[e];
      if (ci < 0) {
        set_error(ws.err, EPOCH_DEVERR_BOUNDS);
        ws.slot[static_cast<size_t>(t) * k + j] = 0;
        continue;
      }
      ws.slot[static_cast<size_t>(t) * k + j] = s_off[e] + pre(ci, c) + __popc(word(ci, c) & below);
    }
  }
#pragma unroll
  for (int q = 0; q < 5; ++q) cnt[q] = __reduce_add_sync(0xffffffffu, cnt[q]);
  bad = __reduce_add_sync(0xffffffffu, bad);
  if (lane == 0) {
#pragma unroll
    for (int q = 0; q < 5; ++q) atomicAdd(&s_cat[q], cnt[q]);
    atomicAdd(&s_cat[5], bad);
  }
  // experts with at least one row (statistics)
  int hit = 0;
  for (int e = tid; e < E; e += kRouteThreads) hit += s_off[e + 1] > s_off[e];
  hit = __reduce_add_sync(0xffffffffu, hit);
  if (lane == 0) atomicAdd(&s_cat[6], hit);
  __syncthreads();
  if (tid == 0) {
    const int nt_sh = d.tn > 0 ? d.n_sh * ((n + d.tn - 1) / d.tn) : 0;
    ws.ctrl->n_hit = s_cat[6];
    ws.stats->n_hit_experts = s_cat[6];
    ws.stats->tiles_up = (d.tn > 0 ? (d.I / 128) * n_tiles : 0) + (d.I_s / 128) * nt_sh;
    ws.stats->tiles_down = (d.tn > 0 ? (d.H / kBmDn) * n_tiles : 0) + (d.H / kBmDn) * nt_sh;
    const int fb = (d.host_fallback ? 1 : 0) | (s_anom ? 2 : 0);
    if (n_fresh * k != n_edges) set_error(ws.err, EPOCH_DEVERR_BOUNDS);
    ws.ctrl->n_fresh = n_fresh;
    ws.ctrl->fallback = fb;
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
    st->n_edges = n_edges;
    st->support_len = fb ? E : ws.ctrl->support_len;
    st->fallback = fb;
    st->bad_flags = s_cat[5];
    if (s_cat[5]) set_error(ws.err, EPOCH_DEVERR_FLAGS);
    if (d.stats_out) *d.stats_out = *st;
  }
  // positions beyond this call's n_pos keep their state
  for (int t = n + tid; t < d.Nmax; t += kRouteThreads) {
    ws.stamp[static_cast<size_t>(wr) * d.Nmax + t] = ws.stamp[static_cast<size_t>(rd) * d.Nmax + t];
    ws.prev_dec[static_cast<size_t>(wr) * d.Nmax + t] = ws.prev_dec[static_cast<size_t>(rd) * d.Nmax + t];
  }
  // the words and the shared-expert tile counters of the next iteration start at zero
  uint32_t *next = ws.sel_words + static_cast<size_t>(rd) * E * cmax;
  for (int q = tid; q < E * cmax; q += kRouteThreads) next[q] = 0u;
  const int nxt = static_cast<int>((d.seq + 1u) & 1u);
  int32_t *sh = ws.sh_ctr + static_cast<size_t>(nxt) * sh_stride(d);
  for (int q = tid; q < sh_stride(d); q += kRouteThreads) sh[q] = 0;
  // ---- 6: publish the bookkeeping (route_done[1] = this call's sequence
  // number, release) for the combine kernel, which reads the fresh index,
  // slots and weights before the expert outputs exist
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(ws.route_done + 1), "r"(d.seq) : "memory");
  }
  if (trace && tid == 0) trace[5] = static_cast<int64_t>(globaltimer_ns());
}

// ---------------------------------------------------------------- permute
// Copies the token rows of the worklist into the compact buffer xp (row l = x
// at wl_pos[l], [W] section "FreshLane Dispatch": compact dispatch), so the
// expert kernel loads each expert's rows as one tiled TMA box. Launched right
// behind the worklist kernel, it waits for the worklist to be published
// (route_done = this call's sequence number), copies its share of the 16-byte
// vectors and adds their count to tile_ctr[2]; the expert kernel's routed up
// tiles start once that count reaches L * (vectors per row). It exits as soon
// as its copies are counted (it does not wait for the worklist kernel to
// finish: its CTAs would hold SMs the expert kernel needs); the combine kernel
// waits for the worklist kernel's bookkeeping through route_done[1].
// One CTA per SM (the block scheduler spreads a grid of one CTA per SM over
// every SM before it stacks any; a larger grid stacked several CTAs on the SMs
// the gate leaves free, and an expert CTA could not start there until they
// left). 384 threads, at most 64 registers: a CTA fits beside a gate CTA or an
// expert CTA. (With fewer registers the scheduler stacked two or three on the
// SMs the gate leaves free, and an SM sub-partition's registers then no longer
// held an expert CTA's warps beside them.)
constexpr int kPermuteThreads = 384;
constexpr int kPermuteVec = 8;  // 16-byte vectors per thread per round
constexpr int kTraceRowPermute = 8;
__global__ void __maxnreg__(64) k_permute(Dims d, Work ws, const uint4 *__restrict__ x, int vpr) {
  pdl_trigger();
  __shared__ int s_ok, s_L;
  const int tid = threadIdx.x;
  int64_t *trace = (d.trace && blockIdx.x < kTraceCtas && tid == 0)
                       ? ws.trace + (static_cast<size_t>(kTraceRowPermute) * kTraceCtas + blockIdx.x) * kTraceFields
                       : nullptr;
  if (trace) {
    trace[0] = static_cast<int64_t>(globaltimer_ns());
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    trace[7] = smid;
  }
  if (tid == 0) {
    int ok = 1;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
      unsigned int v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ws.route_done) : "memory");
      if (v == d.seq) break;
      if (globaltimer_ns() - t0 > static_cast<uint64_t>(d.timeout_ns)) {
        set_error(ws.err, EPOCH_DEVERR_TIMEOUT);
        ok = 0;
        break;
      }
      __nanosleep(32);
    }
    s_ok = ok;
    s_L = ok ? ws.ctrl->n_edges : 0;
    if (trace) trace[1] = static_cast<int64_t>(globaltimer_ns());
  }
  __syncthreads();
  // rows [r0, r1) of the worklist; warp w copies rows r0 + w, r0 + w + 12, ...,
  // lane l the vectors l, l + 32, ... of a row. The warp's row positions are
  // loaded first, one per lane, so the row copies do not wait on them one by one.
  const int L = s_L, lane = lane_id(), wid = warp_id(), nw = kPermuteThreads / 32;
  const int r0 = static_cast<int>(static_cast<long long>(L) * blockIdx.x / gridDim.x);
  const int r1 = static_cast<int>(static_cast<long long>(L) * (blockIdx.x + 1) / gridDim.x);
  uint4 *xp = static_cast<uint4 *>(ws.xp);
  for (int rb = r0 + wid; rb < r1; rb += 32 * nw) {
    int my_pos = 0;
    const int rl = rb + lane * nw;  // this lane's row of the batch
    if (rl < r1) {
      my_pos = ws.wl_pos[rl];
      if (my_pos < 0 || my_pos >= d.n_pos) {
        set_error(ws.err, EPOCH_DEVERR_BOUNDS);
        my_pos = 0;
      }
    }
    const int nb = min(32, (r1 - rb + nw - 1) / nw);  // rows of this batch
#pragma unroll 1
    for (int b = 0; b < nb; ++b) {
      const int row = rb + b * nw;
      const int pos = __shfl_sync(0xffffffffu, my_pos, b);
      const uint4 *src = x + static_cast<size_t>(pos) * vpr;
      uint4 *dst = xp + static_cast<size_t>(row) * vpr;
#pragma unroll 1
      for (int v0 = 0; v0 < vpr; v0 += 32 * kPermuteVec) {
        uint4 buf[kPermuteVec];
#pragma unroll
        for (int q = 0; q < kPermuteVec; ++q) {
          const int v = v0 + lane + 32 * q;
          if (v < vpr) buf[q] = __ldg(src + v);
        }
#pragma unroll
        for (int q = 0; q < kPermuteVec; ++q) {
          const int v = v0 + lane + 32 * q;
          if (v < vpr) dst[v] = buf[q];
        }
      }
    }
  }
  __syncthreads();
  if (tid == 0 && s_ok && r1 > r0) {
    __threadfence();
    atomicAdd(ws.tile_ctr + 2, (r1 - r0) * vpr);
  }
  if (trace) trace[2] = static_cast<int64_t>(globaltimer_ns());
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
// The fresh index, slots and weights come from the worklist kernel's
// bookkeeping and are read while the experts still run (route_done[1] = this
// call's sequence number); once the expert grid has finished, each pass
// requests every row it needs (the k expert-output rows or the cached row,
// the shared outputs, x) before using any of them.
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
  if (threadIdx.x == 0) {
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
      unsigned int v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ws.route_done + 1) : "memory");
      if (v == d.seq) break;
      if (globaltimer_ns() - t0 > static_cast<uint64_t>(d.timeout_ns)) {
        set_error(ws.err, EPOCH_DEVERR_TIMEOUT);
        break;
      }
      __nanosleep(64);
    }
  }
  __syncthreads();
  if (t < d.n_pos) {
    if (threadIdx.x < k) {
      int sl = ws.slot[static_cast<size_t>(t) * k + threadIdx.x];
      slot_s[threadIdx.x] = sl;
      w_s[threadIdx.x] = ws.selw[static_cast<size_t>(t) * k + threadIdx.x];
    }
    if (threadIdx.x == 0) f_s = ws.fidx[t];
  }
  pdl_wait();  // the expert outputs of this call are complete
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
                                int clear_state, int32_t *ids_out, int32_t *len_out, cudaStream_t s) {
  static bool carve_ = (prefer_max_shared(k_plan_support) == cudaSuccess);
  (void)carve_;
  k_plan_support<<<1, 1024, 0, s>>>(d, ws, threshold, all_experts, clear_state, ids_out, len_out);
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

cudaError_t launch_permute(const Dims &d, const Work &ws, const void *x, cudaStream_t s) {
  static bool c_ = (prefer_max_shared(k_permute) == cudaSuccess);
  (void)c_;
  Dims dd = d;
  Work ww = ws;
  const uint4 *xv = static_cast<const uint4 *>(x);
  int vpr = d.H * 2 / 16;
  void *args[] = {&dd, &ww, &xv, &vpr};
  return launch_kernel(reinterpret_cast<void *>(k_permute), dim3(num_sms()), dim3(kPermuteThreads), 0, s, args,
                       true);
}

// One CTA, launched programmatically: it starts while the gate kernel runs and
// waits for it (pdl_wait) before reading its outputs.
cudaError_t launch_route(const Dims &d, const Work &ws, cudaStream_t s) {
  if (d.E > 4 * kRouteThreads) return cudaErrorInvalidConfiguration;
  constexpr size_t kDyn = (2 * kRouteSmemWords + 1024) * 4;  // words, prefixes, group list
  static bool c_ = (prefer_max_shared(k_route) == cudaSuccess &&
                    cudaFuncSetAttribute(k_route, cudaFuncAttributeMaxDynamicSharedMemorySize, kDyn) == cudaSuccess);
  if (!c_) return cudaErrorInvalidConfiguration;
  Dims dd = d;
  Work ww = ws;
  void *args[] = {&dd, &ww};
  return launch_kernel(reinterpret_cast<void *>(k_route), dim3(1), dim3(kRouteThreads), kDyn, s, args, true);
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

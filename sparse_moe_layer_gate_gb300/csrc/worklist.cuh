// The expert-sorted worklist of one iteration, built by every CTA of the
// worklist kernel from the selection words of the classifying kernel (gate or
// select kernel), where the gate does not build it in its own tail
// (gate_tail.cuh): fp32 layers, gates of more than one wave, the hot-update
// path.
//
// Walk-through page "Epoch 完全拆解:把扩散块编译成稀疏 MoE 服务单元", section
// "FreshLane Dispatch": pack the fresh token-expert pairs, exchange per-expert
// counts to get offsets, dispatch the compact rows, and remember for every
// selection where its row went so the combine can return it. On one chip the
// count exchange is a popcount over per-expert bitmasks (bit t of expert e's
// words: fresh position t selected e) and the dispatch a gather of token rows
// into the compact buffer xp.
//
// Every CTA derives the same expert offsets on its own (one round of loads,
// then shared-memory work), so no CTA waits for another. The work comes in two
// phases:
//  A rows per candidate expert (the support, or every expert on a fallback),
//    the expert offsets (a scan over expert ids) and the group list of the
//    expert kernel (experts by row-count class, with token-tile prefixes); CTA
//    0 writes them to global memory;
//  B the CTA's share of the worklist rows (position of each row and, for bf16
//    layers, its row of x copied into xp); then its share of the positions'
//    fresh index, fresh list and selection slots, the statistics (CTA 0), the
//    state of positions beyond n_pos and the cleared words of the next
//    iteration.
// The tcgen05 expert kernel reads the finished worklist once this grid has
// completed. The counters it advances (tile_ctr, done_up) were reset, and the
// anomaly flag set, by block 0 of the classifying kernel before phase A reads
// anything.
#pragma once

#include "common.cuh"
#include "layer.h"
#include "select.cuh"

namespace epoch {

// Threads [0, n) of a CTA (n a multiple of 32, gtid the thread's index among
// them) that synchronise on named barrier `bar` (0 with n = blockDim.x is the
// whole CTA).
struct Group {
  int gtid, n, bar;
  __device__ __forceinline__ void sync() const { asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(n) : "memory"); }
  __device__ __forceinline__ int warp() const { return gtid >> 5; }
  __device__ __forceinline__ int warps() const { return n >> 5; }
};

// Exclusive scan over a group of up to 1024 threads; *total gets the sum.
__device__ __forceinline__ int group_excl_scan(const Group &g, int v, int *warp_tmp, int *total) {
  const int lane = lane_id(), wid = g.warp(), nw = g.warps();
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) warp_tmp[wid] = incl;
  g.sync();
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
  g.sync();
  const int r = warp_tmp[wid] + incl - v;
  *total = warp_tmp[32];
  g.sync();
  return r;
}

// Exclusive scan of four values at once (independent components, one pass).
__device__ __forceinline__ int4 group_excl_scan4(const Group &g, int4 v, int4 *warp_tmp, int4 *total) {
  const int lane = lane_id(), wid = g.warp(), nw = g.warps();
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
  g.sync();
  if (wid == 0) {
    const int4 x = lane < nw ? warp_tmp[lane] : make_int4(0, 0, 0, 0);
    const int4 xi = scan(x);
    warp_tmp[lane] = make_int4(xi.x - x.x, xi.y - x.y, xi.z - x.z, xi.w - x.w);
    if (lane == 31) warp_tmp[32] = xi;
  }
  g.sync();
  const int4 b = warp_tmp[wid];
  *total = warp_tmp[32];
  g.sync();
  return make_int4(b.x + incl.x - v.x, b.y + incl.y - v.y, b.z + incl.z - v.z, b.w + incl.w - v.w);
}

__device__ __forceinline__ int nth_set_bit(uint32_t v, int n) {
  for (int i = 0; i < n; ++i) v &= v - 1u;
  return __ffs(v) - 1;
}

constexpr int kWlStageWords = 1152;  // candidate words kept in shared memory (more are read from L2)
constexpr int kWlChunk = 128;        // worklist rows whose positions are staged together for the copy

// Shared-memory scratch of the worklist build (under 10 KB: it fits in the
// expert kernel's epilogue staging area, unused until the first epilogue).
struct WlSmem {
  int16_t cand[1024];  // candidate experts
  int16_t cidx[1024];  // candidate index of an expert, -1 if none
  uint32_t words[kWlStageWords];
  int32_t pos[kWlChunk];
  int4 tmp4[33];
  int32_t tmp[33];
  int32_t cat[8];
  int32_t fbase;
};

// Phase A's results (the same in every CTA).
struct WlPlan {
  bool force;    // every expert eligible, every position fresh (host or device fallback)
  int anom;      // the classifying kernel saw a decoded -> live transition
  int n_cand;
  bool staged;   // the candidates' words are in WlSmem::words
  int n_edges;   // worklist rows L
  int n_tiles;   // routed token tiles of the expert kernel (groups' rows in tiles of d.tn)
};

// Before the classifying kernel has finished: the block plan's candidates.
__device__ __forceinline__ void wl_prepare(const Dims &d, const Work &ws, WlSmem &sm, int32_t *s_off,
                                           const Group &g) {
  for (int e = g.gtid; e < d.E; e += g.n) {
    sm.cand[e] = static_cast<int16_t>(d.host_fallback ? e : ws.support_ids[e]);
    sm.cidx[e] = -1;
    s_off[e] = 0;
  }
  if (g.gtid < 8) sm.cat[g.gtid] = 0;
}

// Phase A (after the classifying kernel has finished): rows per candidate,
// offsets into s_off [E + 1], and the group list into s_list [E + 1] (when
// given). CTA 0 (`publish`) also writes offsets, group list and tile counts to
// global memory.
__device__ __forceinline__ WlPlan wl_phase_a(const Dims &d, const Work &ws, WlSmem &sm, int32_t *s_off,
                                          int32_t *s_list, bool publish, const Group &g) {
  const int E = d.E, cmax = d.cmax, nch = (d.n_pos + 31) >> 5;
  const uint32_t *words = ws.sel_words + static_cast<size_t>((d.state_rd & 1) ^ 1) * E * cmax;
  WlPlan pl;
  pl.anom = d.host_fallback ? 0 : *reinterpret_cast<volatile const int32_t *>(&ws.ctrl->anom);
  pl.force = d.host_fallback != 0 || pl.anom != 0;
  if (pl.force && !d.host_fallback)  // a decoded -> live anomaly: every expert is a candidate
    for (int e = g.gtid; e < E; e += g.n) sm.cand[e] = static_cast<int16_t>(e);
  pl.n_cand = pl.force ? E : min(E, ws.ctrl->support_len);
  pl.staged = pl.n_cand * nch <= kWlStageWords;
  g.sync();
  for (int i = g.gtid; i < pl.n_cand; i += g.n) sm.cidx[sm.cand[i]] = static_cast<int16_t>(i);
  // the candidates' words in one round of loads; rows per expert. Items are
  // (candidate, block of 32 words); warp w takes items w, w + warps, ..., up to
  // eight at a time, lane l loading word l of each, and adds the block's
  // popcount to its candidate's row count.
  const int lane = lane_id();
  const int nwb = (nch + 31) >> 5;
  const int items = pl.n_cand * nwb;
  const int wid = g.warp(), nw = g.warps();
  for (int i0 = wid; i0 < items; i0 += nw * 8) {
    uint32_t v[8];
#pragma unroll
    for (int bb = 0; bb < 8; ++bb) {
      const int it = i0 + bb * nw;
      v[bb] = 0u;
      if (it < items) {
        const int ci = it / nwb, w = (it - ci * nwb) * 32 + lane;
        if (w < nch) v[bb] = words[static_cast<size_t>(sm.cand[ci]) * cmax + w];
      }
    }
#pragma unroll
    for (int bb = 0; bb < 8; ++bb) {
      const int it = i0 + bb * nw;
      if (it < items) {  // the same for every lane of the warp
        const int ci = it / nwb, w = (it - ci * nwb) * 32 + lane;
        if (pl.staged && w < nch) sm.words[ci * nch + w] = v[bb];
        const int sum = __reduce_add_sync(0xffffffffu, __popc(v[bb]));
        if (lane == 0 && sum) atomicAdd(&s_off[sm.cand[ci]], sum);
      }
    }
  }
  g.sync();
  // One scan over the experts in id order (thread gtid owns [gtid * gpt,
  // gtid * gpt + gpt)) gives the expert offsets and, per row-count class of
  // the group list (2: >= 96 rows, 1: >= 32, 0: fewer; listed in that order,
  // by id within a class), the list positions and token-tile prefixes: .x
  // rows, .y experts of class 0 | class 1 << 16, .z experts of class 2 | its
  // tiles << 16, .w tiles of class 0 | class 1 << 16.
  const int gpt = (E + g.n - 1) / g.n;  // <= 8 (E <= 1024, n >= 128)
  const int g0 = g.gtid * gpt;
  auto cls_of = [](int r) { return r >= 96 ? 2 : r >= 32 ? 1 : 0; };
  int4 v = make_int4(0, 0, 0, 0);
  for (int h = 0; h < gpt && g0 + h < E; ++h) {
    const int r = s_off[g0 + h], k2 = cls_of(r), nt = d.tn > 0 ? (r + d.tn - 1) / d.tn : 0;
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
  const int4 ex = group_excl_scan4(g, v, sm.tmp4, &tot);
  const int n2 = tot.z & 0xffff, n1 = tot.y >> 16;
  const int t2 = tot.z >> 16, t1 = tot.w >> 16, t0 = tot.w & 0xffff;
  int rank0 = ex.y & 0xffff, rank1 = ex.y >> 16, rank2 = ex.z & 0xffff;
  int tb0 = ex.w & 0xffff, tb1 = ex.w >> 16, tb2 = ex.z >> 16;
  int before = ex.x;
  pl.n_edges = tot.x;
  pl.n_tiles = t0 + t1 + t2;
  for (int h = 0; h < gpt && g0 + h < E; ++h) {
    const int e = g0 + h, r = s_off[e], k2 = cls_of(r), nt = d.tn > 0 ? (r + d.tn - 1) / d.tn : 0;
    int entry;
    if (k2 == 2) {
      entry = (tb2 << kGrpIdBits) | e;
      if (s_list) s_list[rank2] = entry;
      if (publish) ws.grp_list[rank2] = entry;
      ++rank2;
      tb2 += nt;
    } else if (k2 == 1) {
      entry = (((t2 + tb1) << kGrpIdBits) | e);
      if (s_list) s_list[n2 + rank1] = entry;
      if (publish) ws.grp_list[n2 + rank1] = entry;
      ++rank1;
      tb1 += nt;
    } else {
      entry = (((t2 + t1 + tb0) << kGrpIdBits) | e);
      if (s_list) s_list[n2 + n1 + rank0] = entry;
      if (publish) ws.grp_list[n2 + n1 + rank0] = entry;
      ++rank0;
      tb0 += nt;
    }
    s_off[e] = before;
    if (publish) ws.offsets[e] = before;
    before += r;
  }
  if (g.gtid == 0) {
    s_off[E] = pl.n_edges;
    if (s_list) s_list[E] = pl.n_tiles << kGrpIdBits;
    if (publish) {
      ws.offsets[E] = pl.n_edges;
      ws.grp_list[E] = pl.n_tiles << kGrpIdBits;
      ws.ctrl->tiles_up = d.tn > 0 ? (d.I / 128) * pl.n_tiles : 0;
      ws.ctrl->tiles_dn = d.tn > 0 ? (d.H / kBmDn) * pl.n_tiles : 0;
      ws.ctrl->n_edges = pl.n_edges;
    }
  }
  g.sync();
  if (pl.n_edges > d.Nmax * d.k) {  // cannot happen with consistent words; never index past the buffers
    if (g.gtid == 0) set_error(ws.err, EPOCH_DEVERR_BOUNDS);
    pl.n_edges = d.Nmax * d.k;
  }
  return pl;
}

// Phase B, rows: CTA b of G's share of the worklist rows: the position of
// each row (wl_pos) and, for bf16 layers, its row of x copied into xp. x: the
// layer input, vpr its 16-byte vectors per row (0: no copy, as for the FFMA
// experts, which read x through wl_pos).
__device__ __forceinline__ void wl_rows(const Dims &d, const Work &ws, WlSmem &sm, const int32_t *s_off,
                                     const WlPlan &pl, const uint4 *__restrict__ x, int vpr, int b, int G,
                                     const Group &g) {
  const int n = d.n_pos, E = d.E, cmax = d.cmax;
  const int nch = (n + 31) >> 5;
  const int wr = (d.state_rd & 1) ^ 1;
  const int lane = lane_id();
  const uint32_t *words = ws.sel_words + static_cast<size_t>(wr) * E * cmax;
  const int n_edges = pl.n_edges;
  // ---- the CTA's rows [r0, r1), kWlChunk at a time (thread gtid <-> row c0 +
  // gtid). The lanes of a warp holding rows of one expert find their positions
  // together: 32 of the expert's words per round (lane j: word w0 + j), a warp
  // scan of their popcounts, then each lane locates its rank among the 32
  // running totals. The group then copies the chunk's rows of x into xp.
  const int r0 = static_cast<int>(static_cast<long long>(n_edges) * b / G);
  const int r1 = static_cast<int>(static_cast<long long>(n_edges) * (b + 1) / G);
  uint4 *xp = static_cast<uint4 *>(ws.xp);
  for (int c0 = r0; c0 < r1; c0 += kWlChunk) {
    const int r = c0 + g.gtid;
    const bool have = g.gtid < kWlChunk && r < r1;
    int my_e = E, my_rank = 0;
    if (have) {
      int lo = 0, hi = E;  // the largest e with s_off[e] <= r
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_off[mid] <= r) lo = mid;
        else hi = mid;
      }
      my_e = lo;
      my_rank = r - s_off[lo];
    }
    int my_pos = -1;
    unsigned todo = __ballot_sync(0xffffffffu, have);
    while (todo) {
      const int e = __shfl_sync(0xffffffffu, my_e, __ffs(todo) - 1);
      const bool mine = have && my_e == e;
      todo &= ~__ballot_sync(0xffffffffu, mine);
      const int ci = sm.cidx[e];
      if (ci < 0) {  // rows of an expert that is not a candidate: the offsets are corrupt
        if (lane == 0) set_error(ws.err, EPOCH_DEVERR_BOUNDS);
        continue;
      }
      int base = 0;  // set bits of e's words before this round
      for (int w0 = 0; w0 < nch; w0 += 32) {
        const int w = w0 + lane;
        const uint32_t v =
            w < nch ? (pl.staged ? sm.words[ci * nch + w] : words[static_cast<size_t>(e) * cmax + w]) : 0u;
        const int cnt = __popc(v);
        int incl = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int u = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += u;
        }
        // j = words of this round whose running total is at or below the lane's
        // rank (the totals ascend with the lane: a binary search over them)
        int j = 0;
#pragma unroll
        for (int step = 16; step >= 1; step >>= 1) {
          const int probe = __shfl_sync(0xffffffffu, incl, j + step - 1);
          if (base + probe <= my_rank) j += step;
        }
        if (base + __shfl_sync(0xffffffffu, incl, 31) <= my_rank) j = 32;
        const int jj = j < 32 ? j : 31;
        const uint32_t vj = __shfl_sync(0xffffffffu, v, jj);
        const int exj = __shfl_sync(0xffffffffu, incl - cnt, jj);
        if (mine && my_pos < 0 && j < 32) my_pos = 32 * (w0 + j) + nth_set_bit(vj, my_rank - base - exj);
        base += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    if (have) {
      if (my_pos < 0 || my_pos >= n) {
        set_error(ws.err, EPOCH_DEVERR_BOUNDS);
        my_pos = 0;
      }
      ws.wl_pos[r] = my_pos;
      sm.pos[g.gtid] = my_pos;
    }
    if (vpr > 0) {
      g.sync();
      // the chunk's rows, one per warp at a time, eight 16-byte vectors per lane in flight
      const int nrows = min(kWlChunk, r1 - c0);
      for (int rr = g.warp(); rr < nrows; rr += g.warps()) {
        const uint4 *src = x + static_cast<size_t>(sm.pos[rr]) * vpr;
        uint4 *dst = xp + static_cast<size_t>(c0 + rr) * vpr;
        for (int v0 = lane; v0 < vpr; v0 += 32 * 8) {
          uint4 buf[8];
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (v0 + 32 * u < vpr) buf[u] = __ldg(src + v0 + 32 * u);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            if (v0 + 32 * u < vpr) dst[v0 + 32 * u] = buf[u];
        }
      }
      g.sync();
    }
  }
}


// Phase B, bookkeeping: CTA b of G's share of the positions (fresh index,
// fresh list, the worklist row of each selection), the statistics (CTA 0), the
// state of positions beyond n_pos and the cleared words of the next
// iteration. trace (CTA 0, nullable): fresh index done, slots done, statistics
// done.
__device__ __forceinline__ void wl_bookkeeping(const Dims &d, const Work &ws, WlSmem &sm, const int32_t *s_off,
                                            const WlPlan &pl, int b, int G, const Group &g, int64_t *trace) {
  trace = (b == 0 && g.gtid == 0) ? trace : nullptr;
  const int n = d.n_pos, E = d.E, k = d.k, cmax = d.cmax;
  const int nch = (n + 31) >> 5;
  const int rd = d.state_rd & 1, wr = rd ^ 1;
  const int lane = lane_id();
  const uint32_t *words = ws.sel_words + static_cast<size_t>(wr) * E * cmax;
  const int n_edges = pl.n_edges;
  const int p0 = static_cast<int>(static_cast<long long>(n) * b / G);
  const int p1 = static_cast<int>(static_cast<long long>(n) * (b + 1) / G);
  auto fresh_code = [&](int code) { return pl.force || (code & 15) != C_REUSE; };
  {
    int before = 0;  // fresh positions in [0, p0)
    for (int t = g.gtid; t < p0; t += g.n) before += fresh_code(ws.cat[t]) ? 1 : 0;
    int tot;
    (void)group_excl_scan(g, before, sm.tmp, &tot);
    if (g.gtid == 0) sm.fbase = tot;
  }
  g.sync();
  if (g.warp() == 0) {
    int f = sm.fbase;
    for (int t0 = p0; t0 < p1; t0 += 32) {
      const int t = t0 + lane;
      const bool fr = t < p1 && fresh_code(ws.cat[t]);
      const unsigned m = __ballot_sync(0xffffffffu, fr);
      if (t < p1) {
        const int mine = f + __popc(m & ((1u << lane) - 1u));
        ws.fidx[t] = fr ? mine : -1;
        if (fr) ws.fresh_pos[mine] = t;
      }
      f += __popc(m);
    }
  }
  if (trace) trace[5] = static_cast<int64_t>(globaltimer_ns());
  for (int it = g.gtid; it < (p1 - p0) * k; it += g.n) {
    const int t = p0 + it / k, j = it - (it / k) * k;
    if (!fresh_code(ws.cat[t])) continue;
    const size_t sj = static_cast<size_t>(t) * k + j;
    const int e = ws.sel[sj];
    const int ci = (e >= 0 && e < E) ? sm.cidx[e] : -1;
    if (ci < 0) {
      set_error(ws.err, EPOCH_DEVERR_BOUNDS);
      ws.slot[sj] = 0;
      continue;
    }
    const int c = t >> 5;
    int rk = 0;
    for (int w = 0; w < c; ++w)
      rk += __popc(pl.staged ? sm.words[ci * nch + w] : words[static_cast<size_t>(e) * cmax + w]);
    const uint32_t own = pl.staged ? sm.words[ci * nch + c] : words[static_cast<size_t>(e) * cmax + c];
    rk += __popc(own & ((1u << (t & 31)) - 1u));
    ws.slot[sj] = s_off[e] + rk;
  }
  if (trace) trace[6] = static_cast<int64_t>(globaltimer_ns());
  if (b == 0) {  // statistics over every position
    int cnt[5] = {0, 0, 0, 0, 0}, bad = 0, fr = 0;
    for (int t = g.gtid; t < n; t += g.n) {
      const int code = ws.cat[t];
#pragma unroll
      for (int q = 0; q < 5; ++q) cnt[q] += (code & 15) == q;
      bad += (code & kCodeBad) ? 1 : 0;
      fr += fresh_code(code) ? 1 : 0;
    }
#pragma unroll
    for (int q = 0; q < 5; ++q) cnt[q] = __reduce_add_sync(0xffffffffu, cnt[q]);
    bad = __reduce_add_sync(0xffffffffu, bad);
    fr = __reduce_add_sync(0xffffffffu, fr);
    int hit = 0;
    for (int e = g.gtid; e < E; e += g.n) hit += s_off[e + 1] > s_off[e];
    hit = __reduce_add_sync(0xffffffffu, hit);
    if (lane == 0) {
#pragma unroll
      for (int q = 0; q < 5; ++q) atomicAdd(&sm.cat[q], cnt[q]);
      atomicAdd(&sm.cat[5], bad);
      atomicAdd(&sm.cat[6], hit);
      atomicAdd(&sm.cat[7], fr);
    }
    g.sync();
    if (g.gtid == 0) {
      const int n_fresh = sm.cat[7];
      const int nt_sh = d.tn > 0 ? d.n_sh * ((n + d.tn - 1) / d.tn) : 0;
      ws.ctrl->n_hit = sm.cat[6];
      const int fb = (d.host_fallback ? 1 : 0) | ((pl.anom & 1) ? 2 : 0) | ((pl.anom & 2) ? 4 : 0);
      if (n_fresh * k != n_edges) set_error(ws.err, EPOCH_DEVERR_BOUNDS);
      ws.ctrl->n_fresh = n_fresh;
      ws.ctrl->fallback = fb;
      epoch_iter_stats *st = ws.stats;
      st->iteration = d.iter;
      st->n_pos = n;
      st->n_live = sm.cat[C_LIVE];
      st->n_new = sm.cat[C_NEW];
      st->n_miss = sm.cat[C_MISS];
      st->n_stale = sm.cat[C_STALE];
      st->n_forced = pl.force ? sm.cat[C_REUSE] : 0;
      st->n_reuse = pl.force ? 0 : sm.cat[C_REUSE];
      st->n_fresh = n_fresh;
      st->n_edges = n_edges;
      st->n_hit_experts = sm.cat[6];
      st->support_len = fb ? E : ws.ctrl->support_len;
      st->fallback = fb;
      st->bad_flags = sm.cat[5];
      st->tiles_up = (d.tn > 0 ? (d.I / 128) * pl.n_tiles : 0) + (d.I_s / 128) * nt_sh;
      st->tiles_down = (d.tn > 0 ? (d.H / kBmDn) * pl.n_tiles : 0) + (d.H / kBmDn) * nt_sh;
      // support coverage of this iteration's fresh positions -> the next iteration
      // (every selection of the call has counted itself; the count restarts for the next call)
      const int under = d.cov_check ? *ws.cov_under : 0;
      *ws.cov_under = 0;
      ws.ctrl->short_next = (d.cov_check && static_cast<float>(under) > (1.f - d.cov_q) * static_cast<float>(n_fresh))
                                ? 1 : 0;
      st->n_under = under;
      if (sm.cat[5]) set_error(ws.err, EPOCH_DEVERR_FLAGS);
      if (d.stats_out) *d.stats_out = *st;
    }
    if (trace) trace[7] = static_cast<int64_t>(globaltimer_ns());
  }
  // positions beyond this call's n_pos keep their state; the words of the next
  // iteration start at zero
  const int gt = b * g.n + g.gtid, gstride = G * g.n;
  for (int t = n + gt; t < d.Nmax; t += gstride) {
    ws.stamp[static_cast<size_t>(wr) * d.Nmax + t] = ws.stamp[static_cast<size_t>(rd) * d.Nmax + t];
    ws.prev_dec[static_cast<size_t>(wr) * d.Nmax + t] = ws.prev_dec[static_cast<size_t>(rd) * d.Nmax + t];
  }
  uint32_t *next = ws.sel_words + static_cast<size_t>(rd) * E * cmax;
  for (int q = gt; q < E * cmax; q += gstride) next[q] = 0u;
}

}  // namespace epoch

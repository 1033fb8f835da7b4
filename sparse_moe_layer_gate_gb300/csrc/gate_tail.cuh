// The iteration's worklist, built in the tail of the tcgen05 gate kernel by
// the gate's own CTAs, each for the positions it classified and routed.
//
// Walk-through page "Epoch 完全拆解:把扩散块编译成稀疏 MoE 服务单元", section
// "FreshLane Dispatch": pack the fresh token-expert pairs, exchange per-expert
// counts to get offsets, dispatch the compact rows, and remember for every
// selection where its row went so the combine can return it. On one chip the
// count exchange is a popcount over per-expert selection bitmasks (bit t of
// expert e's words: fresh position t selected e), and the dispatch copies each
// fresh position's row of x into its k worklist rows.
//
// Every CTA owns a run of positions [p0, p0 + TPC). Once it has arrived at
// the grid barrier it starts bulk copies of its fresh positions' x rows into
// shared memory and adds its positions' category counts to the iteration
// tallies. After the barrier it reads the candidate experts' words once (the block support, or
// every expert on a fallback) and gets, per candidate, its rows in the whole
// iteration and its set bits before p0, plus the words that cover its own
// positions. The expert offsets follow from one scan over expert ids; the row
// of selection (t, j), expert e, is offset(e) + bits of e before p0 + bits of
// e in [p0, t). The CTA then bulk-copies each staged x row to its k worklist
// rows and writes the slots, the fresh index and the fresh list of its
// positions. CTA 0 also publishes the offsets and the expert kernel's group
// list; the combine kernel finishes the statistics. One round of global loads
// after the barrier, no other global read on the way to the expert kernel's
// inputs.
//
// Worklist order: expert-major, positions ascending within an expert (the
// order the oracle defines), reached without any sort.
#pragma once

#include "common.cuh"
#include "layer.h"
#include "select.cuh"
#include "worklist.cuh"

namespace epoch {

// Per-CTA inputs of the tail held outside the operand ring (written while the
// ring is still in use).
struct GateTail {
  const int16_t *sel;   // [TPC][16] selected experts of the own fresh positions
  const uint8_t *fr;    // [TPC] own position j is fresh
  const int *code;      // [TPC] classification codes of the own positions
  const int16_t *cand;  // [E] candidate experts: the block support (or its union over requests)
  const int16_t *cidx;  // [E] candidate index of an expert (valid where cand[cidx[e]] == e)
  int ncand;            // candidates of the plan
  uint32_t x_bar;       // mbarrier of the staged x rows (phase 0)
  int gen0;             // the grid barrier's arrival count when the call began (read at the kernel's start)
};

// Shared-memory bytes of the tail's scratch in the operand ring: staged x
// rows, then rows/offsets per expert, per-candidate counts and words, slots
// and a small scan area.
__host__ __device__ inline int gate_tail_bytes(const Dims &d, int tpc) {
  const int e4 = (d.E + 4) & ~3;
  return tpc * d.H * 2 + 16 * 33 + 4 * e4 + 4 * d.E + 12 * d.E + 4 * tpc * d.k + 4 * 48;
}

constexpr int kTallies = 8;  // Work::tally: categories C_LIVE..C_REUSE, bad flags, fresh positions

__device__ __forceinline__ uint32_t bit_range(int lo, int hi) {  // bits [lo, hi) of a word, 0 <= lo < hi <= 32
  const uint32_t h = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
  return h & ~((1u << lo) - 1u);
}

// All threads of the CTA. x: the layer input (row-major bf16 rows of H);
// smem: the operand ring (free once the cluster's partials are read); p0 the
// CTA's first position, tpc its positions; force: every position fresh and
// every expert a candidate (host fallback or device anomaly), anom the
// device's anomaly bits; trace: CTA 0's timeline row (nullable).
__device__ __forceinline__ void gate_tail(const Dims &d, const Work &ws, const uint8_t *x, uint8_t *smem,
                                          const GateTail &gt, int p0, int tpc, bool force, int anom, int64_t *trace) {
  const int tid = threadIdx.x, wid = tid >> 5, lane = tid & 31, nthr = blockDim.x, nw = nthr >> 5;
  const int n = d.n_pos, E = d.E, k = d.k, cmax = d.cmax;
  const int rowb = d.H * 2;
  const int np = max(0, min(tpc, n - p0));
  const int n_cand = force ? E : min(gt.ncand, E);
  uint8_t *xs = smem;                                                           // [tpc][H] staged rows
  int4 *s_scan = reinterpret_cast<int4 *>(smem + tpc * rowb);                   // [33] scan scratch
  int32_t *s_off = reinterpret_cast<int32_t *>(s_scan + 33);                    // [E + 1]
  int32_t *s_bef = s_off + ((E + 4) & ~3);                                      // [E] by candidate
  uint32_t *s_own = reinterpret_cast<uint32_t *>(s_bef + E);                    // [E][3] by candidate
  int32_t *s_slot = reinterpret_cast<int32_t *>(s_own + 3 * E);                 // [tpc * k]
  int32_t *s_misc = s_slot + tpc * k;  // 36 bits before p0, 40 barrier passed, 41 arrival order
  auto cand_of = [&](int ci) { return force ? ci : static_cast<int>(gt.cand[ci]); };

  // ---- 1. arrive at the grid barrier over the gate's CTAs, then, while it
  // fills: zero the scratch, add the own positions' category counts to the
  // iteration tallies and start bulk copies of the own fresh positions' x rows
  // into the ring. All gate CTAs are resident (one wave of clusters, and no
  // later kernel starts before every gate CTA has). The arrival counter only
  // grows: this call's CTAs wait until it has grown by the grid size from the
  // value it had when the call began (gt.gen0, set by the previous call's CTA 0
  // once its barrier had passed, so it cannot move before every CTA of this
  // call has arrived). Bounded.
  __syncthreads();  // every warp's selections and words are written
  unsigned arrived_raw = 0;
  if (tid == 0) {
    // release: this CTA's selections and words; acquire (the last CTA, which
    // does not wait): every other CTA's
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(arrived_raw) : "l"(ws.gate_arrive) : "memory");
  }
  for (int e = tid; e <= E; e += nthr) s_off[e] = 0;
  for (int c = tid; c < n_cand; c += nthr) {
    s_bef[c] = 0;
    s_own[3 * c] = s_own[3 * c + 1] = s_own[3 * c + 2] = 0u;
  }
  if (tid < 48 && tid != 41) s_misc[tid] = 0;
  if (wid == 0) {  // the own positions' categories, for the statistics
    int cnt[kTallies] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int j = lane; j < np; j += 32) {
      const int code = gt.code[j];
#pragma unroll
      for (int q = 0; q < 5; ++q) cnt[q] += (code & 15) == q;
      cnt[5] += (code & kCodeBad) ? 1 : 0;
      cnt[6] += gt.fr[j] ? 1 : 0;
    }
#pragma unroll
    for (int q = 0; q < 7; ++q) {
      const int c = __reduce_add_sync(0xffffffffu, cnt[q]);
      if (lane == 0 && c) atomicAdd(ws.tally + q, c);
    }
  }
  if (tid == 32) {  // the own fresh positions' rows of x, into the ring
    fence_proxy_async_smem();
    uint32_t bytes = 0;
    for (int j = 0; j < np; ++j) bytes += gt.fr[j] ? static_cast<uint32_t>(rowb) : 0u;
    mbar_arrive_expect_tx(gt.x_bar, bytes);
    const uint64_t pol = policy_evict_first();
    for (int j = 0; j < np; ++j)
      if (gt.fr[j]) bulk_load(smem_u32(xs + j * rowb), x + static_cast<size_t>(p0 + j) * rowb, rowb, gt.x_bar, pol);
  }
  if (tid == 0) s_misc[41] = static_cast<int>(arrived_raw - static_cast<unsigned>(gt.gen0));  // arrival order
  __syncthreads();
  const int arrived = s_misc[41];
  const bool last = arrived == static_cast<int>(gridDim.x) - 1;
  // Steps 2-4 run once after the barrier. The first three CTAs to arrive
  // (not the last) also run one of them each before it -- step 2, 3 or 4 by
  // arrival -- on the data as it stands, with every global write and error
  // check off and their scratch zeroed again afterwards: the other CTAs then
  // find these instructions in L2 (the input flush between iterations evicts
  // code too), not in HBM, when they run the steps for real. One step each
  // keeps every warm-up short enough to end before the barrier opens.
  const int dmask = last || arrived > 2 ? 0 : 1 << arrived;
  bool ok = true;
  int n_tiles = 0, n_hit = 0;
  const uint32_t *words = ws.sel_words + static_cast<size_t>((d.state_rd & 1) ^ 1) * E * cmax;
  const int nch = (n + 31) >> 5, nwb = (nch + 31) >> 5, wa = p0 >> 5;
  const uint32_t m0 = (1u << (p0 & 31)) - 1u;
#pragma unroll 1
  for (int pass = dmask ? 0 : 1; pass < 2; ++pass) {
    const bool dry = pass == 0;
    if (!dry) {
      if (tid == 0) {
        int pass_ok = 1;
        if (!last) {
          const uint64_t t0 = globaltimer_ns();
          for (;;) {
            unsigned v;
            asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ws.gate_arrive) : "memory");
            if (static_cast<int>(v - static_cast<unsigned>(gt.gen0)) >= static_cast<int>(gridDim.x)) break;
            if (globaltimer_ns() - t0 > static_cast<uint64_t>(d.timeout_ns)) {
              set_error(ws.err, EPOCH_DEVERR_TIMEOUT);
              pass_ok = 0;
              break;
            }
            __nanosleep(64);
          }
        }
        if (pass_ok && blockIdx.x == 0)  // the next call's starting count (modulo 2^32)
          ws.gate_arrive[1] = static_cast<int32_t>(static_cast<unsigned>(gt.gen0) + gridDim.x);
        s_misc[40] = pass_ok;
        if (trace) trace[1] = static_cast<int64_t>(globaltimer_ns());
      }
      __syncthreads();
      ok = s_misc[40] != 0;
    }

    // ---- 2. the candidates' words, one round of loads: rows per expert, bits
    // before p0 and the words covering the own positions, per candidate. Items
    // are (candidate, block of 32 words); lane l loads word l of an item.
    const int items = ok && (!dry || (dmask & 1)) ? n_cand * nwb : 0;
    for (int i0 = wid; i0 < items; i0 += nw * 4) {
      uint32_t v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int it = i0 + u * nw;
        v[u] = 0u;
        if (it < items) {
          const int ci = it / nwb, w = (it - ci * nwb) * 32 + lane;
          if (w < nch) v[u] = __ldcg(words + static_cast<size_t>(cand_of(ci)) * cmax + w);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int it = i0 + u * nw;
        if (it < items) {  // the same for every lane of the warp
          const int ci = it / nwb, w = (it - ci * nwb) * 32 + lane;
          const int tot = __reduce_add_sync(0xffffffffu, __popc(v[u]));
          const int bef = __reduce_add_sync(0xffffffffu, __popc(w < wa ? v[u] : (w == wa ? v[u] & m0 : 0u)));
          if (w >= wa && w < wa + 3) s_own[3 * ci + (w - wa)] = v[u];
          if (lane == 0) {
            if (tot) atomicAdd(&s_off[cand_of(ci)], tot);
            if (bef) atomicAdd(&s_bef[ci], bef);
          }
        }
      }
    }
    __syncthreads();
    if (trace && tid == 0) trace[2] = static_cast<int64_t>(globaltimer_ns());

    // ---- 3. one scan over the experts in id order: the expert offsets and,
    // per row-count class of the expert kernel's group list (2: >= 96 rows, 1:
    // >= 32, 0: fewer; listed in that order, by id within a class), each
    // expert's list position and the token tiles of the entries before it
    // (scan components: .x rows, .y experts of class 0 | class 1 << 16, .z
    // experts of class 2 | its tiles << 16, .w tiles of class 0 | class 1 << 16).
    // CTA 0 publishes the offsets and the list.
    auto cls_of = [](int r) { return r >= 96 ? 2 : r >= 32 ? 1 : 0; };
    const int tn = d.tn > 0 ? d.tn : 1;
    n_hit = 0;
    if (!dry || (dmask & 2)) {
      int b = 0;
      for (int c = tid; c < n_cand; c += nthr) b += s_bef[c];
      b = __reduce_add_sync(0xffffffffu, b);
      if (lane == 0 && b) atomicAdd(&s_misc[36], b);
      const int gpt = (E + nthr - 1) / nthr, e0 = tid * gpt;
      int4 v = make_int4(0, 0, 0, 0);
      int hm = 0;  // bit h: expert e0 + h has rows
      for (int h = 0; h < gpt && e0 + h < E; ++h) {
        const int r = s_off[e0 + h], c2 = cls_of(r), nt = (r + tn - 1) / tn;
        hm |= (r > 0 ? 1 : 0) << h;
        v.x += r;
        if (c2 == 0) {
          v.y += 1;
          v.w += nt;
        } else if (c2 == 1) {
          v.y += 1 << 16;
          v.w += nt << 16;
        } else {
          v.z += 1 | (nt << 16);
        }
      }
      int4 tot;
      const Group g{tid, nthr, 0};
      const int4 ex = group_excl_scan4(g, v, s_scan, &tot);
      const int n2 = tot.z & 0xffff, n1 = tot.y >> 16;
      const int t2 = tot.z >> 16, t1 = tot.w >> 16;
      n_tiles = t2 + t1 + (tot.w & 0xffff);
      int rank0 = ex.y & 0xffff, rank1 = ex.y >> 16, rank2 = ex.z & 0xffff;
      int tb0 = ex.w & 0xffff, tb1 = ex.w >> 16, tb2 = ex.z >> 16;
      int run = ex.x;
      const bool publish = blockIdx.x == 0 && ok && !dry;
      for (int h = 0; h < gpt && e0 + h < E; ++h) {
        const int e = e0 + h, r = s_off[e], c2 = cls_of(r), nt = (r + tn - 1) / tn;
        s_off[e] = run;
        if (publish) {
          ws.offsets[e] = run;
          if (c2 == 2) ws.grp_list[rank2++] = (tb2 << kGrpIdBits) | e;
          else if (c2 == 1) ws.grp_list[n2 + rank1++] = ((t2 + tb1) << kGrpIdBits) | e;
          else ws.grp_list[n2 + n1 + rank0++] = ((t2 + t1 + tb0) << kGrpIdBits) | e;
        }
        tb2 += c2 == 2 ? nt : 0;
        tb1 += c2 == 1 ? nt : 0;
        tb0 += c2 == 0 ? nt : 0;
        run += r;
      }
      if (tid == 0) {
        s_off[E] = tot.x;
        if (publish) {
          ws.offsets[E] = tot.x;
          ws.grp_list[E] = n_tiles << kGrpIdBits;
        }
      }
      for (int h = 0; h < gpt; ++h) n_hit += __syncthreads_count((hm >> h) & 1);  // (also a barrier)
    }
    if (trace && tid == 0) trace[4] = static_cast<int64_t>(globaltimer_ns());
    const bool real = ok && !dry;  // global writes and error checks
    if (real && s_off[E] > d.Nmax * k && tid == 0) set_error(ws.err, EPOCH_DEVERR_BOUNDS);  // inconsistent words

    // ---- 4. the own positions: fresh index and list, slots (a warm-up runs
    // the slot arithmetic for every own position, fresh or not)
    const bool step4 = ok && (!dry || (dmask & 4));
    if (step4 && wid == 0) {
      int f = s_misc[36] / k;  // fresh positions before p0 (each sets k bits)
      for (int j0 = 0; j0 < np; j0 += 32) {
        const int j = j0 + lane;
        const bool fr = j < np && gt.fr[j];
        const unsigned m = __ballot_sync(0xffffffffu, fr);
        if (j < np && real) {
          const int mine = f + __popc(m & ((1u << lane) - 1u));
          ws.fidx[p0 + j] = fr ? mine : -1;
          if (fr && mine < d.Nmax) ws.fresh_pos[mine] = p0 + j;
        }
        f += __popc(m);
      }
    }
    const int r0 = p0 & 31;
    for (int q = tid; q < (step4 ? np * k : 0); q += nthr) {
      const int j = q / k, jj = q - j * k, t = p0 + j;
      int slot = -1;
      if (gt.fr[j] || dry) {
        const int e = gt.sel[j * 16 + jj];
        const int ci = (e >= 0 && e < E) ? (force ? e : gt.cidx[e]) : -1;
        if (ci < 0 || ci >= n_cand || cand_of(ci) != e) {
          if (real) set_error(ws.err, EPOCH_DEVERR_BOUNDS);
        } else {
          const int rt = t - (wa << 5);  // bit of t counted from word wa (< 96)
          int rank = s_bef[ci];
#pragma unroll
          for (int w = 0; w < 3; ++w) {
            const int lo = max(r0 - 32 * w, 0), hi = min(rt - 32 * w, 32);
            if (hi > lo) rank += __popc(s_own[3 * ci + w] & bit_range(lo, hi));
          }
          slot = s_off[e] + rank;
          if (slot >= s_off[e + 1] || slot >= d.Nmax * k) {
            if (real) set_error(ws.err, EPOCH_DEVERR_BOUNDS);
            slot = -1;
          }
        }
        if (real) {
          ws.slot[static_cast<size_t>(t) * k + jj] = slot >= 0 ? slot : 0;
          if (slot >= 0) ws.wl_pos[slot] = t;
        }
      }
      s_slot[q] = slot;
    }
    __syncthreads();
    if (dry) {  // the scratch the real pass accumulates into starts at zero again
      for (int e = tid; e <= E; e += nthr) s_off[e] = 0;
      for (int c = tid; c < n_cand; c += nthr) {
        s_bef[c] = 0;
        s_own[3 * c] = s_own[3 * c + 1] = s_own[3 * c + 2] = 0u;
      }
      if (tid == 0) s_misc[36] = 0;
      __syncthreads();
    }
  }
  const int n_edges = s_off[E];
  if (trace && tid == 0) trace[5] = static_cast<int64_t>(globaltimer_ns());

  // ---- 5. the worklist rows: each staged row to its k rows of xp (the
  // staged copies are waited for in any case: none may land after the CTA exits)
  if (np > 0) {
    bool landed = false;
    const uint64_t t0 = globaltimer_ns();
    while (!(landed = mbar_try_wait(gt.x_bar, 0)) && globaltimer_ns() - t0 < static_cast<uint64_t>(d.timeout_ns)) {
    }
    if (!landed) {
      if (tid == 0) set_error(ws.err, EPOCH_DEVERR_TIMEOUT);
    } else if (ok) {
      uint8_t *xp = static_cast<uint8_t *>(ws.xp);
      for (int q = tid; q < np * k; q += nthr) {
        const int slot = s_slot[q];
        if (slot >= 0) bulk_store(xp + static_cast<size_t>(slot) * rowb, smem_u32(xs + (q / k) * rowb), rowb);
      }
    }
  }

  if (trace && tid == 0) trace[6] = static_cast<int64_t>(globaltimer_ns());
  // ---- 6. the control words the statistics need (CTA 0); the statistics
  // themselves are finished by the combine kernel (gate_tail_stats), off the
  // path to the expert kernel
  if (blockIdx.x == 0 && ok && tid == 0) {
    Ctrl *c = ws.ctrl;
    c->tiles_up = d.tn > 0 ? (d.I / 128) * n_tiles : 0;
    c->tiles_dn = d.tn > 0 ? (d.H / kBmDn) * n_tiles : 0;
    c->n_edges = n_edges;
    c->n_hit = n_hit;
  }

  // ---- 7. positions beyond n_pos keep their state; the words of the next
  // iteration start at zero
  {
    const int rd = d.state_rd & 1, wr = rd ^ 1;
    const int gi = blockIdx.x * nthr + tid, gs = gridDim.x * nthr;
    for (int t = n + gi; t < d.Nmax; t += gs) {
      ws.stamp[static_cast<size_t>(wr) * d.Nmax + t] = ws.stamp[static_cast<size_t>(rd) * d.Nmax + t];
      ws.prev_dec[static_cast<size_t>(wr) * d.Nmax + t] = ws.prev_dec[static_cast<size_t>(rd) * d.Nmax + t];
    }
    uint32_t *next = ws.sel_words + static_cast<size_t>(rd) * E * cmax;
    for (int q = gi; q < E * cmax; q += gs) next[q] = 0u;
  }
  if (trace && tid == 0) trace[0] = static_cast<int64_t>(globaltimer_ns());
  bulk_store_wait_read();  // the staged rows are read out before the CTA exits
  if (trace && tid == 0) trace[3] = static_cast<int64_t>(globaltimer_ns());
  if (d.trace && tid == 0 && blockIdx.x < kTraceCtas) ws.trace[(8ull * kTraceCtas + blockIdx.x) * kTraceFields + 3] = static_cast<int64_t>(globaltimer_ns());
}

// The iteration's statistics and control words after a gate-tail worklist,
// by one thread of the combine kernel (which runs once the expert kernel, and
// so the gate, has completed): the tallies every gate CTA added (they restart
// for the next call), the coverage count, and the values gate CTA 0 left in
// the control block. Out of line: one CTA of the combine runs it.
static __device__ __noinline__ void gate_tail_stats(const Dims &d, const Work &ws) {
  const int n = d.n_pos, E = d.E, k = d.k;
  int tl[kTallies];
#pragma unroll
  for (int q = 0; q < kTallies; ++q) tl[q] = __ldcg(ws.tally + q);
  const int under = d.cov_check ? __ldcg(ws.cov_under) : 0;
  Ctrl *c = ws.ctrl;
  const int anom = c->anom, slen = c->support_len, n_edges = c->n_edges, n_hit = c->n_hit;
  const int tiles_up = c->tiles_up, tiles_dn = c->tiles_dn;
#pragma unroll
  for (int q = 0; q < kTallies; ++q) ws.tally[q] = 0;
  *ws.cov_under = 0;
  const bool force = d.host_fallback != 0 || anom != 0;
  const int n_fresh = tl[6];
  const int nt_sh = d.tn > 0 ? d.n_sh * ((n + d.tn - 1) / d.tn) : 0;
  const int fb = (d.host_fallback ? 1 : 0) | ((anom & 1) ? 2 : 0) | ((anom & 2) ? 4 : 0);
  if (n_fresh * k != n_edges) set_error(ws.err, EPOCH_DEVERR_BOUNDS);
  if (tl[5]) set_error(ws.err, EPOCH_DEVERR_FLAGS);
  c->n_fresh = n_fresh;
  c->fallback = fb;
  // support coverage of this iteration's fresh positions -> the next iteration
  c->short_next =
      (d.cov_check && static_cast<float>(under) > (1.f - d.cov_q) * static_cast<float>(n_fresh)) ? 1 : 0;
  epoch_iter_stats st;
  st.iteration = d.iter;
  st.n_pos = n;
  st.n_live = tl[C_LIVE];
  st.n_new = tl[C_NEW];
  st.n_miss = tl[C_MISS];
  st.n_stale = tl[C_STALE];
  st.n_forced = force ? tl[C_REUSE] : 0;
  st.n_reuse = force ? 0 : tl[C_REUSE];
  st.n_fresh = n_fresh;
  st.n_edges = n_edges;
  st.n_hit_experts = n_hit;
  st.support_len = fb ? E : slen;
  st.fallback = fb;
  st.bad_flags = tl[5];
  st.tiles_up = tiles_up + (d.I_s / 128) * nt_sh;
  st.tiles_down = tiles_dn + (d.H / kBmDn) * nt_sh;
  st.n_under = under;
  *ws.stats = st;
  if (d.stats_out) *d.stats_out = st;
}

}  // namespace epoch

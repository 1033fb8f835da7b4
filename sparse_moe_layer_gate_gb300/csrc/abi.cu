// C ABI of the Epoch MoE-layer iteration: argument checks, workspace carve-up,
// the block-plan state machine (cold path, hot iterations, full-fresh
// fallback), the per-iteration launch sequence, and per-kernel profiling.
//
// Lifecycle ([W] = walk-through page "Epoch 完全拆解:把扩散块编译成稀疏 MoE 服务单元",
// section "cold、hot-update、hot-skip"): the cold path runs once per block
// (epoch_plan_block); hot iterations reuse the support mask and recompute
// logits, weights and fresh expert outputs; a missing plan, a skipped
// iteration, a shape mismatch or a liveness anomaly fall back to full fresh
// ([W] section "Two Clocks": the plan can always return to the dense path).
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>
#include <vector>

#include "common.cuh"
#include "layer.h"

using namespace epoch;

struct epoch_layer {
  epoch_layer_config cfg;
  Dims dims;  // static part (n_pos, iter, host_fallback filled per call)
  Weights w;
  Work ws;
  Maps maps;
  bool bf16;
  // block-plan state
  bool planned;
  int32_t n_pos_plan;
  int32_t last_iter;
  int32_t state_rd;  // half of the double-buffered iteration state the next iteration reads
  int64_t n_cold, n_hot, n_fallback, n_launch;
  int64_t n_hot_update, n_refresh;
  // profiling
  bool prof;
  struct Pending {
    int kind;
    cudaEvent_t a, b;
  };
  std::vector<Pending> pending;
  std::vector<cudaEvent_t> pool;
  double total_ms[K_NUM];
  int64_t launches[K_NUM];
};

namespace {

constexpr size_t kAlign = 256;

bool aligned16(const void *p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4_or_null(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool valid_config(const epoch_layer_config *c) {
  if (c == nullptr) return false;
  if (c->hidden <= 0 || c->inter <= 0 || c->n_experts < 1 || c->n_experts > 1024) return false;
  if (c->top_k < 1 || c->top_k > 16 || c->top_k > c->n_experts) return false;
  if (c->n_shared < 0 || c->n_shared > 8 || c->n_experts + c->n_shared > 1024) return false;
  if (c->n_shared > 0 && c->shared_inter <= 0) return false;
  if (c->max_positions < 1 || c->max_positions > 16384) return false;
  if (c->dtype != EPOCH_F32 && c->dtype != EPOCH_BF16) return false;
  if (!(c->tau > 0.0 && c->tau <= 1.0)) return false;
  if (c->refresh_R < 1) return false;
  const int q = c->dtype == EPOCH_BF16 ? 128 : 4;
  if (c->hidden % q || c->inter % q) return false;
  if (c->dtype == EPOCH_BF16 && c->hidden % kBmDn) return false;  // down tiles cover 256 rows of H
  if (c->n_shared > 0 && c->shared_inter % q) return false;
  if (c->router != EPOCH_ROUTER_SOFTMAX && c->router != EPOCH_ROUTER_SIGMOID_GROUP) return false;
  if (c->raw_weights != 0 && c->raw_weights != 1) return false;
  if (c->request_size < 0 || c->request_size > c->max_positions) return false;
  if (c->planner != EPOCH_PLANNER_PREFIX && c->planner != EPOCH_PLANNER_ATLAS) return false;
  if (c->planner == EPOCH_PLANNER_ATLAS &&
      (c->router != EPOCH_ROUTER_SOFTMAX || c->request_size != 0 || c->atlas_m < 0 || c->top_k + c->atlas_m > 32 ||
       c->atlas_B < 1 || c->atlas_c < 1 || !(c->atlas_alpha >= 0.0 && c->atlas_alpha <= 1.0) ||
       !(c->atlas_q >= 0.0 && c->atlas_q <= 1.0) || !(c->atlas_beta >= 0.0)))
    return false;
  if (c->coverage_check && !(c->coverage_alpha >= 0.0 && c->coverage_alpha <= 1.0 && c->coverage_q >= 0.0 &&
                             c->coverage_q <= 1.0))
    return false;
  if (c->router == EPOCH_ROUTER_SIGMOID_GROUP &&
      (c->n_group < 1 || c->n_group > 32 || c->n_experts % c->n_group || c->topk_group < 1 ||
       c->topk_group > c->n_group))
    return false;
  return true;
}

// Lays the workspace out (base == nullptr: only measures). Returns total bytes.
size_t carve(const epoch_layer_config &c, char *base, Work *w) {
  size_t off = 0;
  auto take = [&](size_t bytes) -> void * {
    off = (off + kAlign - 1) & ~(kAlign - 1);
    void *p = base ? base + off : nullptr;
    off += bytes;
    return p;
  };
  const size_t N = c.max_positions, E = c.n_experts, H = c.hidden, I = c.inter, k = c.top_k;
  const size_t nsh = c.n_shared, Is = c.n_shared ? c.shared_inter : 0;
  const size_t act = c.dtype == EPOCH_BF16 ? 2 : 4;
  const size_t chunks = (N + 31) / 32;
  Work t;
  t.stamp = static_cast<int32_t *>(take(2 * N * 4));
  t.prev_dec = static_cast<uint8_t *>(take(2 * N));
  const size_t R = c.request_size > 0 ? (N + c.request_size - 1) / c.request_size : 1;
  t.support_mask = static_cast<uint8_t *>(take(R * E));
  t.support_ids = static_cast<int32_t *>(take(E * 4));
  t.plan_counts = static_cast<int32_t *>(take(R * E * 4));
  t.req_ids = static_cast<int32_t *>(take(R * E * 4));
  t.req_len = static_cast<int32_t *>(take(R * 4));
  const bool atlas = c.planner == EPOCH_PLANNER_ATLAS;
  t.atlas_cand = static_cast<int32_t *>(take(atlas ? N * 32 * 4 : 16));
  t.atlas_w = static_cast<float *>(take(atlas ? N * 32 * 4 : 16));
  t.atlas_r = static_cast<float *>(take(atlas ? N * 4 : 16));
  t.atlas_pop = static_cast<unsigned long long *>(take(E * 8));
  t.atlas_out = static_cast<int32_t *>(take(16));
  t.cache = take(N * H * act);
  t.logits = static_cast<float *>(take(N * E * 4));
  t.cat = static_cast<uint8_t *>(take(N));
  t.fidx = static_cast<int32_t *>(take(N * 4));
  t.fresh_pos = static_cast<int32_t *>(take(N * 4));
  t.sel = static_cast<int32_t *>(take(N * k * 4));
  t.selw = static_cast<float *>(take(N * k * 4));
  t.sel_words = static_cast<uint32_t *>(take(2 * chunks * E * 4));
  t.offsets = static_cast<int32_t *>(take((E + 1) * 4));
  t.grp_list = static_cast<int32_t *>(take((E + nsh + 1) * 4));
  t.done_up = static_cast<int32_t *>(take(E * ((I + 127) / 128) * 4));
  t.cov_under = static_cast<int32_t *>(take(8));
  t.tile_ctr = static_cast<int32_t *>(take(16));
  t.tally = static_cast<int32_t *>(take(32));
  t.gate_arrive = static_cast<int32_t *>(take(8));
  t.sh_ctr = static_cast<int32_t *>(take((1 + nsh * ((N + kTnUp - 1) / kTnUp)) * 4));
  t.wl_pos = static_cast<int32_t *>(take(N * k * 4));
  t.slot = static_cast<int32_t *>(take(N * k * 4));
  t.xp = take(N * k * H * act);
  t.a_int = take(N * k * I * act);
  t.a_sh = take(nsh * N * Is * act + 16);
  t.o_int = take(N * k * H * act);
  t.o_sh = take(nsh * N * H * act + 16);
  if (c.dtype == EPOCH_BF16) {
    t.pk_gu = static_cast<uint8_t *>(take(E * I * H * 2 * 2));
    t.pk_d = static_cast<uint8_t *>(take(E * H * I * 2));
    t.pk_sgu = static_cast<uint8_t *>(take(nsh * Is * H * 2 * 2 + 16));
    t.pk_sd = static_cast<uint8_t *>(take(nsh * H * Is * 2 + 16));
  } else {
    t.pk_gu = t.pk_d = t.pk_sgu = t.pk_sd = nullptr;
  }
  t.trace = static_cast<int64_t *>(take(static_cast<size_t>(kTraceRows) * kTraceCtas * kTraceFields * 8));
  t.timeline = static_cast<unsigned long long *>(take(2ull * K_NUM * 8));
  t.ctrl = static_cast<Ctrl *>(take(sizeof(Ctrl)));
  t.stats = static_cast<epoch_iter_stats *>(take(sizeof(epoch_iter_stats)));
  t.err = static_cast<uint32_t *>(take(16));
  if (w) *w = t;
  return (off + kAlign - 1) & ~(kAlign - 1);
}

cudaStream_t S(epoch_stream s) { return reinterpret_cast<cudaStream_t>(s); }

cudaEvent_t get_event(epoch_layer *L) {
  if (!L->pool.empty()) {
    cudaEvent_t e = L->pool.back();
    L->pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Enqueues one kernel (bracketed by events while profiling) and counts it.
template <typename F>
epoch_status run(epoch_layer *L, Kind kind, cudaStream_t s, F &&launch) {
  cudaEvent_t a = nullptr, b = nullptr;
  if (L->prof) {
    a = get_event(L);
    cudaEventRecord(a, s);
  }
  const cudaError_t e = launch();
  if (L->prof) {
    b = get_event(L);
    cudaEventRecord(b, s);
    L->pending.push_back({kind, a, b});
  }
  ++L->n_launch;
  return e == cudaSuccess ? EPOCH_OK : EPOCH_ECUDA;
}

#define EPOCH_TRY(expr)                       \
  do {                                        \
    const epoch_status st_ = (expr);          \
    if (st_ != EPOCH_OK) return st_;          \
  } while (0)

// Support rows of the plan: one per request with per-request supports, else one.
size_t plan_rows(const epoch_layer_config &c, int32_t n_pos) {
  return c.request_size > 0 ? static_cast<size_t>((n_pos + c.request_size - 1) / c.request_size) : 1;
}

Dims call_dims(const epoch_layer *L, int32_t n_pos, int32_t iter, int host_fallback) {
  Dims d = L->dims;
  d.n_pos = n_pos;
  d.iter = iter;
  d.host_fallback = host_fallback;
  d.state_rd = L->state_rd;
  d.wl_in_gate = 0;
  return d;
}

// G = x W_r^T + b for every position: tcgen05 for bf16 layers (whose gate
// kernel also classifies the positions and takes their top-k, except in plan
// mode), FFMA for fp32 layers (followed by the select kernel). *x_map_up gets
// x with boxes of kTnUp rows (shared-expert up tiles).
epoch_status run_gate(epoch_layer *L, Dims &d, const void *x, const uint8_t *live, const uint8_t *decoded,
                      CUtensorMap *x_map_up, cudaStream_t s) {
  if (L->bf16) {
    if (!encode_kmajor_bf16(x_map_up, x, d.H, d.n_pos, kTnUp)) return EPOCH_ECUDA;
    return run(L, K_GATE, s,
               [&] { return launch_gate_tc(d, L->maps, L->ws, x, L->w.b_router, live, decoded, s); });
  }
  EPOCH_TRY(run(L, K_GATE, s, [&] { return launch_gate_simt(d, L->w, L->ws, x, 0, s); }));
  if (d.plan_mode) return EPOCH_OK;
  return run(L, K_SELECT, s, [&] { return launch_select(d, L->ws, live, decoded, L->w.b_router, s); });
}

// The support from the logits of the plan-mode gate: the hit-count prefix
// rule (one support, or one per request), or the Expert Atlas planner.
// clear_state: a block plan (resets the block's cache state); else a hot update.
epoch_status run_planner(epoch_layer *L, const Dims &d, int clear_state, int32_t *ids_out, int32_t *len_out,
                         cudaStream_t s) {
  if (L->cfg.planner == EPOCH_PLANNER_ATLAS) {
    const AtlasParams a{L->cfg.atlas_m, L->cfg.atlas_B, L->cfg.atlas_c, L->cfg.atlas_alpha, L->cfg.atlas_q,
                        L->cfg.atlas_beta};
    return run(L, K_PLAN_SUPPORT, s, [&] { return launch_atlas(d, L->ws, a, clear_state, ids_out, len_out, s); });
  }
  const int32_t n_pos = d.n_pos;
  if (cudaMemsetAsync(L->ws.plan_counts, 0, sizeof(int32_t) * d.E * plan_rows(L->cfg, n_pos), s) != cudaSuccess)
    return EPOCH_ECUDA;
  EPOCH_TRY(run(L, K_PLAN_TOPK, s, [&] { return launch_plan_topk(d, L->w, L->ws, s); }));
  const double tau = L->cfg.tau;
  const int all = tau >= 1.0;
  const int32_t T = static_cast<int32_t>(std::ceil(tau * static_cast<double>(n_pos * L->cfg.top_k)));
  return run(L, K_PLAN_SUPPORT, s,
             [&] { return launch_plan_support(d, L->ws, T, all, clear_state, ids_out, len_out, tau, s); });
}

}  // namespace

extern "C" {

size_t epoch_workspace_bytes(const epoch_layer_config *cfg) {
  if (!valid_config(cfg)) return 0;
  return carve(*cfg, nullptr, nullptr);
}

epoch_status epoch_layer_create(const epoch_layer_config *cfg, const epoch_layer_weights *w, void *workspace,
                                size_t bytes, epoch_layer **out) {
  if (out == nullptr || w == nullptr || !valid_config(cfg)) return EPOCH_EINVAL;
  if (workspace == nullptr || (reinterpret_cast<uintptr_t>(workspace) & (kAlign - 1))) return EPOCH_EINVAL;
  if (bytes < carve(*cfg, nullptr, nullptr)) return EPOCH_EINVAL;
  if (!aligned16(w->w_router) || !aligned16(w->b_router) || !aligned16(w->w_gate) || !aligned16(w->w_up) ||
      !aligned16(w->w_down))
    return EPOCH_EINVAL;
  if (cfg->n_shared > 0 && (!aligned16(w->ws_gate) || !aligned16(w->ws_up) || !aligned16(w->ws_down)))
    return EPOCH_EINVAL;
  epoch_layer *L = new (std::nothrow) epoch_layer();
  if (L == nullptr) return EPOCH_ECUDA;
  L->cfg = *cfg;
  L->bf16 = cfg->dtype == EPOCH_BF16;
  carve(*cfg, static_cast<char *>(workspace), &L->ws);
  L->w = Weights{w->w_router, w->b_router, w->w_gate, w->w_up, w->w_down, w->ws_gate, w->ws_up, w->ws_down};
  Dims &d = L->dims;
  memset(&d, 0, sizeof(d));
  d.H = cfg->hidden;
  d.E = cfg->n_experts;
  d.I = cfg->inter;
  d.k = cfg->top_k;
  d.n_sh = cfg->n_shared;
  d.I_s = cfg->n_shared ? cfg->shared_inter : 128;
  d.Nmax = cfg->max_positions;
  d.R = cfg->refresh_R;
  d.residual = cfg->residual ? 1 : 0;
  d.router = cfg->router;
  d.n_group = cfg->router ? cfg->n_group : 1;
  d.topk_group = cfg->router ? cfg->topk_group : 1;
  d.raw_weights = cfg->raw_weights;
  d.req_size = cfg->request_size;
  d.cov_check = cfg->coverage_check ? 1 : 0;
  d.cov_alpha = static_cast<float>(cfg->coverage_alpha);
  d.cov_q = static_cast<float>(cfg->coverage_q);
  d.tn = L->bf16 ? kTnUp : 0;
  d.cmax = (cfg->max_positions + 31) / 32;
  d.timeout_ns = 2000000000ll;
  memset(&L->maps, 0, sizeof(L->maps));
  if (L->bf16) {
    if (!tma_encode_init()) {
      delete L;
      return EPOCH_ECUDA;
    }
    const uint64_t H = d.H, E = d.E, I = d.I, N = d.Nmax, k = d.k, nsh = d.n_sh, Is = d.I_s;
    bool ok = encode_kmajor_bf16(&L->maps.w_router, w->w_router, H, E, 128) && gate_tc_supported(d);
    for (int b = 0; ok && b < 4; ++b)
      ok = encode_kmajor_bf16(&L->maps.xp[b], L->ws.xp, H, N * k, kBoxRows[b]) &&
           encode_kmajor_bf16(&L->maps.a_int[b], L->ws.a_int, I, N * k, kBoxRows[b]);
    if (ok && nsh > 0) {
      ok = encode_kmajor_bf16(&L->maps.a_sh, L->ws.a_sh, Is, nsh * N, kTnDn);
    }
    if (!ok) {
      delete L;
      return EPOCH_EINVAL;
    }
  }
  // empty cache, no plan: zero the workspace, stamps = -1, support = every expert
  if (cudaMemset(workspace, 0, bytes) != cudaSuccess ||
      cudaMemset(L->ws.stamp, 0xFF, 2 * sizeof(int32_t) * d.Nmax) != cudaSuccess ||
      cudaMemset(L->ws.support_mask, 1, plan_rows(*cfg, d.Nmax) * d.E) != cudaSuccess) {
    delete L;
    return EPOCH_ECUDA;
  }
  if (L->bf16) {
    // expert weights -> packed swizzled tiles (gate and up tiles interleaved)
    const int64_t H = d.H, E = d.E, I = d.I, nsh = d.n_sh, Is = d.I_s, T = kTileBytes;
    cudaError_t e = launch_pack_tiles(w->w_gate, E * I, H, L->ws.pk_gu, 2 * T, 0, 1, nullptr);
    if (e == cudaSuccess) e = launch_pack_tiles(w->w_up, E * I, H, L->ws.pk_gu, 2 * T, T, 1, nullptr);
    if (e == cudaSuccess) e = launch_pack_tiles(w->w_down, E * H, I, L->ws.pk_d, 2 * T, 0, 2, nullptr);
    if (e == cudaSuccess && nsh > 0) {
      e = launch_pack_tiles(w->ws_gate, nsh * Is, H, L->ws.pk_sgu, 2 * T, 0, 1, nullptr);
      if (e == cudaSuccess) e = launch_pack_tiles(w->ws_up, nsh * Is, H, L->ws.pk_sgu, 2 * T, T, 1, nullptr);
      if (e == cudaSuccess) e = launch_pack_tiles(w->ws_down, nsh * H, Is, L->ws.pk_sd, 2 * T, 0, 2, nullptr);
    }
    if (e != cudaSuccess) {
      delete L;
      return EPOCH_ECUDA;
    }
  }
  Ctrl c0;
  memset(&c0, 0, sizeof(c0));
  c0.support_len = d.E;
  if (cudaMemcpy(L->ws.ctrl, &c0, sizeof(c0), cudaMemcpyHostToDevice) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    delete L;
    return EPOCH_ECUDA;
  }
  L->planned = false;
  L->n_pos_plan = 0;
  L->last_iter = -1;
  L->state_rd = 0;
  L->prof = false;
  for (int i = 0; i < K_NUM; ++i) {
    L->total_ms[i] = 0.0;
    L->launches[i] = 0;
  }
  *out = L;
  return EPOCH_OK;
}

epoch_status epoch_plan_block(epoch_layer *L, const void *x, int32_t n_pos, epoch_stream stream,
                              int32_t *support_ids_dev, int32_t *support_len_dev) {
  if (L == nullptr || !aligned16(x) || n_pos < 1 || n_pos > L->cfg.max_positions) return EPOCH_EINVAL;
  if (!aligned4_or_null(support_ids_dev) || !aligned4_or_null(support_len_dev)) return EPOCH_EINVAL;
  cudaStream_t s = S(stream);
  Dims d = call_dims(L, n_pos, 0, 0);
  d.plan_mode = 1;
  CUtensorMap x_map_up;
  EPOCH_TRY(run_gate(L, d, x, nullptr, nullptr, &x_map_up, s));
  EPOCH_TRY(run_planner(L, d, 1, support_ids_dev, support_len_dev, s));
  L->planned = true;
  L->n_pos_plan = n_pos;
  L->last_iter = -1;
  ++L->n_cold;
  return EPOCH_OK;
}

epoch_status epoch_moe_iter_path(epoch_layer *L, const void *x, const uint8_t *live, const uint8_t *decoded,
                                 int32_t n_pos, int32_t iteration, int32_t path, void *y, epoch_stream stream,
                                 epoch_iter_stats *stats_dev) {
  if (L == nullptr || !aligned16(x) || !aligned16(y) || live == nullptr || decoded == nullptr) return EPOCH_EINVAL;
  if (!aligned4_or_null(stats_dev)) return EPOCH_EINVAL;
  if (n_pos < 1 || n_pos > L->cfg.max_positions || iteration < 0) return EPOCH_EINVAL;
  if ((path & ~(EPOCH_PATH_HOT_UPDATE | EPOCH_PATH_REFRESH)) != 0) return EPOCH_EINVAL;
  cudaStream_t s = S(stream);
  const int host_fallback = !L->planned || iteration != L->last_iter + 1 || n_pos != L->n_pos_plan;
  Dims d = call_dims(L, n_pos, iteration, host_fallback);
  d.stats_out = stats_dev;
  if (path & EPOCH_PATH_REFRESH) d.R = 0;  // every cached row counts as stale: all positions fresh
  if (d.trace) {
    if (cudaMemsetAsync(L->ws.timeline, 0xFF, K_NUM * 8, s) != cudaSuccess ||
        cudaMemsetAsync(L->ws.timeline + K_NUM, 0, K_NUM * 8, s) != cudaSuccess)
      return EPOCH_ECUDA;
  }
  CUtensorMap x_map_up;
  if (path & EPOCH_PATH_HOT_UPDATE) {
    // hot-update path: logits of this iteration, the support rebuilt from them
    // (block-plan rule, state kept), then classification and top-k over it
    d.plan_mode = 1;
    EPOCH_TRY(run_gate(L, d, x, live, decoded, &x_map_up, s));
    EPOCH_TRY(run_planner(L, d, 0, nullptr, nullptr, s));
    d.plan_mode = 0;
    EPOCH_TRY(run(L, K_SELECT, s, [&] { return launch_select(d, L->ws, live, decoded, L->w.b_router, s); }));
    ++L->n_hot_update;
  } else {
    // bf16 gates of one wave build the worklist in their tail
    d.wl_in_gate = L->bf16 && gate_builds_worklist(d) ? 1 : 0;
    EPOCH_TRY(run_gate(L, d, x, live, decoded, &x_map_up, s));
  }
  if (path & EPOCH_PATH_REFRESH) ++L->n_refresh;
  if (L->bf16) {
    if (!d.wl_in_gate)
      EPOCH_TRY(run(L, K_ROUTING, s, [&] { return launch_route(d, L->ws, x, s); }));
    EPOCH_TRY(run(L, K_UP, s, [&] { return launch_experts_tc(d, L->maps, L->ws, x_map_up, s); }));
  } else {
    EPOCH_TRY(run(L, K_ROUTING, s, [&] { return launch_route(d, L->ws, nullptr, s); }));
    EPOCH_TRY(run(L, K_UP, s, [&] { return launch_up_simt(d, L->w, L->ws, x, s); }));
    EPOCH_TRY(run(L, K_DOWN, s, [&] { return launch_down_simt(d, L->w, L->ws, s); }));
  }
  L->state_rd ^= 1;  // this iteration wrote the new state into the other half
  EPOCH_TRY(run(L, K_COMBINE, s, [&] { return launch_combine(d, L->ws, x, y, L->bf16, s); }));
  L->last_iter = iteration;
  if (host_fallback) ++L->n_fallback;
  else ++L->n_hot;
  return EPOCH_OK;
}

epoch_status epoch_moe_iter(epoch_layer *L, const void *x, const uint8_t *live, const uint8_t *decoded,
                            int32_t n_pos, int32_t iteration, void *y, epoch_stream stream,
                            epoch_iter_stats *stats_dev) {
  return epoch_moe_iter_path(L, x, live, decoded, n_pos, iteration, 0, y, stream, stats_dev);
}

epoch_status epoch_block_end(epoch_layer *L) {
  if (L == nullptr) return EPOCH_EINVAL;
  L->planned = false;
  return EPOCH_OK;
}

epoch_status epoch_get_status(epoch_layer *L, epoch_stream stream, uint32_t *word_out) {
  if (L == nullptr) return EPOCH_EINVAL;
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, L->ws.err, sizeof(word), cudaMemcpyDeviceToHost, S(stream)) != cudaSuccess ||
      cudaStreamSynchronize(S(stream)) != cudaSuccess)
    return EPOCH_ECUDA;
  if (word_out) *word_out = word;
  if (word & EPOCH_DEVERR_TIMEOUT) return EPOCH_ETIMEOUT;
  return word ? EPOCH_EDEVICE : EPOCH_OK;
}

epoch_status epoch_clear_status(epoch_layer *L, epoch_stream stream) {
  if (L == nullptr) return EPOCH_EINVAL;
  // the gate's grid barrier too: a call that timed out may leave it part-way
  return cudaMemsetAsync(L->ws.err, 0, sizeof(uint32_t), S(stream)) == cudaSuccess &&
                 cudaMemsetAsync(L->ws.gate_arrive, 0, 2 * sizeof(int32_t), S(stream)) == cudaSuccess
             ? EPOCH_OK
             : EPOCH_ECUDA;
}

epoch_status epoch_read_stats(epoch_layer *L, epoch_iter_stats *out, epoch_stream stream) {
  if (L == nullptr || out == nullptr) return EPOCH_EINVAL;
  if (cudaMemcpyAsync(out, L->ws.stats, sizeof(*out), cudaMemcpyDeviceToHost, S(stream)) != cudaSuccess ||
      cudaStreamSynchronize(S(stream)) != cudaSuccess)
    return EPOCH_ECUDA;
  return EPOCH_OK;
}

epoch_status epoch_debug_pointers(epoch_layer *L, epoch_debug_view *v) {
  if (L == nullptr || v == nullptr) return EPOCH_EINVAL;
  v->support_ids = L->ws.support_ids;
  v->support_len = &L->ws.ctrl->support_len;
  v->plan_counts = L->ws.plan_counts;
  v->logits = L->ws.logits;
  v->fresh_pos = L->ws.fresh_pos;
  v->sel = L->ws.sel;
  v->sel_w = L->ws.selw;
  v->offsets = L->ws.offsets;
  v->wl_pos = L->ws.wl_pos;
  v->slot = L->ws.slot;
  v->stamp = L->ws.stamp + static_cast<size_t>(L->state_rd) * L->cfg.max_positions;
  v->cache = L->ws.cache;
  v->trace = L->ws.trace;
  v->timeline = reinterpret_cast<const int64_t *>(L->ws.timeline);
  v->stats = L->ws.stats;
  v->error_word = L->ws.err;
  v->support_masks = L->ws.support_mask;
  v->request_ids = L->ws.req_ids;
  v->request_len = L->ws.req_len;
  v->atlas_result = L->ws.atlas_out;
  return EPOCH_OK;
}

epoch_status epoch_debug_copy(void *host_dst, const void *dev_src, size_t bytes, epoch_stream stream) {
  if (host_dst == nullptr || dev_src == nullptr) return EPOCH_EINVAL;
  if (bytes == 0) return EPOCH_OK;
  if (cudaMemcpyAsync(host_dst, dev_src, bytes, cudaMemcpyDeviceToHost, S(stream)) != cudaSuccess ||
      cudaStreamSynchronize(S(stream)) != cudaSuccess)
    return EPOCH_ECUDA;
  return EPOCH_OK;
}

epoch_status epoch_path_counters(epoch_layer *L, int64_t *cold, int64_t *hot, int64_t *fallback) {
  if (L == nullptr) return EPOCH_EINVAL;
  if (cold) *cold = L->n_cold;
  if (hot) *hot = L->n_hot;
  if (fallback) *fallback = L->n_fallback;
  return EPOCH_OK;
}

epoch_status epoch_path_counters_ex(epoch_layer *L, int64_t *hot_update, int64_t *refresh) {
  if (L == nullptr) return EPOCH_EINVAL;
  if (hot_update) *hot_update = L->n_hot_update;
  if (refresh) *refresh = L->n_refresh;
  return EPOCH_OK;
}

epoch_status epoch_set_wait_timeout(epoch_layer *L, int64_t timeout_ns) {
  if (L == nullptr || timeout_ns < 1000) return EPOCH_EINVAL;
  L->dims.timeout_ns = timeout_ns;
  return EPOCH_OK;
}

epoch_status epoch_set_tracing(epoch_layer *L, int32_t enable) {
  if (L == nullptr) return EPOCH_EINVAL;
  L->dims.trace = enable ? 1 : 0;
  return EPOCH_OK;
}

epoch_status epoch_set_profiling(epoch_layer *L, int32_t enable) {
  if (L == nullptr) return EPOCH_EINVAL;
  L->prof = enable != 0;
  return EPOCH_OK;
}

epoch_status epoch_read_profile(epoch_layer *L, epoch_profile *out) {
  if (L == nullptr || out == nullptr) return EPOCH_EINVAL;
  for (auto &p : L->pending) {
    if (cudaEventSynchronize(p.b) != cudaSuccess) return EPOCH_ECUDA;
    float ms = 0.f;
    cudaEventElapsedTime(&ms, p.a, p.b);
    L->total_ms[p.kind] += ms;
    L->launches[p.kind] += 1;
    L->pool.push_back(p.a);
    L->pool.push_back(p.b);
  }
  L->pending.clear();
  for (int i = 0; i < EPOCH_PROF_KINDS; ++i) {
    out->name[i] = i < K_NUM ? kKindName[i] : "";
    out->launches[i] = i < K_NUM ? L->launches[i] : 0;
    out->total_ms[i] = i < K_NUM ? L->total_ms[i] : 0.0;
  }
  out->kernels_launched = L->n_launch;
  return EPOCH_OK;
}

epoch_status epoch_reset_profile(epoch_layer *L) {
  if (L == nullptr) return EPOCH_EINVAL;
  epoch_profile tmp;
  const epoch_status st = epoch_read_profile(L, &tmp);
  for (int i = 0; i < K_NUM; ++i) {
    L->total_ms[i] = 0.0;
    L->launches[i] = 0;
  }
  return st;
}

epoch_status epoch_test_wait_timeout(epoch_layer *L, int64_t timeout_ns, epoch_stream stream) {
  if (L == nullptr || timeout_ns < 1000 || timeout_ns > 5000000000ll) return EPOCH_EINVAL;
  return run(L, K_TEST, S(stream), [&] { return launch_wait_test(L->ws.err, timeout_ns, S(stream)); });
}

void epoch_layer_destroy(epoch_layer *L) {
  if (L == nullptr) return;
  for (auto &p : L->pending) {
    cudaEventDestroy(p.a);
    cudaEventDestroy(p.b);
  }
  for (auto e : L->pool) cudaEventDestroy(e);
  delete L;
}

const char *epoch_status_str(epoch_status s) {
  switch (s) {
    case EPOCH_OK: return "ok";
    case EPOCH_EINVAL: return "invalid argument";
    case EPOCH_ESTATE: return "invalid state";
    case EPOCH_ECUDA: return "CUDA runtime error";
    case EPOCH_ETIMEOUT: return "device wait timed out";
    case EPOCH_EDEVICE: return "device-detected error";
  }
  return "unknown status";
}

}  // extern "C"

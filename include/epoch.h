/*
 * epoch.h -- C ABI of the Epoch routed-expert MoE layer iteration on GB300 (sm_103a).
 *
 * Source pages, cited by title and section:
 *   [W] "Epoch 完全拆解:把扩散块编译成稀疏 MoE 服务单元" (pinghaoyang.com.cn walk-through of Epoch)
 *   [A] "Epoch: Compiling Diffusion Blocks for Sparse MoE Serving" (abstract)
 *
 * One layer object holds one MoE layer's block plan (expert support), its
 * per-position routed-output cache with stamps, and the scratch of one
 * iteration. A caller runs, per diffusion block:
 *     epoch_plan_block  (cold path, once)  ->  epoch_moe_iter (i = 0, 1, ...)  ->  epoch_block_end
 * where any iteration may instead take the hot-update or refresh path
 * (epoch_moe_iter_path).
 *
 * Conventions for every entry point:
 *  - Pointers named *_dev or documented as "device" are CUDA device pointers in
 *    the current context; all others are host pointers. Device pointers must be
 *    16-byte aligned.
 *  - Matrices are row-major, contiguous. "dtype" is the layer's epoch_dtype:
 *    EPOCH_F32 (float) or EPOCH_BF16 (bfloat16 bit patterns, 2 bytes).
 *  - The caller owns every buffer it passes (weights, x, masks, y, workspace);
 *    the library keeps the weight and workspace pointers until
 *    epoch_layer_destroy and never frees them. It allocates no device memory.
 *  - Work is enqueued on the given stream (NULL = legacy default stream) and
 *    returns without synchronising, except where a function says it syncs.
 *  - Errors come in three tiers: invalid arguments return EPOCH_EINVAL before
 *    anything is enqueued; state anomalies (no plan, skipped iteration, n_pos
 *    differing from the plan, a decoded->live transition seen on the device)
 *    turn the iteration into a counted full-fresh fallback and still return
 *    EPOCH_OK; device-detected errors set a sticky device error word that
 *    epoch_get_status reports.
 */
#ifndef EPOCH_H
#define EPOCH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *epoch_stream; /* a cudaStream_t */
typedef struct epoch_layer epoch_layer;   /* opaque layer object */

typedef enum {
  EPOCH_OK = 0,
  EPOCH_EINVAL = 1,   /* bad argument; nothing enqueued */
  EPOCH_ESTATE = 2,   /* call not valid in the layer's state (e.g. destroyed workspace too small) */
  EPOCH_ECUDA = 3,    /* a CUDA runtime call failed (launch, copy, driver entry point) */
  EPOCH_ETIMEOUT = 4, /* a bounded device wait gave up (device error word bit 1) */
  EPOCH_EDEVICE = 5   /* other device-detected error (device error word bits 0, 2) */
} epoch_status;

typedef enum { EPOCH_F32 = 0, EPOCH_BF16 = 1 } epoch_dtype;

#define EPOCH_REFRESH_NEVER INT32_MAX

/* Device error word bits (sticky until epoch_clear_status). */
#define EPOCH_DEVERR_FLAGS 1u    /* a position flagged both live and decoded, or neither (treated live) */
#define EPOCH_DEVERR_TIMEOUT 2u  /* a bounded mbarrier wait expired; the kernel returned early */
#define EPOCH_DEVERR_BOUNDS 4u   /* an index failed its range check; the access was skipped */

/* Layer shape and policy.
 *  hidden (H), n_experts (E), inter (I), top_k (k): y_t = sum over the k selected
 *    experts e of w_{t,e} E_e(x_t) ([W] section "MoE 路径为什么成为瓶颈", layer equation),
 *    E_e(x) = W_down,e (silu(W_gate,e x) * (W_up,e x)) (SwiGLU).
 *  n_shared, shared_inter: always-on shared experts added to every position,
 *    untouched by the liveness split ([W] section "Liveness-Shard Parallelism").
 *  max_positions: the largest n_pos any call passes (sizes the workspace).
 *  dtype: element type of weights, x, y and the row cache (router bias is float).
 *  tau in (0, 1]: support coverage fraction; the support is the smallest prefix
 *    of experts ranked by block-start top-k hit count (count desc, id asc) whose
 *    counts reach ceil(tau * n_pos * k) edges, at least k experts; tau = 1 keeps
 *    every expert (the coverage-driven support of [W] section "Expert Atlas").
 *  refresh_R >= 1: a decoded position whose cached routed output is at least R
 *    iterations old is recomputed (EPOCH_REFRESH_NEVER: never) -- the bounded
 *    age of [W] section "decoded-cache 的刷新周期为什么默认取 5".
 *  residual: nonzero makes y = x + routed + shared (chains a stack of layers).
 *  router: EPOCH_ROUTER_SOFTMAX (0): G = x W_r^T + b, top-k of G over the
 *    eligible experts, weights = softmax over the k selected logits.
 *    EPOCH_ROUTER_SIGMOID_GROUP (1), the group-limited rule that [W] section
 *    "Expert Atlas" (step three) runs inside the support: G = x W_r^T (no bias);
 *    scores s = sigmoid(G); selection scores c = s + b; the experts form
 *    n_group groups of consecutive ids, a group's score being the sum of its two
 *    best eligible c; the topk_group best groups (and further ones in that order
 *    while they hold fewer than k eligible experts) are searched for the top-k
 *    of c; weights = the selected s divided by their sum. The block plan's hit
 *    counts use the same rule with every expert eligible.
 *  raw_weights: 0 renormalises the weights over the k selected experts (as
 *    above); 1 keeps the router's own scores -- softmax router: each selected
 *    expert's dense router probability (softmax of G over all E experts);
 *    sigmoid router: the selected s.
 *  coverage_check, coverage_alpha (alpha), coverage_q (q): nonzero checks the
 *    support's coverage every iteration ([W] section "Expert Atlas" defines
 *    it; section "cold、hot-update、hot-skip" sends a layer whose support no
 *    longer covers the routing back to the full fresh path): a fresh position
 *    is under-covered when its dense selection (the router's rule with every
 *    expert eligible) has less than alpha of its raw score mass (dense
 *    probabilities, or sigmoid scores) on support experts; when more than
 *    (1 - q) of the fresh positions are, the next iteration runs full fresh
 *    with every expert eligible (statistics: fallback bit 2, n_under).
 *  request_size: 0 plans one support for all positions of a call. > 0 splits
 *    the positions into requests of request_size consecutive positions (the
 *    last may be shorter), each with its own block plan -- its own hit counts
 *    and threshold ceil(tau * n_r * k) over its n_r positions -- and each
 *    position selects within its request's support ([W] section "cold、
 *    hot-update、hot-skip": a block plan belongs to one diffusion block). The
 *    layer's support (epoch_plan_block's outputs, the statistics) is then the
 *    union of the requests' supports, in ascending expert order.
 *  planner: EPOCH_PLANNER_PREFIX (0) is the hit-count prefix rule of tau.
 *    EPOCH_PLANNER_ATLAS (1) is the planner of [W] section "Expert Atlas"
 *    (softmax router, one support per call; tau unused): every position's
 *    K = min(k + atlas_m, E) best experts by logit are its candidate edges,
 *    weighted by the dense router probabilities W; the coverage floor of a
 *    position is r = atlas_alpha * (mass of its first k candidates); the initial
 *    support is the max(atlas_B, k) experts of largest popularity (sum of W
 *    over their candidate edges); then, while more than (1 - atlas_q) of the
 *    positions have a support coverage C < r, the at most atlas_c experts of
 *    largest positive H_e + atlas_beta * G_e join (G_e: the uncovered mass e
 *    would add, min(W, r - C) summed over under-covered positions; H_e: the
 *    under-covered positions it would lift to r). The support is listed in
 *    the order experts joined.
 * Constraints (else EPOCH_EINVAL): 1 <= top_k <= n_experts <= 1024, top_k <= 16;
 *  bf16: H a multiple of 256, I and shared_inter multiples of 128; f32: multiples of 4;
 *  1 <= max_positions <= 16384; router 1: 1 <= n_group <= 32, n_experts a
 *  multiple of n_group, 1 <= topk_group <= n_group (router 0 ignores both);
 *  raw_weights 0 or 1; with coverage_check, 0 <= coverage_alpha <= 1 and
 *  0 <= coverage_q <= 1; 0 <= request_size <= max_positions; planner 0 or 1; the
 *  Atlas planner needs router 0, request_size 0, atlas_m >= 0, k + atlas_m <= 32,
 *  atlas_B >= 1, atlas_c >= 1, 0 <= atlas_alpha <= 1, 0 <= atlas_q <= 1,
 *  atlas_beta >= 0. */
typedef struct {
  int32_t hidden;
  int32_t n_experts;
  int32_t inter;
  int32_t top_k;
  int32_t n_shared;
  int32_t shared_inter;
  int32_t max_positions;
  int32_t dtype;
  double tau;
  int32_t refresh_R;
  int32_t residual;
  int32_t router;
  int32_t n_group;
  int32_t topk_group;
  int32_t raw_weights;
  int32_t coverage_check;
  double coverage_alpha;
  double coverage_q;
  int32_t request_size;
  int32_t planner;
  int32_t atlas_m;
  int32_t atlas_B;
  int32_t atlas_c;
  double atlas_alpha;
  double atlas_q;
  double atlas_beta;
} epoch_layer_config;

enum { EPOCH_PLANNER_PREFIX = 0, EPOCH_PLANNER_ATLAS = 1 };

enum { EPOCH_ROUTER_SOFTMAX = 0, EPOCH_ROUTER_SIGMOID_GROUP = 1 };

/* Weights, all device pointers of the layer dtype unless noted.
 *  w_router [E][H], b_router [E] (float); w_gate, w_up [E][I][H]; w_down [E][H][I];
 *  ws_gate, ws_up [n_shared][shared_inter][H], ws_down [n_shared][H][shared_inter]
 *  (NULL when n_shared = 0). */
typedef struct {
  const void *w_router;
  const float *b_router;
  const void *w_gate;
  const void *w_up;
  const void *w_down;
  const void *ws_gate;
  const void *ws_up;
  const void *ws_down;
} epoch_layer_weights;

/* Per-iteration statistics, written by the device at the end of each
 * epoch_moe_iter (the block plan's path counters, [W] section "Two Clocks").
 * Categories partition the positions: live + new + miss + stale + forced + reuse = n_pos. */
typedef struct {
  int32_t iteration;
  int32_t n_pos;
  int32_t n_live;      /* still Mask */
  int32_t n_new;       /* decoded now, not at the previous iteration */
  int32_t n_miss;      /* decoded, no cached row */
  int32_t n_stale;     /* decoded, cached row at least R iterations old */
  int32_t n_forced;    /* would have reused its row; made fresh by a fallback */
  int32_t n_reuse;     /* stable decoded, cached row reused */
  int32_t n_fresh;     /* |F_i| */
  int32_t n_edges;     /* worklist length L = k |F_i| */
  int32_t n_hit_experts;
  int32_t support_len; /* experts eligible this iteration (E on a fallback) */
  int32_t fallback;    /* bit 0: host-detected mismatch; bit 1: decoded->live anomaly;
                          bit 2: the previous iteration's support coverage fell short */
  int32_t bad_flags;   /* positions flagged both live and decoded, or neither */
  int32_t tiles_up;    /* grouped-GEMM tiles launched */
  int32_t tiles_down;
  int32_t n_under;     /* fresh positions under the coverage floor (coverage_check; else 0) */
} epoch_iter_stats;

/* Device pointers into the workspace for inspection (valid after the stream
 * that ran the last call has been synchronised; read-only for the caller). */
typedef struct {
  const int32_t *support_ids;  /* [E] experts in rank order (per-request supports: their union,
                                  ascending); first *support_len valid */
  const int32_t *support_len;  /* [1] */
  const int32_t *plan_counts;  /* [E] block-start top-k hit counts */
  const float *logits;         /* [max_positions][E] G of the last iteration, bias included */
  const int32_t *fresh_pos;    /* [n_fresh] ascending fresh positions */
  const int32_t *sel;          /* [max_positions][k] selected experts of position t, selection order
                                  (rows of the fresh positions hold this iteration's values) */
  const float *sel_w;          /* [max_positions][k] routing weights, same rows */
  const int32_t *offsets;      /* [E+1] worklist offsets per expert */
  const int32_t *wl_pos;       /* [n_edges] positions of the expert-sorted worklist */
  const int32_t *slot;         /* [max_positions][k] worklist row of each selection, same rows */
  const int32_t *stamp;        /* [max_positions] iteration of each row's last fresh compute, -1 none */
  const void *cache;           /* [max_positions][H] routed-output cache, layer dtype */
  const epoch_iter_stats *stats;
  const uint32_t *error_word;
  /* [9][1024][8] int64 per-CTA timelines of the last launches while tracing is
   * on (globaltimer ns; unused fields keep older values). Row 0, gate (bf16
   * layers): entry, setup done, first operand stage landed, last MMA issued,
   * epilogue done, position tile, H slice (cluster rank), SM id. Row 1,
   * experts: entry, setup done, producer start, last MMA complete, epilogue
   * done, tiles, ns the producer waited for up tiles, SM id. Row 2, expert
   * epilogue: ns busy, ns waiting for accumulators, longest tile epilogue in
   * ns, that tile's group (bit 30 set: down tile) and valid rows, start and end
   * of the last tile's epilogue, SM id. Row 3, the gate's worklist tail (CTA 0;
   * bf16 layers whose gate grid is one wave): before the final wait, grid
   * barrier passed, candidates' words read, done, offsets scanned, slots
   * written, worklist rows issued. Row 4, gate epilogue: partial sums in shared
   * memory, cluster barrier passed, own rows reduced, exit. Row 5: unused. Row
   * 6, experts: -, ns the producer waited for routed up tiles, for shared-expert
   * up tiles. Row 7, combine (one CTA per position): entry, expert outputs
   * complete, slots checked, end, -, -, -, SM id. Row 8, the gate's worklist
   * tail: field 3, the CTA's end. */
  const int64_t *trace;
  /* [2][EPOCH_PROF_KINDS] while tracing: first CTA entry and last CTA exit
   * (globaltimer ns) of each kernel kind in the last iteration, in the order
   * of epoch_profile.name. */
  const int64_t *timeline;
  /* Support masks [R][E] (1: eligible), R = 1 or, with per-request supports,
   * one row per request; with per-request supports also each request's ranked
   * experts [R][E] and |S| [R] (plan_counts is then [R][E] too). */
  const uint8_t *support_masks;
  const int32_t *request_ids;
  const int32_t *request_len;
  /* Expert Atlas planner: [0] coverage bound met (1) or not, [1] positions
   * left under-covered, [2] repair rounds. */
  const int32_t *atlas_result;
} epoch_debug_view;

/* Per-kernel timing, accumulated while profiling is on. */
#define EPOCH_PROF_KINDS 12
typedef struct {
  const char *name[EPOCH_PROF_KINDS];
  int64_t launches[EPOCH_PROF_KINDS];
  double total_ms[EPOCH_PROF_KINDS];
  int64_t kernels_launched; /* every kernel this layer enqueued since creation */
} epoch_profile;

/* Bytes of device workspace a layer with this config needs (0 on an invalid config). */
size_t epoch_workspace_bytes(const epoch_layer_config *cfg);

/* Validates cfg and weights, carves the caller's device workspace (>= epoch_workspace_bytes,
 * 256-byte aligned) and encodes the TMA descriptors of the weights. Clears the
 * row cache state synchronously (cudaMemset on the legacy stream).
 * Returns EPOCH_EINVAL on a bad config or pointer, EPOCH_ECUDA if the CUDA
 * driver entry point cannot be found. *out is set only on EPOCH_OK. */
epoch_status epoch_layer_create(const epoch_layer_config *cfg, const epoch_layer_weights *w,
                                void *workspace_dev, size_t workspace_bytes, epoch_layer **out);

/* Cold path of a block ([W] section "cold、hot-update、hot-skip"): gate logits
 * G = x W_r^T + b for the n_pos positions of x [n_pos][H] (device, dtype), dense
 * top-k hit counts, the coverage support (see tau), and clears the stamps and
 * previous-decoded flags so that the block starts with an empty cache.
 * Outputs (device, written in stream order; either may be NULL):
 *  support_ids_dev [n_experts] int32: every expert in rank order (hit count
 *    desc, id asc); the first *support_len_dev are the block's support;
 *  support_len_dev [1] int32: |S|.
 * EPOCH_EINVAL if n_pos is not in [1, max_positions] or x (or a non-NULL
 * output) is NULL/misaligned (outputs need 4-byte alignment). */
epoch_status epoch_plan_block(epoch_layer *layer, const void *x_dev, int32_t n_pos, epoch_stream stream,
                              int32_t *support_ids_dev, int32_t *support_len_dev);

/* One refinement iteration ([W] sections "Expert Atlas" step three,
 * "Liveness-Shard Parallelism", "FreshLane Dispatch"):
 *  x_dev [n_pos][H] hidden states; live_dev, decoded_dev [n_pos] uint8 flags
 *  (exactly one nonzero per position); iteration i; y_dev [n_pos][H] output.
 *  Recomputes G for every position; classifies positions (live, newly decoded,
 *  stale or missing row -> fresh; stable decoded -> reuse); takes the top-k of
 *  each fresh position over the support, softmax-weighted; builds the
 *  expert-sorted worklist; runs the SwiGLU experts over it; and writes
 *  y = routed (+ shared) (+ x if residual), routed being the fresh result or the
 *  cached row. Fresh rows refill the cache and get stamp i.
 *  stats_dev (device, may be NULL): receives this iteration's epoch_iter_stats
 *  in stream order, with no host synchronisation (4-byte aligned).
 *  A full-fresh fallback with every expert eligible happens when no plan is
 *  active, i != previous iteration + 1, n_pos differs from the plan, or a
 *  decoded position becomes live. EPOCH_EINVAL on bad sizes or pointers. */
epoch_status epoch_moe_iter(epoch_layer *layer, const void *x_dev, const uint8_t *live_dev,
                            const uint8_t *decoded_dev, int32_t n_pos, int32_t iteration, void *y_dev,
                            epoch_stream stream, epoch_iter_stats *stats_dev);

/* Lifecycle paths of an iteration inside a block ([W] section "cold、hot-update、
 * hot-skip"): 0 is the hot-skip path of epoch_moe_iter (the support of the
 * block plan is reused). EPOCH_PATH_HOT_UPDATE rebuilds the support first,
 * with the block-plan rule (tau), from this iteration's own router logits; the
 * cache, stamps and decoded flags are kept (an update counter or a drifting
 * support is the caller's trigger). EPOCH_PATH_REFRESH is the refresh path:
 * every position goes through the fresh routed path (each cached row counts as
 * stale this iteration, so the selection stays within the support) and every
 * row's age restarts. The two may be combined. */
typedef enum { EPOCH_PATH_HOT_UPDATE = 1, EPOCH_PATH_REFRESH = 2 } epoch_path;

/* epoch_moe_iter on a chosen path (path: a bitwise OR of epoch_path values, or
 * 0). EPOCH_EINVAL for unknown path bits, otherwise as epoch_moe_iter. */
epoch_status epoch_moe_iter_path(epoch_layer *layer, const void *x_dev, const uint8_t *live_dev,
                                 const uint8_t *decoded_dev, int32_t n_pos, int32_t iteration, int32_t path,
                                 void *y_dev, epoch_stream stream, epoch_iter_stats *stats_dev);

/* Ends the block: the plan, cache and stamps become invalid; the next
 * epoch_moe_iter without a new plan runs as a fallback. Host-only, no sync. */
epoch_status epoch_block_end(epoch_layer *layer);

/* Reads the sticky device error word (synchronises the stream). *word_out may be NULL.
 * EPOCH_OK when clear, EPOCH_ETIMEOUT if the timeout bit is set, else EPOCH_EDEVICE. */
epoch_status epoch_get_status(epoch_layer *layer, epoch_stream stream, uint32_t *word_out);

/* Clears the device error word and resets the gate's grid-barrier counter
 * (enqueued on the stream). After a timeout, clear the status before the next
 * call: a call that timed out may leave the barrier part-way. */
epoch_status epoch_clear_status(epoch_layer *layer, epoch_stream stream);

/* Copies the last iteration's statistics to host memory (synchronises the
 * stream; epoch_moe_iter's stats_dev output gives them without a sync). */
epoch_status epoch_read_stats(epoch_layer *layer, epoch_iter_stats *out, epoch_stream stream);

/* Device pointers of the layer's internal arrays (no copy, no sync). */
epoch_status epoch_debug_pointers(epoch_layer *layer, epoch_debug_view *out);

/* Copies bytes from a device pointer (such as one from epoch_debug_pointers)
 * into host memory; synchronises the stream. */
epoch_status epoch_debug_copy(void *host_dst, const void *dev_src, size_t bytes, epoch_stream stream);

/* Host-side counters of the lifecycle paths: plans (cold), normal iterations
 * (hot-skip), host-detected fallbacks. Any pointer may be NULL. */
epoch_status epoch_path_counters(epoch_layer *layer, int64_t *cold, int64_t *hot, int64_t *fallback);

/* Iterations that took the hot-update path, and the refresh path (host-side
 * counts; both also count as hot or fallback above). Any pointer may be NULL. */
epoch_status epoch_path_counters_ex(epoch_layer *layer, int64_t *hot_update, int64_t *refresh);

/* Bounded device waits: a wait that makes no progress for timeout_ns gives up,
 * sets EPOCH_DEVERR_TIMEOUT and lets the kernel return (default 2e9 ns). */
epoch_status epoch_set_wait_timeout(epoch_layer *layer, int64_t timeout_ns);

/* Per-CTA timeline recording in the tcgen05 kernels (see epoch_debug_view.trace). */
epoch_status epoch_set_tracing(epoch_layer *layer, int32_t enable);

/* Per-kernel CUDA-event timing on the launching stream (adds an event pair per launch). */
epoch_status epoch_set_profiling(epoch_layer *layer, int32_t enable);
/* Synchronises pending events, accumulates their times, and copies the totals. */
epoch_status epoch_read_profile(epoch_layer *layer, epoch_profile *out);
epoch_status epoch_reset_profile(epoch_layer *layer);

/* Test hook: launches one kernel whose only work is a bounded wait on an
 * mbarrier that nothing completes, with the given timeout; it must set
 * EPOCH_DEVERR_TIMEOUT and return. Exercises the timeout path without a hang. */
epoch_status epoch_test_wait_timeout(epoch_layer *layer, int64_t timeout_ns, epoch_stream stream);

/* Block planner for callers that cannot allocate device memory (graph capture
 * into a fixed pool, allocator-free runtimes with a pre-planned arena, serving
 * loops that forbid cudaMalloc between requests); it needs no epoch_layer.
 * The pages have no counterpart: this is an interface variant of the cold-path
 * planner of epoch_plan_block (same ranking and coverage rule, see tau) taking
 * the router logits the caller already holds.
 *  logits_dev [n_pos][n_experts] float (device, 16-byte aligned): the router
 *    logits as the layer's gate computes them -- bias included for
 *    EPOCH_ROUTER_SOFTMAX, G = x W_r^T without the bias for
 *    EPOCH_ROUTER_SIGMOID_GROUP;
 *  top_k, tau, router, n_group, topk_group as in epoch_layer_config;
 *  bias_dev [n_experts] float (device): the router bias, used by the
 *    group-limited sigmoid router (may be NULL for the softmax router);
 *  outputs support_ids_dev [n_experts] (experts in rank order) and
 *  support_len_dev [1] (device).
 * Its only scratch, the per-expert hit counts, is a fixed file-scope device
 * array of 1024 int32 (4 KB) that every GPU loading the library holds until
 * exit; n_experts > 1024 or n_pos > 2^26 returns EPOCH_EINVAL. No call
 * allocates memory. Each call made outside stream capture looks up the
 * array's device address; a call under capture reuses the address the last
 * uncaptured call on that device found, so make the first call on each device
 * before any capture. Every call clears the counts it uses. All calls share
 * the array: calls that overlap on the GPU race and must be serialised. */
epoch_status epoch_plan_support_noalloc(const float *logits_dev, int32_t n_pos, int32_t n_experts, int32_t top_k,
                                        double tau, int32_t router, const float *bias_dev, int32_t n_group,
                                        int32_t topk_group, int32_t *support_ids_dev, int32_t *support_len_dev,
                                        epoch_stream stream);

/* Releases host state only (the caller frees the workspace and weights). NULL is ignored. */
void epoch_layer_destroy(epoch_layer *layer);

const char *epoch_status_str(epoch_status s);

#ifdef __cplusplus
}
#endif

#endif /* EPOCH_H */

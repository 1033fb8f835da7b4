// Internal layout of an Epoch MoE layer: workspace carve-up, per-call
// arguments passed to the kernels, and the launchers each .cu file exports.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "epoch.h"

namespace epoch {

// Device-resident control values of one iteration (no host sync inside a call).
struct Ctrl {
  int32_t n_fresh;      // |F_i|
  int32_t fallback;     // bit 0 host mismatch, bit 1 device-detected anomaly
  int32_t n_edges;      // L = k |F_i|
  int32_t n_hit;        // experts with at least one edge
  int32_t tiles_up;     // grouped-GEMM tiles (routed + shared)
  int32_t tiles_dn;
  int32_t support_len;  // |S| of the current plan
  int32_t anom;         // full fresh from the device, set by the classifying kernel: bit 0 a decoded ->
                        // live transition, bit 1 the previous iteration's coverage shortfall
  int32_t short_next;   // the support coverage fell short: the next iteration runs full fresh
};

// Device pointers carved from the caller's workspace.
struct Work {
  // block-lifetime state
  int32_t *stamp;         // [2][Nmax] iteration of the row's last fresh compute, -1 none
  uint8_t *prev_dec;      // [2][Nmax] decoded at the previous iteration
                          // (both double-buffered: an iteration reads half state_rd, writes the other)
  uint8_t *support_mask;  // [R][E] the block's support (R = 1), or one per request (R = requests)
  int32_t *support_ids;   // [E] ranked experts (per-request supports: their union, ascending)
  int32_t *plan_counts;   // [R][E] block-start hit counts (per request)
  int32_t *req_ids;       // [R][E] per-request supports: ranked experts of each request
  int32_t *req_len;       // [R] and each request's |S|
  // Expert Atlas planner
  int32_t *atlas_cand;    // [Nmax][32] candidate experts of each token
  float *atlas_w;         // [Nmax][32] their dense router probabilities
  float *atlas_r;         // [Nmax] coverage floors
  unsigned long long *atlas_pop;  // [E] popularity, fixed point
  int32_t *atlas_out;     // [4] covered_ok, under-covered tokens, repair rounds
  void *cache;            // [Nmax][H] routed-output cache, layer dtype
  // one iteration
  float *logits;          // [Nmax][E] G = x W_r^T + b (gate kernel)
  uint8_t *cat;           // [Nmax] classification code of each position (category | flag bits)
  int32_t *fidx;          // [Nmax] fresh index of a position, -1 if reused
  int32_t *fresh_pos;     // [Nmax] ascending fresh positions
  int32_t *sel;           // [Nmax][k] selected experts of position t (fresh positions only)
  float *selw;            // [Nmax][k] their routing weights
  uint32_t *sel_words;    // [2][E][cmax] bit t%32 of word (e, t/32): fresh position t selected expert e;
                          // the iteration writes half state_rd ^ 1 and clears half state_rd
  int32_t *offsets;       // [E+1]
  int32_t *grp_list;      // [E + n_sh + 1] expert-kernel groups in list order: token tiles of the
                          // groups before << kGrpIdBits | group (shared experts E..E+n_sh-1)
  int32_t *done_up;       // [E][I/128] routed up tiles finished this iteration, per expert and row block
                          // of I (counting token tiles)
  int32_t *cov_under;     // [1] fresh positions of this call under the coverage floor (zeroed by the
                          // worklist bookkeeping once read)
  int32_t *tile_ctr;      // [0] next tile of the expert kernel (dynamic scheduling; reset by the
                          // classifying kernel of the iteration)
  int32_t *tally;         // [8] the gate tail's per-iteration counts (categories, bad flags, fresh),
                          // added by every gate CTA, read and zeroed by CTA 0
  int32_t *gate_arrive;   // grid barrier of the gate before the worklist: [0] arrivals (only grows,
                          // modulo 2^32), [1] its value when the next call begins (set by CTA 0 once
                          // the barrier has passed); both zeroed by the plan and by clearing the status
  int32_t *sh_ctr;        // shared-expert tiles, [sh_stride]: [0] next tile, then the finished up
                          // tiles of each (shared expert, token tile); zeroed by each call's combine
                          // for the next call
  int32_t *wl_pos;        // [Nmax*k] expert-sorted worklist positions
  int32_t *slot;          // [Nmax][k] worklist row of selection (t, j)
  void *xp;               // [Nmax*k][H] token rows of the worklist (x at wl_pos), expert-sorted
  void *a_int;            // [Nmax*k][I] SwiGLU activations of routed edges
  void *a_sh;             // [n_sh*Nmax][I_s] SwiGLU activations of shared experts
  void *o_int;            // [Nmax*k][H] routed expert outputs, layer dtype
  void *o_sh;             // [n_sh*Nmax][H] shared expert outputs, layer dtype
  // expert weights of bf16 layers, packed once at creation into 16 KB tiles of
  // 128 rows x 64 columns in the 128-byte-swizzled K-major layout the tensor
  // cores read, tile (row block rb, K block kb) at index rb * (K / 64) + kb:
  uint8_t *pk_gu;         // routed W_gate/W_up: [E*I/128][H/64] x (gate tile, up tile) = 32 KB
  uint8_t *pk_d;          // routed W_down: [E*H/256][I/64] x (two 128-row tiles) = 32 KB
  uint8_t *pk_sgu;        // shared W_gate/W_up: [n_sh*I_s/128][H/64] x 32 KB
  uint8_t *pk_sd;         // shared W_down: [n_sh*H/256][I_s/64] x 32 KB
  int64_t *trace;         // [kTraceRows][kTraceCtas][8] per-CTA timeline (when tracing)
  unsigned long long *timeline;  // [2][K_NUM]: first CTA entry, last CTA exit per kernel kind (ns)
  Ctrl *ctrl;
  epoch_iter_stats *stats;
  uint32_t *err;
};

// Per-CTA trace record of a tcgen05 kernel (globaltimer ns): entry, setup done,
// first operand stage landed, last MMA committed, epilogue done, tiles, valid
// token columns, SM id.
constexpr int kTraceCtas = 1024;
constexpr int kTraceFields = 8;
constexpr int kTraceRows = 9;

constexpr int kTileBytes = 128 * 64 * 2;  // one packed 128 x 64 bf16 tile
constexpr int kRouteThreads = 256;        // threads per CTA of the worklist kernel

// Shapes and per-call values handed to every kernel by value.
struct Dims {
  int32_t H, E, I, k, n_sh, I_s, Nmax;
  int32_t R;         // refresh period (INT32_MAX = never)
  int32_t residual;
  int32_t n_pos;
  int32_t iter;
  int32_t host_fallback;
  int32_t state_rd;      // half of stamp / prev_dec / sel_words holding the previous iteration's state
  int32_t tn;            // token-tile width of the tcgen05 expert kernel (0 on the SIMT path)
  int32_t cmax;          // words per expert of sel_words: ceil(Nmax / 32)
  int32_t trace;         // nonzero: kernels record per-CTA timelines
  int32_t plan_mode;     // gate kernels: 1 = block plan (logits only), 0 = iteration
  int32_t router;        // 0: softmax over the selected logits (bias in G); 1: group-limited sigmoid
  int32_t n_group, topk_group;  // group rule of router 1
  int32_t raw_weights;   // 1: weights are the router's own scores (no renormalisation over the selection)
  int32_t req_size;      // > 0: positions per request, each request with its own support
  int32_t cov_check;     // support-coverage check: fresh positions with less than cov_alpha of their
  float cov_alpha, cov_q;  // dense selection's mass on the support; more than (1 - cov_q) |F| of them
                           // make the next iteration full fresh
  int32_t wl_in_gate;    // 1: the gate kernel builds the worklist in its tail (bf16 layers whose gate
                         // grid is one wave); 0: the worklist kernel builds it
  int64_t timeout_ns;
  epoch_iter_stats *stats_out;  // caller's copy of this iteration's statistics (nullable)
};

struct Weights {
  const void *w_router;
  const float *b_router;
  const void *w_gate, *w_up, *w_down;
  const void *ws_gate, *ws_up, *ws_down;
};

// TMA descriptors that stay valid for the layer's lifetime.
struct Maps {
  CUtensorMap w_router;   // [E][H], box 64 x 128
  CUtensorMap xp[4];      // [Nmax*k][H], boxes 64 x {32, 64, 128, 256}
  CUtensorMap a_int[4];   // [Nmax*k][I], boxes 64 x {32, 64, 128, 256}
  CUtensorMap a_sh;       // [n_sh*Nmax][I_s], box 64 x 256
};

// Token-box heights of the routed B operands; a tile loads the smallest box
// that holds its valid rows.
constexpr int kBoxRows[4] = {32, 64, 128, 256};

// Parameters of the Expert Atlas planner (see epoch_layer_config).
struct AtlasParams {
  int32_t m, B, c;
  double alpha, q, beta;
};

// Kernel kinds, for profiling and launch counting.
enum Kind {
  K_GATE = 0, K_PLAN_TOPK, K_PLAN_SUPPORT, K_ROUTING, K_UP, K_DOWN, K_COMBINE, K_TEST, K_SELECT, K_NUM
};
extern const char *const kKindName[K_NUM];

#ifdef __CUDACC__
// Records, while tracing, the earliest CTA entry and the latest CTA exit of a
// kernel kind in the workspace timeline (globaltimer ns); a no-op otherwise.
struct KernelMark {
  unsigned long long *tl;
  int kind;
  __device__ __forceinline__ KernelMark(const Dims &d, const Work &ws, int k)
      : tl(d.trace && threadIdx.x == 0 ? ws.timeline : nullptr), kind(k) {
    if (tl) {
      unsigned long long t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)::"memory");
      atomicMin(tl + kind, t);
    }
  }
  __device__ __forceinline__ ~KernelMark() {
    if (tl) {
      unsigned long long t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)::"memory");
      atomicMax(tl + K_NUM + kind, t);
    }
  }
};
#endif

// ------------------------------------------------------------ launchers
// route.cu
cudaError_t launch_gate_simt(const Dims &d, const Weights &w, const Work &ws, const void *x, int bf16,
                             cudaStream_t s);
cudaError_t launch_select(const Dims &d, const Work &ws, const uint8_t *live, const uint8_t *decoded,
                          const float *bias,
                          cudaStream_t s);
cudaError_t launch_plan_topk(const Dims &d, const Weights &w, const Work &ws, cudaStream_t s);
// clear_state: also reset every stamp and decoded flag (a block plan; not a hot update).
// ids_out / len_out: the caller's copies of the ranked experts and |S| (nullable;
// per-request supports: of their union). threshold: the block's (one support);
// per-request thresholds come from tau on the device.
cudaError_t launch_plan_support(const Dims &d, const Work &ws, int32_t threshold, int all_experts,
                                int clear_state, int32_t *ids_out, int32_t *len_out, double tau, cudaStream_t s);
// The worklist kernel: expert offsets, group list, bookkeeping for the combine
// and, for bf16 layers (x non-null), the token rows of the worklist copied into
// xp. Used where the gate does not build the worklist itself.
cudaError_t launch_route(const Dims &d, const Work &ws, const void *x, cudaStream_t s);
// Expert Atlas planner over ws.logits (candidates, then the one-CTA planner).
cudaError_t launch_atlas(const Dims &d, const Work &ws, const AtlasParams &a, int clear_state, int32_t *ids_out,
                         int32_t *len_out, cudaStream_t s);
// CTAs of the worklist kernel: one per SM.
int route_ctas();
cudaError_t launch_combine(const Dims &d, const Work &ws, const void *x, void *y, int bf16, cudaStream_t s);
cudaError_t launch_wait_test(uint32_t *err, int64_t timeout_ns, cudaStream_t s);

// gemm_simt.cu (fp32 layers)
cudaError_t launch_up_simt(const Dims &d, const Weights &w, const Work &ws, const void *x, cudaStream_t s);
cudaError_t launch_down_simt(const Dims &d, const Weights &w, const Work &ws, cudaStream_t s);

// gemm_tc.cu (bf16 layers, tcgen05 + TMA)
// Packs row-major [rows][k] bf16 into swizzled tiles at dst + t * tile_stride + tile_off.
// Tiles of `pair` consecutive row blocks that share a K block are stored adjacent.
cudaError_t launch_pack_tiles(const void *src, int64_t rows, int64_t k, uint8_t *dst, int64_t tile_stride,
                              int64_t tile_off, int pair, cudaStream_t s);
bool tma_encode_init();
bool encode_kmajor_bf16(CUtensorMap *map, const void *base, uint64_t k_elems, uint64_t rows, uint32_t box_rows);
constexpr int kTnUp = 128;    // expert-kernel token tiles (up and down)
constexpr int kTnDn = 128;
// Entries of Work::sh_ctr.
__host__ __device__ inline int sh_stride(const Dims &d) { return 1 + d.n_sh * ((d.Nmax + kTnUp - 1) / kTnUp); }
constexpr int kBmDn = 256;    // rows of H per down tile (two 128-row MMAs)
constexpr int kGrpIdBits = 11;  // group id field of a grp_list entry (E + n_sh <= 1024 < 2^11)

cudaError_t launch_gate_tc(const Dims &d, const Maps &m, const Work &ws, const void *x, const float *bias,
                           const uint8_t *live, const uint8_t *decoded, cudaStream_t s);
// x_map_up: x with boxes of kTnUp rows (shared-expert up tiles). The worklist
// (offsets, group list, xp rows) is complete when the kernel before it in the
// stream has completed.
cudaError_t launch_experts_tc(const Dims &d, const Maps &m, const Work &ws, const CUtensorMap &x_map_up,
                              cudaStream_t s);
// Checks that the gate's thread-block clusters can be scheduled on this device.
bool gate_tc_supported(const Dims &d);
// True when the gate grid of d.n_pos positions is resident all at once (one
// wave of clusters), which its in-kernel grid barrier before the worklist needs.
bool gate_builds_worklist(const Dims &d);

int num_sms();

// cudaLaunchKernelEx of `fn`: programmatic (may start before the previous
// kernel in the stream ends; the kernel calls pdl_wait before touching its
// inputs) and/or with thread-block clusters of `cluster` CTAs along x (0: no
// cluster attribute). When the driver rejects a programmatic launch the kernel
// is launched once more without it, and later launches of this process skip it.
cudaError_t launch_kernel(const void *fn, dim3 grid, dim3 block, size_t smem, cudaStream_t s, void **args,
                          bool programmatic, int cluster = 0);

}  // namespace epoch

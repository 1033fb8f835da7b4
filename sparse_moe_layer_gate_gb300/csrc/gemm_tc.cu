// tcgen05 + TMA GEMMs of the Epoch MoE layer (bf16 in, fp32 accumulate).
//
// Two warp-specialised kernels:
//   k_tc_gate     G = x W_r^T + b for every position: clusters of CTAs split
//                 H, each CTA an (E, position tile) MMA over its slice, the
//                 partials summed over distributed shared memory ([W] section
//                 "Expert Atlas": G in R^{N x E}, recomputed every iteration);
//                 then the classification and top-k of every position, and
//                 the iteration's worklist in the kernel's own tail
//                 (gate_tail.cuh);
//   k_tc_experts  persistent, per group g, UP: A_g = silu(X_g W_gate,g^T) *
//                 (X_g W_up,g^T) and DOWN: O_g = A_g W_down,g^T, both stored as
//                 bf16, in one launch with per-group dependencies.
// Groups are the routed experts with at least one worklist row and the shared
// experts over every position; each routed expert runs once over its compact
// rows (the "light-traffic expert kernel" of [W] section "FreshLane
// Dispatch"); experts with no row produce no tile, so their weights are never
// read (no weight loads for empty slots, same section).
// [W] = walk-through page "Epoch 完全拆解:把扩散块编译成稀疏 MoE 服务单元".
//
// Swap-AB: weight rows are the MMA M dimension (128) and tokens the N
// dimension (16..128, rounded up to 16 per tile), because an expert may hold
// from one to a thousand rows. Roles per expert CTA (192 threads): warp 0
// issues the operand copies into a shared-memory ring (128-byte swizzle,
// K-major), warp 1 issues tcgen05.mma into TMEM accumulators (double-buffered,
// so the epilogue of one tile overlaps the next tile's main loop), warps 2-5
// read TMEM with tcgen05.ld and store. One CTA per SM, persistent over
// device-resident tile counters: no host synchronisation.
#include <cudaTypedefs.h>

#include <cstring>

#include "common.cuh"
#include "layer.h"
#include "select.cuh"
#include "gate_tail.cuh"

namespace epoch {

constexpr int BM = 128;
constexpr int BK = 64;

// Rows of the per-CTA trace: 0 gate, 1 experts, 2 expert epilogue (the gate's worklist tail uses rows 3 and 8).
constexpr int kTraceRowGate = 0;
constexpr int kTraceRowExperts = 1;
constexpr int kTraceRowEpilogue = 2;  // expert-kernel epilogue summary
constexpr int kTraceRowGateEpi = 4;   // gate epilogue steps

struct __align__(128) TcParams {
  CUtensorMap b[4];  // experts: xp (routed up tiles), boxes of 32/64/128/256 rows
  CUtensorMap bs;    // experts: x (shared up tiles), box of kTnUp rows
  CUtensorMap b2[4]; // experts: A (routed down tiles), boxes of 32/64/128/256 rows
  CUtensorMap bs2;   // experts: A (shared down tiles), box of kTnUp rows
  Dims d;
  Work ws;
};

// Waits for a phase without the abort check (teardown after an abort: lets
// copies and MMAs already issued land before the CTA exits).
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity, uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > ns) return;
  }
}

// ---------------------------------------------------------------- gate
// G = x W_r^T + b for every position ([W] section "Expert Atlas": G in
// R^{N x E}, recomputed every iteration), then, in the same launch, each
// position's classification and support-restricted top-k.
//
// A cluster of CS CTAs owns a tile of TN positions and every expert: CTA r of
// the cluster multiplies H-slice r (H / CS columns) on the tensor cores
// (tcgen05.mma, M = 128 experts per block, N = TN positions, fp32 in TMEM),
// writes its fp32 partial sums to its shared memory, and after a cluster
// barrier sums the CS partials of its own TN / CS positions in rank order
// (fixed order: the result does not depend on timing) straight from the other
// CTAs' shared memory, adds the bias (softmax router; the group-limited
// sigmoid router keeps G = x W_r^T and adds the bias to its selection scores)
// and writes G. It then classifies those positions and takes the top-k of the
// fresh ones from the rows it holds.
// Splitting H over the cluster gives 128 CTAs for 1024 positions, each
// streaming 160 KB, instead of a few CTAs streaming all of W_r.
struct __align__(128) GateParams {
  CUtensorMap wr;  // W_r [E][H], box 64 x 128
  CUtensorMap x;   // x [n_pos][H], box 64 x TN
  Dims d;
  Work ws;
  const float *bias;
  const uint8_t *live, *decoded;
  const uint4 *xv;  // x as 16-byte vectors (rows copied into xp by the worklist tail)
  int32_t cs;      // CTAs per cluster (H slices)
  int32_t tn;      // positions per cluster tile (multiple of 16, <= 256, multiple of cs)
  int32_t tcols;   // TMEM columns allocated
  int32_t stages;  // operand ring depth
  int32_t region0; // bytes of the ring / partial-sum region
};

// Shared-memory layout of the gate (from the 1024-aligned base): region0 (the
// operand ring, reused for the fp32 partials [TN][E_pad] once the MMAs are
// done), the reduced rows [TN / CS][E_pad], the support mask [1024], barriers.
__host__ __device__ inline int gate_e_pad(int E) { return ((E + 127) / 128) * 128; }
__host__ __device__ inline int gate_stage_bytes(int E, int TN) { return (gate_e_pad(E) / 128) * kTileBytes + TN * 64 * 2; }

// One position of the gate's epilogue: records its classification and, if it
// is fresh, takes its top-k (one warp; row = its reduced logits).
template <int EPL>
__device__ __forceinline__ void gate_position(const Dims &d, const Work &ws, int t, int code, int32_t stamp,
                                              const float *row, int E_pad, const uint8_t *support, bool force,
                                              uint32_t *words, uint2 *scratch, const float *bias, uint8_t *fr_out,
                                              int16_t *sel_out) {
  const bool fresh = force || (code & 15) != C_REUSE;
  if (lane_id() == 0) {
    record_position(d, ws, t, code, fresh ? d.iter : stamp);
    *fr_out = fresh ? 1 : 0;
  }
  if (!fresh) return;
  float v[EPL];
#pragma unroll
  for (int c = 0; c < EPL; ++c) {
    const int e = lane_id() * EPL + c;
    v[c] = e < E_pad ? row[e] : -INFINITY;
  }
  select_position<EPL>(d, ws, t, v, support, force, words, scratch, bias, sel_out);
}

constexpr int kGateThreads = 384;

// 12 warps: 0 issues the TMA loads, 1 the MMAs, 4-7 read TMEM; all of them
// reduce, and each takes the top-k of one of the CTA's positions (up to 12).

// At most 104 registers a thread: the CTA's 384 threads take 40 K of the SM's
// 64 K registers.
template <int EPL>
__global__ void __maxnreg__(104) k_tc_gate(const __grid_constant__ GateParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base (the 128-byte swizzle pattern repeats every 1024 bytes)
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const Dims &d = p.d;
  const Work &ws = p.ws;
  const int MB = (d.E + 127) / 128, E_pad = MB * 128;
  const int CS = p.cs, TN = p.tn, TPC = TN / CS, STAGES = p.stages;
  const int nkb = d.H / CS / BK;
  const int W_BYTES = MB * kTileBytes, STAGE = W_BYTES + TN * BK * 2;
  float *partial = reinterpret_cast<float *>(smem);                   // [TN][E_pad], after the main loop
  float *rows = reinterpret_cast<float *>(smem + p.region0);          // [TPC][E_pad] reduced rows
  float *s_bias = rows + TPC * E_pad;                                   // [E_pad]
  uint8_t *s_support = reinterpret_cast<uint8_t *>(s_bias + E_pad);       // [1024]
  uint64_t *bars = reinterpret_cast<uint64_t *>(s_support + 1024);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  const uint32_t done_bar = bar0 + 8u * (2 * STAGES);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 2 * STAGES + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int *s_anom = reinterpret_cast<int *>(tmem_slot + 2);
  int *s_code = reinterpret_cast<int *>(tmem_slot + 4);  // [TPC] classification codes of the own positions
  int *s_stamp = s_code + 64;                             // [TPC] their previous stamps
  uint2 *s_scr = reinterpret_cast<uint2 *>(s_stamp + 64);  // [warps][32] top-k scratch
  // for the worklist tail (gate_tail.cuh)
  uint64_t *x_barp = reinterpret_cast<uint64_t *>(s_scr + 32 * (kGateThreads / 32));  // staged x rows
  int *s_ncand = reinterpret_cast<int *>(x_barp + 1);      // [0] candidates, [1] barrier count at the start
  uint8_t *s_fr = reinterpret_cast<uint8_t *>(s_ncand + 2);  // [64] own position fresh
  int16_t *s_sel = reinterpret_cast<int16_t *>(s_fr + 64);   // [64][16] its selected experts
  int16_t *s_cand = s_sel + 64 * 16;                         // [1024] candidate experts
  int16_t *s_cidx = s_cand + 1024;                           // [1024] candidate index of an expert
  const uint32_t x_bar = smem_u32(x_barp);

  const KernelMark mark_(d, ws, K_GATE);
  pdl_wait();
  pdl_trigger();  // the worklist kernel may start its launch; it waits for this grid to finish
  const int tid = threadIdx.x, wid = warp_id(), lane = lane_id();
  const int rank = static_cast<int>(cluster_ctarank());
  const int tile = blockIdx.x / CS;
  const uint64_t tmo = static_cast<uint64_t>(d.timeout_ns);
  // TMEM columns: MB accumulators of TN columns (the readers load 32-column runs)
  const uint32_t tcols = static_cast<uint32_t>(p.tcols);
  int64_t *trace = (d.trace && blockIdx.x < kTraceCtas)
                       ? ws.trace + (static_cast<size_t>(kTraceRowGate) * kTraceCtas + blockIdx.x) * kTraceFields
                       : nullptr;
  if (trace && tid == 0) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    trace[0] = static_cast<int64_t>(globaltimer_ns());
    trace[7] = smid;
  }
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    mbar_init(done_bar, 1);
    mbar_init(x_bar, 1);
    *abort_flag = 0;
    *s_anom = 0;
    mbar_fence_init();
  }
  if (wid == 1) {
    tmem_alloc(smem_u32(tmem_slot), tcols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (trace && tid == 0) trace[1] = static_cast<int64_t>(globaltimer_ns());
  const int k0 = rank * (d.H / CS);

  if (wid == 0) {
    if (lane == 0) {
      // ---------------- TMA producer: MB W_r tiles and one x tile per K block
      tma_prefetch_desc(&p.wr);
      tma_prefetch_desc(&p.x);
      const uint64_t pol_w = policy_evict_last();  // every cluster reads the same W_r slice
      const uint64_t pol_x = policy_evict_last();  // the expert kernel reads x again
      uint32_t armed = 0, armed_par = 0;
      bool ok = true;
      for (int kb = 0; kb < nkb; ++kb) {
        const int stage = kb % STAGES;
        const uint32_t phase = static_cast<uint32_t>(kb / STAGES) & 1u;
        if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, ws.err, tmo)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(full_bar(stage), STAGE);
        const uint32_t st = sbase + stage * STAGE;
        const int kc = k0 + kb * BK;
        for (int mb = 0; mb < MB; ++mb) tma_load_2d(st + mb * kTileBytes, &p.wr, kc, mb * BM, full_bar(stage), pol_w);
        tma_load_2d(st + W_BYTES, &p.x, kc, tile * TN, full_bar(stage), pol_x);
        armed |= 1u << stage;
        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
      }
      if (!ok) {  // let copies already issued land before the region is reused
        for (int s = 0; s < STAGES; ++s)
          if (armed & (1u << s)) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(full_bar(s), (armed_par >> s) & 1u) && globaltimer_ns() - t0 < 50000000ull) {
            }
          }
      }
    }
    __syncwarp();
  } else if (wid == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer: accumulator mb = experts [128 mb, 128 mb + 128) x TN positions
      const uint32_t idesc = idesc_bf16_f32(BM, TN);
      for (int kb = 0; kb < nkb; ++kb) {
        const int stage = kb % STAGES;
        const uint32_t phase = static_cast<uint32_t>(kb / STAGES) & 1u;
        if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, ws.err, tmo)) break;
        tc_fence_after();
        if (trace && kb == 0) trace[2] = static_cast<int64_t>(globaltimer_ns());
        const uint32_t st = sbase + stage * STAGE;
        const uint64_t bd = sw128_kmajor_desc(st + W_BYTES);
        for (int mb = 0; mb < MB; ++mb) {
          const uint64_t ad = sw128_kmajor_desc(st + mb * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma_bf16(tmem_base + static_cast<uint32_t>(mb * TN), ad + 2u * kk, bd + 2u * kk, idesc,
                        (kb | kk) != 0);
        }
        tc_commit(empty_bar(stage));
      }
      tc_commit(done_bar);  // also on an abort, so the readers below never wait forever
      if (trace) trace[3] = static_cast<int64_t>(globaltimer_ns());
    }
    __syncwarp();
  } else {
    // ---------------- warps 2-11, while the operands stream: the support mask,
    // and the decoded -> live scan (any anomaly anywhere makes every position
    // fresh with every expert eligible)
    for (int e = tid - 64; e < E_pad; e += kGateThreads - 64) {
      s_support[e] = e < d.E ? ws.support_mask[e] : 0;
      s_bias[e] = e < d.E ? __ldg(p.bias + e) : 0.f;
    }
    if (!d.plan_mode) {
      const int rd = d.state_rd & 1;
      // classification of this CTA's own positions (the fallback decision comes later)
      const int j = tid - 64, t = tile * TN + rank * TPC + j;
      if (j < TPC && t < d.n_pos) {
        const int st = ws.stamp[static_cast<size_t>(rd) * d.Nmax + t];
        s_stamp[j] = st;
        s_code[j] = classify_code(d, p.live[t] != 0, p.decoded[t] != 0,
                                  ws.prev_dec[static_cast<size_t>(rd) * d.Nmax + t] != 0, st);
      }
      if (any_anomaly(d, p.live, p.decoded, ws.prev_dec + static_cast<size_t>(rd) * d.Nmax, tid - 64,
                      kGateThreads - 64))
        atomicOr(s_anom, 1);
      if (tid == 64 && shortfall_flag(d, ws)) atomicOr(s_anom, 2);
      if (d.wl_in_gate) {  // the plan's candidate experts, for the worklist tail
        const int nc = ws.ctrl->support_len;
        if (tid == 64) {
          s_ncand[0] = nc;
          s_ncand[1] = *reinterpret_cast<volatile const int32_t *>(ws.gate_arrive + 1);  // barrier count at the start
        }
        for (int i = tid - 64; i < d.E; i += kGateThreads - 64) {
          const int e = ws.support_ids[i];
          const bool valid = e >= 0 && e < d.E;
          s_cand[i] = static_cast<int16_t>(valid ? e : 0);
          if (i < nc && valid) s_cidx[e] = static_cast<int16_t>(i);
        }
      }
    }
  }
  if (wid >= 4 && wid < 8) {
    // ---------------- warps 4-7: TMEM -> fp32 partials [position][expert] in shared memory
    if (mbar_wait_bounded(done_bar, 0, abort_flag, ws.err, tmo)) {
      tc_fence_after();
      const int q = wid & 3;  // TMEM lanes 32q.. = experts 32q.. of each block
      for (int mb = 0; mb < MB; ++mb) {
        for (int c0 = 0; c0 < TN; c0 += 32) {
          float v[32];
          tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(mb * TN + c0), v);
          tmem_ld_wait();
          const int nc = min(32, TN - c0);
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (c < nc) partial[(c0 + c) * E_pad + mb * BM + q * 32 + lane] = v[c];
        }
      }
    }
  }
  int64_t *trace2 = trace ? ws.trace + (static_cast<size_t>(kTraceRowGateEpi) * kTraceCtas + blockIdx.x) * kTraceFields
                          : nullptr;
  tc_fence_before();
  __syncthreads();
  if (trace2 && tid == 0) trace2[0] = static_cast<int64_t>(globaltimer_ns());
  if (!d.plan_mode && blockIdx.x == 0) {
    reset_iteration_state(d, ws, *s_anom);
  }
  if (wid == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tcols);
  }
  // every CTA of the cluster has its partials in shared memory
  cluster_arrive();
  cluster_wait();
  if (trace2 && tid == 0) trace2[1] = static_cast<int64_t>(globaltimer_ns());
  // ---------------- reduce positions [rank * TPC, rank * TPC + TPC) of the tile over the cluster
  const int t_own = tile * TN + rank * TPC;
  const int e4n = E_pad / 4;
  const uint32_t pbase = smem_u32(partial);
  const bool vec_out = (d.E & 3) == 0;
  // units of 4 experts x 1 position, kGateBatch per thread at a time: every
  // rank's partials of a batch are requested before any is summed (one round
  // trip over the cluster per batch). One unit a time: the loop runs once per
  // iteration, cold, so short code beats the second unit's overlap.
  constexpr int kGateBatch = 1;
  const int n_units = TPC * e4n;
  for (int u0 = tid; u0 < n_units; u0 += kGateBatch * blockDim.x) {
    float4 v[kGateBatch][8];
#pragma unroll
    for (int b = 0; b < kGateBatch; ++b) {
      const int u = u0 + b * blockDim.x;
      if (u < n_units) {
        const int j = u / e4n, e = (u % e4n) * 4;
        const uint32_t off = static_cast<uint32_t>(((rank * TPC + j) * E_pad + e) * 4);
#pragma unroll
        for (int s = 0; s < 8; ++s)
          if (s < CS) v[b][s] = ld_dsmem_f4(mapa_shared(pbase + off, static_cast<uint32_t>(s)));
      }
    }
#pragma unroll
    for (int b = 0; b < kGateBatch; ++b) {
      const int u = u0 + b * blockDim.x;
      if (u >= n_units) continue;
      const int j = u / e4n, e = (u % e4n) * 4;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int s = 0; s < 8; ++s)
        if (s < CS) {  // rank order
          acc.x += v[b][s].x;
          acc.y += v[b][s].y;
          acc.z += v[b][s].z;
          acc.w += v[b][s].w;
        }
      float g[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
      for (int c = 0; c < 4; ++c) g[c] = e + c < d.E ? (d.router ? g[c] : g[c] + s_bias[e + c]) : -INFINITY;
      *reinterpret_cast<float4 *>(rows + j * E_pad + e) = make_float4(g[0], g[1], g[2], g[3]);
      const int t = t_own + j;
      if (t < d.n_pos && e < d.E) {
        float *dst = ws.logits + static_cast<size_t>(t) * d.E + e;
        if (vec_out) {
          *reinterpret_cast<float4 *>(dst) = make_float4(g[0], g[1], g[2], g[3]);
        } else {
          for (int c = 0; c < 4 && e + c < d.E; ++c) dst[c] = g[c];
        }
      }
    }
  }
  cluster_arrive_relaxed();  // this CTA's reads of the other CTAs' partials are complete
  __syncthreads();   // rows[] complete
  if (trace2 && tid == 0) trace2[2] = static_cast<int64_t>(globaltimer_ns());
  if (!d.plan_mode) {
    // ---------------- classification and top-k of the positions this CTA owns
    const bool force = d.host_fallback != 0 || *s_anom != 0;
    uint32_t *words = words_written(d, ws);
    for (int j = wid; j < TPC; j += kGateThreads / 32) {
      const int t = t_own + j;
      if (t >= d.n_pos) continue;
      // per-request supports: the position's request's mask (read from global memory)
      const uint8_t *mask = d.req_size > 0 ? ws.support_mask + static_cast<size_t>(t / d.req_size) * d.E : s_support;
      gate_position<EPL>(d, ws, t, s_code[j], s_stamp[j], rows + j * E_pad, E_pad, mask, force, words,
                         s_scr + 32 * wid, s_bias, s_fr + j, s_sel + j * 16);
    }
  }
  if (trace && tid == 0) {
    trace[4] = static_cast<int64_t>(globaltimer_ns());
    trace[5] = tile;
    trace[6] = rank;
  }
  cluster_wait();  // no CTA leaves while another may still read its partials
  if (trace2 && tid == 0) trace2[3] = static_cast<int64_t>(globaltimer_ns());
  if (!d.plan_mode && d.wl_in_gate) {
    const GateTail gt{s_sel, s_fr, s_code, s_cand, s_cidx, s_ncand[0], x_bar, s_ncand[1]};
    int64_t *trace_wl = (d.trace && blockIdx.x == 0) ? ws.trace + 3ull * kTraceCtas * kTraceFields : nullptr;
    gate_tail(d, ws, reinterpret_cast<const uint8_t *>(p.xv), smem, gt, tile * TN + rank * TPC, TPC,
              d.host_fallback != 0 || *s_anom != 0, *s_anom, trace_wl);
  }
}

// ---------------------------------------------------------------- fused expert kernel
// Up and down projections of every group in one persistent launch (one CTA
// per SM). The shared experts' up tiles are drawn from their own counter from
// the launch on (they need only the layer input); once the worklist is
// complete, one counter hands out [routed up tiles, shared down tiles, routed
// down tiles] one at a time, so a CTA that drew short tiles draws more. Both
// kinds are two 128-row MMAs sharing one token tile of <= 128 tokens: an up
// tile (group g, 128 rows of I) multiplies the gate and up rows and writes
// silu(gate) * up as bf16, then counts itself done for (g, its row block of
// I); a down tile (g, 256 rows of H) issues its first weight copies, then
// loads its activations one row block of I at a time as the group's up tiles
// of that row block complete, so the down work of lightly loaded experts runs
// while heavy up tiles are still streaming, with no launch in between. Every
// tile uses one 256-column TMEM accumulator buffer, double-buffered; a 48 KB
// stage holds 32 KB of packed weights (one contiguous run) and a 16 KB token
// tile.
constexpr int kExpStages = 4;
constexpr int kExpStage = 48 * 1024;
constexpr int kExpStg = 32 * 80;  // epilogue staging per warp: 32 tokens x 32 bf16 rows, padded
constexpr int kExpSched = 4;  // decoded-tile ring between the producer and the MMA / epilogue warps
constexpr int kExpBars = 2 * kExpStages + 2 * 2 + 1 + 2 * kExpSched;
constexpr int kExpGroups = 1028;  // capacity of the group list and offset copies (E + n_sh + 1 <= 1025)
// shared-memory carve-up, from the 1024-aligned base
constexpr int kExpOffBars = kExpStages * kExpStage + 4 * kExpStg;
constexpr int kExpOffSlot = kExpOffBars + kExpBars * 8;           // TMEM address, abort flag
constexpr int kExpOffRing = (kExpOffSlot + 16 + 15) & ~15;        // int4 [kExpSched]
constexpr int kExpOffPref = kExpOffRing + 16 * kExpSched;         // int32 [kExpGroups] group list
constexpr int kExpOffOffs = kExpOffPref + 4 * kExpGroups;         // int32 [kExpGroups]
constexpr int kExpSmem = 1024 + kExpOffOffs + 4 * kExpGroups;
static_assert(kExpSmem <= 227 * 1024, "shared memory");
static_assert(kTnUp == kTnDn, "up and down tiles share the token tiling");

// Decoded tile as handed through the ring: x = group | kDownBit for a down
// tile (-1 ends the stream), y = row block, z = first token row, w = valid rows.
constexpr int kDownBit = 1 << 30;

// Routed tile q of the list [all up tiles, then all down tiles] -> decoded
// tile and the up-tile count of its group. list = the worklist kernel's group
// list: entry p holds the token tiles of the groups before p (<< kGrpIdBits)
// and the expert of p. offs = expert row offsets. Within a group the tiles run
// row block by row block, token tiles fastest, so tiles drawn close together
// share a weight row block in L2. Up tiles have I / 128 row blocks, down tiles
// H / 256. Returns false when the list and the offsets disagree.
__device__ __forceinline__ bool locate(const Dims &d, const int32_t *list, const int32_t *offs, int q, int n_up,
                                      int4 *td, int *need) {
  auto pref = [&](int p) { return list[p] >> kGrpIdBits; };
  const bool up = q < n_up;
  if (!up) q -= n_up;
  const int mult = up ? d.I / BM : d.H / kBmDn;
  const int key = q / mult;
  // largest p in [0, E) with pref(p) <= key
  int l = 0, h = d.E;
  while (h - l > 1) {
    const int mid = (l + h) >> 1;
    if (pref(mid) <= key) l = mid;
    else h = mid;
  }
  const int nt = pref(l + 1) - pref(l);
  const int qq = q - mult * pref(l);
  if (nt <= 0 || qq < 0 || qq >= mult * nt) return false;
  const int m = qq / nt, tt = qq - m * nt;
  const int g = list[l] & ((1 << kGrpIdBits) - 1);
  if (g >= d.E) return false;
  const int rows = offs[g + 1] - offs[g];
  const int r0 = offs[g] + tt * kTnUp;
  const int n_valid = min(kTnUp, rows - tt * kTnUp);
  if (n_valid <= 0) return false;
  *td = make_int4(g | (up ? 0 : kDownBit), m, r0, n_valid);
  *need = nt;  // down tiles: every token tile of the group, per row block of I
  return true;
}

// Shared-expert tile q: the up tiles of every (shared expert s, token tile
// tt, row block m), then the down tiles, token tiles before row blocks so that
// the down tiles of the first token tiles become ready first. A down tile
// (s, tt) needs the I_s / 128 up tiles of (s, tt).
__device__ __forceinline__ int4 shared_tile(const Dims &d, int q, int *need, int *tt_out) {
  const int nt = (d.n_pos + kTnUp - 1) / kTnUp, mu = d.I_s / BM, md = d.H / kBmDn;
  const int n_up = d.n_sh * nt * mu;
  const bool up = q < n_up;
  if (!up) q -= n_up;
  const int mm = up ? mu : md;
  const int s = q / (nt * mm), r = q - s * nt * mm, tt = r / mm, m = r - tt * mm;
  *need = mu;
  *tt_out = tt;
  return make_int4((d.E + s) | (up ? 0 : kDownBit), m, tt * kTnUp, min(kTnUp, d.n_pos - tt * kTnUp));
}

struct XTile {
  bool up;                // up tile (else down)
  int g;                  // group
  const uint8_t *a_src;   // first packed weight tile of the row block
  int a_bytes;            // weight bytes per K block (32 KB: two 128-row tiles)
  int nk;                 // K blocks
  const CUtensorMap *mb;  // token-operand map (box chosen for the tile)
  bool routed_up;         // token rows come from xp, filled by this kernel's copy phase
  int b_row, b_bytes;
  int n_valid;
  int out_row0, out_rows, ld, col0;
  void *out;
};

__device__ __forceinline__ XTile xdecode(const TcParams &p, int4 td) {
  const Dims &d = p.d;
  const Work &ws = p.ws;
  XTile t;
  t.up = (td.x & kDownBit) == 0;
  const int g = td.x & (kDownBit - 1), m = td.y, r0 = td.z;
  t.g = g;
  t.n_valid = td.w;
  const bool shared = g >= d.E;
  const int s = g - d.E;
  const int bi = t.n_valid <= 32 ? 0 : t.n_valid <= 64 ? 1 : t.n_valid <= 128 ? 2 : 3;
  t.col0 = m * BM;
  if (t.up) {
    const int nkb = d.H / BK;
    const size_t rb = shared ? static_cast<size_t>(s) * (d.I_s / BM) + m : static_cast<size_t>(g) * (d.I / BM) + m;
    t.a_src = (shared ? ws.pk_sgu : ws.pk_gu) + rb * nkb * (2 * kTileBytes);
    t.a_bytes = 2 * kTileBytes;
    t.nk = nkb;
    t.mb = shared ? &p.bs : &p.b[bi];
    t.routed_up = !shared;
    t.b_bytes = (shared ? kTnUp : (32 << bi)) * BK * 2;
    t.b_row = r0;
    t.out_row0 = shared ? s * d.Nmax + r0 : r0;
    t.ld = shared ? d.I_s : d.I;
    t.out = shared ? ws.a_sh : ws.a_int;
    t.out_rows = shared ? d.n_sh * d.Nmax : d.Nmax * d.k;
  } else {
    // 256 rows of H: two 128-row blocks sharing the token tile; the packed pair
    // of a K block is one contiguous 32 KB run
    const int nkb = (shared ? d.I_s : d.I) / BK;
    const size_t pb = shared ? static_cast<size_t>(s) * (d.H / kBmDn) + m : static_cast<size_t>(g) * (d.H / kBmDn) + m;
    t.a_src = (shared ? ws.pk_sd : ws.pk_d) + pb * nkb * (2 * kTileBytes);
    t.a_bytes = 2 * kTileBytes;
    t.nk = nkb;
    t.col0 = m * kBmDn;
    t.mb = shared ? &p.bs2 : &p.b2[bi];
    t.routed_up = false;
    t.b_bytes = (shared ? kTnDn : (32 << bi)) * BK * 2;
    t.b_row = shared ? s * d.Nmax + r0 : r0;
    t.out_row0 = t.b_row;
    t.ld = d.H;
    t.out = shared ? ws.o_sh : ws.o_int;
    t.out_rows = shared ? d.n_sh * d.Nmax : d.Nmax * d.k;
  }
  return t;
}

__global__ void __launch_bounds__(192, 1) k_tc_experts(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base (the 128-byte swizzle pattern repeats every 1024
  // bytes), offset from the __shared__ array itself so that every pointer
  // derived from it stays in the shared state space (shared loads and stores,
  // never ordered behind the epilogue's global stores)
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  uint8_t *stage_out = smem + kExpStages * kExpStage;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kExpOffBars);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kExpStages + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * kExpStages + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * kExpStages + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (2 * kExpStages + 4);
  auto sfull_bar = [&](int i) { return bar0 + 8u * (2 * kExpStages + 5 + i); };
  auto sempty_bar = [&](int i) { return bar0 + 8u * (2 * kExpStages + 5 + kExpSched + i); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kExpOffSlot);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  int4 *s_td = reinterpret_cast<int4 *>(smem + kExpOffRing);
  int32_t *s_list = reinterpret_cast<int32_t *>(smem + kExpOffPref);
  int32_t *s_offs = reinterpret_cast<int32_t *>(smem + kExpOffOffs);

  const Dims &d = p.d;
  const Work &ws = p.ws;
  const KernelMark mark_(d, ws, K_UP);
  const int wid = warp_id(), lane = lane_id();
  const uint64_t tmo = static_cast<uint64_t>(d.timeout_ns);
  int64_t *trace = (d.trace && blockIdx.x < kTraceCtas)
                       ? ws.trace + (static_cast<size_t>(kTraceRowExperts) * kTraceCtas + blockIdx.x) * kTraceFields
                       : nullptr;
  if (trace && threadIdx.x == 0) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    trace[0] = static_cast<int64_t>(globaltimer_ns());
    trace[7] = smid;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kExpStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 128);
    }
    mbar_init(done_bar, 1);
    for (int i = 0; i < kExpSched; ++i) {
      mbar_init(sfull_bar(i), 1);
      mbar_init(sempty_bar(i), 1 + 4);  // the MMA thread and one lane per epilogue warp
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (wid == 0) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  pdl_trigger();  // the combine kernel may start its launch; it waits for this grid to finish
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (trace && threadIdx.x == 0) trace[1] = static_cast<int64_t>(globaltimer_ns());
  // This launch overlaps the kernel before it (programmatic dependent
  // launch): the gate, which builds the iteration's worklist in its tail, or
  // the worklist kernel. The shared experts' up tiles need only the layer
  // input, so the CTAs start on them at once (on the SMs the gate leaves free,
  // while it runs); the producer waits for the kernel before to complete only
  // when they are all taken, then reads the worklist.
  int32_t *shc = ws.sh_ctr;  // [0] shared tile counter, then done counts (zeroed by the previous combine)
  const int nt_max = (d.Nmax + kTnUp - 1) / kTnUp;
  const int nt_sh = (d.n_pos + kTnUp - 1) / kTnUp;
  const int n_sh_up = d.tn > 0 ? d.n_sh * nt_sh * (d.I_s / BM) : 0;
  const int n_sh_dn = d.tn > 0 ? d.n_sh * nt_sh * (d.H / kBmDn) : 0;

  if (wid == 0) {
    // ---------------- producer warp (lane 0 issues): per K block, a 32 KB run of
    // packed weights (bulk copy) and the tile's token rows (tiled TMA load: x
    // for shared-expert up tiles, xp for routed up tiles, activations for down
    // tiles)
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_b = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0, armed = 0, armed_par = 0;
    bool ok = true;
    uint64_t waited = 0;
    int64_t waited_by[3] = {0, 0, 0};  // ns waiting for: (unused), routed up tiles, shared up tiles
    // Issues the operand copies of one tile. Token rows that this launch
    // produces -- the activations of down tiles -- are awaited (counter >=
    // target) after the weight copies of the first stages have gone out. flag:
    // nullptr (no dependency) or the first readiness counter; fstep > 0: K
    // block kb waits for flag[kb / fstep] (the group's up tiles of one row
    // block), 0: every K block waits for flag[0].
    auto issue = [&](const int4 &td, const int32_t *flag, int target, int wait_kind, int fstep) -> bool {
      const XTile t = xdecode(p, td);
      const uint32_t tx = t.a_bytes + t.b_bytes;
      const bool dep = flag != nullptr;
      const int pre = dep ? min(t.nk, kExpStages) : 0;
      int pre_stage[kExpStages] = {0, 0, 0, 0};
      for (int kb = 0; kb < pre; ++kb) {
        if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, ws.err, tmo)) return false;
        mbar_arrive_expect_tx(full_bar(stage), tx);
        bulk_load(sbase + stage * kExpStage, t.a_src + static_cast<size_t>(kb) * t.a_bytes, t.a_bytes,
                  full_bar(stage), pol_w);
        pre_stage[kb] = stage;
        armed |= 1u << stage;
        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
        if (++stage == kExpStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      int ready = -1;  // the counter last seen at its target
      auto tokens = [&](int kb, int st) -> bool {
        if (dep) {
          const int fi = fstep > 0 ? kb / fstep : 0;
          if (fi != ready) {
            const int32_t *f = flag + fi;
            const uint64_t t0 = globaltimer_ns();
            for (;;) {
              int done;
              asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(done) : "l"(f) : "memory");
              if (done >= target) break;
              if (*abort_flag) return false;
              if (globaltimer_ns() - t0 > tmo) {
                set_error(ws.err, EPOCH_DEVERR_TIMEOUT);
                *abort_flag = 1;
                return false;
              }
              __nanosleep(32);
            }
            const int64_t w_ns = static_cast<int64_t>(globaltimer_ns() - t0);
            waited += w_ns;
            waited_by[wait_kind] += w_ns;
            asm volatile("fence.proxy.async.global;" ::: "memory");  // generic writes -> TMA reads
            ready = fi;
          }
        }
        tma_load_2d(sbase + st * kExpStage + 2 * kTileBytes, t.mb, kb * BK, t.b_row, full_bar(st), pol_b);
        return true;
      };
      for (int kb = 0; kb < pre; ++kb)
        if (!tokens(kb, pre_stage[kb])) return false;
      for (int kb = pre; kb < t.nk; ++kb) {
        if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, ws.err, tmo)) return false;
        mbar_arrive_expect_tx(full_bar(stage), tx);
        const uint32_t st = sbase + stage * kExpStage;
        bulk_load(st, t.a_src + static_cast<size_t>(kb) * t.a_bytes, t.a_bytes, full_bar(stage), pol_w);
        armed |= 1u << stage;
        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
        if (!tokens(kb, stage)) return false;
        if (++stage == kExpStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      return true;
    };
    int j = 0;  // tiles handed through the ring
    auto post = [&](const int4 &td) -> bool {
      const int slot = j % kExpSched;
      if (!mbar_wait_bounded(sempty_bar(slot), ((j / kExpSched) & 1) ^ 1u, abort_flag, ws.err, tmo)) return false;
      s_td[slot] = td;
      mbar_arrive(sfull_bar(slot));
      ++j;
      return true;
    };
    if (lane == 0) {
      if (trace) trace[2] = static_cast<int64_t>(globaltimer_ns());
      tma_prefetch_desc(&p.bs);
      tma_prefetch_desc(&p.bs2);
      tma_prefetch_desc(&p.b[0]);
      tma_prefetch_desc(&p.b2[0]);
      // 1. the shared experts' up tiles, from launch (their inputs are the layer input)
      while (ok) {
        const int q = atomicAdd(shc, 1);
        if (q >= n_sh_up) break;
        int need = 0, tt;
        const int4 td = shared_tile(d, q, &need, &tt);
        ok = post(td) && issue(td, nullptr, need, 2, 0);
      }
    }
    __syncwarp();
    // 2. once the worklist of this call is complete (offsets, group list, xp
    // rows), from one counter: the routed up tiles, the shared experts' down
    // tiles, the routed down tiles (down tiles wait for their group's up tiles)
    pdl_wait();
    for (int i = lane; i <= d.E; i += 32) {
      s_list[i] = ws.grp_list[i];
      s_offs[i] = ws.offsets[i];
    }
    __syncwarp();
    if (lane == 0) {
      const int n_tiles = s_list[d.E] >> kGrpIdBits;
      const int n_up = d.tn > 0 ? (d.I / BM) * n_tiles : 0;
      const int total = ok ? n_up + n_sh_dn + (d.tn > 0 ? (d.H / kBmDn) * n_tiles : 0) : 0;
      while (ok) {
        const int q = atomicAdd(ws.tile_ctr, 1);
        if (q >= total) break;
        int4 td;
        int need = 0, kind = 1, fstep = BM / BK;
        const int32_t *flag = nullptr;
        if (q >= n_up && q < n_up + n_sh_dn) {
          int tt;
          td = shared_tile(d, n_sh_up + q - n_up, &need, &tt);
          flag = shc + 1 + ((td.x & (kDownBit - 1)) - d.E) * nt_max + tt;
          kind = 2;
          fstep = 0;
        } else {
          const int qr = q < n_up ? q : q - n_sh_dn;
          if (!locate(d, s_list, s_offs, qr, n_up, &td, &need)) {
            set_error(ws.err, EPOCH_DEVERR_BOUNDS);
            *abort_flag = 1;
            ok = false;
            break;
          }
          // routed up tiles: the rows are in xp; down tiles: their group's up
          // tiles, one row block of I (two K blocks) at a time
          if (q >= n_up) flag = ws.done_up + static_cast<size_t>(td.x & (kDownBit - 1)) * (d.I / BM);
        }
        ok = post(td) && issue(td, flag, need, kind, fstep);
      }
      if (ok) ok = post(make_int4(-1, 0, 0, 0));  // end of the stream
      if (!ok) {
        for (int s = 0; s < kExpStages; ++s)
          if (armed & (1u << s)) mbar_drain(full_bar(s), (armed_par >> s) & 1u, 50000000ull);
      }
      if (trace) {
        int64_t *trace7 = ws.trace + (6ull * kTraceCtas + blockIdx.x) * kTraceFields;
        trace[6] = static_cast<int64_t>(waited);
        trace7[0] = waited_by[0];
        trace7[1] = waited_by[1];
        trace7[2] = waited_by[2];
      }
    }
    __syncwarp();
  }
  if (wid == 1) {


    if (lane == 0) {
      // ---------------- MMA issuer
      int stage = 0, buf = 0;
      uint32_t phase = 0, bphase = 0;
      bool ok = true;
      int64_t n_tiles = 0;
      for (int j = 0; ok; ++j) {
        const int slot = j % kExpSched;
        if (!mbar_wait_bounded(sfull_bar(slot), (j / kExpSched) & 1, abort_flag, ws.err, tmo)) break;
        const int4 td = s_td[slot];
        mbar_arrive(sempty_bar(slot));
        if (td.x < 0) break;
        const XTile t = xdecode(p, td);
        const int n_mma = ((t.n_valid + 15) / 16) * 16;
        const uint32_t idesc = idesc_bf16_f32(BM, n_mma);
        ++n_tiles;
        if (!mbar_wait_bounded(tempty_bar(buf), bphase ^ 1u, abort_flag, ws.err, tmo)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(buf * 256);
        const uint32_t b_off = 2 * kTileBytes;
        for (int kb = 0; kb < t.nk; ++kb) {
          if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, ws.err, tmo)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = sbase + stage * kExpStage;
          const uint64_t ad0 = sw128_kmajor_desc(st);
          const uint64_t ad1 = sw128_kmajor_desc(st + kTileBytes);
          const uint64_t bd = sw128_kmajor_desc(st + b_off);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint32_t acc = (kb | kk) != 0;
            tc_mma_bf16(d0, ad0 + 2u * kk, bd + 2u * kk, idesc, acc);
            tc_mma_bf16(d0 + 128, ad1 + 2u * kk, bd + 2u * kk, idesc, acc);
          }
          tc_commit(empty_bar(stage));
          if (++stage == kExpStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(tfull_bar(buf));
        if (++buf == 2) {
          buf = 0;
          bphase ^= 1u;
        }
      }
      tc_commit(done_bar);
      mbar_drain(done_bar, 0, 50000000ull);
      if (trace) {
        trace[3] = static_cast<int64_t>(globaltimer_ns());
        trace[5] = n_tiles;
      }
    }
    __syncwarp();
  } else if (wid >= 2) {
    // ---------------- epilogue (warps 2..5; warp w reads TMEM lanes 32*(w%4)..)
    const int q = wid & 3;
    uint8_t *stg = stage_out + (wid - 2) * kExpStg;
    int buf = 0;
    uint32_t bphase = 0;
    // epilogue trace (warp 2): ns busy, ns waiting for accumulators, longest tile
    const bool etr = trace != nullptr && wid == 2;
    int64_t e_busy = 0, e_wait = 0, e_max = 0, e_max_x = 0, e_max_n = 0, e_last0 = 0, e_last1 = 0;
    for (int j = 0;; ++j) {
      const int slot = j % kExpSched;
      if (!mbar_wait_bounded(sfull_bar(slot), (j / kExpSched) & 1, abort_flag, ws.err, tmo)) break;
      const int4 td = s_td[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(sempty_bar(slot));
      if (td.x < 0) break;
      const XTile t = xdecode(p, td);
      const int64_t tw0 = etr ? static_cast<int64_t>(globaltimer_ns()) : 0;
      if (!mbar_wait_bounded(tfull_bar(buf), bphase, abort_flag, ws.err, tmo)) break;
      tc_fence_after();
      const int64_t tw1 = etr ? static_cast<int64_t>(globaltimer_ns()) : 0;
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * 256);
      const int esz = 2;  // bf16 outputs (activations and expert outputs)
      const int row_bytes = 80;
      const bool vec_ok = ((t.ld * esz) & 15) == 0;
      const int halves = t.up ? 1 : 2;  // down: the two 128-row blocks are two output column blocks
      for (int hb = 0; hb < halves; ++hb) {
        for (int c0 = 0; c0 < t.n_valid; c0 += 32) {
          const int ncol = min(32, t.n_valid - c0);
          // stage the valid token columns 8 at a time: the loop body is short, so
          // the epilogue fetches few instruction lines when it runs cold (it runs
          // once per tile, while the memory system is saturated by weight reads)
#pragma unroll 1
          for (int cc = 0; cc < ncol; cc += 8) {
            float a[8];
            tmem_ld8(tb + hb * 128 + c0 + cc, a);
            if (t.up) {
              float b[8];
              tmem_ld8(tb + 128 + c0 + cc, b);
              tmem_ld_wait();
#pragma unroll
              for (int c = 0; c < 8; ++c)
                reinterpret_cast<__nv_bfloat16 *>(stg + (cc + c) * row_bytes)[lane] =
                    __float2bfloat16_rn(silu_fast(a[c]) * b[c]);
            } else {
              tmem_ld_wait();
#pragma unroll
              for (int c = 0; c < 8; ++c)
                reinterpret_cast<__nv_bfloat16 *>(stg + (cc + c) * row_bytes)[lane] = __float2bfloat16_rn(a[c]);
            }
          }
          __syncwarp();
          const size_t col_off = static_cast<size_t>(t.col0 + hb * 128 + q * 32);
          if (vec_ok) {
            // a token's 32 outputs of this warp are 32 * esz contiguous bytes: `per`
            // lanes store them together, so one instruction writes whole lines of
            // 32 / per tokens
            const int per = 2 * esz, v = lane % per;
            for (int c = lane / per; c < ncol; c += 32 / per) {
              const int orow = t.out_row0 + c0 + c;
              if (orow < 0 || orow >= t.out_rows) {
                set_error(ws.err, EPOCH_DEVERR_BOUNDS);
                continue;
              }
              *reinterpret_cast<uint4 *>(static_cast<uint8_t *>(t.out) +
                                         (static_cast<size_t>(orow) * t.ld + col_off) * esz + v * 16) =
                  *reinterpret_cast<const uint4 *>(stg + c * row_bytes + v * 16);
            }
          } else if (lane < ncol) {
            const int orow = t.out_row0 + c0 + lane;
            if (orow < 0 || orow >= t.out_rows) {
              set_error(ws.err, EPOCH_DEVERR_BOUNDS);
            } else {
              uint8_t *dst = static_cast<uint8_t *>(t.out) + (static_cast<size_t>(orow) * t.ld + col_off) * esz;
              const uint8_t *src = stg + lane * row_bytes;
              for (int b = 0; b < 32 * esz; b += 2)
                *reinterpret_cast<uint16_t *>(dst + b) = *reinterpret_cast<const uint16_t *>(src + b);
            }
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      mbar_arrive(tempty_bar(buf));
      if (t.up) {
        // all 128 epilogue threads have stored this tile: publish it for the down tiles of g
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (wid == 2 && lane == 0) {
          __threadfence();
          asm volatile("fence.proxy.async.global;" ::: "memory");
          atomicAdd(t.g >= d.E ? shc + 1 + (t.g - d.E) * nt_max + t.b_row / kTnUp
                               : ws.done_up + static_cast<size_t>(t.g) * (d.I / BM) + t.col0 / BM,
                    1);
        }
      }
      if (etr) {
        const int64_t tw2 = static_cast<int64_t>(globaltimer_ns());
        e_wait += tw1 - tw0;
        e_busy += tw2 - tw1;
        if (tw2 - tw1 > e_max) {
          e_max = tw2 - tw1;
          e_max_x = td.x;
          e_max_n = td.w;
        }
        e_last0 = tw1;
        e_last1 = tw2;
      }
      if (++buf == 2) {
        buf = 0;
        bphase ^= 1u;
      }
    }
    if (etr && lane == 0) {
      trace[4] = static_cast<int64_t>(globaltimer_ns());
      int64_t *tr2 = ws.trace + (static_cast<size_t>(kTraceRowEpilogue) * kTraceCtas + blockIdx.x) * kTraceFields;
      tr2[0] = e_busy;
      tr2[1] = e_wait;
      tr2[2] = e_max;
      tr2[3] = e_max_x;
      tr2[4] = e_max_n;
      tr2[5] = e_last0;
      tr2[6] = e_last1;
      tr2[7] = trace[7];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (wid == 0) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

// ---------------------------------------------------------------- weight packing
// One 16-byte chunk per thread: output tile t = rb * (k / 64) + kb holds rows
// [128 rb, 128 rb + 128) x columns [64 kb, 64 kb + 64); row r of the tile sits
// at byte 128 r and its 16-byte chunk c at position c ^ (r % 8) (the 128-byte
// swizzle a TMA load with SWIZZLE_128B would produce in shared memory).
__global__ void k_pack_tiles(const uint4 *__restrict__ src, int64_t rows, int64_t k, uint8_t *__restrict__ dst,
                             int64_t tile_stride, int64_t tile_off, int pair) {
  const int64_t nkb = k / BK;
  const int64_t chunks = rows * k / 8;
  for (int64_t q = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; q < chunks;
       q += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t t = q >> 10;
    const int w = static_cast<int>(q & 1023);
    const int r = w >> 3, pchunk = w & 7;
    const int c8 = pchunk ^ (r & 7);
    const int64_t rb = t / nkb, kb = t % nkb;
    const int64_t row = rb * BM + r;
    const int64_t col = kb * BK + c8 * 8;
    const uint4 v = src[(row * k + col) >> 3];
    // row blocks are grouped by `pair`: the pair's tiles of one K block are adjacent
    const int64_t slot = (rb / pair) * nkb + kb;
    *reinterpret_cast<uint4 *>(dst + slot * tile_stride + (rb % pair) * kTileBytes + tile_off +
                               static_cast<int64_t>(w) * 16) = v;
  }
}

cudaError_t launch_pack_tiles(const void *src, int64_t rows, int64_t k, uint8_t *dst, int64_t tile_stride,
                              int64_t tile_off, int pair, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const int64_t chunks = rows * k / 8;
  int64_t blocks = (chunks + 255) / 256;
  if (blocks > 16 * num_sms()) blocks = 16 * num_sms();
  static bool carve_ = (prefer_max_shared(k_pack_tiles) == cudaSuccess);
  (void)carve_;
  k_pack_tiles<<<static_cast<int>(blocks), 256, 0, s>>>(static_cast<const uint4 *>(src), rows, k, dst, tile_stride,
                                                        tile_off, pair);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

bool tma_encode_init() {
  if (g_encode) return true;
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess || fn == nullptr)
    return false;
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return true;
}

// Row-major [rows][k_elems] bf16 matrix, boxes of 64 (K) x box_rows, 128-byte swizzle.
bool encode_kmajor_bf16(CUtensorMap *map, const void *base, uint64_t k_elems, uint64_t rows, uint32_t box_rows) {
  if (!g_encode || base == nullptr || rows == 0) return false;
  cuuint64_t dims[2] = {k_elems, rows};
  cuuint64_t strides[1] = {k_elems * 2};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
                              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Gate launch geometry. CTAs per cluster (H slices): 8 when H / 8 is a whole
// number of 64-column K blocks, else 4. Positions per cluster tile: as few as
// let every cluster of the launch be resident at once (the device holds a
// limited number of clusters, measured once), at least 32, a multiple of 16,
// at most 256 (one MMA) and within shared memory.
struct GateGeom {
  int tn, cs, tcols, stages, region0, smem;
};
constexpr int kGateSmemCap = 227 * 1024;

static GateGeom gate_geom_for(const Dims &d, int tn) {
  GateGeom g;
  g.cs = (d.H / 8) % BK == 0 ? 8 : 4;
  g.tn = tn;
  const int nkb = d.H / g.cs / BK;
  const int stage = gate_stage_bytes(d.E, tn);
  const int budget = 200 * 1024;
  g.stages = budget / stage < 4 ? budget / stage : 4;
  if (g.stages > nkb) g.stages = nkb;
  if (g.stages < 1) g.stages = 1;
  const int e_pad = gate_e_pad(d.E);
  const int partial = tn * e_pad * 4;
  g.region0 = g.stages * stage > partial ? g.stages * stage : partial;
  const int rows = (tn / g.cs) * e_pad * 4;
  g.smem = 1024 + g.region0 + rows + e_pad * 4 + 1024 + (2 * g.stages + 1) * 8 + 16 + 2 * 64 * 4 +
           (kGateThreads / 32) * 32 * 8 + 8 + 8 + 64 + 64 * 16 * 2 + 2 * 1024 * 2;
  const int cols = (e_pad / BM - 1) * tn + ((tn + 31) / 32) * 32;
  g.tcols = cols <= 32 ? 32 : cols <= 64 ? 64 : cols <= 128 ? 128 : cols <= 256 ? 256 : 512;
  if (cols > 512) g.smem = kGateSmemCap + 1;  // does not fit: rejected by the caller
  return g;
}

static const void *gate_fn(const Dims &d) {
  const int epl = (d.E + 31) / 32;
  if (epl <= 1) return reinterpret_cast<const void *>(k_tc_gate<1>);
  if (epl <= 2) return reinterpret_cast<const void *>(k_tc_gate<2>);
  if (epl <= 4) return reinterpret_cast<const void *>(k_tc_gate<4>);
  if (epl <= 8) return reinterpret_cast<const void *>(k_tc_gate<8>);
  if (epl <= 16) return reinterpret_cast<const void *>(k_tc_gate<16>);
  return reinterpret_cast<const void *>(k_tc_gate<32>);
}

// Shared-memory limits of every instantiation of the gate, set once.
static bool gate_attributes() {
  static const bool ok = [] {
    const void *fns[] = {reinterpret_cast<const void *>(k_tc_gate<1>), reinterpret_cast<const void *>(k_tc_gate<2>),
                         reinterpret_cast<const void *>(k_tc_gate<4>), reinterpret_cast<const void *>(k_tc_gate<8>),
                         reinterpret_cast<const void *>(k_tc_gate<16>), reinterpret_cast<const void *>(k_tc_gate<32>)};
    for (const void *fn : fns)
      if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kGateSmemCap) != cudaSuccess ||
          prefer_max_shared(fn) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
      }
    return true;
  }();
  return ok;
}

// Clusters of the gate's shape the device can hold at once (0: none).
static int gate_max_clusters(const Dims &d, int cs) {
  static int cached[2] = {-1, -1};
  int &c = cached[cs == 8 ? 1 : 0];
  if (c >= 0) return c;
  const void *fn = gate_fn(d);
  if (!gate_attributes()) return 0;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = cs;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs);
  cfg.blockDim = dim3(kGateThreads);
  cfg.dynamicSmemBytes = 160 * 1024;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  c = n;
  return c;
}

static GateGeom gate_geom(const Dims &d) {
  const int cs = (d.H / 8) % BK == 0 ? 8 : 4;
  const int maxc = gate_max_clusters(d, cs);
  int tn = maxc > 0 ? (d.n_pos + maxc - 1) / maxc : 32;
  tn = ((tn + 15) / 16) * 16;
  if (tn < 32) tn = 32;
  if (tn > 256) tn = 256;
  GateGeom g = gate_geom_for(d, tn);
  while (g.smem > kGateSmemCap && tn > 32) {  // large E: narrower tiles, more waves
    tn -= 16;
    g = gate_geom_for(d, tn);
  }
  return g;
}

bool gate_builds_worklist(const Dims &d) {
  const GateGeom g = gate_geom(d);
  const int tiles = (d.n_pos + g.tn - 1) / g.tn, tpc = g.tn / g.cs;
  return g.smem <= kGateSmemCap && g.region0 >= gate_tail_bytes(d, tpc) && tpc <= 64 && d.k <= 16 &&
         d.E <= 1024 && tiles <= gate_max_clusters(d, g.cs);
}

bool gate_tc_supported(const Dims &d) {
  Dims dd = d;
  dd.n_pos = d.Nmax;
  const GateGeom g = gate_geom(dd);
  return gate_max_clusters(d, g.cs) > 0 && g.smem <= kGateSmemCap && gate_geom_for(d, 32).smem <= kGateSmemCap;
}

cudaError_t launch_gate_tc(const Dims &d, const Maps &m, const Work &ws, const void *x, const float *bias,
                           const uint8_t *live, const uint8_t *decoded, cudaStream_t s) {
  const GateGeom g = gate_geom(d);
  if (g.smem > kGateSmemCap || !gate_attributes()) return cudaErrorInvalidConfiguration;
  GateParams p;
  memset(&p, 0, sizeof(p));
  p.wr = m.w_router;
  if (!encode_kmajor_bf16(&p.x, x, d.H, d.n_pos, g.tn)) return cudaErrorInvalidValue;
  p.d = d;
  p.ws = ws;
  p.bias = bias;
  p.live = live;
  p.decoded = decoded;
  p.xv = static_cast<const uint4 *>(x);
  p.cs = g.cs;
  p.tn = g.tn;
  p.tcols = g.tcols;
  p.stages = g.stages;
  p.region0 = g.region0;
  const void *fn = gate_fn(d);
  const int tiles = (d.n_pos + g.tn - 1) / g.tn;
  void *args[] = {&p};
  return launch_kernel(fn, dim3(tiles * g.cs), dim3(kGateThreads), g.smem, s, args, false, g.cs);
}

cudaError_t launch_experts_tc(const Dims &d, const Maps &m, const Work &ws, const CUtensorMap &x_map_up,
                              cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_tc_experts, cudaFuncAttributeMaxDynamicSharedMemorySize, kExpSmem);
    if (e == cudaSuccess) e = prefer_max_shared(k_tc_experts);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  TcParams p;
  memset(&p, 0, sizeof(p));
  p.d = d;
  p.ws = ws;
  for (int i = 0; i < 4; ++i) {
    p.b[i] = m.xp[i];
    p.b2[i] = m.a_int[i];
  }
  p.bs = x_map_up;
  p.bs2 = m.a_sh;
  // Down tiles wait for up tiles of other CTAs, but never for a CTA that has
  // not started: tiles are drawn from one increasing counter and every up tile
  // precedes every down tile, so each awaited up tile is held by a running CTA
  // whose MMA and epilogue finish it independently of its producer's waits.
  // The launch therefore needs no co-residency guarantee.
  void *args[] = {&p};
  return launch_kernel(reinterpret_cast<void *>(k_tc_experts), dim3(num_sms()), dim3(192), kExpSmem, s, args, true);
}

}  // namespace epoch

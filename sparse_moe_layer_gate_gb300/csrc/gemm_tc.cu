// tcgen05 + TMA GEMMs of the Epoch MoE layer (bf16 in, fp32 accumulate).
//
// Two persistent, warp-specialised kernels:
//   k_tc_gate     G = x W_r^T + b for every position, one CTA per (128
//                 experts, 32 tokens) tile over all of H ([W] section "Expert
//                 Atlas": G in R^{N x E}, recomputed every iteration);
//   k_tc_experts  per group g, UP: A_g = silu(X_g W_gate,g^T) * (X_g W_up,g^T)
//                 and DOWN: O_g = A_g W_down,g^T, both stored as bf16, in one
//                 launch with per-group dependencies.
// Groups are the routed experts with at least one worklist row and the shared
// experts over every position; each routed expert runs once over its compact
// rows (the "light-traffic expert kernel" of [W] section "FreshLane
// Dispatch"); experts with no row produce no tile, so their weights are never
// read ("invalid slots load no expert weights", same section).
// [W] = walk-through page "Epoch 完全拆解:把扩散块编译成稀疏 MoE 服务单元".
//
// Swap-AB: weight rows are the MMA M dimension (128) and tokens the N
// dimension (16..128, rounded up to 16 per tile), because an expert may hold
// from one to a thousand rows. Roles per CTA (192 threads): warp 0 issues the
// operand copies into a shared-memory ring (128-byte swizzle, K-major), warp 1
// issues tcgen05.mma into TMEM accumulators (double-buffered, so the epilogue
// of one tile overlaps the next tile's main loop), warps 2-5 read TMEM with
// tcgen05.ld and store. One CTA per SM, persistent over a device-resident tile
// count: no host synchronisation.
#include <cudaTypedefs.h>

#include <cstring>

#include "common.cuh"
#include "layer.h"

namespace epoch {

constexpr int BM = 128;
constexpr int BK = 64;

// Rows of the per-CTA trace: 0 gate, 1 experts, 2 expert epilogue (the routing kernel uses row 3).
constexpr int kTraceRowGate = 0;
constexpr int kTraceRowExperts = 1;
constexpr int kTraceRowEpilogue = 2;  // expert-kernel epilogue summary

struct __align__(128) TcParams {
  CUtensorMap a0;    // gate: W_r [E][H]
  CUtensorMap b[4];  // gate: b[0] = x; experts: Xp (routed up tiles), boxes of 32/64/128/256 rows
  CUtensorMap bs;    // experts: x (shared up tiles), box of kTnUp rows
  CUtensorMap b2[4]; // experts: A (routed down tiles), boxes of 32/64/128/256 rows
  CUtensorMap bs2;   // experts: A (shared down tiles), box of kTnUp rows
  Dims d;
  Work ws;
  int32_t gate_tiles;
  const float *bias;  // gate: router bias [E]
};

// The gate accumulates H in chunks of kGateChunkKb K blocks (256 elements), one
// TMEM accumulator per chunk, and the epilogue adds the chunks in order in fp32:
// a 2048- or 4096-term dot product is not one long tensor-core accumulation.
constexpr int kGateChunkKb = 4;

template <int TN, int STAGES>
struct GateCfg {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = TN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int ACC_COLS = TN;
  static constexpr int NBUF = 2 * ACC_COLS <= 512 ? 2 : 1;
  static constexpr int USED_COLS = NBUF * ACC_COLS;
  static constexpr int TMEM_COLS = USED_COLS <= 32 ? 32 : USED_COLS <= 64 ? 64 : USED_COLS <= 128 ? 128
                                   : USED_COLS <= 256 ? 256 : 512;
  static constexpr int NBARS = 2 * STAGES + 2 * NBUF + 1;
  // epilogue staging: per epilogue warp, 32 token columns x 32 fp32 rows, padded
  static constexpr int STG_ROW = 144;
  static constexpr int STG_BYTES = 32 * STG_ROW;
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + 4 * STG_BYTES + NBARS * 8 + 16;
  static_assert(TN == 32, "the epilogue reads one 32-column accumulator per chunk");
  static_assert(USED_COLS <= 512, "TMEM");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct GateTile {
  int a_row, b_row;  // rows in the W_r and x tensor maps
  int k0, nk;        // first K element, number of BK blocks
  int n_valid;       // valid token columns
  int out_row0;      // output row of column 0
  int col0;          // output column of MMA row 0
  int m_limit;       // valid MMA rows (experts)
  float *out;
};

// Gate tile t = (expert block m, token tile tt), token tiles fastest; the
// whole of H in one accumulator (no split partials, one fixed summation order).
template <int TN>
__device__ __forceinline__ GateTile gate_tile(const TcParams &p, int tile) {
  const Dims &d = p.d;
  GateTile t;
  const int nt = (d.n_pos + TN - 1) / TN;
  const int m = tile / nt, tt = tile % nt;
  t.a_row = m * BM;
  t.b_row = tt * TN;
  t.k0 = 0;
  t.nk = d.H / BK;
  t.n_valid = min(TN, d.n_pos - tt * TN);
  t.out_row0 = tt * TN;
  t.col0 = m * BM;
  t.m_limit = min(BM, d.E - m * BM);
  t.out = p.ws.logits;
  return t;
}

// Waits for a phase without the abort check (teardown after an abort: lets
// copies and MMAs already issued land before the CTA exits).
__device__ __forceinline__ void mbar_drain(uint32_t bar, uint32_t parity, uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > ns) return;
  }
}

template <int TN, int STAGES>
__global__ void __launch_bounds__(192, 1) k_tc_gate(const __grid_constant__ TcParams p) {
  using C = GateCfg<TN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base (the 128-byte swizzle pattern repeats every 1024
  // bytes), offset from the __shared__ array itself so that every pointer
  // derived from it stays in the shared state space (shared loads and stores,
  // never ordered behind the epilogue's global stores)
  uint8_t *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sA = sbase;                          // [STAGES] W_r tiles
  const uint32_t sB = sbase + STAGES * C::A_BYTES;     // [STAGES] x tiles
  uint8_t *stage_out = smem + STAGES * C::STAGE_BYTES;  // [4][STG_BYTES] epilogue transposes
  uint64_t *bars = reinterpret_cast<uint64_t *>(stage_out + 4 * C::STG_BYTES);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * STAGES + C::NBUF + b); };
  const uint32_t done_bar = bar0 + 8u * (2 * STAGES + 2 * C::NBUF);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + C::NBARS);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const Dims &d = p.d;
  const Work &ws = p.ws;
  const KernelMark mark_(d, ws, K_GATE);
  pdl_wait();
  pdl_trigger();  // the routing kernel may start its launch; it waits for this grid to finish
  if (blockIdx.x == 0) {
    // counters of the routing launch that follows: its grid barrier and the
    // count of its finished CTAs (which the expert kernel waits for)
    if (threadIdx.x == 0) {
      *ws.gbar = 0u;
      *ws.route_done = 0u;
    }
  }
  clear_selection_masks(d, ws);
  const int total = p.gate_tiles;
  if (static_cast<int>(blockIdx.x) >= total) return;
  const int wid = warp_id(), lane = lane_id();
  const uint64_t tmo = static_cast<uint64_t>(d.timeout_ns);
  int64_t *trace = (d.trace && blockIdx.x < kTraceCtas)
                       ? ws.trace + (static_cast<size_t>(kTraceRowGate) * kTraceCtas + blockIdx.x) * kTraceFields
                       : nullptr;
  if (trace && threadIdx.x == 0) {
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    trace[0] = static_cast<int64_t>(globaltimer_ns());
    trace[7] = smid;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < C::NBUF; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 128);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (wid == 0) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (trace && threadIdx.x == 0) trace[1] = static_cast<int64_t>(globaltimer_ns());

  if (wid == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      tma_prefetch_desc(&p.a0);
      tma_prefetch_desc(&p.b[0]);
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_b = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const GateTile t = gate_tile<TN>(p, tile);
        const uint32_t tx = C::A_BYTES + C::B_BYTES;
        for (int kb = 0; kb < t.nk; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, ws.err, tmo)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(stage), tx);
          const int kc = t.k0 + kb * BK;
          tma_load_2d(sA + stage * C::A_BYTES, &p.a0, kc, t.a_row, full_bar(stage), pol_w);
          tma_load_2d(sB + stage * C::B_BYTES, &p.b[0], kc, t.b_row, full_bar(stage), pol_b);
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        for (int s = 0; s < STAGES; ++s)
          if (armed & (1u << s)) mbar_drain(full_bar(s), (armed_par >> s) & 1u, 50000000ull);
      }
    }
    __syncwarp();  // the whole warp reaches the final barrier (and the dealloc) together
  } else if (wid == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer
      int stage = 0, buf = 0;
      uint32_t phase = 0, bphase = 0;
      bool ok = true, first = true;
      int64_t n_tiles = 0, n_cols = 0;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const GateTile t = gate_tile<TN>(p, tile);
        const int n_mma = ((t.n_valid + 15) / 16) * 16;
        ++n_tiles;
        n_cols += t.n_valid;
        const uint32_t idesc = idesc_bf16_f32(BM, n_mma);
        uint32_t d0 = 0;
        for (int kb = 0; kb < t.nk; ++kb) {
          if (kb % kGateChunkKb == 0) {  // a new chunk starts in the next accumulator buffer
            if (!mbar_wait_bounded(tempty_bar(buf), bphase ^ 1u, abort_flag, ws.err, tmo)) {
              ok = false;
              break;
            }
            tc_fence_after();
            d0 = tmem_base + static_cast<uint32_t>(buf * C::ACC_COLS);
          }
          if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, ws.err, tmo)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (trace && first) {
            trace[2] = static_cast<int64_t>(globaltimer_ns());
            first = false;
          }
          const uint64_t ad0 = sw128_kmajor_desc(sA + stage * C::A_BYTES);
          const uint64_t bd = sw128_kmajor_desc(sB + stage * C::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint32_t acc = ((kb % kGateChunkKb) | kk) != 0;
            tc_mma_bf16(d0, ad0 + 2u * kk, bd + 2u * kk, idesc, acc);
          }
          tc_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          if (kb % kGateChunkKb == kGateChunkKb - 1 || kb == t.nk - 1) {  // chunk done
            tc_commit(tfull_bar(buf));
            if (++buf == C::NBUF) {
              buf = 0;
              bphase ^= 1u;
            }
          }
        }
        if (!ok) break;
      }
      tc_commit(done_bar);
      mbar_drain(done_bar, 0, 50000000ull);
      if (trace) {
        trace[3] = static_cast<int64_t>(globaltimer_ns());
        trace[5] = n_tiles;
        trace[6] = n_cols;
      }
    }
    __syncwarp();
  } else {
    // ---------------- epilogue (warps 2..5; warp w reads TMEM lanes 32*(w%4)..)
    // Per chunk: one 32-column TMEM load added into registers; then the sums
    // of this warp's 32 rows (+ bias) are staged token by token in shared
    // memory and eight lanes store one token's 32 contiguous logits (128 bytes)
    // together, four tokens per instruction.
    const int q = wid & 3;
    uint8_t *stg = stage_out + (wid - 2) * C::STG_BYTES;
    int buf = 0;
    uint32_t bphase = 0;
    bool ok = true;
    for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
      const GateTile t = gate_tile<TN>(p, tile);
      // sum the chunk accumulators in chunk order (fp32), then add the bias
      float sum[TN];
#pragma unroll
      for (int c = 0; c < TN; ++c) sum[c] = 0.f;
      const int n_chunks = (t.nk + kGateChunkKb - 1) / kGateChunkKb;
      for (int ch = 0; ch < n_chunks; ++ch) {
        if (!mbar_wait_bounded(tfull_bar(buf), bphase, abort_flag, ws.err, tmo)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * C::ACC_COLS);
        float v0[TN];
        tmem_ld32(tb, v0);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < TN; ++c) sum[c] += v0[c];
        tc_fence_before();
        mbar_arrive(tempty_bar(buf));
        if (++buf == C::NBUF) {
          buf = 0;
          bphase ^= 1u;
        }
      }
      if (!ok) break;
      const int rows_valid = min(32, max(0, t.m_limit - q * 32));
      const int e_row = t.col0 + q * 32 + lane;  // this lane's TMEM row = expert
      const float bias_r = e_row < d.E ? __ldg(p.bias + e_row) : 0.f;
      const bool vec_ok = rows_valid == 32 && ((d.E * 4) & 15) == 0;
      {
        const int c0 = 0;
#pragma unroll
        for (int c = 0; c < TN; ++c) reinterpret_cast<float *>(stg + c * C::STG_ROW)[lane] = sum[c] + bias_r;
        __syncwarp();
        const int ncol = min(32, t.n_valid - c0);
        if (vec_ok) {
          const int v = lane & 7;
          for (int c = lane >> 3; c < ncol; c += 4) {
            const int orow = t.out_row0 + c0 + c;
            if (orow < 0 || orow >= d.Nmax) {
              set_error(ws.err, EPOCH_DEVERR_BOUNDS);
              continue;
            }
            reinterpret_cast<uint4 *>(t.out + static_cast<size_t>(orow) * d.E + t.col0 + q * 32)[v] =
                *reinterpret_cast<const uint4 *>(stg + c * C::STG_ROW + v * 16);
          }
        } else if (lane < ncol) {
          const int orow = t.out_row0 + c0 + lane;
          if (orow < 0 || orow >= d.Nmax) {
            set_error(ws.err, EPOCH_DEVERR_BOUNDS);
          } else {
            for (int r = 0; r < rows_valid; ++r)
              t.out[static_cast<size_t>(orow) * d.E + t.col0 + q * 32 + r] =
                  reinterpret_cast<const float *>(stg + lane * C::STG_ROW)[r];
          }
        }
        __syncwarp();
      }
    }
    if (trace && wid == 2 && lane == 0) trace[4] = static_cast<int64_t>(globaltimer_ns());
  }
  tc_fence_before();
  __syncthreads();
  if (wid == 0) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- fused expert kernel
// Up and down projections of every group in one persistent cooperative launch
// (one CTA per SM). Tiles of the list [all up tiles, then all down tiles] are
// handed out one at a time from a global counter, so a CTA that drew short
// tiles draws more. Both kinds are two 128-row MMAs sharing one token tile of
// <= 128 tokens: an up tile (group g, 128 rows of I) multiplies the gate and up
// rows and writes silu(gate) * up as bf16, then counts itself done for g; a
// down tile (g, 256 rows of H) waits until every up tile of g is done before
// loading its activations (its weight copies go out first), so the down work of
// lightly loaded experts runs while heavy up tiles are still streaming, with no
// launch in between. Every tile uses one 256-column TMEM accumulator buffer,
// double-buffered; a 48 KB stage holds 32 KB of packed weights (one contiguous
// run) and a 16 KB token tile.
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

// Tile q of the list [all up tiles, then all down tiles] -> decoded tile and
// the up-tile count of its group. list = the routing kernel's group list:
// entry p holds the token tiles of the groups before p (<< kGrpIdBits) and the
// group of p; the shared experts come first (p < n_sh). offs = expert row
// offsets. Within a group the tiles run row block by row block, token tiles
// fastest, so tiles drawn close together share a weight row block in L2. Up
// tiles of the shared experts come first (I_s / 128 row blocks each), then
// those of the routed experts (I / 128); down tiles have H / 256 row blocks in
// every group. Returns false when the list and the offsets disagree.
__device__ __forceinline__ bool locate(const Dims &d, const int32_t *list, const int32_t *offs, int q, int n_up,
                                      int4 *td, int *need) {
  const int G2 = d.E + d.n_sh;
  auto pref = [&](int p) { return list[p] >> kGrpIdBits; };
  const bool up = q < n_up;
  int base_q = 0, base_t = 0, mult, lo = 0, hi = G2;
  if (up) {
    const int a_sh = (d.I_s / BM) * pref(d.n_sh);
    if (q < a_sh) {
      mult = d.I_s / BM;
      hi = d.n_sh;
    } else {
      base_q = a_sh;
      base_t = pref(d.n_sh);
      mult = d.I / BM;
      lo = d.n_sh;
    }
  } else {
    q -= n_up;
    mult = d.H / kBmDn;
  }
  const int key = base_t + (q - base_q) / mult;
  // largest p in [lo, hi) with pref(p) <= key
  int l = lo, h = hi;
  while (h - l > 1) {
    const int mid = (l + h) >> 1;
    if (pref(mid) <= key) l = mid;
    else h = mid;
  }
  const int nt = pref(l + 1) - pref(l);
  const int qq = q - base_q - mult * (pref(l) - base_t);
  if (nt <= 0 || qq < 0 || qq >= mult * nt) return false;
  const int m = qq / nt, tt = qq - m * nt;
  const int g = list[l] & ((1 << kGrpIdBits) - 1);
  const bool shared = g >= d.E;
  if (shared != (l < d.n_sh) || g >= G2) return false;
  const int rows = shared ? d.n_pos : offs[g + 1] - offs[g];
  const int r0 = (shared ? 0 : offs[g]) + tt * kTnUp;
  const int n_valid = min(kTnUp, rows - tt * kTnUp);
  if (n_valid <= 0) return false;
  *td = make_int4(g | (up ? 0 : kDownBit), m, r0, n_valid);
  *need = nt * ((shared ? d.I_s : d.I) / BM);
  return true;
}

struct XTile {
  bool up;                // up tile (else down)
  int g;                  // group
  const uint8_t *a_src;   // first packed weight tile of the row block
  int a_bytes;            // weight bytes per K block (32 KB: two 128-row tiles)
  int nk;                 // K blocks
  const CUtensorMap *mb;  // token-operand map (box chosen for the tile)
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
  // The prologue above may overlap the routing kernel (programmatic dependent
  // launch); the producer draws tiles from tile_ctr only after it has seen
  // every routing CTA finish (the route_done count) and loaded the group list
  // and expert offsets.

  if (wid == 0) {
    // ---------------- producer: weight bulk copies + token TMA loads (lane 0)
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_b = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0, armed = 0, armed_par = 0;
    bool ok = true;
    uint64_t waited = 0;
    // Issues the operand copies of one tile; a down tile first waits until every
    // up tile of its group (`need` of them) has written its activations.
    auto issue = [&](const int4 &td, int need) -> bool {
      const XTile t = xdecode(p, td);
      const uint32_t tx = t.a_bytes + t.b_bytes;
      // a down tile's weights do not depend on the up tiles: its first stages'
      // weight copies go out before the dependency wait, their token loads after
      const int pre = t.up ? 0 : min(t.nk, 2);
      int pre_stage[2] = {0, 0};
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
      if (!t.up) {
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
          int done;
          asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(done) : "l"(ws.done_up + t.g) : "memory");
          if (done >= need) break;
          if (*abort_flag) return false;
          if (globaltimer_ns() - t0 > tmo) {
            set_error(ws.err, EPOCH_DEVERR_TIMEOUT);
            *abort_flag = 1;
            return false;
          }
          __nanosleep(64);
        }
        waited += globaltimer_ns() - t0;
        asm volatile("fence.proxy.async.global;" ::: "memory");  // generic writes -> TMA reads
        for (int kb = 0; kb < pre; ++kb)
          tma_load_2d(sbase + pre_stage[kb] * kExpStage + 2 * kTileBytes, t.mb, kb * BK, t.b_row,
                      full_bar(pre_stage[kb]), pol_b);
      }
      for (int kb = pre; kb < t.nk; ++kb) {
        if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, ws.err, tmo)) return false;
        mbar_arrive_expect_tx(full_bar(stage), tx);
        const uint32_t st = sbase + stage * kExpStage;
        bulk_load(st, t.a_src + static_cast<size_t>(kb) * t.a_bytes, t.a_bytes, full_bar(stage), pol_w);
        tma_load_2d(st + 2 * kTileBytes, t.mb, kb * BK, t.b_row, full_bar(stage), pol_b);
        armed |= 1u << stage;
        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
        if (++stage == kExpStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      return true;
    };
    if (lane == 0) {
      tma_prefetch_desc(&p.bs);
      tma_prefetch_desc(&p.b[0]);
      tma_prefetch_desc(&p.b2[0]);
    }
    // wait until every routing CTA has counted itself done (acquire: its writes
    // are visible to this warp after the __syncwarp)
    if (lane == 0 && ok) {
      const uint64_t t0 = globaltimer_ns();
      for (;;) {
        unsigned int v;
        asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(ws.route_done) : "memory");
        if (v >= static_cast<unsigned int>(d.route_ctas)) break;
        if (*abort_flag) {
          ok = false;
          break;
        }
        if (globaltimer_ns() - t0 > tmo) {
          set_error(ws.err, EPOCH_DEVERR_TIMEOUT);
          *abort_flag = 1;
          ok = false;
          break;
        }
        __nanosleep(128);
      }
    }
    __syncwarp();
    for (int i = lane; i <= d.E + d.n_sh; i += 32) s_list[i] = ws.grp_list[i];
    for (int i = lane; i <= d.E; i += 32) s_offs[i] = ws.offsets[i];
    const int n_up = ws.ctrl->tiles_up;
    const int total = n_up + ws.ctrl->tiles_dn;
    __syncwarp();
    if (lane == 0) {
      if (trace) trace[2] = static_cast<int64_t>(globaltimer_ns());
      for (int j = 0; ok; ++j) {
        const int slot = j % kExpSched;
        if (!mbar_wait_bounded(sempty_bar(slot), ((j / kExpSched) & 1) ^ 1u, abort_flag, ws.err, tmo)) break;
        const int tile = atomicAdd(ws.tile_ctr, 1);
        int4 td = make_int4(-1, 0, 0, 0);
        int need = 0;
        if (tile < total && !locate(d, s_list, s_offs, tile, n_up, &td, &need)) {
          set_error(ws.err, EPOCH_DEVERR_BOUNDS);
          *abort_flag = 1;
          td.x = -1;
        }
        s_td[slot] = td;
        mbar_arrive(sfull_bar(slot));
        if (td.x < 0) break;
        ok = issue(td, need);
      }
      if (!ok) {
        for (int s = 0; s < kExpStages; ++s)
          if (armed & (1u << s)) mbar_drain(full_bar(s), (armed_par >> s) & 1u, 50000000ull);
      }
      if (trace) trace[6] = static_cast<int64_t>(waited);
    }
    __syncwarp();
  } else if (wid == 1) {
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
  } else {
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
          atomicAdd(ws.done_up + t.g, 1);
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

constexpr int kStGate = 8;  // 20 KB stages (a 128 x 64 W_r tile and a 32 x 64 x tile)

template <int TN, int STAGES>
static cudaError_t launch_gate(const TcParams &p, int grid, cudaStream_t s) {
  using C = GateCfg<TN, STAGES>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(k_tc_gate<TN, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e == cudaSuccess) e = prefer_max_shared(k_tc_gate<TN, STAGES>);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  k_tc_gate<TN, STAGES><<<grid, 192, C::SMEM, s>>>(p);
  return cudaGetLastError();
}

static void base_params(TcParams &p, const Dims &d, const Work &ws) {
  memset(&p, 0, sizeof(p));
  p.d = d;
  p.ws = ws;
}

cudaError_t launch_gate_tc(const Dims &d, const Maps &m, const Work &ws, const CUtensorMap &x_map,
                           const float *bias, cudaStream_t s) {
  TcParams p;
  base_params(p, d, ws);
  p.a0 = m.w_router;
  p.bias = bias;
  p.b[0] = x_map;
  const int tiles = ((d.E + BM - 1) / BM) * ((d.n_pos + kTnGate - 1) / kTnGate);
  p.gate_tiles = tiles;
  const int grid = tiles < num_sms() ? tiles : num_sms();
  return launch_gate<kTnGate, kStGate>(p, grid, s);
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
  base_params(p, d, ws);
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
  return launch_kernel(reinterpret_cast<void *>(k_tc_experts), dim3(num_sms()), dim3(192), kExpSmem, s, args, false,
                       true);
}

}  // namespace epoch

// tcgen05 + TMA grouped GEMMs of the Epoch MoE layer (bf16 in, fp32 accumulate).
//
// Three contractions share one persistent, warp-specialised kernel:
//   GATE  G^T = W_r x^T, split along H (the route kernel sums the splits in a
//         fixed order and adds the bias) -- router logits for every position
//         ([W] section "Expert Atlas": G in R^{N x E}, recomputed every iteration);
//   UP    per group g: A_g = silu(X_g W_gate,g^T) * (X_g W_up,g^T) -> bf16;
//   DOWN  per group g: O_g = A_g W_down,g^T -> fp32.
// Groups are the routed experts with at least one worklist row, then the
// shared experts over every position; each routed expert runs once over its
// compact rows (the "light-traffic expert kernel" of [W] section
// "FreshLane Dispatch"); experts with no row produce no tile, so their weights
// are never read ("invalid slots load no expert weights", same section).
// [W] = walk-through page "Epoch 完全拆解:把扩散块编译成稀疏 MoE 服务单元".
//
// Swap-AB: weight rows are the MMA M dimension (128) and tokens the N
// dimension (16..TN, rounded up to 16 per tile), because an expert may hold
// from one to a thousand rows. Roles per CTA (192 threads): warp 0 issues TMA
// loads into a STAGES-deep shared-memory ring (128-byte swizzle, K-major),
// warp 1 issues tcgen05.mma into TMEM accumulators (double-buffered when they
// fit, so the epilogue of one tile overlaps the next tile's main loop), warps
// 2-5 read TMEM with tcgen05.ld and store. One CTA per SM, persistent over a
// device-resident tile count: no host synchronisation.
#include <cudaTypedefs.h>

#include <cstring>

#include "common.cuh"
#include "layer.h"

namespace epoch {

constexpr int BM = 128;
constexpr int BK = 64;

enum Mode { M_GATE = 0, M_UP = 1, M_DOWN = 2 };

struct __align__(128) TcParams {
  CUtensorMap a0;    // GATE: W_r (UP and DOWN stream packed weight tiles instead)
  CUtensorMap b[4];  // GATE: b[0] = x; UP: Xp; DOWN: A (routed) -- boxes of 32/64/128/256 rows
  CUtensorMap bs;    // UP: x; DOWN: A (shared) -- box of TN rows
  CUtensorMap b2[4]; // fused expert kernel: A (routed) for the down tiles
  CUtensorMap bs2;   // fused expert kernel: A (shared) for the down tiles
  Dims d;
  Work ws;
  int32_t gate_tiles;
};

template <int MODE, int TN, int STAGES>
struct Cfg {
  static constexpr int NA = MODE == M_UP ? 2 : 1;
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int B_BYTES = TN * BK * 2;
  static constexpr int STAGE_BYTES = NA * A_BYTES + B_BYTES;
  static constexpr int ACC_COLS = NA * TN;
  static constexpr int NBUF = 2 * ACC_COLS <= 512 ? 2 : 1;
  static constexpr int USED_COLS = NBUF * ACC_COLS;
  static constexpr int TMEM_COLS = USED_COLS <= 32 ? 32 : USED_COLS <= 64 ? 64 : USED_COLS <= 128 ? 128
                                   : USED_COLS <= 256 ? 256 : 512;
  static constexpr int NBARS = 2 * STAGES + 2 * NBUF + 1;
  // epilogue staging: per epilogue warp, 32 token columns x 32 rows, padded rows
  static constexpr int STG_ROW = MODE == M_UP ? 80 : 144;  // bytes per staged column (64 / 128 B + pad)
  static constexpr int STG_BYTES = 32 * STG_ROW;
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + 4 * STG_BYTES + NBARS * 8 + 16;
  static_assert(TN % 16 == 0 && TN >= 16 && TN <= 256, "MMA N");
  static_assert(USED_COLS <= 512, "TMEM");
  static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct Tile {
  const uint8_t *a_src;   // UP/DOWN: first packed weight tile of the (group, m) row block
  int a_stride;           // bytes between consecutive K blocks of packed weights
  const CUtensorMap *mb;  // B-operand map (box chosen for the tile)
  int a_row, b_row;       // rows in the A (weights) and B (tokens) tensor maps
  int shared;             // group is a shared expert (selects the *s maps)
  int k0, nk;             // first K element, number of BK blocks
  int n_valid;            // valid token columns
  int b_bytes;            // bytes of one B box
  int out_row0;           // output row of column 0
  int out_rows;           // rows in the output buffer (bounds check)
  int ld;                 // output leading dimension
  int col0;               // output column of MMA row 0
  int m_limit;            // valid MMA rows
  void *out;
};

template <int MODE, int TN>
__device__ __forceinline__ Tile decode(const TcParams &p, int tile) {
  const Dims &d = p.d;
  const Work &ws = p.ws;
  Tile t;
  if (MODE == M_GATE) {
    const int mt = (d.E + BM - 1) / BM, nt = (d.n_pos + TN - 1) / TN;
    const int ks = tile / (mt * nt), rem = tile % (mt * nt);
    const int m = rem / nt, tt = rem % nt;
    const int kspan = d.H / d.SK;
    t.mb = &p.b[0];
    t.a_row = m * BM;
    t.b_row = tt * TN;
    t.shared = 0;
    t.k0 = ks * kspan;
    t.nk = kspan / BK;
    t.n_valid = min(TN, d.n_pos - tt * TN);
    t.b_bytes = TN * BK * 2;
    t.out_row0 = tt * TN;
    t.out_rows = d.Nmax;
    t.ld = d.E;
    t.col0 = m * BM;
    t.m_limit = min(BM, d.E - m * BM);
    t.out = ws.gparts + static_cast<size_t>(ks) * d.Nmax * d.E;
    return t;
  }
  const int4 td = MODE == M_UP ? ws.tiles_up[tile] : ws.tiles_dn[tile];
  const int g = td.x, m = td.y, r0 = td.z;
  t.n_valid = td.w;
  t.shared = g >= d.E;
  const int s = g - d.E;
  if (t.shared) {
    t.mb = &p.bs;
    t.b_bytes = TN * BK * 2;
  } else {
    const int bi = t.n_valid <= 32 ? 0 : t.n_valid <= 64 ? 1 : t.n_valid <= 128 ? 2 : 3;
    t.mb = &p.b[bi];
    t.b_bytes = (32 << bi) * BK * 2;  // box rows 32, 64, 128, 256
  }
  t.col0 = m * BM;
  t.m_limit = BM;
  t.k0 = 0;
  if (MODE == M_UP) {
    const int nkb = d.H / BK;
    const size_t rb = t.shared ? static_cast<size_t>(s) * (d.I_s / BM) + m : static_cast<size_t>(g) * (d.I / BM) + m;
    t.a_src = (t.shared ? ws.pk_sgu : ws.pk_gu) + rb * nkb * (2 * kTileBytes);
    t.a_stride = 2 * kTileBytes;
    t.a_row = t.shared ? s * d.I_s + m * BM : g * d.I + m * BM;
    t.b_row = r0;
    t.out_row0 = t.shared ? s * d.Nmax + r0 : r0;
    t.nk = d.H / BK;
    t.ld = t.shared ? d.I_s : d.I;
    t.out = t.shared ? ws.a_sh : ws.a_int;
    t.out_rows = t.shared ? d.n_sh * d.Nmax : d.Nmax * d.k;
  } else {
    const int nkb = (t.shared ? d.I_s : d.I) / BK;
    const size_t rb = t.shared ? static_cast<size_t>(s) * (d.H / BM) + m : static_cast<size_t>(g) * (d.H / BM) + m;
    t.a_src = (t.shared ? ws.pk_sd : ws.pk_d) + rb * nkb * kTileBytes;
    t.a_stride = kTileBytes;
    t.a_row = t.shared ? s * d.H + m * BM : g * d.H + m * BM;
    t.b_row = t.shared ? s * d.Nmax + r0 : r0;
    t.out_row0 = t.b_row;
    t.nk = (t.shared ? d.I_s : d.I) / BK;
    t.ld = d.H;
    t.out = t.shared ? static_cast<void *>(ws.o_sh) : static_cast<void *>(ws.o_int);
    t.out_rows = t.shared ? d.n_sh * d.Nmax : d.Nmax * d.k;
  }
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

template <int MODE, int TN, int STAGES>
__global__ void __launch_bounds__(192, 1) k_tc_gemm(const __grid_constant__ TcParams p) {
  using C = Cfg<MODE, TN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t sA = sbase;                                   // [STAGES][NA] A tiles
  const uint32_t sB = sbase + STAGES * C::NA * C::A_BYTES;     // [STAGES] B tiles
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
  const KernelMark mark_(d, ws, MODE == M_GATE ? K_GATE : MODE == M_UP ? K_UP : K_DOWN);
  if (MODE == M_GATE && blockIdx.x == 0 && threadIdx.x == 0) *ws.gbar = 0u;  // next routing launch
  const int total = MODE == M_GATE ? p.gate_tiles : (MODE == M_UP ? ws.ctrl->tiles_up : ws.ctrl->tiles_dn);
  if (static_cast<int>(blockIdx.x) >= total) return;
  const int wid = warp_id(), lane = lane_id();
  const uint64_t tmo = static_cast<uint64_t>(d.timeout_ns);
  int64_t *trace = (d.trace && blockIdx.x < kTraceCtas)
                       ? ws.trace + (static_cast<size_t>(MODE) * kTraceCtas + blockIdx.x) * kTraceFields
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
      if (MODE == M_GATE) tma_prefetch_desc(&p.a0);
      tma_prefetch_desc(&p.b[0]);
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_b = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
        const Tile t = decode<MODE, TN>(p, tile);
        const CUtensorMap *ma0 = &p.a0;
        const CUtensorMap *mb = t.mb;
        const uint32_t tx = C::NA * C::A_BYTES + t.b_bytes;
        for (int kb = 0; kb < t.nk; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, ws.err, tmo)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(stage), tx);
          const int kc = t.k0 + kb * BK;
          const uint32_t a_dst = sA + stage * C::NA * C::A_BYTES;
          if (MODE == M_GATE) {
            tma_load_2d(a_dst, ma0, kc, t.a_row, full_bar(stage), pol_w);
          } else {
            // packed weights: the stage's A tiles are one contiguous run
            bulk_load(a_dst, t.a_src + static_cast<size_t>(kb) * t.a_stride, C::NA * C::A_BYTES, full_bar(stage),
                      pol_w);
          }
          tma_load_2d(sB + stage * C::B_BYTES, mb, kc, t.b_row, full_bar(stage), pol_b);
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
        const Tile t = decode<MODE, TN>(p, tile);
        const int n_mma = ((t.n_valid + 15) / 16) * 16;
        ++n_tiles;
        n_cols += t.n_valid;
        const uint32_t idesc = idesc_bf16_f32(BM, n_mma);
        if (!mbar_wait_bounded(tempty_bar(buf), bphase ^ 1u, abort_flag, ws.err, tmo)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + static_cast<uint32_t>(buf * C::ACC_COLS);
        for (int kb = 0; kb < t.nk; ++kb) {
          if (!mbar_wait_bounded(full_bar(stage), phase, abort_flag, ws.err, tmo)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (trace && first) {
            trace[2] = static_cast<int64_t>(globaltimer_ns());
            first = false;
          }
          const uint32_t a_src = sA + stage * C::NA * C::A_BYTES;
          const uint64_t ad0 = sw128_kmajor_desc(a_src);
          const uint64_t ad1 = sw128_kmajor_desc(a_src + C::A_BYTES);
          const uint64_t bd = sw128_kmajor_desc(sB + stage * C::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint32_t acc = (kb | kk) != 0;
            tc_mma_bf16(d0, ad0 + 2u * kk, bd + 2u * kk, idesc, acc);
            if (C::NA == 2) tc_mma_bf16(d0 + TN, ad1 + 2u * kk, bd + 2u * kk, idesc, acc);
          }
          tc_commit(empty_bar(stage));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(tfull_bar(buf));
        if (++buf == C::NBUF) {
          buf = 0;
          bphase ^= 1u;
        }
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
    // Per 32 token columns: two 32-column TMEM loads and one wait, the values
    // of this warp's 32 rows staged column-major in shared memory, then lane c
    // writes token column c's 32 contiguous outputs with 16-byte stores.
    const int q = wid & 3;
    uint8_t *stg = stage_out + (wid - 2) * C::STG_BYTES;
    int buf = 0;
    uint32_t bphase = 0;
    for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
      const Tile t = decode<MODE, TN>(p, tile);
      if (!mbar_wait_bounded(tfull_bar(buf), bphase, abort_flag, ws.err, tmo)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * C::ACC_COLS);
      const int rows_valid = min(32, max(0, t.m_limit - q * 32));
      const int esz = MODE == M_UP ? 2 : 4;
      const bool vec_ok = rows_valid == 32 && ((t.ld * esz) & 15) == 0;
      for (int c0 = 0; c0 < t.n_valid; c0 += 32) {
        float v0[32], v1[32];
        tmem_ld32(tb + c0, v0);
        if (C::NA == 2) tmem_ld32(tb + TN + c0, v1);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          if (MODE == M_UP) {
            reinterpret_cast<__nv_bfloat16 *>(stg + c * C::STG_ROW)[lane] =
                __float2bfloat16_rn(silu_fast(v0[c]) * v1[c]);
          } else {
            reinterpret_cast<float *>(stg + c * C::STG_ROW)[lane] = v0[c];
          }
        }
        __syncwarp();
        const int col = c0 + lane;  // token column written by this lane
        const int orow = t.out_row0 + col;
        if (col < t.n_valid) {
          if (orow < 0 || orow >= t.out_rows) {
            set_error(ws.err, EPOCH_DEVERR_BOUNDS);
          } else if (vec_ok) {
            const uint4 *src = reinterpret_cast<const uint4 *>(stg + lane * C::STG_ROW);
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint8_t *>(t.out) +
                                                   (static_cast<size_t>(orow) * t.ld + t.col0 + q * 32) * esz);
#pragma unroll
            for (int v = 0; v < 32 * esz / 16; ++v) dst[v] = src[v];
          } else {
            for (int r = 0; r < rows_valid; ++r) {
              const size_t o = static_cast<size_t>(orow) * t.ld + t.col0 + q * 32 + r;
              if (MODE == M_UP)
                static_cast<__nv_bfloat16 *>(t.out)[o] = reinterpret_cast<const __nv_bfloat16 *>(stg + lane * C::STG_ROW)[r];
              else
                static_cast<float *>(t.out)[o] = reinterpret_cast<const float *>(stg + lane * C::STG_ROW)[r];
            }
          }
        }
        __syncwarp();
      }
      tc_fence_before();
      mbar_arrive(tempty_bar(buf));
      if (++buf == C::NBUF) {
        buf = 0;
        bphase ^= 1u;
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
// (one CTA per SM). Each CTA takes tiles blockIdx.x, + gridDim.x, ... of the
// list [all up tiles, then all down tiles]. Both kinds are two 128-row MMAs
// sharing one token tile of <= 128 tokens: an up tile (group g, 128 rows of I)
// multiplies the gate and up rows and writes silu(gate) * up as bf16, then
// counts itself done for g; a down tile (g, 256 rows of H) waits until every up
// tile of g is done before loading its activations (its weight copies go out
// first), so the down work of lightly loaded experts runs while heavy up tiles
// are still streaming, with no launch in between. Every tile uses one
// 256-column TMEM accumulator buffer, double-buffered; a 48 KB stage holds
// 32 KB of packed weights (one contiguous run) and a 16 KB token tile.
constexpr int kExpStages = 4;
constexpr int kExpStage = 48 * 1024;
constexpr int kExpStg = 32 * 144;  // epilogue staging per warp (fp32 worst case)
constexpr int kExpSched = 4;  // tile-id ring between the producer and the MMA / epilogue warps
constexpr int kExpBars = 2 * kExpStages + 2 * 2 + 1 + 2 * kExpSched;
constexpr int kExpSmem = 1024 + kExpStages * kExpStage + 4 * kExpStg + kExpBars * 8 + 16 + kExpSched * 4;
static_assert(kExpSmem <= 227 * 1024, "shared memory");

struct XTile {
  bool up;                // up tile (else down)
  int g;                  // group
  const uint8_t *a_src;   // first packed weight tile of the row block
  int a_bytes;            // weight bytes per K block (32 KB up, 16 KB down)
  int nk;                 // K blocks
  const CUtensorMap *mb;  // token-operand map (box chosen for the tile)
  int b_row, b_bytes;
  int n_valid;
  int out_row0, out_rows, ld, col0;
  void *out;
};

__device__ __forceinline__ XTile xdecode(const TcParams &p, int tile, int n_up) {
  const Dims &d = p.d;
  const Work &ws = p.ws;
  XTile t;
  t.up = tile < n_up;
  const int4 td = t.up ? ws.tiles_up[tile] : ws.tiles_dn[tile - n_up];
  const int g = td.x, m = td.y, r0 = td.z;
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
    t.b_bytes = (shared ? d.tn_up : (32 << bi)) * BK * 2;
    t.b_row = r0;
    t.out_row0 = shared ? s * d.Nmax + r0 : r0;
    t.ld = shared ? d.I_s : d.I;
    t.out = shared ? ws.a_sh : ws.a_int;
    t.out_rows = shared ? d.n_sh * d.Nmax : d.Nmax * d.k;
  } else {
    // 256 rows of H: two 128-row blocks sharing the token tile; the packed pair
    // of a K block is one contiguous 32 KB run
    const int nkb = (shared ? d.I_s : d.I) / BK;
    const size_t pb = shared ? static_cast<size_t>(s) * (d.H / (2 * BM)) + m : static_cast<size_t>(g) * (d.H / (2 * BM)) + m;
    t.a_src = (shared ? ws.pk_sd : ws.pk_d) + pb * nkb * (2 * kTileBytes);
    t.a_bytes = 2 * kTileBytes;
    t.nk = nkb;
    t.col0 = m * 2 * BM;
    t.mb = shared ? &p.bs2 : &p.b2[bi];
    t.b_bytes = (shared ? d.tn_dn : (32 << bi)) * BK * 2;
    t.b_row = shared ? s * d.Nmax + r0 : r0;
    t.out_row0 = t.b_row;
    t.ld = d.H;
    t.out = shared ? static_cast<void *>(ws.o_sh) : static_cast<void *>(ws.o_int);
    t.out_rows = shared ? d.n_sh * d.Nmax : d.Nmax * d.k;
  }
  return t;
}

__global__ void __launch_bounds__(192, 1) k_tc_experts(const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  uint8_t *stage_out = smem + kExpStages * kExpStage;
  uint64_t *bars = reinterpret_cast<uint64_t *>(stage_out + 4 * kExpStg);
  const uint32_t bar0 = smem_u32(bars);
  auto full_bar = [&](int s) { return bar0 + 8u * s; };
  auto empty_bar = [&](int s) { return bar0 + 8u * (kExpStages + s); };
  auto tfull_bar = [&](int b) { return bar0 + 8u * (2 * kExpStages + b); };
  auto tempty_bar = [&](int b) { return bar0 + 8u * (2 * kExpStages + 2 + b); };
  const uint32_t done_bar = bar0 + 8u * (2 * kExpStages + 4);
  auto sfull_bar = [&](int i) { return bar0 + 8u * (2 * kExpStages + 5 + i); };
  auto sempty_bar = [&](int i) { return bar0 + 8u * (2 * kExpStages + 5 + kExpSched + i); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + kExpBars);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  volatile int *s_tile = reinterpret_cast<volatile int *>(tmem_slot + 4);  // [kExpSched]

  const Dims &d = p.d;
  const Work &ws = p.ws;
  const KernelMark mark_(d, ws, K_UP);
  const int n_up = ws.ctrl->tiles_up;
  const int total = n_up + ws.ctrl->tiles_dn;
  const int wid = warp_id(), lane = lane_id();
  const uint64_t tmo = static_cast<uint64_t>(d.timeout_ns);
  int64_t *trace = (d.trace && blockIdx.x < kTraceCtas)
                       ? ws.trace + (static_cast<size_t>(M_UP) * kTraceCtas + blockIdx.x) * kTraceFields
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
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  if (trace && threadIdx.x == 0) trace[1] = static_cast<int64_t>(globaltimer_ns());

  if (wid == 0) {
    if (lane == 0) {
      // ---------------- producer: weight bulk copies + token TMA loads
      tma_prefetch_desc(&p.b[0]);
      tma_prefetch_desc(&p.b2[0]);
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_b = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_par = 0;
      bool ok = true;
      uint64_t waited = 0;
      for (int j = 0; ok; ++j) {
        // next tile from the global counter, handed to the MMA and epilogue warps
        const int slot = j % kExpSched;
        if (!mbar_wait_bounded(sempty_bar(slot), ((j / kExpSched) & 1) ^ 1u, abort_flag, ws.err, tmo)) break;
        int tile = atomicAdd(ws.tile_ctr, 1);
        if (tile >= total) tile = -1;
        s_tile[slot] = tile;
        mbar_arrive(sfull_bar(slot));
        if (tile < 0) break;
        const XTile t = xdecode(p, tile, n_up);
        const uint32_t tx = t.a_bytes + t.b_bytes;
        // a down tile's weights do not depend on the up tiles: its first stages'
        // weight copies go out before the dependency wait, their token loads after
        const int pre = t.up ? 0 : min(t.nk, 2);
        int pre_stage[2] = {0, 0};
        for (int kb = 0; kb < pre; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, ws.err, tmo)) {
            ok = false;
            break;
          }
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
        if (!ok) break;
        if (!t.up) {
          // wait until every up tile of this group has written its activations
          const int need = ws.up_needed[t.g];
          const uint64_t t0 = globaltimer_ns();
          for (;;) {
            int done;
            asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(done) : "l"(ws.done_up + t.g) : "memory");
            if (done >= need) break;
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
            __nanosleep(64);
          }
          if (!ok) break;
          waited += globaltimer_ns() - t0;
          asm volatile("fence.proxy.async.global;" ::: "memory");  // generic writes -> TMA reads
          for (int kb = 0; kb < pre; ++kb)
            tma_load_2d(sbase + pre_stage[kb] * kExpStage + 2 * kTileBytes, t.mb, kb * BK, t.b_row,
                        full_bar(pre_stage[kb]), pol_b);
        }
        for (int kb = pre; kb < t.nk; ++kb) {
          if (!mbar_wait_bounded(empty_bar(stage), phase ^ 1u, abort_flag, ws.err, tmo)) {
            ok = false;
            break;
          }
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
      bool ok = true, first = true;
      int64_t n_tiles = 0;
      for (int j = 0; ok; ++j) {
        const int slot = j % kExpSched;
        if (!mbar_wait_bounded(sfull_bar(slot), (j / kExpSched) & 1, abort_flag, ws.err, tmo)) break;
        const int tile = s_tile[slot];
        mbar_arrive(sempty_bar(slot));
        if (tile < 0) break;
        const XTile t = xdecode(p, tile, n_up);
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
          if (trace && first) {
            trace[2] = static_cast<int64_t>(globaltimer_ns());
            first = false;
          }
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
    for (int j = 0;; ++j) {
      const int slot = j % kExpSched;
      if (!mbar_wait_bounded(sfull_bar(slot), (j / kExpSched) & 1, abort_flag, ws.err, tmo)) break;
      const int tile = s_tile[slot];
      __syncwarp();
      if (lane == 0) mbar_arrive(sempty_bar(slot));
      if (tile < 0) break;
      const XTile t = xdecode(p, tile, n_up);
      if (!mbar_wait_bounded(tfull_bar(buf), bphase, abort_flag, ws.err, tmo)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(buf * 256);
      const int esz = t.up ? 2 : 4;
      const int row_bytes = t.up ? 80 : 144;
      const bool vec_ok = ((t.ld * esz) & 15) == 0;
      const int halves = t.up ? 1 : 2;  // down: the two 128-row blocks are two output column blocks
      for (int hb = 0; hb < halves; ++hb) {
        for (int c0 = 0; c0 < t.n_valid; c0 += 32) {
          float v0[32];
          tmem_ld32(tb + hb * 128 + c0, v0);
          if (t.up) {
            float v1[32];
            tmem_ld32(tb + 128 + c0, v1);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c)
              reinterpret_cast<__nv_bfloat16 *>(stg + c * row_bytes)[lane] =
                  __float2bfloat16_rn(silu_fast(v0[c]) * v1[c]);
          } else {
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) reinterpret_cast<float *>(stg + c * row_bytes)[lane] = v0[c];
          }
          __syncwarp();
          const int col = c0 + lane;
          const int orow = t.out_row0 + col;
          if (col < t.n_valid) {
            if (orow < 0 || orow >= t.out_rows) {
              set_error(ws.err, EPOCH_DEVERR_BOUNDS);
            } else {
              uint8_t *dst = static_cast<uint8_t *>(t.out) +
                             (static_cast<size_t>(orow) * t.ld + t.col0 + hb * 128 + q * 32) * esz;
              const uint8_t *src = stg + lane * row_bytes;
              if (vec_ok) {
                for (int v = 0; v < 32 * esz / 16; ++v)
                  reinterpret_cast<uint4 *>(dst)[v] = reinterpret_cast<const uint4 *>(src)[v];
              } else {
                for (int b = 0; b < 32 * esz; b += 2)
                  *reinterpret_cast<uint16_t *>(dst + b) = *reinterpret_cast<const uint16_t *>(src + b);
              }
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
      if (++buf == 2) {
        buf = 0;
        bphase ^= 1u;
      }
    }
    if (trace && wid == 2 && lane == 0) trace[4] = static_cast<int64_t>(globaltimer_ns());
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

constexpr int kStGate = 6;

// Split count of the gate along H: enough (m, n, split) tiles to cover the SMs,
// each split a whole number of 64-wide K blocks.
int tc_gate_splits(const Dims &d) {
  const int tiles_mn = ((d.E + BM - 1) / BM) * ((d.n_pos + kTnGate - 1) / kTnGate);
  const int kb = d.H / BK;
  int target = num_sms() / (tiles_mn > 0 ? tiles_mn : 1);
  if (target < 1) target = 1;
  if (target > 16) target = 16;
  int sk = 1;
  for (int c = 1; c <= target; ++c)
    if (kb % c == 0) sk = c;
  return sk;
}

template <int MODE, int TN, int STAGES>
static cudaError_t launch_tc(const TcParams &p, int grid, cudaStream_t s) {
  using C = Cfg<MODE, TN, STAGES>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e =
        cudaFuncSetAttribute(k_tc_gemm<MODE, TN, STAGES>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e == cudaSuccess) e = prefer_max_shared(k_tc_gemm<MODE, TN, STAGES>);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  k_tc_gemm<MODE, TN, STAGES><<<grid, 192, C::SMEM, s>>>(p);
  return cudaGetLastError();
}

static void base_params(TcParams &p, const Dims &d, const Work &ws) {
  memset(&p, 0, sizeof(p));
  p.d = d;
  p.ws = ws;
}

cudaError_t launch_gate_tc(const Dims &d, const Maps &m, const Work &ws, const CUtensorMap &x_map,
                           cudaStream_t s) {
  TcParams p;
  base_params(p, d, ws);
  p.a0 = m.w_router;
  p.b[0] = x_map;
  const int tiles = ((d.E + BM - 1) / BM) * ((d.n_pos + kTnGate - 1) / kTnGate) * d.SK;
  p.gate_tiles = tiles;
  const int grid = tiles < num_sms() ? tiles : num_sms();
  return launch_tc<M_GATE, kTnGate, kStGate>(p, grid, s);
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
  // every CTA must be resident: down tiles wait for up tiles of other CTAs
  void *args[] = {&p};
  return cudaLaunchCooperativeKernel(reinterpret_cast<void *>(k_tc_experts), dim3(num_sms()), dim3(192), args,
                                     kExpSmem, s);
}

}  // namespace epoch

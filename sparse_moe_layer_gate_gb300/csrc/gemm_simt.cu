// SwiGLU experts over the worklist for fp32 layers, on the FFMA pipes.
//
// The tensor cores have no fp32-input MMA, and TF32 inputs would not hold the
// 1e-5 relative bar of an fp32 layer, so fp32 layers run these kernels; bf16
// layers use the tcgen05 kernels in gemm_tc.cu. Each expert runs once over its
// compact rows ("light-traffic expert kernel", walk-through page
// "Epoch 完全拆解:把扩散块编译成稀疏 MoE 服务单元", section "FreshLane Dispatch").
//
// Rows: [0, L) are worklist edges (expert from the offsets, token row of x
// from the worklist position), then n_shared blocks of n_pos rows for the
// shared experts over every position.
#include "common.cuh"
#include "layer.h"

namespace epoch {

__device__ __forceinline__ int expert_of_row(const int32_t *__restrict__ offsets, int E, int r) {
  int lo = 0, hi = E;  // offsets[lo] <= r < offsets[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (offsets[mid] <= r) lo = mid;
    else hi = mid;
  }
  return lo;
}

// A[row] = silu(W_gate x) * (W_up x); one CTA per row, one warp per output column.
__global__ void __launch_bounds__(256) k_up_simt(Dims d, Weights w, Work ws, const float *__restrict__ x) {
  extern __shared__ float xs[];
  const int L = ws.ctrl->n_edges;
  const int rows = L + d.n_sh * d.n_pos;
  const int lane = lane_id(), wid = warp_id(), nw = blockDim.x >> 5;
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const float *src;
    const float *wg;
    const float *wu;
    float *dst;
    int inter;
    if (r < L) {
      const int e = expert_of_row(ws.offsets, d.E, r);
      int tp = ws.wl_pos[r];  // worklist row r is fresh position tp
      if (tp < 0 || tp >= d.n_pos) {
        if (threadIdx.x == 0) set_error(ws.err, EPOCH_DEVERR_BOUNDS);
        tp = 0;
      }
      src = x + static_cast<size_t>(tp) * d.H;
      wg = static_cast<const float *>(w.w_gate) + static_cast<size_t>(e) * d.I * d.H;
      wu = static_cast<const float *>(w.w_up) + static_cast<size_t>(e) * d.I * d.H;
      dst = static_cast<float *>(ws.a_int) + static_cast<size_t>(r) * d.I;
      inter = d.I;
    } else {
      const int s = (r - L) / d.n_pos, t = (r - L) % d.n_pos;
      src = x + static_cast<size_t>(t) * d.H;
      wg = static_cast<const float *>(w.ws_gate) + static_cast<size_t>(s) * d.I_s * d.H;
      wu = static_cast<const float *>(w.ws_up) + static_cast<size_t>(s) * d.I_s * d.H;
      dst = static_cast<float *>(ws.a_sh) + (static_cast<size_t>(s) * d.Nmax + t) * d.I_s;
      inter = d.I_s;
    }
    __syncthreads();
    for (int h = threadIdx.x; h < d.H; h += blockDim.x) xs[h] = src[h];
    __syncthreads();
    for (int i = wid; i < inter; i += nw) {
      const float *gr = wg + static_cast<size_t>(i) * d.H;
      const float *ur = wu + static_cast<size_t>(i) * d.H;
      float g = 0.f, u = 0.f;
      for (int h = lane; h < d.H; h += 32) {
        g = fmaf(xs[h], gr[h], g);
        u = fmaf(xs[h], ur[h], u);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        g += __shfl_xor_sync(0xffffffffu, g, o);
        u += __shfl_xor_sync(0xffffffffu, u, o);
      }
      if (lane == 0) dst[i] = silu(g) * u;
    }
  }
}

// O[row] = W_down a; one CTA per row, one warp per output element.
__global__ void __launch_bounds__(256) k_down_simt(Dims d, Weights w, Work ws) {
  extern __shared__ float as[];
  const int L = ws.ctrl->n_edges;
  const int rows = L + d.n_sh * d.n_pos;
  const int lane = lane_id(), wid = warp_id(), nw = blockDim.x >> 5;
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const float *src;
    const float *wd;
    float *dst;
    int inter;
    if (r < L) {
      const int e = expert_of_row(ws.offsets, d.E, r);
      src = static_cast<const float *>(ws.a_int) + static_cast<size_t>(r) * d.I;
      wd = static_cast<const float *>(w.w_down) + static_cast<size_t>(e) * d.H * d.I;
      dst = static_cast<float *>(ws.o_int) + static_cast<size_t>(r) * d.H;
      inter = d.I;
    } else {
      const int s = (r - L) / d.n_pos, t = (r - L) % d.n_pos;
      src = static_cast<const float *>(ws.a_sh) + (static_cast<size_t>(s) * d.Nmax + t) * d.I_s;
      wd = static_cast<const float *>(w.ws_down) + static_cast<size_t>(s) * d.H * d.I_s;
      dst = static_cast<float *>(ws.o_sh) + (static_cast<size_t>(s) * d.Nmax + t) * d.H;
      inter = d.I_s;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < inter; i += blockDim.x) as[i] = src[i];
    __syncthreads();
    for (int h = wid; h < d.H; h += nw) {
      const float *dr = wd + static_cast<size_t>(h) * inter;
      float o = 0.f;
      for (int i = lane; i < inter; i += 32) o = fmaf(as[i], dr[i], o);
#pragma unroll
      for (int q = 16; q > 0; q >>= 1) o += __shfl_xor_sync(0xffffffffu, o, q);
      if (lane == 0) dst[h] = o;
    }
  }
}

cudaError_t launch_up_simt(const Dims &d, const Weights &w, const Work &ws, const void *x, cudaStream_t s) {
  const int blocks = 2 * num_sms();
  static bool carve_ = (prefer_max_shared(k_up_simt) == cudaSuccess);
  (void)carve_;
  k_up_simt<<<blocks, 256, d.H * sizeof(float), s>>>(d, w, ws, static_cast<const float *>(x));
  return cudaGetLastError();
}

cudaError_t launch_down_simt(const Dims &d, const Weights &w, const Work &ws, cudaStream_t s) {
  const int blocks = 2 * num_sms();
  const int inter = d.I > d.I_s ? d.I : d.I_s;
  static bool carve_ = (prefer_max_shared(k_down_simt) == cudaSuccess);
  (void)carve_;
  k_down_simt<<<blocks, 256, inter * sizeof(float), s>>>(d, w, ws);
  return cudaGetLastError();
}

}  // namespace epoch

// Block planner that allocates nothing: epoch_plan_support_noalloc.
//
// Some callers cannot allocate device memory at the point where they plan a
// block: code running while a CUDA graph is being captured into a fixed memory
// pool, allocator-free inference runtimes that hand the library only the
// buffers of a pre-planned arena, or real-time serving loops that forbid
// cudaMalloc (it may synchronise the device) between requests. They also may
// not want to keep a whole epoch_layer workspace for a one-off plan. This file
// gives them the block planner (dense top-k hit counts -> coverage support)
// over logits they already hold, with its only scratch -- the per-expert hit
// counts -- in a fixed file-scope device array instead of caller memory.
//
// The scratch array is shared by every call in the process on a device: calls
// that overlap on the GPU (different streams without ordering) race on it and
// produce wrong supports; serialise them. Each call clears the counts it uses
// before counting. The array lives on every GPU that loads the library, for
// the life of the process (kNoAllocMaxExperts * 4 bytes).
//
// Both routers of the layer are covered: the softmax router ranks the logits
// as given (bias included), the group-limited sigmoid router ranks
// sigmoid(G) + b within the chosen groups, exactly as epoch_plan_block counts.
#include <cmath>
#include <mutex>

#include "common.cuh"
#include "layer.h"
#include "topk.cuh"

namespace epoch {

constexpr int kNoAllocMaxExperts = 1024;
constexpr int kNoAllocMaxPositions = 1 << 26;  // keeps n_pos * top_k and every count within int32
constexpr int kNoAllocMaxDevices = 64;

// Hit counts of the planner, one per expert.
static __device__ __align__(256) int32_t g_noalloc_counts[kNoAllocMaxExperts];

// Device address of g_noalloc_counts on the current device, through
// cudaGetSymbolAddress; host code must never pass the symbol itself to a
// kernel (in host code it names a host-side stand-in). The address is looked
// up again on every call made outside stream capture (so a new primary context
// after a device reset is picked up); a call under capture uses the address
// of the last uncaptured call on that device, hence the first call on a device
// must come before any capture.
static int32_t *counts_address(int device, bool capturing, cudaError_t *err) {
  static std::mutex mu;
  static int32_t *addr[kNoAllocMaxDevices] = {};
  std::lock_guard<std::mutex> lock(mu);
  if (addr[device] == nullptr || !capturing) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_counts);
    if (e != cudaSuccess) {
      *err = e;
      return nullptr;
    }
    addr[device] = static_cast<int32_t *>(p);
  }
  *err = cudaSuccess;
  return addr[device];
}

// Dense top-k of every position over all E experts (the router's rule with
// every expert eligible); one warp per position.
template <int EPL>
__global__ void k_noalloc_topk(const float *__restrict__ logits, int n_pos, int E, int k, int router,
                               const float *__restrict__ bias, int n_group, int topk_group, int32_t *counts) {
  __shared__ uint2 s_scr[8][32];  // top-k scratch of each warp (256 threads)
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int lane = lane_id();
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < n_pos; t += warps) {
    float v[EPL];
    bool ok[EPL];
    lane_logits<EPL>(logits + static_cast<size_t>(t) * E, E, v);
#pragma unroll
    for (int c = 0; c < EPL; ++c) ok[c] = lane * EPL + c < E;
    int sel;
    float val;
    if (router != 0) {  // selection scores sigmoid(G) + b, within the chosen groups
#pragma unroll
      for (int c = 0; c < EPL; ++c) {
        const int e = lane * EPL + c;
        v[c] = e < E ? 1.f / (1.f + expf(-v[c])) + bias[e] : -INFINITY;
      }
      warp_group_limit<EPL>(v, ok, E, n_group, topk_group, k);
    }
    warp_topk<EPL>(v, ok, k, &sel, &val, s_scr[warp_id()]);
    if (lane < k && sel >= 0) atomicAdd(&counts[sel], 1);
  }
}

// One CTA: experts ranked by (count desc, id asc); the support is the
// smallest prefix whose counts reach `threshold` (at least k; every expert
// when all_experts).
__global__ void __launch_bounds__(1024) k_noalloc_support(const int32_t *__restrict__ counts, int E, int k,
                                                          int32_t threshold, int all_experts, int32_t *support_ids,
                                                          int32_t *support_len) {
  __shared__ int32_t cnt[kNoAllocMaxExperts];
  __shared__ int32_t csum[kNoAllocMaxExperts];
  __shared__ int32_t len_s;
  const int tid = threadIdx.x;
  if (tid < E) cnt[tid] = counts[tid];
  if (tid == 0) len_s = E;
  __syncthreads();
  if (tid < E) {
    const int c = cnt[tid];
    int rank = 0;
    for (int e = 0; e < E; ++e) rank += (cnt[e] > c) || (cnt[e] == c && e < tid);
    support_ids[rank] = tid;
    csum[rank] = c;
  }
  __syncthreads();
  for (int off = 1; off < E; off <<= 1) {
    int add = 0;
    if (tid < E && tid >= off) add = csum[tid - off];
    __syncthreads();
    if (tid < E) csum[tid] += add;
    __syncthreads();
  }
  if (!all_experts && tid < E && csum[tid] >= threshold && (tid == 0 || csum[tid - 1] < threshold)) len_s = tid + 1;
  __syncthreads();
  if (tid == 0) *support_len = min(max(len_s, k), E);
}

static int epl_noalloc(int E) {
  const int epl = (E + 31) / 32;
  return epl <= 1 ? 1 : epl <= 2 ? 2 : epl <= 4 ? 4 : epl <= 8 ? 8 : epl <= 16 ? 16 : 32;
}

}  // namespace epoch

using namespace epoch;

extern "C" epoch_status epoch_plan_support_noalloc(const float *logits_dev, int32_t n_pos, int32_t n_experts,
                                                   int32_t top_k, double tau, int32_t router, const float *bias_dev,
                                                   int32_t n_group, int32_t topk_group, int32_t *support_ids_dev,
                                                   int32_t *support_len_dev, epoch_stream stream) {
  if (logits_dev == nullptr || support_ids_dev == nullptr || support_len_dev == nullptr) return EPOCH_EINVAL;
  if (n_pos < 1 || n_pos > kNoAllocMaxPositions || n_experts < 1 || n_experts > kNoAllocMaxExperts)
    return EPOCH_EINVAL;
  if (top_k < 1 || top_k > 16 || top_k > n_experts || !(tau > 0.0 && tau <= 1.0)) return EPOCH_EINVAL;
  if ((reinterpret_cast<uintptr_t>(logits_dev) & 15u) != 0) return EPOCH_EINVAL;
  if (router != EPOCH_ROUTER_SOFTMAX && router != EPOCH_ROUTER_SIGMOID_GROUP) return EPOCH_EINVAL;
  if (router == EPOCH_ROUTER_SIGMOID_GROUP &&
      (bias_dev == nullptr || n_group < 1 || n_group > 32 || n_experts % n_group || topk_group < 1 ||
       topk_group > n_group))
    return EPOCH_EINVAL;
  int device = 0;
  if (cudaGetDevice(&device) != cudaSuccess || device < 0 || device >= kNoAllocMaxDevices) return EPOCH_ECUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return EPOCH_ECUDA;
  cudaError_t e;
  int32_t *counts = counts_address(device, cap != cudaStreamCaptureStatusNone, &e);
  if (counts == nullptr) return EPOCH_ECUDA;
  if (cudaMemsetAsync(counts, 0, sizeof(int32_t) * n_experts, s) != cudaSuccess) return EPOCH_ECUDA;
  int blocks = (n_pos + 7) / 8;
  if (blocks > 8 * num_sms()) blocks = 8 * num_sms();
  const int ng = router ? n_group : 1, tg = router ? topk_group : 1;
  switch (epl_noalloc(n_experts)) {
#define EPOCH_CASE(N)                                                                                     \
  case N:                                                                                                 \
    k_noalloc_topk<N><<<blocks, 256, 0, s>>>(logits_dev, n_pos, n_experts, top_k, router, bias_dev, ng, tg, \
                                             counts);                                                     \
    break;
    EPOCH_CASE(1) EPOCH_CASE(2) EPOCH_CASE(4) EPOCH_CASE(8) EPOCH_CASE(16) EPOCH_CASE(32)
#undef EPOCH_CASE
  }
  if (cudaGetLastError() != cudaSuccess) return EPOCH_ECUDA;
  const int all = tau >= 1.0;
  // ceil(tau * (n_pos * top_k)) in float64, the edge count formed exactly first
  // (n_pos * top_k <= 2^30), the same order of operations as the layer's planner
  const int64_t edges = static_cast<int64_t>(n_pos) * top_k;
  const int32_t threshold = static_cast<int32_t>(std::ceil(tau * static_cast<double>(edges)));
  k_noalloc_support<<<1, 1024, 0, s>>>(counts, n_experts, top_k, threshold, all, support_ids_dev, support_len_dev);
  return cudaGetLastError() == cudaSuccess ? EPOCH_OK : EPOCH_ECUDA;
}

// Batch-level budget (global top-N of prefix confidences, prefix-closed) and the serial cut
// with the chosen depths.  One warp per request; every CTA rebuilds the confidence table.
#include "spec_device.cuh"

namespace sv {

constexpr int kBudgetThreads = 1024;

// key (c2, m2, b2) precedes key (c, m, b): c descending, then m ascending, then b ascending
__device__ __forceinline__ bool precedes(float c2, int m2, int b2, float c, int m, int b) {
  return c2 > c || (c2 == c && (m2 < m || (m2 == m && b2 < b)));
}

__global__ void __launch_bounds__(kBudgetThreads) budget_cut_kernel(const __grid_constant__ BudgetParams P) {
  extern __shared__ float conf[];   // [B, K] prefix confidences
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the row kernel's records are complete
  const int B = P.B, K = P.K;
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    float cp = 1.f;
    for (int k = 0; k < K; ++k) {
      const float a = P.alpha_in ? P.alpha_in[static_cast<size_t>(b) * K + k]
                                 : __ldcg(&P.recs[static_cast<size_t>(b) * P.U + k].alpha);
      cp *= fminf(fmaxf(a, 0.f), 1.f);          // NaN -> 0
      conf[b * K + k] = cp;
    }
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * (kBudgetThreads / 32) + warp;
  if (b >= B) return;

  // rank of key (b, m) in the total order; within each request b' the preceding keys form a
  // prefix (conf is non-increasing in m'), found by binary search; lanes split the requests.
  auto rank_of = [&](int m) {
    const float cv = conf[b * K + m];
    int cnt = 0;
    for (int bp = lane; bp < B; bp += 32) {
      int lo = 0, hi = K;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (precedes(conf[bp * K + mid], mid, bp, cv, m, b)) lo = mid + 1; else hi = mid;
      }
      cnt += lo;
    }
    return warp_sum_int(cnt);
  };
  // d_b = number of m whose key ranks below N (a prefix of m)
  int lo = 0, hi = K;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (rank_of(mid) < P.N) lo = mid + 1; else hi = mid;
  }
  const int d = lo;
  if (P.out_depth && lane == 0) P.out_depth[b] = d;
  if (P.out_conf)
    for (int k = lane; k < K; k += 32) P.out_conf[static_cast<size_t>(b) * K + k] = conf[b * K + k];
  if (P.do_cut)
    cut_request(b, d, P.greedy != 0, P.stats_only != 0, P.recs, P.U, K, P.V, P.tokens, P.uniforms,
                P.out_tokens, P.out_accepted, P.out_alpha, P.out_cum, P.out_E, P.status, lane);
}

// Serial cut only (no budget): one warp per request, depth from the caller or K.
constexpr int kCutThreads = 128;
__global__ void __launch_bounds__(kCutThreads) cut_kernel(const __grid_constant__ BudgetParams P,
                                                          const int32_t* depth) {
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the row kernel's records are complete
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * (kCutThreads / 32) + warp;
  if (b >= P.B) return;
  const int d = depth ? min(max(depth[b], 0), P.K) : P.K;
  cut_request(b, d, P.greedy != 0, P.stats_only != 0, P.recs, P.U, P.K, P.V, P.tokens, P.uniforms,
              P.out_tokens, P.out_accepted, P.out_alpha, P.out_cum, P.out_E, P.status, lane);
}

// Launch chained to the previous kernel on the stream (programmatic dependent launch): the
// grid may start while the previous one drains and waits for it in griddepcontrol.wait.
static cudaError_t launch_pdl(const void* fn, int grid, int block, size_t smem, cudaStream_t stream,
                              void** args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_budget_cut(const BudgetParams& p, cudaStream_t stream) {
  const int per = kBudgetThreads / 32;
  const int grid = (p.B + per - 1) / per;
  const size_t smem = static_cast<size_t>(p.B) * p.K * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(budget_cut_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  BudgetParams q = p;
  void* args[] = {&q};
  return launch_pdl(reinterpret_cast<const void*>(&budget_cut_kernel), grid, kBudgetThreads, smem, stream, args);
}

cudaError_t launch_cut(const BudgetParams& p, const int32_t* depth, cudaStream_t stream) {
  const int per = kCutThreads / 32;
  const int grid = (p.B + per - 1) / per;
  BudgetParams q = p;
  const int32_t* d = depth;
  void* args[] = {&q, &d};
  return launch_pdl(reinterpret_cast<const void*>(&cut_kernel), grid, kCutThreads, 0, stream, args);
}

}  // namespace sv

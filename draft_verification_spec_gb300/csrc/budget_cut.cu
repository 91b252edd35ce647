// The small kernels chained after the row kernel:
//  * cut_kernel: the serial first-rejection cut of each request (one warp per request);
//  * budget_cut_kernel: the batch-level budget -- the global top-N of prefix confidences
//    prod_{k<=m} alpha_k, prefix-closed per request -- then the cut at the chosen depths.
// Both start with griddepcontrol.wait, so they may be scheduled while the row kernel drains.
#include "argmax_kernel.cuh"
#include "cut_sampling.cuh"
#include "spec_device.cuh"

namespace sv {

constexpr int kBudgetThreads = 512;
constexpr int kCutThreads = 128;

// key (c2, m2, b2) precedes key (c, m, b): c descending, then m ascending, then b ascending
__device__ __forceinline__ bool precedes(float c2, int m2, int b2, float c, int m, int b) {
  return c2 > c || (c2 == c && (m2 < m || (m2 == m && b2 < b)));
}

__device__ __forceinline__ float alpha_of(const BudgetParams& P, int b, int k) {
  if (P.alpha_in) return P.alpha_in[static_cast<size_t>(b) * P.K + k];
  const unsigned long long* kb = reinterpret_cast<const unsigned long long*>(P.keys) +
                                 (static_cast<size_t>(b) * (P.K + 1) + k) * 2;
  return key_index(__ldcg(kb)) == key_index(__ldcg(kb + 1)) ? 1.f : 0.f;
}

// q_k(x_k) of request b from the draft statistics kernel's partials of row (b, k), merged in part
// order: 2^((z_x - M) c) / S, or [x_k == first argmax] at T = 0; 0 for a token outside [0, V).
__device__ __forceinline__ float draft_q(const BudgetParams& P, int b, int k) {
  const size_t r = static_cast<size_t>(b) * P.K + k;
  const int x = P.tokens[r];
  if (x < 0 || x >= P.V) return 0.f;
  const float4* pr = P.draft_part + r * P.nparts;
  float M = ninf();
  for (int j = 0; j < P.nparts; ++j) M = fmaxf(M, __ldcg(&pr[j].x));
  if (P.draft_greedy) {
    unsigned I = 0xffffffffu;
    for (int j = 0; j < P.nparts; ++j)
      if (__ldcg(&pr[j].x) == M) I = min(I, __float_as_uint(__ldcg(&pr[j].z)));
    return static_cast<unsigned>(x) == I ? 1.f : 0.f;
  }
  const float ref = M == ninf() ? 0.f : M;
  float S = 0.f;
  for (int j = 0; j < P.nparts; ++j) S += __ldcg(&pr[j].y) * ex2((__ldcg(&pr[j].x) - ref) * P.c);
  const void* row = static_cast<const uint8_t*>(P.draft) + r * P.V * (P.bf16 ? 2 : 4);
  const float q = ex2((logit_at(row, x, P.bf16 != 0) - ref) * P.c) / S;
  return fminf(fmaxf(q, 0.f), 1.f);   // NaN (a row with no finite logit) -> 0
}

// The cost of verifying n positions: the table interpolated piecewise-linearly, held constant
// beyond its ends.
__device__ __forceinline__ float cost_at(float n, const float* cn, const float* ct, int nc) {
  if (n <= cn[0]) return ct[0];
  if (n >= cn[nc - 1]) return ct[nc - 1];
  int i = 0;
  while (i + 2 < nc && cn[i + 1] <= n) ++i;
  return ct[i] + (ct[i + 1] - ct[i]) * (n - cn[i]) / (cn[i + 1] - cn[i]);
}

// The budget N with the largest expected tokens per unit of verification cost: the first N
// maximising (B + S(N)) / cost(B + N), S(N) the sum of the N largest prefix confidences.  Every
// thread of the CTA calls it and gets the same N (the confidences are sorted in shared memory by
// a bitonic network, descending -- exchange steps with strides of 32 and more through shared
// memory with a barrier each, the shorter ones in registers, a warp per 32 consecutive elements
// exchanging by shuffle -- then one scan).
__device__ int choose_budget(const BudgetParams& P, const float* conf, float* sb, float* cn, float* ct,
                             float* red_u, int* red_n, int* n_out) {
  const int BK = P.B * P.K, tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5;
  const int nw = nt >> 5;
  int n2 = 32;
  while (n2 < BK) n2 <<= 1;
  for (int i = tid; i < n2; i += nt) sb[i] = i < BK ? conf[i] : -1.f;
  for (int i = tid; i < P.n_cost; i += nt) {
    cn[i] = P.cost_n[i];
    ct[i] = P.cost_t[i];
  }
  __syncthreads();
  // the exchange steps of stages kmin .. kmax with strides below 32, in registers
  auto warp_steps = [&](int kmin, int kmax) {
    for (int base = warp * 32; base < n2; base += nw * 32) {
      const int i = base + lane;
      float a = sb[i];
      for (int k = kmin; k <= kmax; k <<= 1)
        for (int j = min(k >> 1, 16); j > 0; j >>= 1) {
          const float bv = __shfl_xor_sync(0xffffffffu, a, j);
          a = (((i & j) == 0) == ((i & k) == 0)) ? fmaxf(a, bv) : fminf(a, bv);   // descending blocks keep the larger first
        }
      sb[i] = a;
    }
    __syncthreads();
  };
  warp_steps(2, 32);
  for (int k = 64; k <= n2; k <<= 1) {
    for (int j = k >> 1; j >= 32; j >>= 1) {
      for (int i = tid; i < n2; i += nt) {
        const int l = i ^ j;
        if (l > i) {
          const float a = sb[i], bv = sb[l];
          if (((i & k) == 0) ? a < bv : a > bv) {
            sb[i] = bv;
            sb[l] = a;
          }
        }
      }
      __syncthreads();
    }
    warp_steps(k, k);
  }
  // S(N): each thread sums a contiguous run of the sorted values; a scan of the runs' totals
  const int per = (BK + nt - 1) / nt;
  const int i0 = min(BK, tid * per), i1 = min(BK, i0 + per);
  float run = 0.f;
  for (int i = i0; i < i1; ++i) run += sb[i];
  const float incl = warp_incl_scan(run, lane);
  if (lane == 31) red_u[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const float t = lane < nw ? red_u[lane] : 0.f;
    const float ti = warp_incl_scan(t, lane);
    if (lane < nw) red_u[lane] = ti - t;
  }
  __syncthreads();
  float S = red_u[warp] + incl - run;
  float bu = ninf();
  int bn = 0x7fffffff;
  auto consider = [&](int N, float SN) {
    const float u = (static_cast<float>(P.B) + SN) / cost_at(static_cast<float>(P.B + N), cn, ct, P.n_cost);
    if (u > bu || (u == bu && N < bn)) {
      bu = u;
      bn = N;
    }
  };
  if (tid == 0) consider(0, 0.f);
  for (int i = i0; i < i1; ++i) {
    S += sb[i];
    consider(i + 1, S);
  }
  // the largest utility, then the smallest N
  for (int o = 16; o; o >>= 1) {
    const float ou = __shfl_xor_sync(0xffffffffu, bu, o);
    const int on = __shfl_xor_sync(0xffffffffu, bn, o);
    if (ou > bu || (ou == bu && on < bn)) {
      bu = ou;
      bn = on;
    }
  }
  __syncthreads();   // every thread is done with the scan offsets in red_u
  if (lane == 0) {
    red_u[warp] = bu;
    red_n[warp] = bn;
  }
  __syncthreads();
  if (tid == 0) {
    float u = red_u[0];
    int n = red_n[0];
    for (int w = 1; w < nw; ++w)
      if (red_u[w] > u || (red_u[w] == u && red_n[w] < n)) {
        u = red_u[w];
        n = red_n[w];
      }
    *n_out = n;
  }
  __syncthreads();
  return *n_out;
}

// One CTA builds the whole confidence table; its warps take requests b = warp, warp + nwarps, ...
// (grid > 1 only when every CTA can rebuild the table from inputs nobody clears).  The tables are
// stored position-major ([K][B]), so lanes that read different requests at one position -- or at
// different positions -- hit different banks.
__global__ void __launch_bounds__(kBudgetThreads) budget_cut_kernel(const __grid_constant__ BudgetParams P) {
  // [K, B] prefix confidences, [K, B] per-position confidences; then, for the utility / cost
  // choice of N, the sort buffer (next power of two >= B K), the cost table and reduction slots
  extern __shared__ float conf[];
  float* const alpha_s = conf + P.B * P.K;
  __shared__ int n_choice;
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the row kernel's results are complete
  const int B = P.B, K = P.K;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  if (P.alpha_in || P.greedy) {
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
      float cp = 1.f;
      for (int k = 0; k < K; ++k) {
        cp *= fminf(fmaxf(alpha_of(P, b, k), 0.f), 1.f);   // clamp; NaN -> 0
        conf[k * B + b] = cp;
      }
    }
  } else {
    // sampling path (alpha from the row records) or draft-side confidences: every row in
    // parallel (a thread per row), then the prefix products
    for (int r = threadIdx.x; r < B * K; r += blockDim.x) {
      const int b = r / K, k = r - b * K;
      alpha_s[k * B + b] = P.draft_part ? draft_q(P, b, k) : alpha_of_row(P, b, k);
    }
    __syncthreads();
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
      float cp = 1.f;
      for (int k = 0; k < K; ++k) {
        cp *= alpha_s[k * B + b];
        conf[k * B + b] = cp;
      }
    }
  }
  __syncthreads();
  int Nsel = P.N;
  if (P.n_cost > 0) {
    int n2 = 32;
    while (n2 < B * K) n2 <<= 1;
    float* const sb = conf + 2 * B * K;
    float* const cn = sb + n2;
    float* const ct = cn + kBudgetMaxCost;
    float* const red_u = ct + kBudgetMaxCost;
    int* const red_n = reinterpret_cast<int*>(red_u + 32);
    Nsel = choose_budget(P, conf, sb, cn, ct, red_u, red_n, &n_choice);
    if (blockIdx.x == 0 && threadIdx.x == 0 && P.out_N) *P.out_N = Nsel;
  }
  for (int b = blockIdx.x * nw + warp; b < B; b += gridDim.x * nw) {
    // rank of key (b, m): within each request b' the keys that precede it form a prefix
    // (conf is non-increasing in m'), found by binary search; lanes split the requests.
    auto rank_of = [&](int m) {
      const float cv = conf[m * B + b];
      int cnt = 0;
      for (int bp = lane; bp < B; bp += 32) {
        int lo = 0, hi = K;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (precedes(conf[mid * B + bp], mid, bp, cv, m, b)) lo = mid + 1; else hi = mid;
        }
        cnt += lo;
      }
      return warp_sum_int(cnt);
    };
    // d_b = number of m whose key ranks below N (a prefix of m)
    int lo = 0, hi = K;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (rank_of(mid) < Nsel) lo = mid + 1; else hi = mid;
    }
    const int d = lo;
    if (P.out_depth && lane == 0) P.out_depth[b] = d;
    if (P.out_conf)
      for (int k = lane; k < K; k += 32) P.out_conf[static_cast<size_t>(b) * K + k] = conf[k * B + b];
    if (P.do_cut) {
      if (P.greedy)
        cut_request(b, d, P.stats_only != 0, P.keys, P.draft_keys != 0, false, P.U, K, P.V, P.tokens,
                    P.out_tokens, P.out_accepted, P.out_alpha, P.out_cum, P.out_E, P.status, lane);
      else
        cut_sampling(P, b, d, lane, true, lane < K ? alpha_s[lane * B + b] : 0.f);
    }
  }
  if (P.greedy && P.keys) {   // every warp of the (single) CTA is done with the keys: clear them
    __syncthreads();
    unsigned long long* k = reinterpret_cast<unsigned long long*>(P.keys);
    for (int i = threadIdx.x; i < B * (K + 1) * 2; i += blockDim.x) k[i] = 0ull;
  }
}

__global__ void __launch_bounds__(kCutThreads) cut_kernel(const __grid_constant__ BudgetParams P,
                                                          const int32_t* depth) {
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the row kernel's results are complete
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x * (kCutThreads / 32) + warp;
  if (b >= P.B) return;
  const int d = depth ? min(max(depth[b], 0), P.K) : P.K;
  if (P.greedy)
    cut_request(b, d, P.stats_only != 0, P.keys, P.draft_keys != 0, true, P.U, P.K, P.V, P.tokens,
                P.out_tokens, P.out_accepted, P.out_alpha, P.out_cum, P.out_E, P.status, lane);
  else
    cut_sampling(P, b, d, lane);
}

// Launch chained to the previous kernel on the stream (programmatic dependent launch): the
// grid may start while the previous one drains and waits for it in griddepcontrol.wait.
static cudaError_t launch_pdl(const void* fn, int grid, int block, size_t smem, cudaStream_t stream,
                              void** args, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t launch_budget_cut(const BudgetParams& p, cudaStream_t stream, bool pdl) {
  const int per = kBudgetThreads / 32;
  // the greedy path clears the keys it reads, so one CTA must own the whole table; otherwise every
  // CTA builds the table and a warp cuts one request
  const int grid = (p.greedy && p.keys) ? 1 : (p.B + per - 1) / per;
  size_t smem = static_cast<size_t>(p.B) * p.K * sizeof(float) * 2;
  if (p.n_cost > 0) {
    size_t n2 = 32;
    while (n2 < static_cast<size_t>(p.B) * p.K) n2 <<= 1;
    smem += (n2 + 2 * kBudgetMaxCost + 64) * sizeof(float);
  }
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(budget_cut_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  BudgetParams q = p;
  void* args[] = {&q};
  return launch_pdl(reinterpret_cast<const void*>(&budget_cut_kernel), grid > 0 ? grid : 1, kBudgetThreads,
                    smem, stream, args, pdl);
}

cudaError_t launch_cut(const BudgetParams& p, const int32_t* depth, cudaStream_t stream, bool pdl) {
  const int per = kCutThreads / 32;
  const int grid = (p.B + per - 1) / per;
  BudgetParams q = p;
  const int32_t* d = depth;
  void* args[] = {&q, &d};
  return launch_pdl(reinterpret_cast<const void*>(&cut_kernel), grid, kCutThreads, 0, stream, args, pdl);
}

cudaError_t argmax_blocks_per_sm(bool bf16, int* out) {
  const void* fn = bf16 ? reinterpret_cast<const void*>(&argmax_kernel<true>)
                        : reinterpret_cast<const void*>(&argmax_kernel<false>);
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(out, fn, 256, 0);
}

cudaError_t launch_argmax(bool bf16, const ArgmaxParams& p, int grid, cudaStream_t stream) {
  ArgmaxParams q = p;
  void* args[] = {&q};
  const void* fn = bf16 ? reinterpret_cast<const void*>(&argmax_kernel<true>)
                        : reinterpret_cast<const void*>(&argmax_kernel<false>);
  // programmatic dependent launch: the grid may be scheduled while the preceding kernel drains;
  // it waits (griddepcontrol.wait) for that kernel's completion before its first memory access
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace sv

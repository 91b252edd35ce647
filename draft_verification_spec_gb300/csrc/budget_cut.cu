// The small kernels chained after the row kernel:
//  * cut_kernel: the serial first-rejection cut of each request (one warp per request);
//  * budget_cut_kernel: the batch-level budget -- the global top-N of prefix confidences
//    prod_{k<=m} alpha_k, prefix-closed per request -- then the cut at the chosen depths.
// Both wait (griddepcontrol.wait) for the preceding kernel before they read its results, so they
// may be scheduled while it drains.
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

// The draft-side confidence q_k(x_k) of row r = b K + k, in two halves.  What comes from the
// caller -- the token and the draft logit at it -- is read first; then the statistics kernel's
// partials of the row are merged in part order into 2^((z_x - M) c) / S, or [x_k == first argmax]
// at T = 0.  A token outside [0, V) has confidence 0.
struct DraftPick {
  int x;     // the token, or -1 when it lies outside [0, V)
  float z;   // its draft logit (T > 0)
};

__device__ __forceinline__ DraftPick draft_pick(const BudgetParams& P, int r) {
  DraftPick d{P.tokens[r], 0.f};
  if (d.x < 0 || d.x >= P.V) {
    d.x = -1;
  } else if (!P.draft_greedy) {
    const void* row = static_cast<const uint8_t*>(P.draft) + static_cast<size_t>(r) * P.V * (P.bf16 ? 2 : 4);
    d.z = logit_at(row, d.x, P.bf16 != 0);
  }
  return d;
}

__device__ __forceinline__ float draft_q(const BudgetParams& P, int r, DraftPick d) {
  if (d.x < 0) return 0.f;
  const float4* pr = P.draft_part + static_cast<size_t>(r) * P.nparts;
  if (P.draft_greedy) {
    // the parts cover increasing index ranges: the first part with the row maximum holds the
    // first argmax (a part of -inf logits reports no index)
    float M = ninf();
    unsigned I = 0xffffffffu;
#pragma unroll 4
    for (int j = 0; j < P.nparts; ++j) {
      const float4 v = __ldcg(pr + j);
      if (v.x > M) {
        M = v.x;
        I = __float_as_uint(v.z);
      }
    }
    return static_cast<unsigned>(d.x) == I ? 1.f : 0.f;
  }
  // online (max, sum): the running sum is rescaled to each new maximum (reference 0 while every
  // logit so far is -inf)
  float M = ninf(), S = 0.f;
#pragma unroll 4
  for (int j = 0; j < P.nparts; ++j) {
    const float4 v = __ldcg(pr + j);
    const float nm = fmaxf(M, v.x);
    const float ref = nm == ninf() ? 0.f : nm;
    S = S * ex2((M - ref) * P.c) + v.y * ex2((v.x - ref) * P.c);
    M = nm;
  }
  const float ref = M == ninf() ? 0.f : M;
  const float q = ex2((d.z - ref) * P.c) / S;
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

// Bitonic sort, descending, of n2 confidences (a power of two, at least 32) by the first ts = n2 / E
// threads of the CTA, E values each: thread t holds positions t E .. t E + E - 1.  The exchange
// steps of stride j run inside a thread below E, between the lanes of a warp by shuffle below 32 E,
// and between threads through the exchange area xb (two halves of n2 values, used in turn, so one
// barrier -- named, over the ts sorting threads -- a step) from 32 E up.
template <int E>
__device__ void sort_desc(float (&v)[E], int n2, int ts, float* xb) {
  const int tid = threadIdx.x;
  int half = 0;
  for (int k = 2; k <= n2; k <<= 1) {
    for (int j = k >> 1; j >= 32 * E; j >>= 1) {
      float* const x = xb + half * n2;
#pragma unroll
      for (int e = 0; e < E; ++e) x[e * ts + tid] = v[e];
      asm volatile("bar.sync 1, %0;" ::"r"(ts) : "memory");
      const int partner = tid ^ (j / E);
      const bool keep_max = (((tid * E) & j) == 0) == (((tid * E) & k) == 0);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float o = x[e * ts + partner];
        v[e] = keep_max ? fmaxf(v[e], o) : fminf(v[e], o);
      }
      half ^= 1;
    }
    for (int j = min(k >> 1, 16 * E); j >= E; j >>= 1) {
      const bool keep_max = (((tid * E) & j) == 0) == (((tid * E) & k) == 0);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float o = __shfl_xor_sync(0xffffffffu, v[e], j / E);
        v[e] = keep_max ? fmaxf(v[e], o) : fminf(v[e], o);
      }
    }
#pragma unroll
    for (int j = E / 2; j >= 1; j >>= 1) {
      if (j < k) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if ((e & j) == 0) {
            const float a = v[e], b = v[e | j];
            const bool desc = ((tid * E + e) & k) == 0;   // this block of the stage runs descending
            v[e] = desc ? fmaxf(a, b) : fminf(a, b);
            v[e | j] = desc ? fminf(a, b) : fmaxf(a, b);
          }
        }
      }
    }
  }
}

// Shared scratch of the choice of N: the cost table, scan and reduction slots, the results.
struct BudgetShared {
  float cn[kBudgetMaxCost], ct[kBudgetMaxCost];
  float run[32], offset[32], best_u[32];
  int best_n[32], ties[32], tie_off[32], above[32];
  int n, above_all, r_last;
};

__device__ __forceinline__ int warp_incl_scan_int(int v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// The budget N with the largest expected tokens per unit of verification cost: the first N
// maximising (B + S(N)) / cost(B + N), S(N) the sum of the N largest prefix confidences, from the
// sorted confidences srt (one scan, each thread over a contiguous run).  Every thread gets N.
__device__ int choose_budget(const BudgetParams& P, const float* srt, BudgetShared& sh) {
  const int BK = P.B * P.K, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int per = (BK + blockDim.x - 1) / blockDim.x;
  const int i0 = min(BK, tid * per), i1 = min(BK, i0 + per);
  float run = 0.f;
  for (int i = i0; i < i1; ++i) run += srt[i];
  const float incl = warp_incl_scan(run, lane);
  if (lane == 31) sh.run[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    const float t = lane < nw ? sh.run[lane] : 0.f;
    const float ti = warp_incl_scan(t, lane);
    if (lane < nw) sh.offset[lane] = ti - t;
  }
  __syncthreads();
  float S = sh.offset[warp] + incl - run;
  float bu = ninf();
  int bn = 0x7fffffff;
  auto consider = [&](int N, float SN) {
    const float u = (static_cast<float>(P.B) + SN) / cost_at(static_cast<float>(P.B + N), sh.cn, sh.ct, P.n_cost);
    if (u > bu || (u == bu && N < bn)) {
      bu = u;
      bn = N;
    }
  };
  if (tid == 0) consider(0, 0.f);
  for (int i = i0; i < i1; ++i) {
    S += srt[i];
    consider(i + 1, S);
  }
  // the largest utility, then the smallest N
  auto fold = [&]() {
    for (int o = 16; o; o >>= 1) {
      const float ou = __shfl_xor_sync(0xffffffffu, bu, o);
      const int on = __shfl_xor_sync(0xffffffffu, bn, o);
      if (ou > bu || (ou == bu && on < bn)) {
        bu = ou;
        bn = on;
      }
    }
  };
  fold();
  if (lane == 0) {
    sh.best_u[warp] = bu;
    sh.best_n[warp] = bn;
  }
  __syncthreads();
  if (warp == 0) {
    bu = lane < nw ? sh.best_u[lane] : ninf();
    bn = lane < nw ? sh.best_n[lane] : 0x7fffffff;
    fold();
    if (lane == 0) sh.n = bn;
  }
  __syncthreads();
  return sh.n;
}

// The last key the budget takes, in its order (c descending, then m ascending, then b ascending,
// i.e. r = m B + b ascending): key (b, m) is taken when c(b, m) > c_last, or c(b, m) == c_last and
// m B + b <= r_last.
struct BudgetCut {
  float c_last;
  int r_last;
};

// The utility / cost choice of N over the [K, B] table `conf`, and the cut of the first N keys:
// the confidences sorted (one bitonic sort by the first n2 / E threads), S(N) and the first
// maximum of U(N); c_last is then the N-th largest confidence, and of the ties at c_last the
// first N - #{c > c_last} in increasing r are taken (one block count and scan).  All keys for
// N >= B K, none for N = 0.  Writes N to *n_out.
template <int E>
__device__ BudgetCut adaptive_cut(const BudgetParams& P, const float* conf, int n2, float* xb, BudgetShared& sh,
                                  int* n_out) {
  const int BK = P.B * P.K, tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  const int ts = n2 / E;
  float* const srt = xb + 2 * n2;   // the sorted confidences, descending
  if (tid < ts) {
    float v[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {   // any start placement will do: lanes read consecutive words
      const int r = e * ts + tid;
      v[e] = r < BK ? conf[r] : -1.f;   // padding below every confidence (all >= 0)
    }
    sort_desc<E>(v, n2, ts, xb);
#pragma unroll
    for (int e = 0; e < E; ++e) srt[tid * E + e] = v[e];
  }
  __syncthreads();
  const int N = choose_budget(P, srt, sh);
  *n_out = N;
  if (N <= 0) return BudgetCut{2.f, -1};
  if (N >= BK) return BudgetCut{-1.f, -1};
  const float cl = srt[N - 1];
  // each thread counts a contiguous run of positions: above c_last, and ties with it
  const int per = (BK + nt - 1) / nt;
  const int r0 = min(BK, tid * per), r1 = min(BK, r0 + per);
  int above = 0, ties = 0;
  for (int r = r0; r < r1; ++r) {
    const float c = conf[r];
    above += c > cl;
    ties += c == cl;
  }
  const int ties_incl = warp_incl_scan_int(ties, lane);
  const int above_w = warp_sum_int(above);
  if (lane == 31) sh.ties[warp] = ties_incl;
  if (lane == 0) sh.above[warp] = above_w;
  __syncthreads();
  if (warp == 0) {
    const int t = lane < nw ? sh.ties[lane] : 0;
    const int ti = warp_incl_scan_int(t, lane);
    if (lane < nw) sh.tie_off[lane] = ti - t;
    const int a = warp_sum_int(lane < nw ? sh.above[lane] : 0);
    if (lane == 0) sh.above_all = a;
  }
  __syncthreads();
  const int want = N - sh.above_all;   // ties taken: at least 1, at most the ties there are
  int seen = sh.tie_off[warp] + ties_incl - ties;
  if (seen < want && seen + ties >= want) {
    for (int r = r0; r < r1; ++r)
      if (conf[r] == cl && ++seen == want) {
        sh.r_last = r;
        break;
      }
  }
  __syncthreads();
  return BudgetCut{cl, sh.r_last};
}

// Values per sorting thread of the choice of N: n2 / 256 within [1, 16] (at most 256 sorting threads
// up to n2 = 4096; fewer threads with more values each issue fewer instructions a step).
__host__ __device__ constexpr int budget_values_per_thread(int n2) {
  return n2 <= 256 ? 1 : (n2 / 256 > 16 ? 16 : n2 / 256);
}

// One CTA builds the whole confidence table; its warps take requests b = warp, warp + nwarps, ...
// (grid > 1 only when every CTA can rebuild the table from inputs nobody clears).  The tables are
// stored position-major ([K][B]), so lanes that read different requests at one position -- or at
// different positions -- hit different banks.
__global__ void __launch_bounds__(kBudgetThreads) budget_cut_kernel(const __grid_constant__ BudgetParams P) {
  // [K, B] prefix confidences, [K, B] per-position confidences, [K, B] accept-test failures (one
  // byte each, sampling path), then for the choice of N the sort's exchange area (2 n2 floats) and
  // the sorted confidences (n2 floats)
  extern __shared__ __align__(16) float conf[];
  __shared__ BudgetShared sh;
  const int B = P.B, K = P.K, BK = B * K;
  float* const alpha_s = conf + BK;
  uint8_t* const rej_s = reinterpret_cast<uint8_t*>(conf + 2 * BK);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  auto load_costs = [&]() {
    for (int i = threadIdx.x; i < P.n_cost; i += blockDim.x) {
      sh.cn[i] = P.cost_n[i];
      sh.ct[i] = P.cost_t[i];
    }
  };
  // The draft-side budget runs after the statistics kernel, which starts only once the caller's
  // work is complete: the tokens, the draft logits and the cost table are read before the wait
  // for that kernel's partials.
  constexpr int kEarlyRows = 4;
  DraftPick pick[kEarlyRows];
  if (P.draft_part) {
    load_costs();
#pragma unroll
    for (int j = 0; j < kEarlyRows; ++j) {
      const int r = threadIdx.x + j * blockDim.x;
      pick[j] = r < BK ? draft_pick(P, r) : DraftPick{-1, 0.f};
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the preceding kernel's results are complete
  if (!P.draft_part) load_costs();
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
    // parallel (a thread per row r = b K + k), then the prefix products
    if (P.draft_part) {
#pragma unroll
      for (int j = 0; j < kEarlyRows; ++j) {
        const int r = threadIdx.x + j * blockDim.x;
        if (r < BK) {
          const int b = r / K, k = r - b * K;
          alpha_s[k * B + b] = draft_q(P, r, pick[j]);
        }
      }
      for (int r = threadIdx.x + kEarlyRows * blockDim.x; r < BK; r += blockDim.x) {
        const int b = r / K, k = r - b * K;
        alpha_s[k * B + b] = draft_q(P, r, draft_pick(P, r));
      }
    } else {
      // each row's alpha, and the outcome of its accept test as the row kernel evaluated it (the
      // cuts read it from shared memory): the record's second 16-byte word, (mode, alpha, rej, -)
      for (int r = threadIdx.x; r < BK; r += blockDim.x) {
        const int b = r / K, k = r - b * K;
        const float4 w = __ldcg(reinterpret_cast<const float4*>(P.recs + static_cast<size_t>(b) * P.U + k) + 1);
        alpha_s[k * B + b] = w.y;
        rej_s[k * B + b] = __float_as_int(w.z) != 0 ? 1 : 0;
      }
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
  // with N chosen by utility / cost the keys are sorted anyway, and the cut of the first N comes
  // from the sorted order; with a given N, each request ranks its own keys (below)
  int Nsel = P.N;
  BudgetCut cut = {0.f, 0};
  if (P.n_cost > 0) {
    int n2 = 32;
    while (n2 < BK) n2 <<= 1;
    float* const xb = conf + 2 * BK + (BK + 3) / 4;
    switch (budget_values_per_thread(n2)) {
      case 1: cut = adaptive_cut<1>(P, conf, n2, xb, sh, &Nsel); break;
      case 2: cut = adaptive_cut<2>(P, conf, n2, xb, sh, &Nsel); break;
      case 4: cut = adaptive_cut<4>(P, conf, n2, xb, sh, &Nsel); break;
      case 8: cut = adaptive_cut<8>(P, conf, n2, xb, sh, &Nsel); break;
      default: cut = adaptive_cut<16>(P, conf, n2, xb, sh, &Nsel); break;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0 && P.out_N) *P.out_N = Nsel;
  }
  for (int b = blockIdx.x * nw + warp; b < B; b += gridDim.x * nw) {
    // rank of key (b, m): within each request b' the keys that precede it form a prefix (conf
    // is non-increasing in m'), found by binary search; lanes split the requests
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
    int d;
    if (P.n_cost > 0) {
      // the positions at or above the cut, a prefix of m (c never grows with m, and among ties
      // the smaller m comes first)
      const float cm = lane < K ? conf[lane * B + b] : -1.f;
      d = __popc(__ballot_sync(0xffffffffu,
                               lane < K && (cm > cut.c_last || (cm == cut.c_last && lane * B + b <= cut.r_last))));
    } else {
      // d_b = the number of m whose key ranks below N (a prefix of m)
      int lo = 0, hi = K;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (rank_of(mid) < Nsel) lo = mid + 1; else hi = mid;
      }
      d = lo;
    }
    if (P.out_depth && lane == 0) P.out_depth[b] = d;
    if (P.out_conf)
      for (int k = lane; k < K; k += 32) P.out_conf[static_cast<size_t>(b) * K + k] = conf[k * B + b];
    if (P.do_cut) {
      if (P.greedy)
        cut_request(b, d, P.stats_only != 0, P.keys, P.draft_keys != 0, false, P.U, K, P.V, P.tokens,
                    P.out_tokens, P.out_accepted, P.out_alpha, P.out_cum, P.out_E, P.status, lane);
      else
        cut_sampling(P, b, d, lane, true, lane < K ? alpha_s[lane * B + b] : 0.f, rej_s);
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
  const int BK = p.B * p.K;
  size_t smem = static_cast<size_t>(BK) * sizeof(float) * 2 + static_cast<size_t>((BK + 3) / 4) * sizeof(float);
  if (p.n_cost > 0) {   // the choice of N sorts: its exchange area and the sorted values
    int n2 = 32;
    while (n2 < BK) n2 <<= 1;
    smem += 3 * static_cast<size_t>(n2) * sizeof(float);
  }
  // beyond 48 KB in all (the kernel's static scratch included) a launch needs the opt-in
  if (smem + sizeof(BudgetShared) + 256 > 48 * 1024) {
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

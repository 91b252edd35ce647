// C ABI of the verification library: argument checks, launch planning, launches.
// The declarations and their contracts are in include/spec_verify.h.
//
// The library keeps no mutable state between calls except two per-device caches (kernel
// attributes set, occupancy answers), guarded by a mutex.  Tuning and test knobs travel with
// the call (spec_tuning_t), never through process-wide settings.
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

#include "../../include/spec_verify.h"
#include "api_range.h"
#include "spec_internal.h"

namespace sv {
const void* sample_kernel_bf16(bool aligned);
const void* sample_kernel_f32(bool aligned);
}  // namespace sv

namespace {

using sv::BudgetParams;
using sv::RowParams;
using sv::UnitRec;

constexpr long long kDefaultWaitNs = 200000000ll;   // wall time per bounded on-device wait
constexpr size_t kAlign = 256;
constexpr int kMaxV = 262144;
constexpr int kBudgetMaxKeys = 8192;
constexpr int kSampThreads = 256;
constexpr int kItemBytes = sv::kSampItemBytes;       // bytes of one row per item of the sampling kernel

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace layout, a function of the buffer size only (so the greedy keys, which the cut
// kernel clears after every call, never overlap bytes another call shape wrote):
//   [status word | pad to 256] [argmax keys: cap rows x 16 B] [request counters: cap x 4 B]
//   [row records: cap rows x 32 B] [row mass tables: cap rows x kMassRowFloats x 4 B]
// where cap = the number of (request, position) rows the buffer can hold.
constexpr size_t kKeyBytes = 2 * sizeof(uint64_t);
constexpr size_t kMassBytes = sizeof(float) * sv::kMassRowFloats;
constexpr size_t kRowBytes = kKeyBytes + sizeof(int32_t) + sizeof(UnitRec) + kMassBytes;
struct WsLayout {
  size_t status, keys, counters, recs, mass, cap_rows;
};
WsLayout ws_layout_for(size_t ws_bytes) {
  WsLayout L;
  L.status = 0;
  L.keys = kAlign;
  const size_t avail = ws_bytes > 5 * kAlign ? ws_bytes - 5 * kAlign : 0;
  L.cap_rows = avail / kRowBytes;
  L.counters = align_up(L.keys + L.cap_rows * kKeyBytes, kAlign);
  L.recs = align_up(L.counters + L.cap_rows * sizeof(int32_t), kAlign);
  L.mass = align_up(L.recs + L.cap_rows * sizeof(UnitRec), kAlign);
  return L;
}
size_t ws_bytes_needed(int B, int K) {
  const size_t rows = static_cast<size_t>(B > 0 ? B : 1) * (K + 1);
  return 5 * kAlign + rows * kRowBytes;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The knobs of one call: defaults, or the caller's spec_tuning_t.
struct Knobs {
  long long wait_ns = kDefaultWaitNs;
  int cluster = 0;
  int variant = 0;
  int32_t* plan_out = nullptr;
  cudaEvent_t split = nullptr;
};
Knobs knobs_of(const spec_tuning_t* t) {
  Knobs k;
  if (!t) return k;
  if (t->wait_limit_us > 0) k.wait_ns = t->wait_limit_us * 1000;
  if (t->wait_limit_us < 0) k.wait_ns = 0;
  k.cluster = t->cluster;
  k.variant = t->greedy_variant & 7;
  k.plan_out = t->plan_out;
  k.split = static_cast<cudaEvent_t>(t->split_event);
  return k;
}
void report_plan(const Knobs& kn, const int (&rec)[8]) {
  if (kn.plan_out) std::memcpy(kn.plan_out, rec, sizeof(rec));
}

// Per-device caches: kernel attributes set once, and occupancy answers.
std::mutex g_mu;
std::map<std::tuple<int, const void*>, bool> g_attr_done;
std::map<std::tuple<int, const void*, int, int>, int> g_maxc;
std::map<int, std::tuple<int, int, size_t>> g_dev;   // SMs, L2 bytes
// chosen sampling plan per call shape
struct PlanChoice {
  int cluster, nclusters, maxc;
};
std::map<std::tuple<int, const void*, int, int, int, int, int>, PlanChoice> g_plans;

cudaError_t device_info(int dev, int* sms, size_t* l2) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_dev.find(dev);
    if (it != g_dev.end()) {
      *sms = std::get<0>(it->second);
      *l2 = std::get<2>(it->second);
      return cudaSuccess;
    }
  }
  int s = 0, l = 0;
  cudaError_t e = cudaDeviceGetAttribute(&s, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&l, cudaDevAttrL2CacheSize, dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mu);
  g_dev[dev] = std::make_tuple(s, 0, static_cast<size_t>(l));
  *sms = s;
  *l2 = static_cast<size_t>(l);
  return cudaSuccess;
}

cudaError_t prepare_kernel(int dev, const void* fn, int smem_max) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_tuple(dev, fn);
  if (g_attr_done.count(key)) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_max);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  g_attr_done[key] = true;
  return cudaSuccess;
}

// Largest number of clusters of `cluster` sampling CTAs, each with `smem` bytes of dynamic shared
// memory, that can be resident at once.
cudaError_t max_clusters(int dev, const void* fn, int smem_max, int cluster, int smem, int* out) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_maxc.find(std::make_tuple(dev, fn, cluster, smem));
    if (it != g_maxc.end()) {
      *out = it->second;
      return cudaSuccess;
    }
  }
  cudaError_t e = prepare_kernel(dev, fn, smem_max);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(cluster, 1, 1);
  cfg.blockDim = dim3(kSampThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(smem);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mu);
  g_maxc[std::make_tuple(dev, fn, cluster, smem)] = n;
  *out = n;
  return cudaSuccess;
}

struct RowPlan {
  const void* fn;
  int cluster, nclusters, maxc, smem;
  RowParams p;
};

// Estimated duration (seconds) of the sampling kernel with clusters of C CTAs: units go
// round-robin to the clusters (pairs first); a CTA reads its slice of a unit's rows at its share
// of the HBM bandwidth (bw_total over all CTAs, at most bw_cta each) and every step pays a fixed
// cost t_step for the cluster exchange and the normalisers.
double plan_cost(int C, int ncl, int npairs, int nsingle, double row_bytes, double bw_total, double bw_cta,
                 double t_step) {
  const int units = npairs + nsingle;
  if (ncl < 1) return 1e300;
  const double bw = std::fmin(bw_total / (static_cast<double>(ncl) * C), bw_cta);
  const double t_row = row_bytes / C / bw;
  double worst = 0.0;
  for (int j = 0; j < ncl && j < units; ++j) {
    double t = t_step;
    for (int u = j; u < units; u += ncl) t += (u < npairs ? 2.0 : 1.0) * t_row + t_step;
    worst = std::fmax(worst, t);
  }
  return worst;
}
// Fitted to timings of the verification configurations on a GB300.
constexpr double kPlanBw = 6.5e12, kPlanBwCta = 2.5e10, kPlanStep = 1.5e-6;

spec_status_t plan_rows(const void* target, const void* draft, int dtype, int B, int K, int V, float T,
                        bool need_draft, bool stats_only, const Knobs& kn, RowPlan* plan) {
  const bool bf16 = dtype == SPEC_BF16;
  const int esz = bf16 ? 2 : 4;
  const bool aligned = (static_cast<size_t>(V) * esz) % 16 == 0 && aligned16(target) &&
                       (!need_draft || aligned16(draft));
  const void* fn = bf16 ? sv::sample_kernel_bf16(aligned) : sv::sample_kernel_f32(aligned);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
  const int npairs = need_draft ? B * K : 0;
  const int nsingle = stats_only ? 0 : (need_draft ? B : B * (K + 1));
  const int units = npairs + nsingle;
  const double row_bytes = static_cast<double>(V) * esz;
  const int item_logits = kItemBytes / esz;
  auto slice_of = [&](int C) { return static_cast<int>(align_up((V + C - 1) / C, sv::kChunk)); };
  auto items_of = [&](int C) { return (slice_of(C) + item_logits - 1) / item_logits; };
  PlanChoice best = {0, 0, 0};
  const auto key = std::make_tuple(dev, fn, B, K, V, static_cast<int>(need_draft) | (stats_only ? 2 : 0), kn.cluster);
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_plans.find(key);
    if (it != g_plans.end()) best = it->second;
  }
  if (best.cluster == 0) {
    // among the cluster sizes whose slice fits the slab, the cheapest estimated schedule
    double best_cost = 1e300;
    for (int C = 1; C <= sv::kMaxCluster; C *= 2) {
      if (kn.cluster && C != kn.cluster) continue;
      const int itmax = items_of(C);
      if (itmax > sv::kSampMaxItems || C * itmax > sv::kMassMaxSegments) continue;
      int maxc = 0;
      if (max_clusters(dev, fn, sv::kSampMaxSlabBytes, C, sv::samp_slab_bytes(itmax), &maxc) != cudaSuccess)
        return SPEC_ERR_CUDA;
      if (maxc < 1) continue;
      const int ncl = units < maxc ? units : maxc;
      const double cost = plan_cost(C, ncl, npairs, nsingle, row_bytes, kPlanBw, kPlanBwCta, kPlanStep);
      if (best.cluster == 0 || cost < best_cost * 0.97) {
        best_cost = cost;
        best = {C, ncl, maxc};
      }
    }
    if (best.cluster == 0) return SPEC_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    g_plans[key] = best;
  }
  const int slice = slice_of(best.cluster);
  const int itmax = items_of(best.cluster);
  plan->fn = fn;
  plan->cluster = best.cluster;
  plan->nclusters = best.nclusters;
  plan->maxc = best.maxc;
  plan->smem = sv::samp_slab_bytes(itmax);
  RowParams& p = plan->p;
  std::memset(&p, 0, sizeof(p));
  p.target = target;
  p.draft = draft;
  p.B = B;
  p.K = K;
  p.V = V;
  p.U = stats_only ? K : K + 1;
  p.total_units = units;
  p.slice = slice;
  p.itmax = itmax;
  p.flags = (need_draft ? sv::F_NEED_DRAFT : 0) | (stats_only ? sv::F_STATS_ONLY : 0) |
            (aligned ? sv::F_ALIGNED : 0);
  p.c = static_cast<float>(1.4426950408889634 / static_cast<double>(T));
  p.wait_limit = kn.wait_ns;
  return SPEC_OK;
}

spec_status_t launch_plan(RowPlan* plan, const Knobs& kn, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
  if (prepare_kernel(dev, plan->fn, sv::kSampMaxSlabBytes) != cudaSuccess) return SPEC_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = plan->cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the grid's prologue overlaps the preceding kernel's tail; it
  // waits (griddepcontrol.wait) for that kernel before touching memory
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(plan->nclusters * plan->cluster, 1, 1);
  cfg.blockDim = dim3(kSampThreads, 1, 1);
  cfg.dynamicSmemBytes = static_cast<size_t>(plan->smem);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  void* args[] = {&plan->p};
  if (cudaLaunchKernelExC(&cfg, plan->fn, args) != cudaSuccess) return SPEC_ERR_CUDA;
  const int rec[8] = {kSampThreads, plan->cluster, plan->nclusters, plan->maxc, plan->p.slice,
                      plan->p.itmax, plan->smem, plan->p.flags};
  report_plan(kn, rec);
  return SPEC_OK;
}

bool bad_T(float T) { return !(T >= 0.f) || std::isinf(T); }

// Greedy path: the streaming argmax kernel over target rows (and draft rows when need_draft).
std::map<int, int> g_argmax_grid;
spec_status_t launch_greedy(const void* target, const void* draft, int dtype, int B, int K, int V,
                            bool need_draft, bool stats_only, bool fused_cut, uint64_t* keys,
                            sv::ArgmaxParams cut, const Knobs& kn, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
  int grid_cap;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    const int gkey = dev * 2 + (dtype == SPEC_BF16);
    auto it = g_argmax_grid.find(gkey);
    if (it == g_argmax_grid.end()) {
      int sms = 0, per_sm = 0;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SPEC_ERR_CUDA;
      // one wave of resident CTAs (the bf16 and fp32 instances differ only in registers)
      if (sv::argmax_blocks_per_sm(dtype == SPEC_BF16, &per_sm) != cudaSuccess) return SPEC_ERR_CUDA;
      g_argmax_grid[gkey] = sms * (per_sm > 0 ? per_sm : 1);
      it = g_argmax_grid.find(gkey);
    }
    grid_cap = it->second;
  }
  sv::ArgmaxParams p = cut;   // fused-cut arguments (tokens, depth, outputs, counters, status)
  p.target = target;
  p.draft = need_draft ? draft : nullptr;
  p.keys = keys;
  p.B = B;
  p.K = K;
  p.V = V;
  p.rows_t = stats_only ? K : K + 1;
  p.drows = need_draft ? K : 0;
  const int tile = dtype == SPEC_BF16 ? 2048 : 1024;   // the argmax kernel's warp tile
  p.tpr = (V + tile - 1) / tile;
  p.total_tiles = static_cast<long long>(B) * (p.rows_t + p.drows) * p.tpr;
  if (p.total_tiles >= (1ll << 31)) return SPEC_ERR_UNSUPPORTED;
  p.fused_cut = fused_cut && !(kn.variant & 2);
  p.stats_only = stats_only;
  p.wait_limit = kn.wait_ns;
  const int esz = dtype == SPEC_BF16 ? 2 : 4;
  p.aligned = (static_cast<size_t>(V) * esz) % 16 == 0 && aligned16(target) && (!need_draft || aligned16(draft));
  // every warp takes the same number of tiles (the fewest one resident wave allows), so no
  // warp is left with an extra tile after the others finish
  const long long per_warp = (p.total_tiles + 8ll * grid_cap - 1) / (8ll * grid_cap);
  long long grid = (p.total_tiles + 8 * per_warp - 1) / (8 * per_warp);
  if (kn.variant & 4) grid = (p.total_tiles + 7) / 8;   // every resident CTA slot, tiles spread evenly
  if (grid > grid_cap) grid = grid_cap;
  if (grid < 1) grid = 1;
  if (sv::launch_argmax(dtype == SPEC_BF16, p, static_cast<int>(grid), stream) != cudaSuccess) return SPEC_ERR_CUDA;
  const int rec[8] = {256, 1, static_cast<int>(grid), grid_cap, tile, 0, 0, -1};
  report_plan(kn, rec);
  return SPEC_OK;
}

spec_status_t check_ws(void* ws, size_t ws_bytes, int B, int K) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return SPEC_ERR_WORKSPACE;
  if (ws_bytes < ws_bytes_needed(B, K)) return SPEC_ERR_WORKSPACE;
  if (ws_layout_for(ws_bytes).cap_rows < static_cast<size_t>(B) * (K + 1)) return SPEC_ERR_WORKSPACE;
  return SPEC_OK;
}

// What the cut kernels need to read the sampling kernel's records and redo its one draw.
void set_sampling_geometry(sv::BudgetParams* bp, const RowPlan& plan, const float* mass, int dtype) {
  bp->mass = mass;
  bp->target = plan.p.target;
  bp->draft = plan.p.draft;
  bp->c = plan.p.c;
  bp->bf16 = dtype == SPEC_BF16;
  bp->aligned = (plan.p.flags & sv::F_ALIGNED) != 0;
  bp->ncta = plan.cluster;
  bp->slice = plan.p.slice;
  bp->itmax = plan.p.itmax;
}

struct VerifyArgs {
  const void* target;
  const void* draft;
  int dtype;
  const int32_t* tokens;
  const float* uniforms;
  int B, K, V;
  float T;
  const int32_t* depth;
  int budget;
  int32_t* out_tokens;
  int32_t* out_accepted;
  float* out_alpha;
  float* out_cum;
  float* out_E;
  int32_t* out_depth;
  void* ws;
  size_t ws_bytes;
  cudaStream_t stream;
};

spec_status_t run_verify(const VerifyArgs& a, const Knobs& kn) {
  if (a.dtype != SPEC_F32 && a.dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (a.B < 0 || a.K < 0 || a.V < 1 || bad_T(a.T)) return SPEC_ERR_INVALID_ARG;
  if (a.K > sv::kMaxK || a.V > kMaxV) return SPEC_ERR_UNSUPPORTED;
  if (a.B == 0) return SPEC_OK;
  const bool greedy = a.T == 0.f;
  const bool budget = a.budget >= 0;
  if (budget && a.depth) return SPEC_ERR_INVALID_ARG;
  if (budget && static_cast<long long>(a.B) * a.K > kBudgetMaxKeys) return SPEC_ERR_UNSUPPORTED;
  const bool want_alpha = a.out_alpha || a.out_cum || a.out_E || budget;
  const bool need_draft = a.K > 0 && (!greedy || want_alpha);
  if (!a.target || !a.out_tokens || !a.out_accepted) return SPEC_ERR_INVALID_ARG;
  if (a.K > 0 && !a.tokens) return SPEC_ERR_INVALID_ARG;
  if (need_draft && !a.draft) return SPEC_ERR_INVALID_ARG;
  if (!greedy && !a.uniforms) return SPEC_ERR_INVALID_ARG;
  spec_status_t st = check_ws(a.ws, a.ws_bytes, a.B, a.K);
  if (st != SPEC_OK) return st;

  const WsLayout L = ws_layout_for(a.ws_bytes);
  uint8_t* ws = static_cast<uint8_t*>(a.ws);
  UnitRec* recs = reinterpret_cast<UnitRec*>(ws + L.recs);
  float* mass = reinterpret_cast<float*>(ws + L.mass);
  uint64_t* keys = reinterpret_cast<uint64_t*>(ws + L.keys);
  int32_t* counters = reinterpret_cast<int32_t*>(ws + L.counters);
  int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
  RowPlan plan;
  std::memset(&plan, 0, sizeof(plan));
  if (greedy) {
    sv::ArgmaxParams cut;
    std::memset(&cut, 0, sizeof(cut));
    cut.counters = counters;
    cut.status = status;
    cut.tokens = a.tokens;
    cut.depth = a.depth;
    cut.out_tokens = a.out_tokens;
    cut.out_accepted = a.out_accepted;
    cut.out_alpha = a.out_alpha;
    cut.out_cum = a.out_cum;
    cut.out_E = a.out_E;
    st = launch_greedy(a.target, a.draft, a.dtype, a.B, a.K, a.V, need_draft, false, !budget, keys, cut, kn,
                       a.stream);
    if (st != SPEC_OK) return st;
    if (!budget && (kn.variant & 2) == 0) return SPEC_OK;   // the cut ran inside the argmax kernel
  } else {
    st = plan_rows(a.target, a.draft, a.dtype, a.B, a.K, a.V, a.T, need_draft, false, kn, &plan);
    if (st != SPEC_OK) return st;
    RowParams& p = plan.p;
    p.tokens = a.tokens;
    p.uniforms = a.uniforms;
    p.depth = a.depth;
    p.recs = recs;
    p.mass = mass;
    p.status = status;
    if (budget) p.flags |= sv::F_ALL_PDRAWS;
    st = launch_plan(&plan, kn, a.stream);
    if (st != SPEC_OK) return st;
  }

  BudgetParams bp;
  std::memset(&bp, 0, sizeof(bp));
  bp.alpha_in = nullptr;
  bp.recs = recs;
  bp.keys = keys;
  bp.draft_keys = greedy && need_draft;
  bp.U = a.K + 1;
  bp.B = a.B;
  bp.K = a.K;
  bp.V = a.V;
  bp.N = a.budget;
  bp.greedy = greedy;
  bp.do_cut = 1;
  bp.stats_only = 0;
  bp.tokens = a.tokens;
  bp.uniforms = a.uniforms;
  bp.out_depth = a.out_depth;
  bp.out_tokens = a.out_tokens;
  bp.out_accepted = a.out_accepted;
  bp.out_alpha = a.out_alpha;
  bp.out_cum = a.out_cum;
  bp.out_E = a.out_E;
  bp.status = status;
  set_sampling_geometry(&bp, plan, mass, a.dtype);
  if (kn.split && cudaEventRecord(kn.split, a.stream) != cudaSuccess) return SPEC_ERR_CUDA;
  const bool pdl = kn.split == nullptr;
  const cudaError_t e = budget ? sv::launch_budget_cut(bp, a.stream, pdl) : sv::launch_cut(bp, a.depth, a.stream, pdl);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status_t run_overlap(const void* target_logits, const void* draft_logits, int dtype, int B, int K, int V,
                          float temperature, float* out_alpha, float* out_cum_alpha, float* out_expected_len,
                          void* workspace, size_t ws_bytes, cudaStream_t stream, const Knobs& kn) {
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (B < 0 || K < 0 || V < 1 || bad_T(temperature)) return SPEC_ERR_INVALID_ARG;
  if (K > sv::kMaxK || V > kMaxV) return SPEC_ERR_UNSUPPORTED;
  if (B == 0 || K == 0) return SPEC_OK;
  if (!target_logits || !draft_logits || !out_alpha) return SPEC_ERR_INVALID_ARG;
  spec_status_t st = check_ws(workspace, ws_bytes, B, K);
  if (st != SPEC_OK) return st;
  const WsLayout L = ws_layout_for(ws_bytes);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  UnitRec* recs = reinterpret_cast<UnitRec*>(ws + L.recs);
  float* mass = reinterpret_cast<float*>(ws + L.mass);
  uint64_t* keys = reinterpret_cast<uint64_t*>(ws + L.keys);
  int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
  const bool greedy = temperature == 0.f;
  RowPlan plan;
  std::memset(&plan, 0, sizeof(plan));
  if (greedy) {
    sv::ArgmaxParams cut;
    std::memset(&cut, 0, sizeof(cut));
    cut.counters = reinterpret_cast<int32_t*>(ws + L.counters);
    cut.status = status;
    cut.out_alpha = out_alpha;
    cut.out_cum = out_cum_alpha;
    cut.out_E = out_expected_len;
    st = launch_greedy(target_logits, draft_logits, dtype, B, K, V, true, true, true, keys, cut, kn, stream);
    if (st != SPEC_OK || (kn.variant & 2) == 0) return st;
  } else {
    st = plan_rows(target_logits, draft_logits, dtype, B, K, V, temperature, true, true, kn, &plan);
    if (st != SPEC_OK) return st;
    plan.p.recs = recs;
    plan.p.mass = mass;
    plan.p.status = status;
    st = launch_plan(&plan, kn, stream);
  }
  if (st != SPEC_OK) return st;
  BudgetParams bp;
  std::memset(&bp, 0, sizeof(bp));
  bp.recs = recs;
  bp.keys = keys;
  bp.draft_keys = greedy;
  bp.U = K;
  bp.B = B;
  bp.K = K;
  bp.V = V;
  bp.greedy = greedy;
  bp.stats_only = 1;
  bp.out_alpha = out_alpha;
  bp.out_cum = out_cum_alpha;
  bp.out_E = out_expected_len;
  bp.status = status;
  set_sampling_geometry(&bp, plan, mass, dtype);
  if (kn.split && cudaEventRecord(kn.split, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  return sv::launch_cut(bp, nullptr, stream, kn.split == nullptr) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace

extern "C" {

int spec_version(void) { return 200; }

const char* spec_error_string(int status) {
  switch (status) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_UNSUPPORTED: return "unsupported size";
    case SPEC_ERR_CUDA: return "CUDA launch or runtime error";
    case SPEC_ERR_DEVICE_TIMEOUT: return "a bounded device wait ran out";
    case SPEC_ERR_TOKEN_RANGE: return "draft token id outside [0, V)";
    case SPEC_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
    default: return "unknown status";
  }
}

size_t spec_workspace_bytes(int B, int K, int V, int dtype) {
  (void)V;
  (void)dtype;
  if (B < 0 || K < 0) return 0;
  return ws_bytes_needed(B, K);
}

spec_status_t spec_workspace_init(void* workspace, size_t ws_bytes, void* stream) {
  const sv::ApiRange range("spec_workspace_init");
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0) return SPEC_ERR_WORKSPACE;
  return cudaMemsetAsync(workspace, 0, ws_bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}

spec_status_t spec_get_status(void* workspace, void* stream, int32_t* out_status) {
  const sv::ApiRange range("spec_get_status");
  if (!workspace || !out_status) return SPEC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t h = 0;
  if (cudaMemcpyAsync(&h, workspace, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return SPEC_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SPEC_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(h), s) != cudaSuccess) return SPEC_ERR_CUDA;
  *out_status = (h & sv::kStatusTimeout) ? SPEC_ERR_DEVICE_TIMEOUT
                : (h & sv::kStatusTokenRange) ? SPEC_ERR_TOKEN_RANGE
                                              : SPEC_OK;
  return SPEC_OK;
}

spec_status_t spec_verify_chain(const void* target_logits, const void* draft_logits, int dtype,
                                const int32_t* tokens, const float* uniforms, int B, int K, int V,
                                float temperature, const int32_t* depth, int32_t* out_tokens,
                                int32_t* out_accepted, float* out_alpha, void* workspace,
                                size_t ws_bytes, void* stream) {
  const sv::ApiRange range("spec_verify_chain");
  VerifyArgs a = {target_logits, draft_logits, dtype, tokens, uniforms, B, K, V, temperature,
                  depth, -1, out_tokens, out_accepted, out_alpha, nullptr, nullptr, nullptr,
                  workspace, ws_bytes, static_cast<cudaStream_t>(stream)};
  return run_verify(a, Knobs());
}

spec_status_t spec_verify_block(const void* target_logits, const void* draft_logits, int dtype,
                                const int32_t* tokens, const float* uniforms, int B, int K, int V,
                                float temperature, const int32_t* depth, int budget_N,
                                int32_t* out_tokens, int32_t* out_accepted, float* out_alpha,
                                float* out_cum_alpha, float* out_expected_len, int32_t* out_depth,
                                void* workspace, size_t ws_bytes, void* stream) {
  const sv::ApiRange range("spec_verify_block");
  VerifyArgs a = {target_logits, draft_logits, dtype, tokens, uniforms, B, K, V, temperature,
                  depth, budget_N, out_tokens, out_accepted, out_alpha, out_cum_alpha,
                  out_expected_len, out_depth, workspace, ws_bytes, static_cast<cudaStream_t>(stream)};
  return run_verify(a, Knobs());
}

spec_status_t spec_overlap_alpha(const void* target_logits, const void* draft_logits, int dtype,
                                 int B, int K, int V, float temperature, float* out_alpha,
                                 float* out_cum_alpha, float* out_expected_len, void* workspace,
                                 size_t ws_bytes, void* stream) {
  const sv::ApiRange range("spec_overlap_alpha");
  return run_overlap(target_logits, draft_logits, dtype, B, K, V, temperature, out_alpha, out_cum_alpha,
                     out_expected_len, workspace, ws_bytes, static_cast<cudaStream_t>(stream), Knobs());
}

spec_status_t spec_verify_tuned(const void* target_logits, const void* draft_logits, int dtype,
                                const int32_t* tokens, const float* uniforms, int B, int K, int V,
                                float temperature, const int32_t* depth, int budget_N, int stats_only,
                                int32_t* out_tokens, int32_t* out_accepted, float* out_alpha,
                                float* out_cum_alpha, float* out_expected_len, int32_t* out_depth,
                                void* workspace, size_t ws_bytes, void* stream, const spec_tuning_t* tuning) {
  const sv::ApiRange range("spec_verify_tuned");
  const Knobs kn = knobs_of(tuning);
  if (tuning && tuning->cluster != 0) {
    const int c = tuning->cluster;
    if (c < 1 || c > sv::kMaxCluster || (c & (c - 1)) != 0) return SPEC_ERR_INVALID_ARG;
  }
  if (stats_only)
    return run_overlap(target_logits, draft_logits, dtype, B, K, V, temperature, out_alpha, out_cum_alpha,
                       out_expected_len, workspace, ws_bytes, static_cast<cudaStream_t>(stream), kn);
  VerifyArgs a = {target_logits, draft_logits, dtype, tokens, uniforms, B, K, V, temperature,
                  depth, budget_N, out_tokens, out_accepted, out_alpha, out_cum_alpha,
                  out_expected_len, out_depth, workspace, ws_bytes, static_cast<cudaStream_t>(stream)};
  return run_verify(a, kn);
}

spec_status_t spec_alloc_budget(const float* alpha, int B, int K, int budget_N, int32_t* out_depth,
                                float* out_conf, void* workspace, size_t ws_bytes, void* stream) {
  const sv::ApiRange range("spec_alloc_budget");
  if (B < 0 || K < 0 || budget_N < 0) return SPEC_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * K > kBudgetMaxKeys) return SPEC_ERR_UNSUPPORTED;
  if (B == 0) return SPEC_OK;
  if (!out_depth || (K > 0 && !alpha)) return SPEC_ERR_INVALID_ARG;
  spec_status_t st = check_ws(workspace, ws_bytes, B, K);
  if (st != SPEC_OK) return st;
  BudgetParams bp;
  std::memset(&bp, 0, sizeof(bp));
  bp.alpha_in = alpha;
  bp.B = B;
  bp.K = K;
  bp.N = budget_N;
  bp.do_cut = 0;
  bp.out_depth = out_depth;
  bp.out_conf = out_conf;
  bp.status = static_cast<int32_t*>(workspace);
  return sv::launch_budget_cut(bp, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SPEC_OK
                                                                                      : SPEC_ERR_CUDA;
}

spec_status_t spec_alloc_budget_adaptive(const float* alpha, int B, int K, const float* cost_n,
                                         const float* cost_t, int n_cost, int32_t* out_N, int32_t* out_depth,
                                         float* out_conf, void* workspace, size_t ws_bytes, void* stream) {
  const sv::ApiRange range("spec_alloc_budget_adaptive");
  if (B < 0 || K < 0 || n_cost < 1) return SPEC_ERR_INVALID_ARG;
  if (n_cost > sv::kBudgetMaxCost) return SPEC_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * K > kBudgetMaxKeys) return SPEC_ERR_UNSUPPORTED;
  if (B == 0) return SPEC_OK;
  if (!out_depth || !cost_n || !cost_t || (K > 0 && !alpha)) return SPEC_ERR_INVALID_ARG;
  spec_status_t st = check_ws(workspace, ws_bytes, B, K);
  if (st != SPEC_OK) return st;
  sv::BudgetParams bp;
  std::memset(&bp, 0, sizeof(bp));
  bp.alpha_in = alpha;
  bp.B = B;
  bp.K = K;
  bp.do_cut = 0;
  bp.cost_n = cost_n;
  bp.cost_t = cost_t;
  bp.n_cost = n_cost;
  bp.out_N = out_N;
  bp.out_depth = out_depth;
  bp.out_conf = out_conf;
  bp.status = static_cast<int32_t*>(workspace);
  return sv::launch_budget_cut(bp, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status_t spec_draft_budget(const void* draft_logits, int dtype, const int32_t* tokens, int B, int K, int V,
                                float temperature, int budget_N, const float* cost_n, const float* cost_t,
                                int n_cost, int32_t* out_N, int32_t* out_depth, float* out_conf,
                                void* workspace, size_t ws_bytes, void* stream) {
  const sv::ApiRange range("spec_draft_budget");
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (B < 0 || K < 0 || V < 1 || bad_T(temperature) || n_cost < 0) return SPEC_ERR_INVALID_ARG;
  if (n_cost == 0 && budget_N < 0) return SPEC_ERR_INVALID_ARG;
  if (n_cost > sv::kBudgetMaxCost || V > kMaxV) return SPEC_ERR_UNSUPPORTED;
  if (static_cast<long long>(B) * K > kBudgetMaxKeys) return SPEC_ERR_UNSUPPORTED;
  if (B == 0) return SPEC_OK;
  if (!out_depth || (n_cost > 0 && (!cost_n || !cost_t)) || (K > 0 && (!draft_logits || !tokens)))
    return SPEC_ERR_INVALID_ARG;
  spec_status_t st = check_ws(workspace, ws_bytes, B, K);
  if (st != SPEC_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf16 = dtype == SPEC_BF16;
  const int esz = bf16 ? 2 : 4;
  const bool greedy = temperature == 0.f;
  const float c = greedy ? 0.f : static_cast<float>(1.4426950408889634 / static_cast<double>(temperature));
  // the partials of every draft row live in the workspace's mass tables (at most 16 x 16 B a row)
  const WsLayout L = ws_layout_for(ws_bytes);
  float4* part = reinterpret_cast<float4*>(static_cast<uint8_t*>(workspace) + L.mass);
  int nparts = static_cast<int>((static_cast<size_t>(V) * esz + 65535) / 65536);
  nparts = nparts < 1 ? 1 : (nparts > 16 ? 16 : nparts);
  const int part_len = static_cast<int>(align_up((V + nparts - 1) / nparts, sv::kChunk));
  nparts = (V + part_len - 1) / part_len;
  if (K > 0) {
    sv::DraftStatsParams dp;
    dp.draft = draft_logits;
    dp.rows = B * K;
    dp.V = V;
    dp.nparts = nparts;
    dp.part_len = part_len;
    dp.c = c;
    dp.out = part;
    const bool aligned = (static_cast<size_t>(V) * esz) % 16 == 0 && aligned16(draft_logits);
    if (sv::launch_draft_stats(bf16, greedy, aligned, dp, s) != cudaSuccess) return SPEC_ERR_CUDA;
  }
  sv::BudgetParams bp;
  std::memset(&bp, 0, sizeof(bp));
  bp.draft_part = part;
  bp.nparts = nparts;
  bp.draft_greedy = greedy ? 1 : 0;
  bp.draft = draft_logits;
  bp.bf16 = bf16 ? 1 : 0;
  bp.c = c;
  bp.tokens = tokens;
  bp.U = K + 1;
  bp.B = B;
  bp.K = K;
  bp.V = V;
  bp.N = budget_N;
  bp.do_cut = 0;
  bp.cost_n = cost_n;
  bp.cost_t = cost_t;
  bp.n_cost = n_cost;
  bp.out_N = out_N;
  bp.out_depth = out_depth;
  bp.out_conf = out_conf;
  bp.status = static_cast<int32_t*>(workspace);
  return sv::launch_budget_cut(bp, s) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // extern "C"

// C ABI of the verification library: argument checks, launch configuration, launches.
// The declarations and their contracts are in include/spec_verify.h.
#include <atomic>
#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

#include "../../include/spec_verify.h"
#include "spec_internal.h"

namespace sv {
const void* sample_kernel_bf16(int nt);
const void* sample_kernel_f32(int nt);
}  // namespace sv

namespace {

using sv::BudgetParams;
using sv::RowParams;
using sv::UnitRec;

constexpr long long kDefaultWaitLimit = 200000000ll;   // ns of wall time per bounded on-device wait
std::atomic<long long> g_wait_limit{kDefaultWaitLimit};

constexpr size_t kAlign = 256;
constexpr int kMaxV = 262144;
constexpr int kBudgetMaxKeys = 8192;
constexpr size_t kRingBudgetLarge = 200 * 1024;   // per CTA when one CTA fills an SM

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace layout, a function of the buffer size only (so the greedy keys, which the cut
// kernel clears after every call, never overlap bytes another call shape wrote):
//   [status word | pad to 256] [argmax keys: cap rows x 16 B] [request counters: cap x 4 B]
//   [row records: cap rows x 32 B]
// where cap = the number of (request, position) rows the buffer can hold.
constexpr size_t kKeyBytes = 2 * sizeof(uint64_t);
constexpr size_t kRowBytes = kKeyBytes + sizeof(int32_t) + sizeof(UnitRec);
struct WsLayout {
  size_t status, keys, counters, recs, cap_rows;
};
WsLayout ws_layout_for(size_t ws_bytes) {
  WsLayout L;
  L.status = 0;
  L.keys = kAlign;
  const size_t avail = ws_bytes > 4 * kAlign ? ws_bytes - 4 * kAlign : 0;
  L.cap_rows = avail / kRowBytes;
  L.counters = align_up(L.keys + L.cap_rows * kKeyBytes, kAlign);
  L.recs = align_up(L.counters + L.cap_rows * sizeof(int32_t), kAlign);
  return L;
}
size_t ws_bytes_needed(int B, int K) {
  const size_t rows = static_cast<size_t>(B > 0 ? B : 1) * (K + 1);
  return 4 * kAlign + rows * kRowBytes;
}

// Test and tuning hooks: the last row-kernel plan, and optional overrides (0 = automatic).
std::atomic<int> g_force_nt{0}, g_force_cluster{0}, g_force_nstage{0};
std::atomic<int> g_variant{0};   // greedy path: bit 1 separate cut kernel, bit 2 one full resident wave
int g_last_plan[8] = {0};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// One-time per (device, kernel) attribute setup and a cache of the cluster occupancy.
std::mutex g_mu;
std::map<std::tuple<int, const void*>, bool> g_attr_done;
std::map<std::tuple<int, const void*, int, size_t>, int> g_occ;

cudaError_t prepare_kernel(int dev, const void* fn) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_tuple(dev, fn);
  if (g_attr_done.count(key)) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kRingBudgetLarge + 4096));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  g_attr_done[key] = true;
  return cudaSuccess;
}

cudaError_t max_clusters(int dev, const void* fn, int nt, int cluster, size_t smem, int* out) {
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_occ.find(std::make_tuple(dev, fn, cluster, smem));
    if (it != g_occ.end()) {
      *out = it->second;
      return cudaSuccess;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(cluster, 1, 1);
  cfg.blockDim = dim3(nt, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  cudaError_t e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mu);
  g_occ[std::make_tuple(dev, fn, cluster, smem)] = n;
  *out = n;
  return cudaSuccess;
}

struct RowPlan {
  const void* fn;
  int nt, cluster, nclusters;
  size_t smem;
  RowParams p;
};

// Chooses threads per CTA, cluster size, slice and staging depth for a (dtype, V) pair.
// Resident CTAs of the row kernel on this device (SMs x CTAs per SM), cached per kernel and size.
std::map<std::tuple<int, const void*, size_t>, int> g_resident;
cudaError_t resident_ctas(const void* fn, int nt, size_t smem, int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = g_resident.find(std::make_tuple(dev, fn, smem));
    if (it != g_resident.end()) {
      *out = it->second;
      return cudaSuccess;
    }
  }
  e = prepare_kernel(dev, fn);
  if (e != cudaSuccess) return e;
  int sms = 0, per_sm = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, nt, smem);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(g_mu);
  g_resident[std::make_tuple(dev, fn, smem)] = sms * per_sm;
  *out = sms * per_sm;
  return cudaSuccess;
}

spec_status_t plan_rows(const void* target, const void* draft, int dtype, int B, int K, int V,
                        float T, bool need_draft, bool stats_only, RowPlan* plan) {
  const bool bf16 = dtype == SPEC_BF16;
  const bool greedy = T == 0.f;
  const int esz = bf16 ? 2 : 4;
  // clusters of C CTAs, each CTA streaming a slice of V / C logits per row in 4096-logit items
  const int nt = 256;                       // 8 warps, each thread streaming its own chunks
  const int item = 4096;
  const void* fn = bf16 ? sv::sample_kernel_bf16(nt) : sv::sample_kernel_f32(nt);
  const int units = B * (stats_only ? K : K + 1);
  int cluster = 0;
  if (g_force_cluster.load()) {
    if (g_force_cluster.load() * 32 * item < V) return SPEC_ERR_UNSUPPORTED;
    cluster = g_force_cluster.load();
  } else {
    // The kernel is issue-bound and a unit's CTAs work in lockstep.  Split rows across more CTAs
    // while each slice keeps at least 7 items (so per-unit exchanges stay small against the
    // streaming) and there are at most 2.5 CTA-tasks (units x C) per resident CTA slot (beyond
    // that the extra per-unit rounds cost more than the finer balance gains).  A slice holds at
    // most 32 items.
    int slots = 0;
    if (resident_ctas(fn, nt, 2 * static_cast<size_t>(item) * esz * sv::kStreamStagesHost, &slots) != cudaSuccess)
      return SPEC_ERR_CUDA;
    const int cmin = (V + 32 * item - 1) / (32 * item);
    cluster = 1;
    while (cluster * 2 <= sv::kMaxCluster && static_cast<long long>(V) >= 2ll * cluster * 7 * item &&
           static_cast<long long>(units) * cluster * 2 * 2 <= 5ll * slots)
      cluster *= 2;
    while (cluster < cmin) cluster *= 2;
  }
  if (cluster > sv::kMaxCluster) return SPEC_ERR_UNSUPPORTED;
  int slice = (V + cluster - 1) / cluster;
  slice = static_cast<int>(align_up(slice, sv::kChunk));
  if (slice > 32 * item) return SPEC_ERR_UNSUPPORTED;
  const bool tma = (static_cast<size_t>(V) * esz) % 16 == 0 && aligned16(target) &&
                   (!need_draft || aligned16(draft));
  const int stage_row_bytes = item * esz;
  const size_t stage_bytes = 2 * static_cast<size_t>(stage_row_bytes);
  // the kernel's copy pipeline is kStreamStages items deep: bf16 64 KB per CTA (three CTAs per
  // SM), fp32 128 KB (one CTA per SM)
  const int nstage = sv::kStreamStagesHost;
  (void)greedy;
  plan->fn = fn;
  plan->nt = nt;
  plan->cluster = cluster;
  plan->smem = static_cast<size_t>(nstage) * stage_bytes;
  RowParams& p = plan->p;
  std::memset(&p, 0, sizeof(p));
  p.target = target;
  p.draft = draft;
  p.B = B;
  p.K = K;
  p.V = V;
  p.U = stats_only ? K : K + 1;
  p.total_units = B * p.U;
  p.slice = slice;
  p.nstage = nstage;
  p.stage_row_bytes = stage_row_bytes;
  p.flags = (need_draft ? sv::F_NEED_DRAFT : 0) | (stats_only ? sv::F_STATS_ONLY : 0) |
            (tma ? sv::F_TMA : 0);
  p.c = greedy ? 0.f : static_cast<float>(1.4426950408889634 / static_cast<double>(T));
  p.wait_limit = g_wait_limit.load();
  return SPEC_OK;
}

spec_status_t launch_plan(RowPlan* plan, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
  if (prepare_kernel(dev, plan->fn) != cudaSuccess) return SPEC_ERR_CUDA;
  int maxc = 0;
  if (max_clusters(dev, plan->fn, plan->nt, plan->cluster, plan->smem, &maxc) != cudaSuccess)
    return SPEC_ERR_CUDA;
  if (maxc < 1) return SPEC_ERR_UNSUPPORTED;
  const int ncl = plan->p.total_units < maxc ? plan->p.total_units : maxc;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = plan->cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(ncl * plan->cluster, 1, 1);
  cfg.blockDim = dim3(plan->nt, 1, 1);
  cfg.dynamicSmemBytes = plan->smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {&plan->p};
  if (cudaLaunchKernelExC(&cfg, plan->fn, args) != cudaSuccess) return SPEC_ERR_CUDA;
  const int rec[8] = {plan->nt, plan->cluster, ncl, maxc, plan->p.slice, plan->p.nstage,
                      static_cast<int>(plan->smem), plan->p.flags};
  std::memcpy(g_last_plan, rec, sizeof(rec));
  return SPEC_OK;
}

bool bad_T(float T) { return !(T >= 0.f) || std::isinf(T); }

// Greedy path: the streaming argmax kernel over target rows (and draft rows when need_draft).
// Ring: stages of 8 tiles (16 KB bf16 / 32 KB fp32); about 64 KB per CTA.
std::map<int, int> g_argmax_grid;
spec_status_t launch_greedy(const void* target, const void* draft, int dtype, int B, int K, int V,
                            bool need_draft, bool stats_only, bool fused_cut, uint64_t* keys,
                            sv::ArgmaxParams cut, cudaStream_t stream) {
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
      if (sv::argmax_blocks_per_sm(dtype == SPEC_BF16, 0, &per_sm) != cudaSuccess)
        return SPEC_ERR_CUDA;
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
  const int variant = g_variant.load();
  p.fused_cut = fused_cut && !(variant & 2);
  p.stats_only = stats_only;
  p.wait_limit = g_wait_limit.load();
  const int esz = dtype == SPEC_BF16 ? 2 : 4;
  p.aligned = (static_cast<size_t>(V) * esz) % 16 == 0 && aligned16(target) && (!need_draft || aligned16(draft));
  // every warp takes the same number of tiles (the fewest one resident wave allows), so no
  // warp is left with an extra tile after the others finish
  const long long per_warp = (p.total_tiles + 8ll * grid_cap - 1) / (8ll * grid_cap);
  long long grid = (p.total_tiles + 8 * per_warp - 1) / (8 * per_warp);
  if (variant & 4) grid = (p.total_tiles + 7) / 8;   // every resident CTA slot, tiles spread evenly
  if (grid > grid_cap) grid = grid_cap;
  if (grid < 1) grid = 1;
  if (sv::launch_argmax(dtype == SPEC_BF16, p, static_cast<int>(grid), stream) != cudaSuccess) return SPEC_ERR_CUDA;
  const int rec[8] = {256, 1, static_cast<int>(grid), grid_cap, tile, 0,
                      0, -1};
  std::memcpy(g_last_plan, rec, sizeof(rec));
  return SPEC_OK;
}

spec_status_t check_ws(void* ws, size_t ws_bytes, int B, int K) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) % kAlign) != 0) return SPEC_ERR_WORKSPACE;
  if (ws_bytes < ws_bytes_needed(B, K)) return SPEC_ERR_WORKSPACE;
  if (ws_layout_for(ws_bytes).cap_rows < static_cast<size_t>(B) * (K + 1)) return SPEC_ERR_WORKSPACE;
  return SPEC_OK;
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

spec_status_t run_verify(const VerifyArgs& a) {
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
  uint64_t* keys = reinterpret_cast<uint64_t*>(ws + L.keys);
  int32_t* counters = reinterpret_cast<int32_t*>(ws + L.counters);
  int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
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
    st = launch_greedy(a.target, a.draft, a.dtype, a.B, a.K, a.V, need_draft, false, !budget, keys, cut,
                       a.stream);
    if (st != SPEC_OK) return st;
    if (!budget && (g_variant.load() & 2) == 0) return SPEC_OK;   // the cut ran inside the argmax kernel
  } else {
    RowPlan plan;
    st = plan_rows(a.target, a.draft, a.dtype, a.B, a.K, a.V, a.T, need_draft, false, &plan);
    if (st != SPEC_OK) return st;
    RowParams& p = plan.p;
    p.tokens = a.tokens;
    p.uniforms = a.uniforms;
    p.depth = a.depth;
    p.recs = recs;
    p.status = status;
    if (budget) p.flags |= sv::F_ALL_PDRAWS;
    st = launch_plan(&plan, a.stream);
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
  const cudaError_t e = budget ? sv::launch_budget_cut(bp, a.stream) : sv::launch_cut(bp, a.depth, a.stream);
  return e == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace

extern "C" {

int spec_version(void) { return 100; }

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
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) % kAlign) != 0) return SPEC_ERR_WORKSPACE;
  return cudaMemsetAsync(workspace, 0, ws_bytes, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SPEC_OK
             : SPEC_ERR_CUDA;
}

spec_status_t spec_get_status(void* workspace, void* stream, int32_t* out_status) {
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
  VerifyArgs a = {target_logits, draft_logits, dtype, tokens, uniforms, B, K, V, temperature,
                  depth, -1, out_tokens, out_accepted, out_alpha, nullptr, nullptr, nullptr,
                  workspace, ws_bytes, static_cast<cudaStream_t>(stream)};
  return run_verify(a);
}

spec_status_t spec_verify_block(const void* target_logits, const void* draft_logits, int dtype,
                                const int32_t* tokens, const float* uniforms, int B, int K, int V,
                                float temperature, const int32_t* depth, int budget_N,
                                int32_t* out_tokens, int32_t* out_accepted, float* out_alpha,
                                float* out_cum_alpha, float* out_expected_len, int32_t* out_depth,
                                void* workspace, size_t ws_bytes, void* stream) {
  VerifyArgs a = {target_logits, draft_logits, dtype, tokens, uniforms, B, K, V, temperature,
                  depth, budget_N, out_tokens, out_accepted, out_alpha, out_cum_alpha,
                  out_expected_len, out_depth, workspace, ws_bytes, static_cast<cudaStream_t>(stream)};
  return run_verify(a);
}

spec_status_t spec_overlap_alpha(const void* target_logits, const void* draft_logits, int dtype,
                                 int B, int K, int V, float temperature, float* out_alpha,
                                 float* out_cum_alpha, float* out_expected_len, void* workspace,
                                 size_t ws_bytes, void* stream) {
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
  uint64_t* keys = reinterpret_cast<uint64_t*>(ws + L.keys);
  int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
  const bool greedy = temperature == 0.f;
  if (greedy) {
    sv::ArgmaxParams cut;
    std::memset(&cut, 0, sizeof(cut));
    cut.counters = reinterpret_cast<int32_t*>(ws + L.counters);
    cut.status = status;
    cut.out_alpha = out_alpha;
    cut.out_cum = out_cum_alpha;
    cut.out_E = out_expected_len;
    st = launch_greedy(target_logits, draft_logits, dtype, B, K, V, true, true, true, keys, cut,
                       static_cast<cudaStream_t>(stream));
    if (st != SPEC_OK || (g_variant.load() & 2) == 0) return st;
  } else {
    RowPlan plan;
    st = plan_rows(target_logits, draft_logits, dtype, B, K, V, temperature, true, true, &plan);
    if (st != SPEC_OK) return st;
    plan.p.recs = recs;
    plan.p.status = status;
    st = launch_plan(&plan, static_cast<cudaStream_t>(stream));
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
  return sv::launch_cut(bp, nullptr, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status_t spec_alloc_budget(const float* alpha, int B, int K, int budget_N, int32_t* out_depth,
                                float* out_conf, void* workspace, size_t ws_bytes, void* stream) {
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

void spec_debug_set_wait_limit(long long limit_us) {
  g_wait_limit.store(limit_us < 0 ? kDefaultWaitLimit : limit_us * 1000);
}

void spec_debug_set_plan(int threads, int cluster, int nstage) {
  g_force_nt.store(threads == 256 || threads == 512 ? threads : 0);
  g_force_cluster.store(cluster > 0 && cluster <= sv::kMaxCluster ? cluster : 0);
  g_force_nstage.store(nstage > 0 && nstage <= 16 ? nstage : 0);
}

void spec_debug_set_variant(int variant) { g_variant.store(variant & 7); }

void spec_debug_last_plan(int32_t* out8) {
  if (out8) std::memcpy(out8, g_last_plan, sizeof(g_last_plan));
}

}  // extern "C"

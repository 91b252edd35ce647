// Greedy chain verification that allocates nothing and takes no workspace.
//
// Some callers cannot hand the library a device workspace: engines that reserve all of their
// device memory at start-up through their own pool and expose no allocator to plug-ins, hosts
// that forbid device allocations after initialisation because cudaMalloc / cudaFree can
// synchronise the whole device and stall every stream, and embedders whose memory budget is
// fixed per model.  For them this entry point keeps its scratch (status word, per-row argmax
// slots, per-request completion counters) in one file-scope device array of fixed size that
// every GPU loading the library holds until the process exits.
#include "../../include/spec_verify.h"
#include "api_range.h"
#include "spec_internal.h"

namespace {

// Largest batch the fixed scratch serves: B * (K + 1) rows.
constexpr int kStaticMaxRows = SPEC_STATIC_MAX_ROWS;
constexpr size_t kStatusBytes = 256;
constexpr size_t kKeysBytes = static_cast<size_t>(kStaticMaxRows) * 2 * sizeof(uint64_t);
constexpr size_t kCountersBytes = static_cast<size_t>(kStaticMaxRows) * sizeof(int32_t);
constexpr size_t kStaticBytes = kStatusBytes + kKeysBytes + kCountersBytes;   // 80.25 KiB

// The scratch itself.  In host code this name is only a stand-in for the device object: its
// device address comes from cudaGetSymbolAddress on each device.
static __device__ __align__(256) unsigned char g_static_scratch[kStaticBytes];

// Device address of the scratch in the current device's context, looked up on every call (a
// host-side table lookup once the module is loaded).  Nothing is cached: after a device reset, or
// in another context on the same device, the module is loaded again and the array can move.
spec_status_t scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return SPEC_ERR_CUDA;
  *out = p;
  return SPEC_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" spec_status_t spec_verify_chain_greedy_static(const void* target_logits, const void* draft_logits,
                                                         int dtype, const int32_t* tokens, int B, int K, int V,
                                                         const int32_t* depth, int32_t* out_tokens,
                                                         int32_t* out_accepted, float* out_alpha,
                                                         int32_t* out_status, void* stream) {
  const sv::ApiRange range("spec_verify_chain_greedy_static");
  if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_ERR_INVALID_ARG;
  if (B < 0 || K < 0 || V < 1) return SPEC_ERR_INVALID_ARG;
  if (K > sv::kMaxK || V > 262144) return SPEC_ERR_UNSUPPORTED;
  if (B == 0) return SPEC_OK;
  if (static_cast<long long>(B) * (K + 1) > kStaticMaxRows) return SPEC_ERR_UNSUPPORTED;
  if (!target_logits || !out_tokens || !out_accepted) return SPEC_ERR_INVALID_ARG;
  if (K > 0 && !tokens) return SPEC_ERR_INVALID_ARG;
  const bool need_draft = K > 0 && out_alpha != nullptr;
  if (need_draft && !draft_logits) return SPEC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  void* base = nullptr;
  spec_status_t st = scratch_address(&base);
  if (st != SPEC_OK) return st;
  uint8_t* scratch = static_cast<uint8_t*>(base);
  int32_t* status = reinterpret_cast<int32_t*>(scratch);
  uint64_t* keys = reinterpret_cast<uint64_t*>(scratch + kStatusBytes);
  int32_t* counters = reinterpret_cast<int32_t*>(scratch + kStatusBytes + kKeysBytes);
  // the array keeps the previous call's contents: clear the status word, the slots and the
  // counters this call uses
  const size_t rows = static_cast<size_t>(B) * (K + 1);
  if (cudaMemsetAsync(status, 0, sizeof(int32_t), s) != cudaSuccess) return SPEC_ERR_CUDA;
  if (cudaMemsetAsync(keys, 0, rows * 2 * sizeof(uint64_t), s) != cudaSuccess) return SPEC_ERR_CUDA;
  if (cudaMemsetAsync(counters, 0, static_cast<size_t>(B) * sizeof(int32_t), s) != cudaSuccess) return SPEC_ERR_CUDA;

  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SPEC_ERR_CUDA;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return SPEC_ERR_CUDA;
  if (sv::argmax_blocks_per_sm(dtype == SPEC_BF16, &per_sm) != cudaSuccess) return SPEC_ERR_CUDA;

  sv::ArgmaxParams p = {};
  p.target = target_logits;
  p.draft = need_draft ? draft_logits : nullptr;
  p.keys = keys;
  p.counters = counters;
  p.status = status;
  p.tokens = tokens;
  p.depth = depth;
  p.out_tokens = out_tokens;
  p.out_accepted = out_accepted;
  p.out_alpha = out_alpha;
  p.B = B;
  p.K = K;
  p.V = V;
  p.rows_t = K + 1;
  p.drows = need_draft ? K : 0;
  const int tile = dtype == SPEC_BF16 ? 2048 : 1024;   // the argmax kernel's warp tile
  p.tpr = (V + tile - 1) / tile;
  p.total_tiles = static_cast<long long>(B) * (p.rows_t + p.drows) * p.tpr;
  const int esz = dtype == SPEC_BF16 ? 2 : 4;
  p.aligned = (static_cast<size_t>(V) * esz) % 16 == 0 && aligned16(target_logits) &&
              (!need_draft || aligned16(draft_logits));
  p.wait_limit = 200000000ll;   // ns (this kernel has no waits)
  p.fused_cut = 1;
  p.stats_only = 0;
  long long grid = (p.total_tiles + 7) / 8;
  const long long cap = static_cast<long long>(sms) * (per_sm > 0 ? per_sm : 1);
  if (grid > cap) grid = cap;
  if (grid < 1) grid = 1;
  if (sv::launch_argmax(dtype == SPEC_BF16, p, static_cast<int>(grid), s) != cudaSuccess) return SPEC_ERR_CUDA;
  if (out_status &&
      cudaMemcpyAsync(out_status, status, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return SPEC_ERR_CUDA;
  return SPEC_OK;
}

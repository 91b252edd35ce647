// Internal declarations shared by the kernels and the C-ABI host code.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

constexpr int kChunk = 8;         // logits held per register chunk
constexpr int kMaxCluster = 16;   // CTAs that share one row (non-portable cluster size)
constexpr int kMaxK = 31;         // drafted positions per request (lanes 0..K of one warp in the cut)
// Sampling kernel geometry: 8 warps per CTA; per item every lane loads kSampPieces 16-byte pieces
// of each row straight into registers.
#ifndef SPEC_SAMP_PIECES
#define SPEC_SAMP_PIECES 4
#endif
#ifndef SPEC_SAMP_MINB
#define SPEC_SAMP_MINB 3
#endif
constexpr int kSampWarps = 8;
constexpr int kSampPieces = SPEC_SAMP_PIECES;
constexpr int kSampWarpBytes = kSampPieces * 512;                    // one row, one item, one warp
constexpr int kSampItemBytes = kSampWarps * kSampWarpBytes;           // one row, one item
constexpr int kSampMinBlocks = SPEC_SAMP_MINB;                        // resident CTAs per SM the registers allow
// A CTA's slice of a unit (target and draft row) stays in a shared-memory slab of at most
// kSampMaxItems items per row (192 KB) between the two passes.
constexpr int samp_slab_bytes(int items) { return kSampWarps * items * 2 * kSampWarpBytes; }
constexpr int kSampMaxItems = (192 * 1024) / samp_slab_bytes(1);
constexpr int kSampMaxSlabBytes = samp_slab_bytes(kSampMaxItems);

// Status bits in the workspace's device status word.
constexpr int kStatusTimeout = 1;
constexpr int kStatusTokenRange = 2;

// Per (request, position) results of the sampling row kernel; 32 bytes.  Written by CTA 0 of the
// unit's cluster once the row normalisers are known.
struct UnitRec {
  float px, qx;      // p_k(x_k), q_k(x_k)
  float offt, offd;  // p_v = 2^(z_T[v] c - offt), q_v = 2^(z_D[v] c - offd)
  int32_t mode;      // pass-2 work done: kModeAlpha, kModeFull or kModeSingle
  float alpha;       // sum_v min(p_v, q_v) of a pair, clamped to [0, 1] (written after the next exchange)
  int32_t rej;       // 1: the accept test u_k q_k(x_k) < p_k(x_k) fails at this position (k < K)
  int32_t pad;
};
static_assert(sizeof(UnitRec) == 32 && offsetof(UnitRec, alpha) == 20 && offsetof(UnitRec, rej) == 24,
              "the budget kernel reads (mode, alpha, rej) as the record's second 16-byte word");
enum : int32_t { kModeAlpha = 0, kModeFull = 1, kModeSingle = 2 };

// Per-row mass table of the sampling kernel, written by every warp of every CTA of the unit's
// cluster for rows that may draw (full / single mode), floats:
//   m[((c * itmax + it) * kSampWarps + w) * 2]  (R, P): residual mass sum max(0, p - q) and sum p of
//                                      item `it` of warp w of CTA c
// in vocabulary order (c, it, w).  The cut kernels draw from these.  (The draft-side budget
// reuses the region for its per-part row partials.)
constexpr int kMassMaxSegments = 80;                     // CTA x item segments of a row
constexpr int kMassRowFloats = kMassMaxSegments * kSampWarps * 2;

// Greedy path: per (request, position) two 64-bit argmax keys (target row, draft row), folded
// with atomicMax by the argmax kernel and cleared by the kernel that consumes them.

struct ArgmaxParams {
  const void* target;        // [B, K+1, V]
  const void* draft;         // [B, K, V] or null
  uint64_t* keys;            // [B, K+1, 2]
  int32_t* counters;         // [B] finished tiles per request (zero between calls)
  int32_t* status;
  const int32_t* tokens;     // [B, K] (fused cut)
  const int32_t* depth;      // [B] or null (fused cut)
  int32_t* out_tokens;
  int32_t* out_accepted;
  float* out_alpha;
  float* out_cum;
  float* out_E;
  int B, K, V;
  int rows_t;                // target rows scanned per request (K+1, or K for overlap stats)
  int drows;                 // draft rows scanned per request (K when the one-hot alpha is wanted)
  int tpr;                   // tiles per row
  long long total_tiles;     // B * (rows_t + drows) * tpr
  int aligned;               // rows start on 16-byte boundaries: 16-byte vector loads
  long long wait_limit;      // ns of wall time per bounded wait; 0 = give up at once
  int fused_cut;             // the warp that completes a request runs its cut
  int stats_only;            // overlap statistics only (no tokens)
};

enum : int {
  F_NEED_DRAFT = 1,   // draft rows are read for positions k < K
  F_STATS_ONLY = 2,   // rows k < K only; alpha, no draws
  F_ALIGNED = 8,      // rows start on 16-byte boundaries: staged by 16-byte asynchronous copies
  F_ALL_PDRAWS = 16,  // draw from p at every row (the verified depth is chosen afterwards)
};

struct RowParams {
  const void* target;        // [B, K+1, V]
  const void* draft;         // [B, K, V] or null
  const int32_t* tokens;     // [B, K]
  const float* uniforms;     // [B, K+1]
  const int32_t* depth;      // [B] or null
  int32_t* out_tokens;       // [B, K+1] or null
  int32_t* out_accepted;     // [B] or null
  float* out_alpha;          // [B, K] or null
  float* out_cum;            // [B, K] or null
  float* out_E;              // [B] or null
  UnitRec* recs;             // [B, U]
  float* mass;               // [B, U] mass tables of kMassRowFloats
  int32_t* status;           // 1 word
  int B, K, V;
  int U;                     // rows (units) per request: K+1, or K in stats-only mode
  int total_units;           // B * U
  int slice;                 // logits per CTA slice (multiple of kChunk)
  int itmax;                 // items of the first (longest) slice
  int flags;
  float c;                   // log2(e) / T  (T > 0)
  long long wait_limit;      // ns of wall time per bounded wait; 0 = give up at once
};

struct BudgetParams {
  const float* alpha_in;     // [B, K] caller alpha, or null: from recs / keys
  const UnitRec* recs;
  const float* mass;         // sampling path: [B, U] mass tables
  const void* target;        // sampling path: logits, for the one draw per request
  const void* draft;
  float c;                   // log2(e) / T
  int bf16, aligned;         // logits element type; rows start on 16-byte boundaries
  int ncta, slice, itmax;    // the sampling kernel's cluster size, slice and items per slice
  uint64_t* keys;            // greedy path: argmax keys [B, K+1, 2] (cleared after use)
  int draft_keys;            // greedy path: draft keys were produced (one-hot alpha)
  int U;
  int B, K, V, N;
  int greedy, do_cut, stats_only;
  const int32_t* tokens;
  const float* uniforms;
  int32_t* out_depth;        // [B] or null
  float* out_conf;           // [B, K] or null
  int32_t* out_tokens;
  int32_t* out_accepted;
  float* out_alpha;
  float* out_cum;
  float* out_E;
  int32_t* status;
  // draft-side confidence: per-row partials of the draft statistics kernel (alpha_k is then
  // q_k(x_k), read from the draft row), or null
  const float4* draft_part;  // [B*K, nparts]: (max, sum of 2^((z - max) c), first argmax index, 0)
  int nparts;
  int draft_greedy;          // T = 0: q_k(x_k) = [x_k == argmax]
  // the utility / cost choice of N (n_cost > 0; N is then ignored)
  const float* cost_n;       // [n_cost] strictly increasing
  const float* cost_t;       // [n_cost]
  int n_cost;
  int32_t* out_N;            // the chosen N, or null
};

// Per-row partials of the draft rows alone: one CTA per (row, part) of part_len logits.
struct DraftStatsParams {
  const void* draft;         // [rows, V]
  int rows, V, nparts, part_len;
  float c;                   // log2(e) / T (unused at T = 0)
  float4* out;               // [rows, nparts]
};
constexpr int kDraftStatsThreads = 256;
constexpr int kBudgetMaxCost = 64;     // cost-table points

// Host-side launchers of the small kernels (defined next to them).
cudaError_t launch_draft_stats(bool bf16, bool greedy, bool aligned, const DraftStatsParams& p, cudaStream_t stream);
cudaError_t launch_argmax(bool bf16, const ArgmaxParams& p, int grid, cudaStream_t stream);
cudaError_t argmax_blocks_per_sm(bool bf16, int* out);
cudaError_t launch_budget_cut(const BudgetParams& p, cudaStream_t stream, bool pdl = true);
cudaError_t launch_cut(const BudgetParams& p, const int32_t* depth, cudaStream_t stream, bool pdl = true);

}  // namespace sv

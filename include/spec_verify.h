/*
 * spec_verify.h - C ABI of the batched draft-verification library (sm_103a).
 *
 * The operation is speculative-decoding verification as described on the
 * AngelSpec / DFly pages (agifrontier tutorial, section "KL to end-to-end
 * TV loss"; abstract; section on verification as a shared batch-level pool):
 *
 *   p_k = softmax(z_T[b,k,:] / T),  q_k = softmax(z_D[b,k,:] / T)
 *   alpha_k = sum_v min(p_k(v), q_k(v)) = 1 - TV(p_k, q_k)
 *   c_m = prod_{k<=m} alpha_k,   E = sum_{m<K} c_m (expected accepted drafts)
 *   serial test at k = 0..d_b-1:  accept x_k iff u[b,k] * q_k(x_k) < p_k(x_k);
 *   the first rejection at n emits a draw from norm(max(0, p_n - q_n)),
 *   full acceptance emits a bonus draw from p_{d_b};
 *   T == 0: accept iff x_k == argmax z_T[b,k] (lowest index on ties); the
 *   emitted token is the target argmax at the first mismatch or at d_b.
 * Draws use the inverse CDF in vocabulary order: the smallest v whose
 * inclusive prefix mass is strictly above u[b,K] * (total mass).
 * The budget spends N verified positions on the N best prefix confidences
 * c[b,m] over the whole batch (order: c desc, m asc, b asc), which is
 * prefix-closed and yields a per-request depth d_b.
 *
 * Conventions for every entry point
 * - Pointers named *_logits, tokens, uniforms, depth, out_* and workspace
 *   are DEVICE pointers (cudaMalloc / torch CUDA memory) on the current
 *   device; tensors are dense row-major: target [B, K+1, V], draft [B, K, V],
 *   tokens [B, K] int32, uniforms [B, K+1] float32, outputs as stated.
 * - The caller owns every buffer.  The library allocates no device memory,
 *   keeps no per-call state, and never synchronises the stream except in
 *   spec_get_status.  Every call is asynchronous on `stream` (a cudaStream_t
 *   passed as void*, NULL = legacy default stream).
 * - Argument errors are returned synchronously (nothing is launched).
 *   Data errors found on the device (a draft token outside [0, V), a wait
 *   that ran out) are recorded in a status word inside the workspace and
 *   read with spec_get_status.
 * - The workspace (at least spec_workspace_bytes) holds the status word,
 *   per-row intermediate records and per-row argmax slots that every call
 *   leaves zeroed.  Its layout depends only on ws_bytes: zero-fill it
 *   (spec_workspace_init) before its first use and again whenever the same
 *   buffer is passed with a different ws_bytes.  Calls that share a
 *   workspace must be ordered on one stream.
 * - Launches on `stream`: at T == 0 without a budget one kernel (the argmax,
 *   with the serial cut fused in); otherwise the row kernel and a small kernel
 *   (the serial cut, or the budget and the cut) chained to it with
 *   programmatic dependent launch.
 * - Logits may contain -inf (probability 0); each row needs one finite
 *   value.  NaN / +inf give unspecified tokens (they are not scanned for).
 * - Limits: 1 <= V <= 262144 (fp32 logits at T > 0: V <= 131072),
 *   0 <= K <= 31, B >= 0 (B == 0 is a no-op), T >= 0 and finite.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SPEC_OK = 0,
  SPEC_ERR_INVALID_ARG = 1,     /* bad pointer, size, dtype, temperature */
  SPEC_ERR_UNSUPPORTED = 2,     /* shape outside the limits above */
  SPEC_ERR_CUDA = 3,            /* a launch or runtime call failed */
  SPEC_ERR_DEVICE_TIMEOUT = 4,  /* a bounded on-device wait ran out */
  SPEC_ERR_TOKEN_RANGE = 5,     /* a draft token id outside [0, V) */
  SPEC_ERR_WORKSPACE = 6        /* workspace too small or misaligned */
} spec_status_t;

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype_t;

/* Library version (major*10000 + minor*100 + patch). */
int spec_version(void);

/* Static text for a status code. */
const char* spec_error_string(int status);

/* Bytes of workspace a call with these sizes needs (256-byte aligned start). */
size_t spec_workspace_bytes(int B, int K, int V, int dtype);

/* Zero-fill a workspace once before its first use (cudaMemsetAsync). */
spec_status_t spec_workspace_init(void* workspace, size_t ws_bytes, void* stream);

/*
 * Read and clear the device status word of a workspace.  Synchronises
 * `stream`.  *out_status receives SPEC_OK, SPEC_ERR_TOKEN_RANGE or
 * SPEC_ERR_DEVICE_TIMEOUT (the first two bits found, in that priority:
 * timeout first).  After SPEC_ERR_DEVICE_TIMEOUT re-initialise the
 * workspace before reuse.
 */
spec_status_t spec_get_status(void* workspace, void* stream, int32_t* out_status);

/*
 * Verify an MTP chain (K = drafting depth).  Serial acceptance, first
 * rejection cut, residual / bonus draw (AngelSpec pages, "KL to end-to-end
 * TV loss": alpha = 1 - TV and the multiplicative, serial acceptance).
 *
 *   target_logits [B, K+1, V] dtype; row K is the bonus position.
 *   draft_logits  [B, K, V] dtype; may be NULL iff temperature == 0 and
 *                 out_alpha == NULL.
 *   tokens        [B, K] int32 drafted ids.
 *   uniforms      [B, K+1] float32 in [0, 1); u[b,k] tests position k,
 *                 u[b,K] drives the final draw.  Ignored at T == 0 (may be
 *                 NULL then).
 *   temperature   T > 0 stochastic, T == 0 greedy; negative or NaN ->
 *                 SPEC_ERR_INVALID_ARG.
 *   depth         [B] int32 in [0, K] (e.g. from spec_alloc_budget) or NULL
 *                 (= K): positions >= depth[b] are not tested and the bonus
 *                 is drawn at depth[b].  Values outside [0, K] are clamped.
 *   out_tokens    [B, K+1] int32: accepted drafts, then the emitted token,
 *                 then -1.
 *   out_accepted  [B] int32: number n_b of accepted drafts (emitted = n+1).
 *   out_alpha     [B, K] float32 or NULL (at T == 0: 1 if the argmaxes of
 *                 target and draft agree, else 0).
 */
spec_status_t spec_verify_chain(const void* target_logits, const void* draft_logits, int dtype,
                                const int32_t* tokens, const float* uniforms,
                                int B, int K, int V, float temperature,
                                const int32_t* depth,
                                int32_t* out_tokens, int32_t* out_accepted, float* out_alpha,
                                void* workspace, size_t ws_bytes, void* stream);

/*
 * Verify a DFly block (K = block size) with the same rule as the chain
 * (block drafts are accepted left to right, AngelSpec pages, DFly section),
 * plus the block statistics and, optionally, the batch-level budget:
 *
 *   out_cum_alpha    [B, K] float32 prod_{k<=m} alpha_k, or NULL.
 *   out_expected_len [B] float32 sum_m prod_{k<=m} alpha_k, or NULL
 *                    (the L_e2e summand of the "KL to end-to-end TV loss"
 *                    section).
 *   budget_N         < 0: no budget (depth as in spec_verify_chain);
 *                    >= 0: spend N verified positions over the batch on the
 *                    best prefix confidences (the D-cut shared pool, section
 *                    on verification as a shared batch-level resource); the
 *                    depth argument must then be NULL.  The logits are read
 *                    once: alpha of every position, the budget and the
 *                    decisions come from that one pass.
 *   out_depth        [B] int32 chosen depth d_b, or NULL.
 * B * K <= 8192 when budget_N >= 0.  draft_logits is required when
 * budget_N >= 0 (alpha needs it, also at T == 0).
 */
spec_status_t spec_verify_block(const void* target_logits, const void* draft_logits, int dtype,
                                const int32_t* tokens, const float* uniforms,
                                int B, int K, int V, float temperature,
                                const int32_t* depth, int budget_N,
                                int32_t* out_tokens, int32_t* out_accepted, float* out_alpha,
                                float* out_cum_alpha, float* out_expected_len, int32_t* out_depth,
                                void* workspace, size_t ws_bytes, void* stream);

/*
 * Overlap statistics only (no decisions): alpha_k for k < K, the prefix
 * confidences and the expected accepted length (AngelSpec pages, "KL to
 * end-to-end TV loss", inline formula and L_e2e summand).  Reads target
 * rows 0..K-1 of the [B, K+1, V] tensor and the [B, K, V] draft tensor.
 * out_alpha [B, K] required; out_cum_alpha [B, K] and out_expected_len [B]
 * may be NULL.  T == 0 gives the one-hot limit.
 */
spec_status_t spec_overlap_alpha(const void* target_logits, const void* draft_logits, int dtype,
                                 int B, int K, int V, float temperature,
                                 float* out_alpha, float* out_cum_alpha, float* out_expected_len,
                                 void* workspace, size_t ws_bytes, void* stream);

/*
 * Batch-level verification budget (AngelSpec abstract and the section on
 * verification as a shared batch-level resource): alpha [B, K] (device,
 * float32; clamped to [0, 1], NaN read as 0) -> prefix confidences
 * c[b,m] = prod_{k<=m} alpha[b,k]; the first min(N, B*K) keys in the order
 * (c desc, m asc, b asc) are selected; out_depth[b] = number selected in
 * row b (prefix-closed).  out_conf [B, K] may be NULL.  N >= 0.
 * B * K <= 8192.  Needs no workspace contents beyond its status word.
 */
spec_status_t spec_alloc_budget(const float* alpha, int B, int K, int budget_N,
                                int32_t* out_depth, float* out_conf,
                                void* workspace, size_t ws_bytes, void* stream);

/*
 * The budget with N chosen online (AngelSpec, section on verification as a
 * shared pool: verification is spent where it pays against a profiled cost
 * of verifying more positions).  With the keys and selection of
 * spec_alloc_budget and S(N) the sum of the N largest prefix confidences,
 * N = the first N in 0 .. B*K maximising
 *     (B + S(N)) / cost(B + N),
 * B + N being the positions the batch verifies (every request verifies its
 * first emitted position).  cost is the table (cost_n [n_cost] strictly
 * increasing, cost_t [n_cost]; device, float32) interpolated piecewise-
 * linearly and held constant beyond its ends.  1 <= n_cost <= 64.
 * out_N (device int32, nullable) receives N; out_depth and out_conf as in
 * spec_alloc_budget.  B * K <= 8192.
 */
spec_status_t spec_alloc_budget_adaptive(const float* alpha, int B, int K,
                                         const float* cost_n, const float* cost_t, int n_cost,
                                         int32_t* out_N, int32_t* out_depth, float* out_conf,
                                         void* workspace, size_t ws_bytes, void* stream);

/*
 * The budget chosen from the draft alone, before the target runs (AngelSpec,
 * section on verification as a shared pool: the budget is decided from the
 * draft model's output distribution).  The confidence of drafted position
 * (b, k) is q_k(x_k) = softmax(draft_logits[b, k] / T)[tokens[b, k]] (at
 * T == 0 the one-hot [tokens[b, k] == argmax], lowest index on ties; 0 for a
 * token outside [0, V)), and the keys are its prefix products
 * c[b, m] = prod_{k<=m} q_k(x_k), selected as in spec_alloc_budget: with
 * n_cost == 0 the first min(budget_N, B*K) keys (budget_N >= 0), with
 * n_cost > 0 the N of spec_alloc_budget_adaptive (budget_N ignored).
 *   draft_logits  device [B, K, V], dtype SPEC_BF16 or SPEC_F32; one pass
 *   tokens        device int32 [B, K]
 *   out_N         device int32 or NULL: the N spent
 *   out_depth     device int32 [B]: per-request verification depth d_b
 *   out_conf      device float32 [B, K] or NULL: the prefix confidences
 * The caller then runs the target on the selected depths and verifies with
 * spec_verify_chain / spec_verify_block and `depth`.  B * K <= 8192.
 * Workspace as for spec_verify_block (spec_workspace_bytes(B, K, V, dtype)).
 */
spec_status_t spec_draft_budget(const void* draft_logits, int dtype, const int32_t* tokens,
                                int B, int K, int V, float temperature, int budget_N,
                                const float* cost_n, const float* cost_t, int n_cost,
                                int32_t* out_N, int32_t* out_depth, float* out_conf,
                                void* workspace, size_t ws_bytes, void* stream);

/*
 * Greedy (T == 0) chain verification that allocates nothing and needs no
 * workspace.  The pages have no counterpart: this entry point exists for
 * callers that cannot give the library device memory -- serving engines that
 * reserve all device memory up front in their own pool and expose no
 * allocator, and hosts that forbid cudaMalloc / cudaFree after start-up
 * because those calls can synchronise the whole device.
 *
 * Same result as spec_verify_chain at temperature 0 (tokens, accepted
 * counts, one-hot alpha when out_alpha is given; draft_logits needed only
 * then).  Its scratch (status word, argmax slots, request counters) is one
 * fixed device array of 80.25 KiB inside the library, held by every GPU that
 * loads it until the process exits:
 * - B * (K + 1) <= SPEC_STATIC_MAX_ROWS (4096), else SPEC_ERR_UNSUPPORTED;
 * - every call looks up the array's device address in the current device's
 *   context (cudaGetSymbolAddress); the first call on a device may load the
 *   module, so make it before any stream capture;
 * - every call clears the parts it uses (cudaMemsetAsync) and shares the one
 *   array, so calls that overlap on the GPU (other streams, other threads)
 *   race: order them on one stream;
 * - out_status (device int32, nullable) receives the raw status bits of the
 *   call: 1 = a bounded wait ran out, 2 = a draft token outside [0, V).
 * It calls no cudaMalloc, cudaFree or allocating library routine.
 */
#define SPEC_STATIC_MAX_ROWS 4096
spec_status_t spec_verify_chain_greedy_static(const void* target_logits, const void* draft_logits, int dtype,
                                              const int32_t* tokens, int B, int K, int V,
                                              const int32_t* depth, int32_t* out_tokens,
                                              int32_t* out_accepted, float* out_alpha,
                                              int32_t* out_status, void* stream);

/*
 * Test and tuning knobs of one call (no process-wide settings exist).  A
 * zero-filled struct means the defaults everywhere.
 *   wait_limit_us   0: default wall-time limit of every bounded on-device wait
 *                   (200 ms, read from the GPU's global timer); > 0: that
 *                   limit; < 0: every such wait gives up at once, which sets
 *                   SPEC_ERR_DEVICE_TIMEOUT in the status word (the kernel
 *                   then waits once more, up to 100 ms, so its copies and
 *                   cluster exchanges still complete before it returns).
 *   cluster         T > 0: CTAs per row of the sampling kernel (1, 2, 4, 8 or
 *                   16; a CTA's slice of a row must fit 6 items of 16 KB,
 *                   else SPEC_ERR_UNSUPPORTED); 0: chosen per call shape.
 *   greedy_variant  T == 0: bit 1 runs the cut in its own kernel instead of
 *                   fusing it into the argmax kernel; bit 2 launches every
 *                   resident CTA slot with the tiles spread evenly.
 *   split_event     a cudaEvent_t (as void*) or NULL: recorded on the stream
 *                   between the row kernel and the kernel chained after it
 *                   (which is then launched without programmatic dependent
 *                   launch), so a caller can time the two apart.
 *   plan_out        host int32[8] or NULL: receives the launched plan,
 *                   sampling kernel {threads, cluster, clusters launched, max
 *                   co-resident clusters, slice, items per slice, dynamic
 *                   shared memory bytes, flags};
 *                   argmax kernel {threads, 1, grid, resident CTAs, tile, 0,
 *                   0, -1}.
 */
typedef struct spec_tuning {
  long long wait_limit_us;
  int cluster;
  int greedy_variant;
  int32_t* plan_out;
  void* split_event;
} spec_tuning_t;

/*
 * spec_verify_block with per-call knobs (tuning may be NULL = defaults).
 * stats_only != 0 computes what spec_overlap_alpha computes (tokens,
 * uniforms, depth, budget_N, out_tokens, out_accepted and out_depth are then
 * ignored).  Same argument meaning, ownership and errors as those calls;
 * SPEC_ERR_INVALID_ARG for a cluster size that is not a power of two in
 * [1, 16].
 */
spec_status_t spec_verify_tuned(const void* target_logits, const void* draft_logits, int dtype,
                                const int32_t* tokens, const float* uniforms,
                                int B, int K, int V, float temperature,
                                const int32_t* depth, int budget_N, int stats_only,
                                int32_t* out_tokens, int32_t* out_accepted, float* out_alpha,
                                float* out_cum_alpha, float* out_expected_len, int32_t* out_depth,
                                void* workspace, size_t ws_bytes, void* stream,
                                const spec_tuning_t* tuning);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */

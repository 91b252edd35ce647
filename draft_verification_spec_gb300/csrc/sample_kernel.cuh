// Sampling-path row kernel (T > 0): two streaming passes per (request, position) unit.
//
// A thread-block cluster of C CTAs works on one unit at a time -- target row k and, for k < K,
// draft row k -- looping over units (persistent).  CTA r owns the vocabulary slice
// [r*slice, (r+1)*slice) of every row and walks it in items of kSampItemBytes per row.  Warp w of
// the CTA owns bytes [w*kSampWarpBytes, (w+1)*kSampWarpBytes) of every item and streams them itself:
// one lane issues a 1-D bulk copy (cp.async.bulk) per row into the warp's own ring of kSampStages
// stages, completing on the warp's own mbarrier, kSampStages - 1 items ahead, across pass and unit
// boundaries.  No producer warp, no shared stages, no per-thread copy bookkeeping: a lane reads
// its kSampPieces 16-byte pieces of each row with as many shared loads.
//
// Per unit:
//   pass 1 (from HBM): per-lane online (max, sum of 2^((z - m) c)) of the target and draft rows ->
//     warp butterfly merge -> exchange #1 with st.async into every CTA of the cluster, completing
//     on its mbarrier -> the row normalisers of p and q, merged in one fixed order so every warp of
//     every CTA holds bitwise-identical values; p_k(x_k), q_k(x_k) and the accept test, exactly as
//     the cut kernel evaluates them afterwards
//   pass 2 (the same bytes again, L2 hits while the data streamed in between fits in L2): per
//     logit p = 2^(z c - offt), q = 2^(z c - offd).  A pair that passes the test and needs no draw
//     only needs alpha = sum 2^min(a, b) (one exp2 per logit pair); otherwise per (item, warp)
//     masses of r = max(0, p - q) and of p -> CTA totals -> exchange #2 -> residual mass R,
//     alpha = sum p - R, and the owner of each needed inverse-CDF draw in vocabulary order
//     (CTA, item, warp), whose warp reloads its segment and walks piece / lane / element sums.
// A target row that no draw needs is skipped entirely.  DRAM reads each needed logit once.  The
// serial cut runs afterwards in a small kernel chained with programmatic dependent launch.
//
// Every wait is bounded by wall time.  A wait that runs out records SPEC_ERR_DEVICE_TIMEOUT and
// then waits once more with a long limit, so the exchange and copy protocol stays consistent and
// no copy or peer store lands in shared memory after the CTA has left.  Only if that second wait
// also runs out does the CTA stop waiting (abort mode), drain its own copies and leave.
#pragma once

#include <cuda_bf16.h>

#include "spec_async.cuh"

namespace sv {

constexpr int kSampThreads = 32 * kSampWarps;
constexpr long long kDrainNs = 100000000ll;            // second, long wait after a timeout (100 ms)

template <bool BF16>
struct SampGeo {
  static constexpr int ESZ = BF16 ? 2 : 4;
  static constexpr int EPP = 16 / ESZ;                 // logits per 16-byte piece
  static constexpr int NPC = kSampPieces;              // pieces per lane per row per item
  static constexpr int NWD = 4 * NPC;                  // 32-bit words per lane per row per item
  static constexpr int NP = BF16 ? NWD : NWD / 2;      // logit pairs per lane per row per item
  static constexpr int IL = kSampItemBytes / ESZ;      // logits per row per item
  static constexpr int WS = kSampWarpBytes / ESZ;      // logits per row per item per warp
  static constexpr int PS = 32 * EPP;                  // piece j of lane l: [j*PS + l*EPP, +EPP) of the warp's logits
};
__device__ __forceinline__ float lg2f(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed fp32 pairs (one 64-bit register pair) and Blackwell's paired fp32 FMA / add.
__device__ __forceinline__ uint64_t pk(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void upk(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// Logits 2i and 2i+1 of a lane's item words as a packed pair (bf16 halves widen exactly).
template <bool BF16, int N>
__device__ __forceinline__ uint64_t pair_of(const uint32_t (&w)[N], int i) {
  if constexpr (BF16) return pk(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
  else return pk(__uint_as_float(w[2 * i]), __uint_as_float(w[2 * i + 1]));
}
// Largest logit of a lane's item words.
template <bool BF16, int N>
__device__ __forceinline__ float words_max(const uint32_t (&w)[N]) {
  if constexpr (BF16) {
    __nv_bfloat162 a[4], t;
#pragma unroll
    for (int i = 0; i < 4; ++i) memcpy(&a[i], &w[i], 4);
#pragma unroll
    for (int i = 4; i < N; ++i) {
      memcpy(&t, &w[i], 4);
      a[i & 3] = __hmax2(a[i & 3], t);
    }
    a[0] = __hmax2(__hmax2(a[0], a[1]), __hmax2(a[2], a[3]));
    return fmaxf(__low2float(a[0]), __high2float(a[0]));
  } else {
    float a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = __uint_as_float(w[i]);
#pragma unroll
    for (int i = 4; i < N; ++i) a[i & 3] = fmaxf(a[i & 3], __uint_as_float(w[i]));
    return fmaxf(fmaxf(a[0], a[1]), fmaxf(a[2], a[3]));
  }
}

// Every warp of the CTA.
__device__ __forceinline__ void samp_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kSampThreads) : "memory");
}

// 1-D bulk copy global -> this CTA's shared memory, completing (in bytes) on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// One elected lane of the warp arms `bar` for `tx` bytes and issues the item's copies: `bytes`
// from src_t to dst and, when `two`, from src_d to dst + WB (no copy when bytes == 0).  No branch.
template <int WB>
__device__ __forceinline__ void issue_item(uint32_t bar, uint32_t tx, uint32_t dst, const void* src_t,
                                           const void* src_d, uint32_t bytes, uint32_t two) {
  asm volatile(
      "{\n\t.reg .pred e, pb, pt;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t"
      "setp.ne.and.u32 pb, %5, 0, e;\n\t"
      "@pb cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%2], [%3], %5, [%0];\n\t"
      "setp.ne.and.u32 pt, %6, 0, pb;\n\t"
      "@pt cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%7], [%4], %5, [%0];\n\t"
      "}" ::"r"(bar),
      "r"(tx), "r"(dst), "l"(src_t), "l"(src_d), "r"(bytes), "r"(two), "r"(dst + WB)
      : "memory");
}

// First entry (vocabulary order: lane-major, EPL entries per lane) whose running prefix
// cum0 + sum(..) crosses t; if rounding leaves none, the last entry with positive mass; -1 if
// none has mass.  Uniform across the warp.  *cum_before = cum0 + mass before the chosen entry.
template <int EPL>
__device__ __forceinline__ int select_entry(const float (&m)[EPL], float cum0, float t, int lane,
                                            float* cum_before) {
  float loc = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) loc += m[i];
  const float incl = warp_incl_scan(loc, lane);
  float excl = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) excl = 0.f;
  int first = -1, lastpos = -1;
  float run = cum0 + excl, before = 0.f, lb = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    if (first < 0 && run + m[i] > t) { first = i; before = run; }
    if (m[i] > 0.f) { lastpos = i; lb = run; }
    run += m[i];
  }
  const unsigned hit = __ballot_sync(0xffffffffu, first >= 0);
  int sel = -1;
  float cb = cum0;
  if (hit) {
    const int l = __ffs(hit) - 1;
    sel = l * EPL + __shfl_sync(0xffffffffu, first, l);
    cb = __shfl_sync(0xffffffffu, before, l);
  } else {
    const unsigned pos = __ballot_sync(0xffffffffu, lastpos >= 0);
    if (pos) {
      const int l = 31 - __clz(pos);
      sel = l * EPL + __shfl_sync(0xffffffffu, lastpos, l);
      cb = __shfl_sync(0xffffffffu, lb, l);
    }
  }
  *cum_before = cb;
  return sel;
}

template <bool BF16>
__global__ void __launch_bounds__(kSampThreads, kSampRingBytes <= 65536 ? 3 : 2) sample_kernel(const __grid_constant__ RowParams P) {
  using G = SampGeo<BF16>;
  constexpr int ESZ = G::ESZ, EPP = G::EPP, NPC = G::NPC, NWD = G::NWD, NP = G::NP;
  constexpr int IL = G::IL, WS = G::WS, PS = G::PS;
  constexpr int NWARP = kSampWarps;
  constexpr int S = kSampStages;
  constexpr int WB = kSampWarpBytes, IB = kSampItemBytes;
  constexpr int ENT = kMaxCluster * NWARP;         // exchange #1 entries per row: (CTA c, warp w) at c*NWARP + w
  constexpr int EPL = ENT / 32;
  constexpr int EP = kSampMaxItems * NWARP / 32;   // (item, warp) entries per lane in the owner search
  constexpr uint32_t NEG = BF16 ? 0xff80ff80u : 0xff800000u;

  // warp w's ring: stage s, row r at byte ((w * S + s) * 2 + r) * WB
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(16) float4 mbox1[2][ENT];               // (m_t, s_t, m_d, s_d) per (CTA, warp)
  __shared__ __align__(16) float2 mbox2[2][kMaxCluster];       // (R, P) per CTA
  __shared__ float2 part[2][kSampMaxItems][NWARP];             // (R, P) per (item, warp) of this CTA
  __shared__ __align__(8) uint64_t full_bar[NWARP][S];
  __shared__ __align__(8) uint64_t x1_bar[2];
  __shared__ __align__(8) uint64_t x2_bar[2];
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank(), C = cluster_ncta();
  const uint32_t cid = cluster_idx(), ncl = cluster_count();
  const int K = P.K, V = P.V;
  const int lo = static_cast<int>(rank) * P.slice;
  const int n = max(0, min(P.slice, V - lo));                  // this CTA's slice length
  const int nitems = (n + IL - 1) / IL;
  const bool aligned = (P.flags & F_ALIGNED) != 0;
  const bool need_draft = (P.flags & F_NEED_DRAFT) != 0;
  const bool stats_only = (P.flags & F_STATS_ONLY) != 0;
  const bool all_pdraws = (P.flags & F_ALL_PDRAWS) != 0;
  const float c = P.c;
  const int nent = static_cast<int>(C) * NWARP;
  const int nunits = static_cast<int>(cid) < P.total_units
                         ? (P.total_units - static_cast<int>(cid) + static_cast<int>(ncl) - 1) / static_cast<int>(ncl)
                         : 0;
  const int npairs = need_draft ? P.B * K : 0;   // units [0, npairs) are (target, draft) pairs
  // valid logits of this warp's bytes in the last item of the slice (all of them in the others)
  const int last_nval = nitems > 0 ? min(WS, max(0, n - (nitems - 1) * IL - warp * WS)) : 0;

  // unit u -> (b, k): the pairs first (b-major), then the target rows k = K (or, without draft
  // rows, every target row); larger units first gives round-robin assignment a short tail
  auto unit_of = [&](int i, int& u, int& b, int& k) {
    u = static_cast<int>(cid) + i * static_cast<int>(ncl);
    if (u < npairs) {
      b = u / K;
      k = u - b * K;
    } else if (need_draft) {
      b = u - npairs;
      k = K;
    } else {
      b = u / (K + 1);
      k = u - b * (K + 1);
    }
  };
  // the draw from p this row needs: at the verified depth, or at every row when the depth is
  // chosen afterwards (budget)
  auto pdraw_row = [&](int b, int k) {
    if (stats_only) return false;
    if (all_pdraws) return true;
    const int dep = P.depth ? min(max(P.depth[b], 0), K) : K;
    return k == dep;
  };
  auto row_ptr = [&](bool draft, int b, int k) {
    return draft ? static_cast<const uint8_t*>(P.draft) + ((static_cast<size_t>(b) * K + k) * static_cast<size_t>(V) + lo) * ESZ
                 : static_cast<const uint8_t*>(P.target) + ((static_cast<size_t>(b) * (K + 1) + k) * static_cast<size_t>(V) + lo) * ESZ;
  };

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid < NWARP * S) mbar_init(smem_addr(&full_bar[tid / S][tid % S]), 1);
  if (tid == 0) {
    for (int p = 0; p < 2; ++p) {
      mbar_init(smem_addr(&x1_bar[p]), 1);
      mbar_init(smem_addr(&x2_bar[p]), 1);
    }
    abort_flag = 0;
  }
  mbar_fence_init();
  __syncthreads();
  cluster_sync();   // every CTA's barriers exist before any peer sends into them
  // launched with programmatic serialization: the logits, tokens and records are touched only
  // once the preceding grid on the stream has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const long long wlimit = P.wait_limit;
  // A bounded wait on a phase; on timeout record it, then wait with the long limit; if that also
  // runs out, switch the CTA to abort mode (no more waiting, results unspecified).  CLUSTER: the
  // phase completes on peers' stores (acquire at cluster scope); otherwise on this warp's own bulk
  // copies.  The common case -- the phase is complete, or completes while the hardware holds the
  // poll -- reads no clock.
  auto wait_slow = [&](uint32_t bar, uint32_t parity, bool cluster) {
    if (*static_cast<volatile int*>(&abort_flag)) return cluster ? mbar_try_cluster(bar, parity) : mbar_try(bar, parity);
    if (cluster ? mbar_wait_for<true>(bar, parity, wlimit) : mbar_wait_for<false>(bar, parity, wlimit)) return true;
    atomicOr(P.status, kStatusTimeout);
    if (cluster ? mbar_wait_for<true>(bar, parity, kDrainNs) : mbar_wait_for<false>(bar, parity, kDrainNs)) return true;
    *static_cast<volatile int*>(&abort_flag) = 1;
    return false;
  };
  auto wait_phase = [&](uint32_t bar, uint32_t parity) {
    return (wlimit > 0 && mbar_try_cluster(bar, parity)) || wait_slow(bar, parity, true);
  };

  // ---- this warp's copy ring over the CTA's (unit, pass, item) sequence, S - 1 items ahead
  const uint32_t ring_w = smem_addr(ring) + static_cast<uint32_t>(warp * S * 2 * WB);
  const uint32_t fbar0 = smem_addr(&full_bar[warp][0]);
  const uint32_t last_bytes = static_cast<uint32_t>(last_nval) * ESZ;
  int iu = 0, ileft = 0, ipass = 0, istage = 0;     // issue cursor
  bool ipair = false, idone = !(aligned && nitems > 0);
  const uint8_t* isrc_t = nullptr;
  const uint8_t* isrc_d = nullptr;
  uint32_t issued = 0;                               // copies issued by this warp (for the final drain)
  auto issue_unit = [&]() {                          // the next needed unit at or after iu
    for (; iu < nunits; ++iu) {
      int u, b, k;
      unit_of(iu, u, b, k);
      ipair = need_draft && k < K;
      if (!(ipair || pdraw_row(b, k))) continue;
      isrc_t = row_ptr(false, b, k) + warp * WB;
      isrc_d = row_ptr(true, b, ipair ? k : 0) + warp * WB;
      ileft = nitems;
      return;
    }
    idone = true;
  };
  if (!idone) issue_unit();
  // arm the next stage with this warp's bytes of the next item (0 bytes past the slice end)
  auto issue_next = [&]() {
    if (idone) return;
    const uint32_t bytes = ileft == 1 ? last_bytes : static_cast<uint32_t>(WB);
    issue_item<WB>(fbar0 + istage * 8u, ipair ? 2u * bytes : bytes, ring_w + static_cast<uint32_t>(istage * 2 * WB),
                   isrc_t, isrc_d, bytes, ipair ? 1u : 0u);
    ++issued;
    istage = istage == S - 1 ? 0 : istage + 1;
    if (--ileft) {
      isrc_t += IB;
      isrc_d += IB;
    } else if (ipass == 0) {                          // the same rows again for pass 2
      ipass = 1;
      ileft = nitems;
      isrc_t -= static_cast<size_t>(nitems - 1) * IB;
      isrc_d -= static_cast<size_t>(nitems - 1) * IB;
    } else {
      ipass = 0;
      ++iu;
      issue_unit();
    }
  };
  for (int q = 0; q < S - 1; ++q) issue_next();

  // consume cursor
  int cstage = 0;
  uint32_t cphase = 0;                      // bit s: parity of stage s's next phase
  // The next item's stage: issue the item S - 1 further on (into the stage consumed last step,
  // whose words every lane has used), then wait for this one.  Returns the lane's byte address of
  // row 0 in the stage (row 1 at + WB).
  auto acquire = [&]() -> uint32_t {
    __syncwarp();
    issue_next();
    const uint32_t bar = fbar0 + cstage * 8u, par = (cphase >> cstage) & 1u;
    if (!(wlimit > 0 && mbar_try(bar, par))) wait_slow(bar, par, false);
    const uint32_t base = ring_w + static_cast<uint32_t>(cstage * 2 * WB) + static_cast<uint32_t>(lane) * 16u;
    cphase ^= 1u << cstage;
    cstage = cstage == S - 1 ? 0 : cstage + 1;
    return base;
  };
  // -inf over the logits of piece j of a lane's words that lie past the slice end
  auto mask_piece = [&](uint32_t (&W)[4], int j) {
#pragma unroll
    for (int e = 0; e < EPP; ++e) {
      if (j * PS + lane * EPP + e >= last_nval) {
        if constexpr (BF16) {
          const int q = e >> 1;
          W[q] = (e & 1) ? ((W[q] & 0x0000ffffu) | 0xff800000u) : ((W[q] & 0xffff0000u) | 0x0000ff80u);
        } else {
          W[e] = NEG;
        }
      }
    }
  };
  // piece j of this lane's words of item `it` of one row: from the stage (aligned rows) or
  // element-wise from global memory with -inf past the slice end
  auto piece = [&](uint32_t (&W)[4], uint32_t base, int j, bool ragged, const uint8_t* grow, int it) {
    if (aligned) {
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(W[0]), "=r"(W[1]), "=r"(W[2]), "=r"(W[3])
                   : "r"(base + j * 512));
      if (ragged) mask_piece(W, j);
      return;
    }
    const int o = it * IL + warp * WS + j * PS + lane * EPP;   // first logit of the piece in the slice
#pragma unroll
    for (int q = 0; q < 4; ++q) W[q] = NEG;
#pragma unroll
    for (int e = 0; e < EPP; ++e) {
      if (o + e < n) {
        if constexpr (BF16) {
          const uint32_t h16 = reinterpret_cast<const uint16_t*>(grow)[o + e];
          uint32_t& w = W[e >> 1];
          w = (e & 1) ? ((w & 0x0000ffffu) | (h16 << 16)) : ((w & 0xffff0000u) | h16);
        } else {
          W[e] = reinterpret_cast<const uint32_t*>(grow)[o + e];
        }
      }
    }
  };
  auto row_words = [&](uint32_t (&W)[NWD], uint32_t base, bool ragged, const uint8_t* grow, int it) {
#pragma unroll
    for (int j = 0; j < NPC; ++j) {
      uint32_t T[4];
      piece(T, base, j, ragged, grow, it);
#pragma unroll
      for (int q = 0; q < 4; ++q) W[4 * j + q] = T[q];
    }
  };

  const uint64_t c2 = pk(c, c);
  // online (max, sum) update with one item of one row, without branches: the sum is rescaled to
  // the new running maximum (reference 0 while every logit so far is -inf)
  auto fold = [&](const uint32_t (&W)[NWD], float& m, float& s) {
    const float nm = fmaxf(m, words_max<BF16>(W));
    const float ref = nm == ninf() ? 0.f : nm;
    s *= ex2((m - ref) * c);
    const uint64_t nref = pk(-ref * c, -ref * c);
    uint64_t acc0 = pk(0.f, 0.f), acc1 = acc0;
#pragma unroll
    for (int i = 0; i < NP; i += 2) {
      float x0, x1, y0, y1;
      upk(ffma2(pair_of<BF16>(W, i), c2, nref), x0, x1);
      upk(ffma2(pair_of<BF16>(W, i + 1), c2, nref), y0, y1);
      acc0 = fadd2(acc0, pk(ex2(x0), ex2(x1)));
      acc1 = fadd2(acc1, pk(ex2(y0), ex2(y1)));
    }
    float s0, s1;
    upk(fadd2(acc0, acc1), s0, s1);
    s += s0 + s1;
    m = nm;
  };

  uint32_t x2ph = 0;
  int j = 0;                                 // processed units (exchange parity)
  for (int i = 0; i < nunits; ++i) {
    int u, b, k;
    unit_of(i, u, b, k);
    const bool pair = need_draft && k < K;
    const bool pdraw = pdraw_row(b, k);
    if (!(pair || pdraw)) continue;          // nothing of this row is needed
    const int rec = b * P.U + k;             // the row's record, where the cut kernel reads it
    const int par = j & 1;
    ++j;
    const uint8_t* gt = row_ptr(false, b, k);
    const uint8_t* gd = row_ptr(true, b, pair ? k : 0);
    if (tid == 0) mbar_arrive_tx(smem_addr(&x1_bar[par]), static_cast<uint32_t>(nent) * 16u);
    // scalars this unit needs later (issued now, consumed after pass 1)
    const float uK = stats_only ? 0.f : P.uniforms[static_cast<size_t>(b) * (K + 1) + K];
    const float uk = (stats_only || k >= K) ? 0.f : P.uniforms[static_cast<size_t>(b) * (K + 1) + k];
    bool xin = false;
    float ztx = 0.f, zdx = 0.f;
    if (!stats_only && k < K && lane == 0) {
      const int x = P.tokens[static_cast<size_t>(b) * K + k];
      xin = (x >= 0 && x < V);
      if (xin) {
        const size_t ot = (static_cast<size_t>(b) * (K + 1) + k) * V + x;
        const size_t od = (static_cast<size_t>(b) * K + k) * V + x;
        if constexpr (BF16) {
          ztx = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(P.target)[ot]) << 16);
          zdx = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(P.draft)[od]) << 16);
        } else {
          ztx = reinterpret_cast<const float*>(P.target)[ot];
          zdx = reinterpret_cast<const float*>(P.draft)[od];
        }
      }
    }

    // ---- pass 1: online (max, sum) of both rows, item by item
    float mt = ninf(), st = 0.f, md = ninf(), sd = 0.f;
    for (int it = 0; it < nitems; ++it) {
      const uint32_t base = aligned ? acquire() : 0u;
      const bool ragged = it == nitems - 1 && last_nval < WS;
      uint32_t W[NWD];
      row_words(W, base, ragged, gt, it);
      fold(W, mt, st);
      if (pair) {
        row_words(W, base + WB, ragged, gd, it);
        fold(W, md, sd);
      }
    }
    // warp partials: the warp maximum, then every lane's sum rescaled to it and summed
    {
      const float wt = warp_max(mt), wd = warp_max(md);
      const float rt = wt == ninf() ? 0.f : wt, rd = wd == ninf() ? 0.f : wd;
      st = warp_sum(st * ex2((mt - rt) * c));
      sd = warp_sum(sd * ex2((md - rd) * c));
      mt = wt;
      md = wd;
    }
    if (lane < static_cast<int>(C)) {
      const uint32_t dst = smem_addr(&mbox1[par][rank * NWARP + warp]);
      st_async_v4(peer_addr(dst, lane), mt, st, md, sd, peer_addr(smem_addr(&x1_bar[par]), lane));
    }
    wait_phase(smem_addr(&x1_bar[par]), ((j - 1) >> 1) & 1);
    float Mt = ninf(), Md = ninf();
#pragma unroll
    for (int q = 0; q < EPL; ++q) {
      const int e = lane * EPL + q;
      if (e < nent) {
        const float4 v = mbox1[par][e];
        Mt = fmaxf(Mt, v.x);
        Md = fmaxf(Md, v.z);
      }
    }
    Mt = warp_max(Mt);
    Md = warp_max(Md);
    float St = 0.f, Sd = 0.f;
    {
      const float rt = (Mt == ninf()) ? 0.f : Mt, rd = (Md == ninf()) ? 0.f : Md;
#pragma unroll
      for (int q = 0; q < EPL; ++q) {
        const int e = lane * EPL + q;
        if (e < nent) {
          const float4 v = mbox1[par][e];
          St += v.y * ex2((v.x - rt) * c);
          Sd += v.w * ex2((v.z - rd) * c);
        }
      }
    }
    St = warp_sum(St);
    Sd = warp_sum(Sd);
    // p_v = 2^(z c - offt), q_v = 2^(z c - offd): the normalisers folded into the exponent
    const float offt = (Mt == ninf() ? 0.f : Mt * c) + lg2f(St);
    const float offd = (Md == ninf() ? 0.f : Md * c) + lg2f(Sd);
    float px = 0.f, qx = 0.f;
    if (lane == 0 && xin) {
      px = ex2(fmaf(ztx, c, -offt));
      qx = ex2(fmaf(zdx, c, -offd));
    }
    px = __shfl_sync(0xffffffffu, px, 0);
    qx = __shfl_sync(0xffffffffu, qx, 0);
    const bool xin_all = __shfl_sync(0xffffffffu, xin ? 1 : 0, 0) != 0;
    const bool rejects = !stats_only && k < K && !(xin_all && uk * qx < px);
    // a pair that passes the test and draws nothing needs only alpha = sum min(p, q), and
    // min(2^a, 2^b) = 2^min(a, b): one exp2 per logit pair, no per-item masses, and only CTA 0
    // (which writes the record) receives the CTA totals
    const bool alpha_only = pair && !rejects && !pdraw;
    const bool all_recv = !alpha_only;
    const bool recv = all_recv || rank == 0;
    if (tid == 0 && recv) mbar_arrive_tx(smem_addr(&x2_bar[par]), static_cast<uint32_t>(C) * 8u);

    // ---- pass 2: residual and p masses per (item, warp) -> CTA totals -> exchange #2
    const uint64_t noff_t = pk(-offt, -offt), noff_d = pk(-offd, -offd);
    if (alpha_only) {
      uint64_t aacc = pk(0.f, 0.f), bacc = aacc;
      for (int it = 0; it < nitems; ++it) {
        const uint32_t base = aligned ? acquire() : 0u;
        const bool ragged = it == nitems - 1 && last_nval < WS;
#pragma unroll
        for (int jp = 0; jp < NPC; ++jp) {
          uint32_t Wt[4], Wd[4];
          piece(Wt, base, jp, ragged, gt, it);
          piece(Wd, base + WB, jp, ragged, gd, it);
#pragma unroll
          for (int q = 0; q < (BF16 ? 4 : 2); q += 2) {
            float a0, a1, b0, b1, a2, a3, b2, b3;
            upk(ffma2(pair_of<BF16>(Wt, q), c2, noff_t), a0, a1);
            upk(ffma2(pair_of<BF16>(Wd, q), c2, noff_d), b0, b1);
            upk(ffma2(pair_of<BF16>(Wt, q + 1), c2, noff_t), a2, a3);
            upk(ffma2(pair_of<BF16>(Wd, q + 1), c2, noff_d), b2, b3);
            aacc = fadd2(aacc, pk(ex2(fminf(a0, b0)), ex2(fminf(a1, b1))));
            bacc = fadd2(bacc, pk(ex2(fminf(a2, b2)), ex2(fminf(a3, b3))));
          }
        }
      }
      float a0, a1;
      upk(fadd2(aacc, bacc), a0, a1);
      const float aw = warp_sum(a0 + a1);
      if (lane == 0) part[par][0][warp] = make_float2(aw, 0.f);
    } else {
      const uint64_t neg1 = pk(-1.f, -1.f);
      for (int it = 0; it < nitems; ++it) {
        const uint32_t base = aligned ? acquire() : 0u;
        const bool ragged = it == nitems - 1 && last_nval < WS;
        uint64_t pacc = pk(0.f, 0.f), racc = pacc;
#pragma unroll
        for (int jp = 0; jp < NPC; ++jp) {
          uint32_t Wt[4], Wd[4];
          piece(Wt, base, jp, ragged, gt, it);
          if (pair) {
            piece(Wd, base + WB, jp, ragged, gd, it);
#pragma unroll
            for (int q = 0; q < (BF16 ? 4 : 2); ++q) {
              float a0, a1, b0, b1, d0, d1;
              upk(ffma2(pair_of<BF16>(Wt, q), c2, noff_t), a0, a1);
              const uint64_t p = pk(ex2(a0), ex2(a1));     // p of logits 2q, 2q+1
              pacc = fadd2(pacc, p);
              upk(ffma2(pair_of<BF16>(Wd, q), c2, noff_d), b0, b1);
              upk(ffma2(pk(ex2(b0), ex2(b1)), neg1, p), d0, d1);   // p - q
              racc = fadd2(racc, pk(fmaxf(d0, 0.f), fmaxf(d1, 0.f)));
            }
          } else {
#pragma unroll
            for (int q = 0; q < (BF16 ? 4 : 2); ++q) {
              float a0, a1;
              upk(ffma2(pair_of<BF16>(Wt, q), c2, noff_t), a0, a1);
              pacc = fadd2(pacc, pk(ex2(a0), ex2(a1)));
            }
          }
        }
        float p0, p1, r0, r1;
        upk(pacc, p0, p1);
        upk(racc, r0, r1);
        // lanes 0-15 end with the warp's R, lanes 16-31 with its P (one exchange of each at 16)
        const bool hi = (lane & 16) != 0;
        float keep = hi ? p0 + p1 : r0 + r1;
        keep += __shfl_xor_sync(0xffffffffu, hi ? r0 + r1 : p0 + p1, 16);
#pragma unroll
        for (int o = 8; o; o >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, o);
        if ((lane & 15) == 0) reinterpret_cast<float*>(&part[par][it][warp])[lane >> 4] = keep;
      }
    }
    // (item, warp) masses in `part`: alpha-only units have one item row holding sum min(p, q)
    const int pitems = alpha_only ? 1 : nitems;
    samp_sync();                             // every warp's (item, warp) masses are in `part`
    if (warp == 0) {
      // CTA totals: lane l sums entries l*EP .. l*EP+EP-1 in (item, warp) order, then a scan
      // across lanes -- the same grouping the owner search below uses
      float rl = 0.f, pl = 0.f;
#pragma unroll
      for (int q = 0; q < EP; ++q) {
        const int e = lane * EP + q, iti = e / NWARP, wi = e - iti * NWARP;
        if (iti < pitems) {
          const float2 v = part[par][iti][wi];
          rl += v.x;
          pl += v.y;
        }
      }
      const float rc = __shfl_sync(0xffffffffu, warp_incl_scan(rl, lane), 31);
      const float pc = __shfl_sync(0xffffffffu, warp_incl_scan(pl, lane), 31);
      if (lane < (all_recv ? static_cast<int>(C) : 1)) {
        const uint32_t dst = smem_addr(&mbox2[par][rank]);
        const uint32_t rdst = peer_addr(dst, lane);
        const uint32_t rbar = peer_addr(smem_addr(&x2_bar[par]), lane);
        st_async_f32(rdst, rc, rbar);
        st_async_f32(rdst + 4, pc, rbar);
      }
    }
    if (!recv) continue;                     // CTA r > 0 of an alpha-only unit: done with it
    wait_phase(smem_addr(&x2_bar[par]), (x2ph >> par) & 1u);
    x2ph ^= 1u << par;
    const float2 e2 = lane < static_cast<int>(C) ? mbox2[par][lane] : make_float2(0.f, 0.f);
    // totals over CTAs: inclusive scans (CTA order), the last lane holds the totals
    const float rin = warp_incl_scan(e2.x, lane), pin = warp_incl_scan(e2.y, lane);
    const float Rtot = __shfl_sync(0xffffffffu, rin, 31);
    const float Ptot = __shfl_sync(0xffffffffu, pin, 31);

    // ---- the draws this unit may need
    const bool need_r = pair && rejects && Rtot > 0.f;
    const bool need_p = pdraw || (rejects && !(Rtot > 0.f));   // p == q: the residual is empty
    for (int which = 0; which < 2; ++which) {
      const bool resid = which == 0;
      if (resid ? !need_r : !need_p) continue;
      const float total = resid ? Rtot : Ptot;
      const float t = uK * total;
      // owner CTA (vocabulary order), then owner (item, warp) inside it, from the same sums
      float mc[1] = {lane < static_cast<int>(C) ? (resid ? e2.x : e2.y) : 0.f};
      float cum_c = 0.f;
      const int oc = select_entry<1>(mc, 0.f, t, lane, &cum_c);
      if (oc != static_cast<int>(rank)) {
        if (oc < 0 && rank == 0 && tid == 0) {
          if (resid) P.recs[rec].rs = -1; else P.recs[rec].ps = -1;
        }
        continue;
      }
      // (item, warp) entries of this CTA in order: lane l holds entries l*EP .. l*EP+EP-1
      float mw[EP];
#pragma unroll
      for (int q = 0; q < EP; ++q) {
        const int e = lane * EP + q, iti = e / NWARP, wi = e - iti * NWARP;
        mw[q] = iti < nitems ? (resid ? part[par][iti][wi].x : part[par][iti][wi].y) : 0.f;
      }
      float cum_w = 0.f;
      const int ow = select_entry<EP>(mw, cum_c, t, lane, &cum_w);
      const int ow_it = ow < 0 ? 0 : ow / NWARP, ow_w = ow < 0 ? 0 : ow % NWARP;
      if (warp != ow_w) continue;
      // the owner warp reloads its segment of this item and walks pieces, lanes, elements
      const int e0 = ow_it * IL + ow_w * WS;
      auto mass_at = [&](int v) {                    // the draw's mass of logit v of the slice
        if (v >= n) return 0.f;
        float zt, zd = 0.f;
        if constexpr (BF16) {
          zt = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(gt)[v]) << 16);
          if (resid) zd = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(gd)[v]) << 16);
        } else {
          zt = reinterpret_cast<const float*>(gt)[v];
          if (resid) zd = reinterpret_cast<const float*>(gd)[v];
        }
        const float p = ex2(fmaf(zt, c, -offt));
        return resid ? fmaxf(p - ex2(fmaf(zd, c, -offd)), 0.f) : p;
      };
      // pieces in vocabulary order, then the lane, then the element
      float sj[NPC], tot[NPC];
#pragma unroll
      for (int jj = 0; jj < NPC; ++jj) {
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < EPP; ++e) a += mass_at(e0 + jj * PS + lane * EPP + e);
        sj[jj] = a;
        tot[jj] = warp_sum(a);
      }
      float cum = cum_w, cumj = cum_w;
      int js = -1;
#pragma unroll
      for (int jj = 0; jj < NPC; ++jj) {
        if (js < 0 && cum + tot[jj] > t) { js = jj; cumj = cum; }
        cum += tot[jj];
      }
      if (js < 0) {
        cum = cum_w;
#pragma unroll
        for (int jj = 0; jj < NPC; ++jj) {
          if (tot[jj] > 0.f) { js = jj; cumj = cum; }
          cum += tot[jj];
        }
        if (js < 0) { js = 0; cumj = cum_w; }
      }
      float mine = 0.f;
#pragma unroll
      for (int jj = 0; jj < NPC; ++jj) if (jj == js) mine = sj[jj];
      float m1[1] = {mine};
      float cl = cumj;
      int l = select_entry<1>(m1, cumj, t, lane, &cl);
      if (l < 0) l = 0;
      if (lane == l) {
        float run = cl;
        int first = -1, lastpos = -1;
        for (int e = 0; e < EPP; ++e) {
          const float me = mass_at(e0 + js * PS + l * EPP + e);
          run += me;
          if (first < 0 && run > t) first = e;
          if (me > 0.f) lastpos = e;
        }
        const int es = first >= 0 ? first : (lastpos >= 0 ? lastpos : 0);
        const int idx = lo + e0 + js * PS + l * EPP + es;
        if (resid) P.recs[rec].rs = idx; else P.recs[rec].ps = idx;
      }
    }
    if (rank == 0 && tid == 0) {
      UnitRec* r = P.recs + rec;
      r->px = px;
      r->qx = qx;
      // alpha-only units carry sum min(p, q) in the first total; R is then only informative
      const float alpha = alpha_only ? Rtot : Ptot - Rtot;
      r->alpha = pair ? fminf(fmaxf(alpha, 0.f), 1.f) : 0.f;
      r->R = alpha_only ? fmaxf(1.f - Rtot, 0.f) : Rtot;
    }
  }
  // every copy this warp issued has landed (normally all were consumed; in abort mode some may
  // still be in flight) before the CTA leaves
  if (aligned && lane == 0) {
    for (uint32_t q = 0; q < static_cast<uint32_t>(S) && q < issued; ++q) {
      // the most recent copy into stage s = (issued - 1 - q) mod S, its phase parity
      const uint32_t qi = issued - 1 - q;
      const uint32_t s = qi % S, ph = (qi / S) & 1u;
      mbar_wait_for<false>(fbar0 + s * 8u, ph, kDrainNs);
    }
  }
}

}  // namespace sv

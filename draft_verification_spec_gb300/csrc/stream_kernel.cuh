// Sampling-path row kernel (T > 0): two streaming passes per (request, position) unit.
//
// A thread-block cluster of C CTAs works on one unit at a time -- target row k and, for k < K,
// draft row k -- looping over units (persistent).  CTA r owns the vocabulary slice
// [r*slice, (r+1)*slice) of every row and streams it in items of 4096 logits per row through a
// shared-memory ring: a producer warp issues one-thread bulk copies into free stages (full /
// empty mbarriers), eight consumer warps read them.  Inside an item, consumer warp w owns logits
// [w*512, (w+1)*512), lane-interleaved in 8-logit chunks.
//
// Per unit:
//   pass 1 (from HBM, kept in L2 with an evict-last hint): per-thread online (max, sum of
//     2^((z - m) c)) of the target and draft rows -> warp partials -> exchange #1 with st.async
//     into every CTA of the cluster, completing on its mbarrier -> the row's normalisers of p and
//     q, merged in one fixed order so every warp of every CTA holds bitwise-identical values;
//     p_k(x_k), q_k(x_k) and the accept test, as the cut kernel will evaluate them
//   pass 2 (the same bytes again, now L2 hits, evict-first): per element p = 2^(z c - offt),
//     q = 2^(z c - offd); per (item, warp) masses of r = max(0, p - q) and of p -> CTA totals ->
//     exchange #2 -> residual mass R, alpha = sum p - R (= sum min(p, q)), and the owner of each
//     needed inverse-CDF draw, found in vocabulary order (CTA, item, warp)
//   the owner warp reloads its 512 logits of the row(s) and walks slot / lane / element prefix
//     sums to the drawn index.  The residual is drawn only where the test fails, the p draw only
//     at the verified depth (or at every row when the depth is chosen afterwards).
// DRAM reads each logit once; the second pass is served by L2.  The serial cut runs afterwards in
// a small kernel chained with programmatic dependent launch.
#pragma once

#include <cuda_bf16.h>

#include "spec_async.cuh"

namespace sv {

constexpr int kStreamWarps = 8;                                 // consumer warps
constexpr int kStreamThreads = 32 * (kStreamWarps + 1);         // + the producer warp
constexpr int kStreamNV = 2;                                    // 8-logit chunks per lane per item
constexpr int kStreamWarpSpan = 32 * kStreamNV * kChunk;        // logits of one warp per item (512)
constexpr int kStreamItem = kStreamWarps * kStreamWarpSpan;     // logits per row per item (4096)
constexpr int kStreamMaxItems = 32;                             // items per slice (slice <= 131072)

template <bool BF16>
__device__ __forceinline__ float chunk_elem(const uint4 (&w)[BF16 ? 1 : 2], int e) {   // logit e of a chunk
  if constexpr (BF16) {
    const uint32_t word = (e < 2) ? w[0].x : (e < 4) ? w[0].y : (e < 6) ? w[0].z : w[0].w;
    return __uint_as_float((e & 1) ? (word & 0xffff0000u) : (word << 16));
  } else {
    const uint4 v = w[e >> 2];
    const uint32_t word = ((e & 3) == 0) ? v.x : ((e & 3) == 1) ? v.y : ((e & 3) == 2) ? v.z : v.w;
    return __uint_as_float(word);
  }
}

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
// logits 2i and 2i+1 of a lane's item words as a packed pair (bf16 halves widen exactly)
template <bool BF16>
__device__ __forceinline__ uint64_t pair_of(const uint32_t* w, int i) {
  if constexpr (BF16) return pk(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
  else return pk(__uint_as_float(w[2 * i]), __uint_as_float(w[2 * i + 1]));
}

__device__ __forceinline__ uint64_t l2_evict_last_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Named barrier among the consumer warps (the producer warp never joins it).
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kStreamWarps) : "memory");
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
__global__ void __launch_bounds__(kStreamThreads, BF16 ? 3 : 1) stream_kernel(const __grid_constant__ RowParams P) {
  constexpr int ESZ = BF16 ? 2 : 4;
  constexpr int NW = kStreamWarps;
  constexpr int ENT = kMaxCluster * NW;   // exchange #1 entries per row: (CTA c, warp w) at c*NW + w
  constexpr int EPL = ENT / 32;
  constexpr int ITEM_BYTES = kStreamItem * ESZ;   // one row of one item in the ring
  using Chunk = uint4[BF16 ? 1 : 2];

  extern __shared__ __align__(128) uint8_t ring[];            // [nstage][2 rows][ITEM_BYTES]
  __shared__ __align__(16) float4 mbox1[2][ENT];               // (m_t, s_t, m_d, s_d) per (CTA, warp)
  __shared__ __align__(16) float2 mbox2[2][kMaxCluster];       // (R, P) per CTA
  __shared__ float2 part[2][kStreamMaxItems][NW];              // (R, P) per (item, warp) of this CTA
  __shared__ __align__(8) uint64_t full_bar[kMaxStreamStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStreamStages];
  __shared__ __align__(8) uint64_t x1_bar[2];
  __shared__ __align__(8) uint64_t x2_bar[2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank(), C = cluster_ncta();
  const uint32_t cid = cluster_idx(), ncl = cluster_count();
  const int K = P.K, V = P.V, U = P.U;
  const int lo = static_cast<int>(rank) * P.slice;
  const int n = max(0, min(P.slice, V - lo));                  // this CTA's slice length
  const int nitems = (n + kStreamItem - 1) / kStreamItem;
  const bool tma = (P.flags & F_TMA) != 0;
  const bool need_draft = (P.flags & F_NEED_DRAFT) != 0;
  const bool stats_only = (P.flags & F_STATS_ONLY) != 0;
  const bool all_pdraws = (P.flags & F_ALL_PDRAWS) != 0;
  const float c = P.c;
  const int nstage = P.nstage;
  const int nent = static_cast<int>(C) * NW;
  const int nunits = static_cast<int>(cid) < P.total_units
                         ? (P.total_units - static_cast<int>(cid) + static_cast<int>(ncl) - 1) / static_cast<int>(ncl)
                         : 0;

  // what a unit needs: pass 2 for alpha (pairs) or for a p draw at this row
  auto unit_of = [&](int i, int& u, int& b, int& k) {
    u = static_cast<int>(cid) + i * static_cast<int>(ncl);
    b = u / U;
    k = u - b * U;
  };
  auto pdraw_row = [&](int b, int k) {
    if (stats_only) return false;
    const int dep = P.depth ? min(max(P.depth[b], 0), K) : K;
    return all_pdraws || k == dep;
  };
  auto needs_p2 = [&](bool pair, bool pdraw) { return pair || pdraw; };

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int s = 0; s < nstage; ++s) {
      mbar_init(smem_addr(&full_bar[s]), 1);
      mbar_init(smem_addr(&empty_bar[s]), NW);
    }
    for (int p = 0; p < 2; ++p) {
      mbar_init(smem_addr(&x1_bar[p]), 1);
      mbar_init(smem_addr(&x2_bar[p]), 1);
    }
    mbar_fence_init();
  }
  __syncthreads();
  cluster_sync();   // every CTA's barriers exist before any peer sends into them

  if (warp == NW) {
    // ================= producer warp: stream (unit, pass, item) into the ring =================
    if (tma && lane == 0) {
      const uint64_t keep = l2_evict_last_policy(), drop = l2_evict_first_policy();
      int slot = 0;                          // running item count
      bool give_up = false;
      for (int i = 0; i < nunits && !give_up; ++i) {
        int u, b, k;
        unit_of(i, u, b, k);
        const bool pair = need_draft && k < K;
        const int passes = needs_p2(pair, pdraw_row(b, k)) ? 2 : 1;
        const uint8_t* rt = static_cast<const uint8_t*>(P.target) +
                            ((static_cast<size_t>(b) * (K + 1) + k) * static_cast<size_t>(V) + lo) * ESZ;
        const uint8_t* rd = static_cast<const uint8_t*>(P.draft) +
                            ((static_cast<size_t>(b) * K + k) * static_cast<size_t>(V) + lo) * ESZ;
        for (int pass = 0; pass < passes && !give_up; ++pass) {
          for (int it = 0; it < nitems; ++it, ++slot) {
            const int s = slot % nstage;
            if (slot >= nstage &&            // stage s free once every consumer warp released it
                !mbar_wait_bounded(smem_addr(&empty_bar[s]), ((slot / nstage) - 1) & 1, 1ll << 17)) {
              atomicOr(P.status, kStatusTimeout);
              give_up = true;
              break;
            }
            const int e0 = it * kStreamItem;
            const uint32_t bytes = static_cast<uint32_t>(min(kStreamItem, n - e0)) * ESZ;
            const uint32_t bar = smem_addr(&full_bar[s]);
            mbar_arrive_tx(bar, bytes * (pair ? 2u : 1u));
            const uint64_t pol = pass == 0 ? keep : drop;
            const uint32_t dst = smem_addr(ring) + s * 2 * ITEM_BYTES;
            bulk_g2s(dst, rt + static_cast<size_t>(e0) * ESZ, bytes, bar, pol);
            if (pair) bulk_g2s(dst + ITEM_BYTES, rd + static_cast<size_t>(e0) * ESZ, bytes, bar, pol);
          }
        }
      }
      // every copy issued is waited for by the consumers before they leave
    }
    cluster_sync_relaxed();
    return;
  }

  // ======================= consumer warps =======================
  bool tabort = false;   // a staged-data wait gave up once (test hook or a lost copy)
  bool xabort = false;   // gave up waiting for an exchange
  const long long xlimit = 1ll << 17;   // polls of up to kWaitSliceNs each
  uint32_t x2ph = 0;

  constexpr uint32_t NEG = BF16 ? 0xff80ff80u : 0xff800000u;
  constexpr int WPC = BF16 ? 4 : 8;                  // 32-bit words per 8-logit chunk
  constexpr int IW = kStreamNV * WPC;                // words per lane per row per item
  constexpr int NP = kStreamNV * kChunk / 2;         // logit pairs per lane per row per item
  // this lane's logits of item `it` of one row, as raw words: 16-byte reads from the ring, or
  // element-wise reads (ragged slice end, unaligned rows) with -inf past the slice end
  auto read_item = [&](uint32_t (&W)[IW], const uint8_t* st, const uint8_t* grow, int it) {
    const int e0 = it * kStreamItem;
    const int nval = min(kStreamItem, n - e0);
    if (tma && nval == kStreamItem) {
#pragma unroll
      for (int j = 0; j < kStreamNV; ++j) {
        const int o = warp * kStreamWarpSpan + (j * 32 + lane) * kChunk;
#pragma unroll
        for (int h = 0; h < WPC / 4; ++h) {
          const uint4 v = *reinterpret_cast<const uint4*>(st + o * ESZ + h * 16);
          W[j * WPC + h * 4] = v.x;
          W[j * WPC + h * 4 + 1] = v.y;
          W[j * WPC + h * 4 + 2] = v.z;
          W[j * WPC + h * 4 + 3] = v.w;
        }
      }
      return;
    }
    const uint8_t* src = tma ? st : grow + static_cast<size_t>(e0) * ESZ;
#pragma unroll
    for (int j = 0; j < kStreamNV; ++j) {
      const int o = warp * kStreamWarpSpan + (j * 32 + lane) * kChunk;
      const int nv = min(kChunk, max(0, nval - o));
#pragma unroll
      for (int q = 0; q < WPC; ++q) W[j * WPC + q] = NEG;
#pragma unroll
      for (int e = 0; e < kChunk; ++e) {
        if (e < nv) {
          if constexpr (BF16) {
            const uint32_t h16 = reinterpret_cast<const uint16_t*>(src)[o + e];
            uint32_t& w = W[j * WPC + (e >> 1)];
            w = (e & 1) ? ((w & 0x0000ffffu) | (h16 << 16)) : ((w & 0xffff0000u) | h16);
          } else {
            W[j * WPC + e] = reinterpret_cast<const uint32_t*>(src)[o + e];
          }
        }
      }
    }
  };
  // ring position of the next item, advanced without divisions
  int stage = 0;
  uint32_t fpar = 0;
  // a wait that gives up (the test hook, or a lost copy) records the timeout, then still drains
  // the copy with a long bound so no copy lands in a stage after it is reused or after exit
  auto wait_item = [&]() {
    if (!tma) return;
    const uint32_t bar = smem_addr(&full_bar[stage]);
    if (!tabort && mbar_wait_bounded(bar, fpar, P.wait_limit)) return;
    if (!tabort) atomicOr(P.status, kStatusTimeout);
    tabort = true;
    if (!mbar_wait_bounded(bar, fpar, 1ll << 17)) atomicOr(P.status, kStatusTimeout);
  };
  auto release_item = [&]() {
    __syncwarp();
    if (tma && lane == 0) mbar_arrive(smem_addr(&empty_bar[stage]));
    if (++stage == nstage) { stage = 0; fpar ^= 1u; }
  };
  const uint64_t c2 = pk(c, c);
  // online (max, sum) update with one item of one row: one max, one rescale, paired FMA / add
  auto fold_item = [&](const uint32_t (&W)[IW], float& m, float& sum) {
    float im;
    if constexpr (BF16) {
      __nv_bfloat162 a0, a1, t0, t1;
      memcpy(&a0, &W[0], 4);
      memcpy(&a1, &W[1], 4);
#pragma unroll
      for (int q = 2; q < IW; q += 2) {
        memcpy(&t0, &W[q], 4);
        memcpy(&t1, &W[q + 1], 4);
        a0 = __hmax2(a0, t0);
        a1 = __hmax2(a1, t1);
      }
      a0 = __hmax2(a0, a1);
      im = fmaxf(__low2float(a0), __high2float(a0));
    } else {
      float a0 = ninf(), a1 = ninf();
#pragma unroll
      for (int q = 0; q < IW; q += 2) {
        a0 = fmaxf(a0, __uint_as_float(W[q]));
        a1 = fmaxf(a1, __uint_as_float(W[q + 1]));
      }
      im = fmaxf(a0, a1);
    }
    const float nm = fmaxf(m, im);
    if (nm == ninf()) return;                          // nothing finite yet
    const float scale = (m == ninf()) ? 0.f : ex2((m - nm) * c);
    const uint64_t nref = pk(-nm * c, -nm * c);
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
    sum = fmaf(sum, scale, s0 + s1);
    m = nm;
  };

  for (int i = 0; i < nunits; ++i) {
    int u, b, k;
    unit_of(i, u, b, k);
    const bool pair = need_draft && k < K;
    const bool pdraw = pdraw_row(b, k);
    const bool p2 = needs_p2(pair, pdraw);
    const int par = i & 1;
    const uint8_t* gt = static_cast<const uint8_t*>(P.target) +
                        ((static_cast<size_t>(b) * (K + 1) + k) * static_cast<size_t>(V) + lo) * ESZ;
    const uint8_t* gd = static_cast<const uint8_t*>(P.draft) +
                        ((static_cast<size_t>(b) * K + k) * static_cast<size_t>(V) + lo) * ESZ;
    if (tid == 0) {   // arm this unit's exchanges (their previous phases completed two units ago)
      mbar_arrive_tx(smem_addr(&x1_bar[par]), static_cast<uint32_t>(nent) * 16u);
      if (p2) mbar_arrive_tx(smem_addr(&x2_bar[par]), static_cast<uint32_t>(C) * 8u);
    }
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

    // ---- pass 1: online (max, sum) of both rows, item by item from the ring
    float mt = ninf(), st = 0.f, md = ninf(), sd = 0.f;
    for (int it = 0; it < nitems; ++it) {
      wait_item();
      const uint8_t* rt_st = ring + (stage * 2) * ITEM_BYTES;
      uint32_t Wt[IW];
      read_item(Wt, rt_st, gt, it);
      if (pair) {
        uint32_t Wd[IW];
        read_item(Wd, rt_st + ITEM_BYTES, gd, it);
        release_item();
        fold_item(Wt, mt, st);
        fold_item(Wd, md, sd);
      } else {
        release_item();
        fold_item(Wt, mt, st);
      }
    }
    // warp partials (symmetric butterfly merges) -> exchange #1
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float om1 = __shfl_xor_sync(0xffffffffu, mt, o), os1 = __shfl_xor_sync(0xffffffffu, st, o);
      const float om2 = __shfl_xor_sync(0xffffffffu, md, o), os2 = __shfl_xor_sync(0xffffffffu, sd, o);
      ms_merge(mt, st, om1, os1, c);
      ms_merge(md, sd, om2, os2, c);
    }
    if (lane < static_cast<int>(C)) {
      const uint32_t dst = smem_addr(&mbox1[par][rank * NW + warp]);
      st_async_v4(peer_addr(dst, lane), mt, st, md, sd, peer_addr(smem_addr(&x1_bar[par]), lane));
    }
    if (!xabort && !mbar_wait_cluster_bounded(smem_addr(&x1_bar[par]), (i >> 1) & 1, xlimit)) {
      xabort = true;
      atomicOr(P.status, kStatusTimeout);
    }
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

    // ---- pass 2: residual and p masses per (item, warp) -> CTA totals -> exchange #2
    float Rtot = 0.f, Ptot = 0.f;
    if (p2) {
      const uint64_t noff_t = pk(-offt, -offt), noff_d = pk(-offd, -offd), neg1 = pk(-1.f, -1.f);
      for (int it = 0; it < nitems; ++it) {
        wait_item();
        const uint8_t* rt_st = ring + (stage * 2) * ITEM_BYTES;
        uint32_t Wt[IW], Wd[IW];
        read_item(Wt, rt_st, gt, it);
        if (pair) read_item(Wd, rt_st + ITEM_BYTES, gd, it);
        release_item();
        uint64_t pacc = pk(0.f, 0.f), racc = pacc;
#pragma unroll
        for (int i = 0; i < NP; ++i) {
          float a0, a1;
          upk(ffma2(pair_of<BF16>(Wt, i), c2, noff_t), a0, a1);
          const uint64_t p = pk(ex2(a0), ex2(a1));     // p of logits 2i, 2i+1
          pacc = fadd2(pacc, p);
          if (pair) {
            float b0, b1, d0, d1;
            upk(ffma2(pair_of<BF16>(Wd, i), c2, noff_d), b0, b1);
            upk(ffma2(pk(ex2(b0), ex2(b1)), neg1, p), d0, d1);   // p - q
            racc = fadd2(racc, pk(fmaxf(d0, 0.f), fmaxf(d1, 0.f)));
          }
        }
        float p0, p1, r0, r1;
        upk(pacc, p0, p1);
        upk(racc, r0, r1);
        const float rw = warp_sum(r0 + r1), pw = warp_sum(p0 + p1);
        if (lane == 0) part[par][it][warp] = make_float2(rw, pw);
      }
      consumers_sync();                       // every warp's (item, warp) masses are in `part`
      float rc = 0.f, pc = 0.f;               // CTA totals, summed in (item, warp) order
      for (int it = 0; it < nitems; ++it)
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          const float2 v = part[par][it][w];
          rc += v.x;
          pc += v.y;
        }
      if (warp == 0 && lane < static_cast<int>(C)) {
        const uint32_t dst = smem_addr(&mbox2[par][rank]);
        const uint32_t rdst = peer_addr(dst, lane);
        const uint32_t rbar = peer_addr(smem_addr(&x2_bar[par]), lane);
        st_async_f32(rdst, rc, rbar);
        st_async_f32(rdst + 4, pc, rbar);
      }
      if (!xabort && !mbar_wait_cluster_bounded(smem_addr(&x2_bar[par]), (x2ph >> par) & 1u, xlimit)) {
        xabort = true;
        atomicOr(P.status, kStatusTimeout);
      }
      x2ph ^= 1u << par;
      float2 e2 = lane < static_cast<int>(C) ? mbox2[par][lane] : make_float2(0.f, 0.f);
      // totals over CTAs: inclusive scans (CTA order), the last lane holds the totals
      const float rin = warp_incl_scan(e2.x, lane), pin = warp_incl_scan(e2.y, lane);
      Rtot = __shfl_sync(0xffffffffu, rin, 31);
      Ptot = __shfl_sync(0xffffffffu, pin, 31);

      // ---- record and the draws this unit may need
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
            if (resid) P.recs[u].rs = -1; else P.recs[u].ps = -1;
          }
          continue;
        }
        // (item, warp) entries of this CTA in order: lane l holds entries l*EP .. l*EP+EP-1
        constexpr int EP = kStreamMaxItems * NW / 32;
        float mw[EP];
#pragma unroll
        for (int q = 0; q < EP; ++q) {
          const int e = lane * EP + q, iti = e / NW, wi = e - iti * NW;
          mw[q] = iti < nitems ? (resid ? part[par][iti][wi].x : part[par][iti][wi].y) : 0.f;
        }
        float cum_w = 0.f;
        const int ow = select_entry<EP>(mw, cum_c, t, lane, &cum_w);
        const int ow_it = ow < 0 ? 0 : ow / NW, ow_w = ow < 0 ? 0 : ow % NW;
        if (warp != ow_w) continue;
        // the owner warp reloads its 512 logits of this item and walks slots, lanes, elements
        const int e0 = ow_it * kStreamItem + ow_w * kStreamWarpSpan;
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
        // slots in vocabulary order, then the lane, then the element
        float sj[kStreamNV], tot[kStreamNV];
#pragma unroll
        for (int j = 0; j < kStreamNV; ++j) {
          float a = 0.f;
#pragma unroll
          for (int e = 0; e < kChunk; ++e) a += mass_at(e0 + (j * 32 + lane) * kChunk + e);
          sj[j] = a;
          tot[j] = warp_sum(a);
        }
        float cum = cum_w, cumj = cum_w;
        int js = -1;
#pragma unroll
        for (int j = 0; j < kStreamNV; ++j) {
          if (js < 0 && cum + tot[j] > t) { js = j; cumj = cum; }
          cum += tot[j];
        }
        if (js < 0) {
          cum = cum_w;
#pragma unroll
          for (int j = 0; j < kStreamNV; ++j) {
            if (tot[j] > 0.f) { js = j; cumj = cum; }
            cum += tot[j];
          }
          if (js < 0) { js = 0; cumj = cum_w; }
        }
        float mine = 0.f;
#pragma unroll
        for (int j = 0; j < kStreamNV; ++j) if (j == js) mine = sj[j];
        float m1[1] = {mine};
        float cl = cumj;
        int l = select_entry<1>(m1, cumj, t, lane, &cl);
        if (l < 0) l = 0;
        int es = 0;
        if (lane == l) {
          float run = cl;
          int first = -1, lastpos = -1;
          for (int e = 0; e < kChunk; ++e) {
            const float me = mass_at(e0 + (js * 32 + l) * kChunk + e);
            run += me;
            if (first < 0 && run > t) first = e;
            if (me > 0.f) lastpos = e;
          }
          es = first >= 0 ? first : (lastpos >= 0 ? lastpos : 0);
          const int idx = lo + e0 + (js * 32 + l) * kChunk + es;
          if (resid) P.recs[u].rs = idx; else P.recs[u].ps = idx;
        }
      }
    }
    if (rank == 0 && tid == 0) {
      UnitRec* r = P.recs + u;
      r->px = px;
      r->qx = qx;
      r->alpha = pair ? fminf(fmaxf(Ptot - Rtot, 0.f), 1.f) : 0.f;
      r->R = Rtot;
    }
  }
  cluster_sync_relaxed();   // no CTA leaves while a peer may still write into its shared memory
}

}  // namespace sv

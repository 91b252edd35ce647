// Sampling-path row kernel (T > 0): two streaming passes per (request, position) unit.
//
// A thread-block cluster of C CTAs works on one unit at a time -- target row k and, for k < K,
// draft row k -- looping over units (persistent).  CTA r owns the vocabulary slice
// [r*slice, (r+1)*slice) of every row and walks it in items of 4096 logits per row.  Inside an
// item, warp w owns logits [w*512, (w+1)*512), lane-interleaved in 8-logit chunks, and every
// thread fetches its own chunks with 16-byte cp.async copies into its own shared-memory slots,
// kStreamStages - 1 items ahead of the one it computes on, across pass and unit boundaries: no
// producer warp and no CTA-wide staging barrier.
//
// Per unit:
//   pass 1 (from HBM): per-thread online (max, sum of
//     2^((z - m) c)) of the target and draft rows -> warp partials -> exchange #1 with st.async
//     into every CTA of the cluster, completing on its mbarrier -> the row's normalisers of p and
//     q, merged in one fixed order so every warp of every CTA holds bitwise-identical values;
//     p_k(x_k), q_k(x_k) and the accept test, as the cut kernel will evaluate them
//   pass 2 (the same bytes again, L2 hits while the data streamed in between fits in L2): per element p = 2^(z c - offt),
//     q = 2^(z c - offd); per (item, warp) masses of r = max(0, p - q) and of p -> CTA totals ->
//     exchange #2 -> residual mass R, alpha = sum p - R (= sum min(p, q)), and the owner of each
//     needed inverse-CDF draw, found in vocabulary order (CTA, item, warp).  A pair that passes
//     the test and draws nothing only needs alpha = sum 2^min(a, b) (one exp2 per logit pair).
//   the owner warp reloads its 512 logits of the row(s) and walks slot / lane / element prefix
//     sums to the drawn index.  The residual is drawn only where the test fails, the p draw only
//     at the verified depth (or at every row when the depth is chosen afterwards).
// DRAM reads each logit once; the second pass is served by L2.  The serial cut runs afterwards in
// a small kernel chained with programmatic dependent launch.
#pragma once

#include <cuda_bf16.h>

#include "spec_async.cuh"

namespace sv {

constexpr int kStreamWarps = 8;                                 // warps per CTA
constexpr int kStreamThreads = 32 * kStreamWarps;
constexpr int kStreamStages = kStreamStagesHost;                // items in each thread's cp.async pipeline
constexpr int kStreamNV = 2;                                    // 8-logit chunks per lane per item
constexpr int kStreamWarpSpan = 32 * kStreamNV * kChunk;        // logits of one warp per item (512)
constexpr int kStreamItem = kStreamWarps * kStreamWarpSpan;     // logits per row per item (4096)
constexpr int kStreamMaxItems = 32;                             // items per slice (slice <= 131072)

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



// Every warp of the CTA.
__device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kStreamWarps) : "memory");
}

// 16-byte asynchronous global -> shared copy by this thread (L1 bypassed), `src_bytes` <= 16 of
// them read from global and the rest of the 16 zero-filled; completion tracked per commit group.
// (No L2 cache-policy operand: the form carrying both a source size and a cache policy faulted.)
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
// The same copy, full 16 bytes, with compile-time byte offsets on both addresses.
template <uint32_t SO, uint32_t GO>
__device__ __forceinline__ void cp_async16_at(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0+%2], [%1+%3], 16;" ::"r"(dst), "l"(src), "n"(SO), "n"(GO)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

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
  constexpr int EP = kStreamMaxItems * NW / 32;   // (item, warp) entries per lane in the owner search
  using Chunk = uint4[BF16 ? 1 : 2];

  // each thread's own copies: stage s, row r, chunk j, 16-byte piece h of (warp, lane) at uint4
  // index (((s * 2 + r) * NV + j) * HP + h) * 256 + warp * 32 + lane (a warp reads 512 B at once)
  extern __shared__ __align__(128) uint4 stage_buf[];
  __shared__ __align__(16) float4 mbox1[2][ENT];               // (m_t, s_t, m_d, s_d) per (CTA, warp)
  __shared__ __align__(16) float2 mbox2[2][kMaxCluster];       // (R, P) per CTA
  __shared__ float2 part[2][kStreamMaxItems][NW];              // (R, P) per (item, warp) of this CTA
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
    for (int p = 0; p < 2; ++p) {
      mbar_init(smem_addr(&x1_bar[p]), 1);
      mbar_init(smem_addr(&x2_bar[p]), 1);
    }
    mbar_fence_init();
  }
  __syncthreads();
  cluster_sync();   // every CTA's barriers exist before any peer sends into them

  bool xabort = false;   // gave up waiting for an exchange (test hook or a lost peer)
  const long long xlimit = P.wait_limit;   // ns per exchange wait; 0 gives up at once
  uint32_t x2ph = 0;

  constexpr uint32_t NEG = BF16 ? 0xff80ff80u : 0xff800000u;
  constexpr int WPC = BF16 ? 4 : 8;                  // 32-bit words per 8-logit chunk
  constexpr int IW = kStreamNV * WPC;                // words per lane per row per item
  constexpr int NP = kStreamNV * kChunk / 2;         // logit pairs per lane per row per item
  constexpr int NV = kStreamNV;
  constexpr int HP = WPC / 4;                        // 16-byte pieces per 8-logit chunk
  constexpr int S = kStreamStages;
  // ---- per-thread copy pipeline over the CTA's (unit, pass, item) sequence, S - 1 items ahead;
  // every step commits one group (possibly empty) so wait_group(S - 1) retires the oldest
  int iu = 0, ipass = 0, iit = 0, ipasses = 0;       // issue cursor
  bool ipair = false;
  const uint8_t* irt = nullptr;
  const uint8_t* ird = nullptr;
  auto issue_unit = [&]() {
    if (iu >= nunits) return;
    int u, b, k;
    unit_of(iu, u, b, k);
    ipair = need_draft && k < K;
    ipasses = needs_p2(ipair, pdraw_row(b, k)) ? 2 : 1;
    irt = static_cast<const uint8_t*>(P.target) + ((static_cast<size_t>(b) * (K + 1) + k) * static_cast<size_t>(V) + lo) * ESZ;
    ird = static_cast<const uint8_t*>(P.draft) + ((static_cast<size_t>(b) * K + k) * static_cast<size_t>(V) + lo) * ESZ;
  };
  int istage = 0;
  // this thread's first logit of an item and its first 16-byte slot of stage 0, row 0
  const int tofs = warp * kStreamWarpSpan + lane * kChunk;
  const uint32_t sbase = smem_addr(&stage_buf[warp * 32 + lane]);
  constexpr uint32_t kRowBytes = NV * HP * 256 * 16;                // one row of one stage
  auto issue_whole = [&](uint32_t s0, const uint8_t* src) {         // every piece of an item
    static_assert(kStreamNV == 2, "two chunks per lane");
    constexpr uint32_t GJ = 32 * kChunk * ESZ;                      // chunk j + 1 of a lane, in bytes
    cp_async16_at<0u, 0u>(s0, src);
    if constexpr (HP == 1) {
      cp_async16_at<4096u, GJ>(s0, src);
    } else {
      cp_async16_at<4096u, 16u>(s0, src);
      cp_async16_at<8192u, GJ>(s0, src);
      cp_async16_at<12288u, GJ + 16u>(s0, src);
    }
  };
  auto issue_next = [&]() {
    if (tma && iu < nunits && nitems > 0) {
      const int e0 = iit * kStreamItem;
      const int nval = min(kStreamItem, n - e0);
      if (nval == kStreamItem) {
        const size_t g0 = static_cast<size_t>(e0 + tofs) * ESZ;
        const uint32_t s0 = sbase + static_cast<uint32_t>(istage) * (2u * kRowBytes);
        issue_whole(s0, irt + g0);
        if (ipair) issue_whole(s0 + kRowBytes, ird + g0);
      } else {
#pragma unroll
      for (int j = 0; j < NV; ++j) {
        const int o = warp * kStreamWarpSpan + (j * 32 + lane) * kChunk;
        const int vb = (nval - o) * ESZ;             // valid bytes from this chunk on
#pragma unroll
        for (int h = 0; h < HP; ++h) {
          const int sb = min(max(vb - h * 16, 0), 16);
          if (sb > 0) {
            const size_t go = static_cast<size_t>(e0 + o) * ESZ + h * 16;
            const int q = (((istage * 2) * NV + j) * HP + h) * 256 + warp * 32 + lane;
            cp_async16(smem_addr(&stage_buf[q]), irt + go, static_cast<uint32_t>(sb));
            if (ipair)
              cp_async16(smem_addr(&stage_buf[q + NV * HP * 256]), ird + go, static_cast<uint32_t>(sb));
          }
        }
      }
      }
      if (++iit == nitems) {
        iit = 0;
        if (++ipass == ipasses) {
          ipass = 0;
          ++iu;
          issue_unit();
        }
      }
    }
    cp_async_commit();
    if (++istage == S) istage = 0;
  };
  issue_unit();
  for (int q = 0; q < S - 1; ++q) issue_next();
  int stage = 0;   // stage of the next item to consume
  // the next item of the sequence is in this thread's stage: issue the one S - 1 further on
  // (into the stage consumed last step, whose words are already in registers), then retire it
  auto next_item = [&]() {
    issue_next();
    cp_async_wait<S - 1>();
  };
  auto done_item = [&]() {
    if (++stage == S) stage = 0;
  };
  // this lane's logits of item `it` of row r (0 target, 1 draft), as raw words: 16-byte reads
  // of its own copies, -inf past the slice end; element-wise global reads for unaligned rows
  auto read_item = [&](uint32_t (&W)[IW], int r, const uint8_t* grow, int it) {
    const int e0 = it * kStreamItem;
    const int nval = min(kStreamItem, n - e0);
    if (tma) {
#pragma unroll
      for (int j = 0; j < NV; ++j) {
#pragma unroll
        for (int h = 0; h < HP; ++h) {
          const uint4 v = stage_buf[(((stage * 2 + r) * NV + j) * HP + h) * 256 + warp * 32 + lane];
          W[j * WPC + h * 4] = v.x;
          W[j * WPC + h * 4 + 1] = v.y;
          W[j * WPC + h * 4 + 2] = v.z;
          W[j * WPC + h * 4 + 3] = v.w;
        }
      }
      if (nval < kStreamItem) {
#pragma unroll
        for (int j = 0; j < NV; ++j) {
          const int o = warp * kStreamWarpSpan + (j * 32 + lane) * kChunk;
#pragma unroll
          for (int e = 0; e < kChunk; ++e) {
            if (o + e >= nval) {
              if constexpr (BF16) {
                uint32_t& w = W[j * WPC + (e >> 1)];
                w = (e & 1) ? ((w & 0x0000ffffu) | 0xff800000u) : ((w & 0xffff0000u) | 0x0000ff80u);
              } else {
                W[j * WPC + e] = NEG;
              }
            }
          }
        }
      }
      return;
    }
    const uint8_t* src = grow + static_cast<size_t>(e0) * ESZ;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
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

    // ---- pass 1: online (max, sum) of both rows, item by item
    float mt = ninf(), st = 0.f, md = ninf(), sd = 0.f;
    for (int it = 0; it < nitems; ++it) {
      next_item();
      uint32_t Wt[IW];
      read_item(Wt, 0, gt, it);
      if (pair) {
        uint32_t Wd[IW];
        read_item(Wd, 1, gd, it);
        done_item();
        fold_item(Wt, mt, st);
        fold_item(Wd, md, sd);
      } else {
        done_item();
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
    // a pair that passes the test and draws nothing needs only alpha = sum min(p, q), and
    // min(2^a, 2^b) = 2^min(a, b): one exp2 per logit pair, no per-item masses
    const bool alpha_only = pair && !rejects && !pdraw;
    if (p2) {
      const uint64_t noff_t = pk(-offt, -offt), noff_d = pk(-offd, -offd), neg1 = pk(-1.f, -1.f);
      if (alpha_only) {
        uint64_t aacc = pk(0.f, 0.f);
        for (int it = 0; it < nitems; ++it) {
          next_item();
          uint32_t Wt[IW], Wd[IW];
          read_item(Wt, 0, gt, it);
          read_item(Wd, 1, gd, it);
          done_item();
#pragma unroll
          for (int i = 0; i < NP; ++i) {
            float a0, a1, b0, b1;
            upk(ffma2(pair_of<BF16>(Wt, i), c2, noff_t), a0, a1);
            upk(ffma2(pair_of<BF16>(Wd, i), c2, noff_d), b0, b1);
            aacc = fadd2(aacc, pk(ex2(fminf(a0, b0)), ex2(fminf(a1, b1))));
          }
        }
        float a0, a1;
        upk(aacc, a0, a1);
        const float aw = warp_sum(a0 + a1);
        if (lane == 0) part[par][0][warp] = make_float2(aw, 0.f);
      } else {
      for (int it = 0; it < nitems; ++it) {
        next_item();
        uint32_t Wt[IW], Wd[IW];
        read_item(Wt, 0, gt, it);
        if (pair) read_item(Wd, 1, gd, it);
        done_item();
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
      consumers_sync();                       // every warp's (item, warp) masses are in `part`
      if (warp == 0) {
        // CTA totals: lane l sums entries l*EP .. l*EP+EP-1 in (item, warp) order, then a scan
        // across lanes -- the same grouping the owner search below uses
        float rl = 0.f, pl = 0.f;
#pragma unroll
        for (int q = 0; q < EP; ++q) {
          const int e = lane * EP + q, iti = e / NW, wi = e - iti * NW;
          if (iti < pitems) {
            const float2 v = part[par][iti][wi];
            rl += v.x;
            pl += v.y;
          }
        }
        const float rc = __shfl_sync(0xffffffffu, warp_incl_scan(rl, lane), 31);
        const float pc = __shfl_sync(0xffffffffu, warp_incl_scan(pl, lane), 31);
        if (lane < static_cast<int>(C)) {
          const uint32_t dst = smem_addr(&mbox2[par][rank]);
          const uint32_t rdst = peer_addr(dst, lane);
          const uint32_t rbar = peer_addr(smem_addr(&x2_bar[par]), lane);
          st_async_f32(rdst, rc, rbar);
          st_async_f32(rdst + 4, pc, rbar);
        }
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
      // alpha-only units carry sum min(p, q) in the first total; R is then only informative
      const float alpha = alpha_only ? Rtot : Ptot - Rtot;
      r->alpha = pair ? fminf(fmaxf(alpha, 0.f), 1.f) : 0.f;
      r->R = alpha_only ? fmaxf(1.f - Rtot, 0.f) : Rtot;
    }
  }
  cp_async_wait<0>();        // only empty groups remain; retire them before leaving
  cluster_sync_relaxed();   // no CTA leaves while a peer may still write into its shared memory
}

}  // namespace sv

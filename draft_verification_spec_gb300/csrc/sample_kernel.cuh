// Sampling-path row kernel (T > 0): two passes per (request, position) unit over a CTA's slice of
// the unit's rows, which stays in shared memory between them, so HBM is read once.
//
// A thread-block cluster of C CTAs works on a sequence of units -- target row k and, for k < K,
// draft row k -- (persistent; units go round-robin to clusters, pairs first).  CTA r owns the
// vocabulary slice [r*slice, (r+1)*slice) of every row and holds its bytes of the current unit in
// a shared-memory slab of itmax items of kSampItemBytes per row.  Warp w owns bytes
// [w*kSampWarpBytes, (w+1)*kSampWarpBytes) of every item and each lane its kSampPieces 16-byte
// pieces of those, so the lane that copies a piece is the only one that ever reads it: no barrier
// sits between a copy and its use, and a wait is one cp.async.wait_group.
//   pass 1, as the unit's asynchronous copies land (one commit group per item): per-lane online
//     (max, sum of 2^((z - m) c)) of the target and draft rows -> warp maximum and rescaled warp
//     sum -> the CTA's partial, merged by warp 0 in warp order -> one st.async into every CTA of
//     the cluster, completing on its mbarrier -> the row normalisers of p and q, merged in rank
//     order by warp 0 of every CTA (bitwise-identical values everywhere); p_k(x_k), q_k(x_k) and
//     the accept test, exactly as the cut kernel evaluates them afterwards
//   pass 2, from shared memory: per logit p = 2^(z c - offt), q = 2^(z c - offd).  A pair that
//     passes the test and needs no draw only needs alpha = sum 2^min(a, b) (one exp2 per logit
//     pair); otherwise every warp writes its (item, warp) masses of r = max(0, p - q) and of p to
//     the row's mass table.  As soon as a lane is done with an item, it copies its pieces of the
//     next unit's item into the same bytes.  The CTA's alpha partial (its warps' in warp order)
//     reaches rank 0 with the next exchange (the last unit's in an exchange of its own), and rank
//     0 writes the row's alpha, summed in rank order, to its record.
// The draws themselves are made by the chained cut kernel from the mass tables.  While a CTA
// waits on its cluster's exchange, the other CTAs resident on its SM keep HBM busy.  A target row
// that no draw needs is skipped entirely.  Rows that do not start on 16-byte boundaries are read
// element-wise in pass 1 and stored to the slab for pass 2.
//
// Every wait is bounded by wall time.  A wait that runs out records SPEC_ERR_DEVICE_TIMEOUT and
// then waits once more with a long limit, so the exchange protocol stays consistent and no peer
// store lands in shared memory after the CTA has left.  Only if that second wait also runs out
// does the CTA stop waiting (abort mode; results unspecified).  Every phase a CTA arms it also
// waits for, and the kernel ends with a cluster barrier, so no CTA exits while a store it sent or
// a store sent to it may still be in flight.
#pragma once

#include <type_traits>

#include <cuda_bf16.h>

#include "packed_math.cuh"
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
  static constexpr int IL = kSampItemBytes / ESZ;      // logits per row per item
  static constexpr int WS = kSampWarpBytes / ESZ;      // logits per row per item per warp
  static constexpr int PS = 32 * EPP;                  // piece j of lane l: [j*PS + l*EPP, +EPP) of the warp's logits
};

// 16-byte asynchronous copy global -> shared by this thread (cached in L2 only, evict-first: every
// byte is read from global memory once).  The form without a source-size operand: a piece is
// either copied whole or not at all.
__device__ __forceinline__ void cp_async16(uint32_t dst, const uint8_t* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "l"(policy)
               : "memory");
}
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
// wait_group with a run-time depth (uniform across the CTA); deeper than 15 waits for everything
__device__ __forceinline__ void cp_async_wait_upto(int n) {
  switch (n) {
    case 15: cp_async_wait<15>(); break;
    case 14: cp_async_wait<14>(); break;
    case 13: cp_async_wait<13>(); break;
    case 12: cp_async_wait<12>(); break;
    case 11: cp_async_wait<11>(); break;
    case 10: cp_async_wait<10>(); break;
    case 9: cp_async_wait<9>(); break;
    case 8: cp_async_wait<8>(); break;
    case 7: cp_async_wait<7>(); break;
    case 6: cp_async_wait<6>(); break;
    case 5: cp_async_wait<5>(); break;
    case 4: cp_async_wait<4>(); break;
    case 3: cp_async_wait<3>(); break;
    case 2: cp_async_wait<2>(); break;
    case 1: cp_async_wait<1>(); break;
    default: cp_async_wait<0>(); break;
  }
}

__device__ __forceinline__ void lds16(uint32_t* w, uint32_t addr) {
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
               : "r"(addr));
}
__device__ __forceinline__ void sts16(uint32_t addr, const uint32_t* w) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3])
               : "memory");
}

// A unit as a CTA walks it: its row slices, its record, its exchange slot.
struct SampUnit {
  const uint8_t* gt;       // target row slice (this CTA's part)
  const uint8_t* gd;       // draft row slice (pairs)
  int b, k, rec, idx;      // request, position, record index, needed-unit ordinal of this CTA
  bool pair, pdraw;
  int x = -1;              // drafted token (thread 0 of a tested pair; -1 otherwise)
  float uk;                // its accept uniform
  float ztx, zdx;          // target and draft logits at x (lane 0)
};

template <bool BF16, bool ALIGNED>
__global__ void __launch_bounds__(kSampThreads, kSampMinBlocks) sample_kernel(const __grid_constant__ RowParams P) {
  using G = SampGeo<BF16>;
  constexpr int ESZ = G::ESZ, EPP = G::EPP, NPC = G::NPC, NWD = G::NWD;
  constexpr int IL = G::IL, WS = G::WS, PS = G::PS;
  constexpr int NWARP = kSampWarps;
  constexpr int IB = kSampItemBytes, WB = kSampWarpBytes;
  constexpr int NQ = BF16 ? NWD : NWD / 2;         // logit pairs per lane per row per item
  constexpr uint32_t NEG = BF16 ? 0xff80ff80u : 0xff800000u;

  // the slab: warp w, item it, row r (0 target, 1 draft) at byte ((w * itmax + it) * 2 + r) * WB
  extern __shared__ __align__(128) uint8_t slab[];
  __shared__ __align__(16) float4 mbox1[2][kMaxCluster];       // (m_t, s_t, m_d, s_d) per CTA of the cluster
  __shared__ float abox[2][kMaxCluster];                       // rank 0: the previous unit's alpha per CTA
  __shared__ __align__(16) float4 part_sh[NWARP];              // this CTA's warp partials
  __shared__ float apart_sh[NWARP];                            // this CTA's warp alpha partials
  __shared__ __align__(8) uint64_t x1_bar[2];
  __shared__ float norm_sh[2];                                 // offt, offd of the current unit
  __shared__ int mode_sh;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank(), C = cluster_ncta();
  const uint32_t cid = cluster_idx(), ncl = cluster_count();
  const int K = P.K, V = P.V;
  const int itmax = P.itmax;
  const int lo = static_cast<int>(rank) * P.slice;
  const int n = max(0, min(P.slice, V - lo));                  // this CTA's slice length
  const int nitems = (n + IL - 1) / IL;
  const bool need_draft = (P.flags & F_NEED_DRAFT) != 0;
  const bool stats_only = (P.flags & F_STATS_ONLY) != 0;
  const bool all_pdraws = (P.flags & F_ALL_PDRAWS) != 0;
  const float c = P.c;
  const int nc = static_cast<int>(C);                          // exchange entries per unit: one per CTA
  const int nunits = static_cast<int>(cid) < P.total_units
                         ? (P.total_units - static_cast<int>(cid) + static_cast<int>(ncl) - 1) / static_cast<int>(ncl)
                         : 0;
  const int npairs = need_draft ? P.B * K : 0;   // units [0, npairs) are (target, draft) pairs
  // this lane's byte offset of piece j of item it in a row slice: it * IB + wl + j * 512; its
  // first logit there: it * IL + el + j * PS
  const int wl = warp * WB + lane * 16;
  const int el = warp * WS + lane * EPP;
  // logits of this warp's part of the last item that lie inside the slice
  const int last_nval = nitems > 0 ? min(WS, max(0, n - (nitems - 1) * IL - warp * WS)) : 0;
  const uint32_t slab_l = smem_addr(slab) + static_cast<uint32_t>(warp * itmax * 2 * WB + lane * 16);
  auto slot = [&](int it, int r) -> uint32_t { return slab_l + static_cast<uint32_t>((it * 2 + r) * WB); };

  // unit u -> (b, k): the pairs first (b-major), then the target rows k = K (or, without draft
  // rows, every target row); larger units first gives round-robin assignment a short tail
  auto unit_of = [&](int i, int& b, int& k) {
    const int u = static_cast<int>(cid) + i * static_cast<int>(ncl);
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

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    for (int p = 0; p < 2; ++p) mbar_init(smem_addr(&x1_bar[p]), 1);
    abort_flag = 0;
  }
  mbar_fence_init();
  // pieces of the last item past the slice end are never copied: they hold -inf for good
  if (nitems > 0) {
    const uint32_t neg[4] = {NEG, NEG, NEG, NEG};
#pragma unroll
    for (int j = 0; j < NPC; ++j)
      if (j * PS + lane * EPP >= last_nval) {
        sts16(slot(nitems - 1, 0) + j * 512, neg);
        sts16(slot(nitems - 1, 1) + j * 512, neg);
      }
  }
  __syncthreads();
  cluster_sync();   // every CTA's barriers exist before any peer sends into them
  // launched with programmatic serialization: the logits, tokens and records are touched only
  // once the preceding grid on the stream has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const long long wlimit = P.wait_limit;
  // A bounded wait on an exchange phase (completed by peers' stores; acquire at cluster scope), by
  // one thread while the rest of the CTA waits at a barrier without issuing.  On timeout record
  // it, then wait with the long limit; if that also runs out, switch the CTA to abort mode (no
  // more waiting).  The common case reads no clock.
  auto wait_phase = [&](uint32_t bar, uint32_t parity) {
    if (wlimit > 0 && mbar_try_cluster(bar, parity)) return true;
    if (*static_cast<volatile int*>(&abort_flag)) return mbar_try_cluster(bar, parity);
    if (mbar_wait_for<true>(bar, parity, wlimit)) return true;
    atomicOr(P.status, kStatusTimeout);
    if (mbar_wait_for<true>(bar, parity, kDrainNs)) return true;
    *static_cast<volatile int*>(&abort_flag) = 1;
    return false;
  };

  // rows not on 16-byte boundaries: this lane's words of item `it` of a row (slice base g),
  // element by element, -inf past the slice end
  auto row_words = [&](uint32_t (&W)[NWD], const uint8_t* g, int it) {
#pragma unroll
    for (int j = 0; j < NPC; ++j) {
      const int o = it * IL + el + j * PS;       // first logit of the piece in the slice
#pragma unroll
      for (int q = 0; q < 4; ++q) W[4 * j + q] = NEG;
#pragma unroll
      for (int e = 0; e < EPP; ++e) {
        if (o + e < n) {
          if constexpr (BF16) {
            const uint32_t h16 = reinterpret_cast<const uint16_t*>(g)[o + e];
            uint32_t& w = W[4 * j + (e >> 1)];
            w = (e & 1) ? ((w & 0x0000ffffu) | (h16 << 16)) : ((w & 0xffff0000u) | h16);
          } else {
            W[4 * j + e] = reinterpret_cast<const uint32_t*>(g)[o + e];
          }
        }
      }
    }
  };
  auto slab_words = [&](uint32_t (&W)[NWD], uint32_t addr) {
#pragma unroll
    for (int j = 0; j < NPC; ++j) lds16(&W[4 * j], addr + j * 512);
  };
  auto slab_store = [&](uint32_t addr, const uint32_t (&W)[NWD]) {
#pragma unroll
    for (int j = 0; j < NPC; ++j) sts16(addr + j * 512, &W[4 * j]);
  };

  // one item of a unit into the slab (t, d: this lane's first byte of the row slices; d null for
  // a target row alone)
  const uint64_t policy = l2_evict_first_policy();
  auto issue_item = [&](const uint8_t* t, const uint8_t* d, int it) {
    const size_t off = static_cast<size_t>(it) * IB;
    const uint32_t dst = slot(it, 0);
    const bool full = it != nitems - 1;
#pragma unroll
    for (int j = 0; j < NPC; ++j) {
      if (full || j * PS + lane * EPP < last_nval) {
        cp_async16(dst + j * 512, t + off + j * 512, policy);
        if (d) cp_async16(dst + WB + j * 512, d + off + j * 512, policy);
      }
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
    for (int i = 0; i < NQ; i += 2) {
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

  // ---------------------------------------------------------------- the unit sequence
  int iu = 0;                                // next unit index to look at
  int taken = 0;                             // needed units taken so far
  auto take_unit = [&](SampUnit& U) -> bool {   // the next needed unit, if any
    for (; iu < nunits; ++iu) {
      int b, k;
      unit_of(iu, b, k);
      const bool pair = need_draft && k < K;
      const bool pdraw = pdraw_row(b, k);
      if (!(pair || pdraw)) continue;
      ++iu;
      U.b = b;
      U.k = k;
      U.rec = b * P.U + k;
      U.pair = pair;
      U.pdraw = pdraw;
      U.idx = taken++;
      U.gt = static_cast<const uint8_t*>(P.target) +
             ((static_cast<size_t>(b) * (K + 1) + k) * static_cast<size_t>(V) + lo) * ESZ;
      U.gd = pair ? static_cast<const uint8_t*>(P.draft) +
                        ((static_cast<size_t>(b) * K + k) * static_cast<size_t>(V) + lo) * ESZ
                  : U.gt;
      // the accept test's operands (warp 0 runs it)
      const bool tested = !stats_only && k < K && warp == 0;
      U.x = (tested && lane == 0) ? __ldg(&P.tokens[static_cast<size_t>(b) * K + k]) : -1;
      U.uk = tested ? __ldg(&P.uniforms[static_cast<size_t>(b) * (K + 1) + k]) : 0.f;
      U.ztx = U.zdx = 0.f;
      return true;
    }
    return false;
  };
  // thread 0: the logits at the drafted token of a tested pair (no other unit reads the draft)
  auto fetch_at_token = [&](SampUnit& U) {
    if (tid == 0 && U.pair && U.x >= 0 && U.x < V) {
      const size_t ot = (static_cast<size_t>(U.b) * (K + 1) + U.k) * V + U.x;
      const size_t od = (static_cast<size_t>(U.b) * K + U.k) * V + U.x;
      if constexpr (BF16) {
        U.ztx = __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const uint16_t*>(P.target) + ot)) << 16);
        U.zdx = __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const uint16_t*>(P.draft) + od)) << 16);
      } else {
        U.ztx = __ldg(reinterpret_cast<const float*>(P.target) + ot);
        U.zdx = __ldg(reinterpret_cast<const float*>(P.draft) + od);
      }
    }
  };

  // pass 1 of a unit over the slab; PAIR: the draft row too
  auto pass1 = [&](auto pair_tag, const SampUnit& A, float& mt, float& st, float& md, float& sd) {
    constexpr bool PAIR = decltype(pair_tag)::value;
    for (int it = 0; it < nitems; ++it) {
      uint32_t Wt[NWD], Wd[NWD];
      if constexpr (ALIGNED) {
        cp_async_wait_upto(nitems - 1 - it);        // this lane's pieces of the item have landed
        slab_words(Wt, slot(it, 0));
        if constexpr (PAIR) slab_words(Wd, slot(it, 1));
      } else {
        row_words(Wt, A.gt, it);
        slab_store(slot(it, 0), Wt);
        if constexpr (PAIR) {
          row_words(Wd, A.gd, it);
          slab_store(slot(it, 1), Wd);
        }
      }
      fold(Wt, mt, st);
      if constexpr (PAIR) fold(Wd, md, sd);
    }
  };

  // pass 2 of a unit from the slab; each item, once consumed, takes the next unit's copies
  // (nT / nD: this lane's first byte of its row slices, nT null if there is none).  MODE: alpha
  // only, full masses, or target masses alone.  Returns the warp's alpha partial (lane-uniform).
  auto pass2 = [&](auto mode_tag, float offt, float offd, float* mrow, const uint8_t* nT, const uint8_t* nD) -> float {
    constexpr int MODE = decltype(mode_tag)::value;
    const uint64_t noff_t = pk(-offt, -offt), noff_d = pk(-offd, -offd);
    const uint64_t neg1 = pk(-1.f, -1.f);
    uint64_t aacc = pk(0.f, 0.f), bacc = aacc;
    float pw = 0.f, rw = 0.f;                      // full / single: the warp's totals (lanes 16 / 0)
    for (int it = 0; it < nitems; ++it) {
      uint32_t Wt[NWD], Wd[NWD];
      slab_words(Wt, slot(it, 0));
      if constexpr (MODE != kModeSingle) slab_words(Wd, slot(it, 1));
      if constexpr (MODE == kModeAlpha) {
#pragma unroll
        for (int q = 0; q < NQ; q += 2) {
          float a0, a1, b0, b1, a2, a3, b2, b3;
          upk(ffma2(pair_of<BF16>(Wt, q), c2, noff_t), a0, a1);
          upk(ffma2(pair_of<BF16>(Wd, q), c2, noff_d), b0, b1);
          upk(ffma2(pair_of<BF16>(Wt, q + 1), c2, noff_t), a2, a3);
          upk(ffma2(pair_of<BF16>(Wd, q + 1), c2, noff_d), b2, b3);
          aacc = fadd2(aacc, pk(ex2(fminf(a0, b0)), ex2(fminf(a1, b1))));
          bacc = fadd2(bacc, pk(ex2(fminf(a2, b2)), ex2(fminf(a3, b3))));
        }
      } else {
        uint64_t pacc = pk(0.f, 0.f), racc = pacc;
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          float a0, a1;
          upk(ffma2(pair_of<BF16>(Wt, q), c2, noff_t), a0, a1);
          const uint64_t p = pk(ex2(a0), ex2(a1));     // p of logits 2q, 2q+1
          pacc = fadd2(pacc, p);
          if constexpr (MODE == kModeFull) {
            float b0, b1, d0, d1;
            upk(ffma2(pair_of<BF16>(Wd, q), c2, noff_d), b0, b1);
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
        if ((lane & 15) == 0) {
          mrow[((static_cast<int>(rank) * itmax + it) * NWARP + warp) * 2 + (lane >> 4)] = keep;
          if (hi) pw += keep; else rw += keep;
        }
      }
      if constexpr (ALIGNED) {
        // the item's words are in registers and used: the next unit's copies take its bytes
        if (nT) issue_item(nT, nD, it);
        cp_async_commit();
      }
    }
    if constexpr (MODE == kModeAlpha) {
      float a0, a1;
      upk(fadd2(aacc, bacc), a0, a1);
      return warp_sum(a0 + a1);
    } else {
      // sum p - R over this warp's items (lane 16 holds P, lane 0 holds R)
      return __shfl_sync(0xffffffffu, pw, 16) - __shfl_sync(0xffffffffu, rw, 0);
    }
  };

  SampUnit A;
  bool hasA = take_unit(A);
  if (hasA) fetch_at_token(A);
  if constexpr (ALIGNED) {
    // the first unit's slice, one commit group per item; pass 2 commits one group per item too,
    // so when pass 1 consumes item it, the groups after it are items it+1 .. nitems-1
    if (hasA)
      for (int it = 0; it < nitems; ++it) {
        issue_item(A.gt + wl, A.pair ? A.gd + wl : nullptr, it);
        cp_async_commit();
      }
  }

  // alpha of a pair: each CTA's partial of unit i (its warps' partials summed in warp order)
  // travels to rank 0 with the exchange of unit i + 1 (or a last exchange of its own), where warp 0
  // sums the CTAs' partials in rank order
  bool has_prev = false;
  float prev_aw = 0.f;
  int prev_rec = 0;
  auto alpha_to_record = [&](int par) {
    const float s = warp_sum(lane < nc ? abox[par][lane] : 0.f);
    if (lane == 0) P.recs[prev_rec].alpha = fminf(fmaxf(s, 0.f), 1.f);   // NaN -> 0
  };
  // warp 0: the sum of the CTA's warp alpha partials in warp order
  auto cta_alpha = [&]() { return warp_sum(lane < NWARP ? apart_sh[lane] : 0.f); };

  while (hasA) {
    const int apar = A.idx & 1;
    if (tid == 0)
      mbar_arrive_tx(smem_addr(&x1_bar[apar]), static_cast<uint32_t>(nc) * (rank == 0 && has_prev ? 20u : 16u));

    // ---- pass 1, then the warp partials (warp maximum, every lane's sum rescaled to it), merged
    // by warp 0 in warp order into the CTA's partial, which goes to every CTA of the cluster (with
    // the previous unit's alpha partial to rank 0)
    float mt = ninf(), st = 0.f, md = ninf(), sd = 0.f;
    if (A.pair) pass1(std::true_type(), A, mt, st, md, sd);
    else pass1(std::false_type(), A, mt, st, md, sd);
    {
      const float wt = warp_maxf(mt), wd = warp_maxf(md);
      const float rt = wt == ninf() ? 0.f : wt, rd = wd == ninf() ? 0.f : wd;
      st = warp_sum(st * ex2((mt - rt) * c));
      sd = warp_sum(sd * ex2((md - rd) * c));
      if (lane == 0) {
        part_sh[warp] = make_float4(wt, st, wd, sd);
        apart_sh[warp] = prev_aw;
      }
    }
    __syncthreads();
    if (warp == 0) {
      const float4 v = lane < NWARP ? part_sh[lane] : make_float4(ninf(), 0.f, ninf(), 0.f);
      const float Mt = warp_maxf(v.x), Md = warp_maxf(v.z);
      const float rt = Mt == ninf() ? 0.f : Mt, rd = Md == ninf() ? 0.f : Md;
      const float St = warp_sum(lane < NWARP ? v.y * ex2((v.x - rt) * c) : 0.f);
      const float Sd = warp_sum(lane < NWARP ? v.w * ex2((v.z - rd) * c) : 0.f);
      const float Ac = cta_alpha();
      if (lane < nc)
        st_async_v4(peer_addr(smem_addr(&mbox1[apar][rank]), lane), Mt, St, Md, Sd,
                    peer_addr(smem_addr(&x1_bar[apar]), lane));
      if (has_prev && lane == 0)
        st_async_f32(peer_addr(smem_addr(&abox[apar][rank]), 0), Ac, peer_addr(smem_addr(&x1_bar[apar]), 0));
    }

    // ---- the next unit (while the exchange completes), then the row normalisers and the accept
    // test, by warp 0 alone while the other warps wait at the barrier; the barrier carries thread
    // 0's acquire of the peers' partials and warp 0's results to the whole CTA
    SampUnit N;
    const bool hasN = take_unit(N);
    if (hasN) fetch_at_token(N);
    if (warp == 0) {
      if (lane == 0) wait_phase(smem_addr(&x1_bar[apar]), (A.idx >> 1) & 1);
      __syncwarp();
      const float4 v = lane < nc ? mbox1[apar][lane] : make_float4(ninf(), 0.f, ninf(), 0.f);
      const float Mt = warp_maxf(v.x), Md = warp_maxf(v.z);
      const float rt = (Mt == ninf()) ? 0.f : Mt, rd = (Md == ninf()) ? 0.f : Md;
      const float St = warp_sum(lane < nc ? v.y * ex2((v.x - rt) * c) : 0.f);
      const float Sd = warp_sum(lane < nc ? v.w * ex2((v.z - rd) * c) : 0.f);
      if (lane == 0) {
        // p_v = 2^(z c - offt), q_v = 2^(z c - offd): the normalisers folded into the exponent
        const float offt = (Mt == ninf() ? 0.f : Mt * c) + lg2f(St);
        const float offd = (Md == ninf() ? 0.f : Md * c) + lg2f(Sd);
        float px = 0.f, qx = 0.f;
        const bool xin = A.x >= 0 && A.x < V;
        if (xin) {
          px = ex2(fmaf(A.ztx, c, -offt));
          qx = ex2(fmaf(A.zdx, c, -offd));
        }
        const bool rejects = !stats_only && A.k < K && !(xin && A.uk * qx < px);
        // a pair that passes the test and draws nothing needs only alpha = sum min(p, q), and
        // min(2^a, 2^b) = 2^min(a, b): one exp2 per logit pair and no mass table
        const int mode = A.pair ? ((!rejects && !A.pdraw) ? kModeAlpha : kModeFull) : kModeSingle;
        norm_sh[0] = offt;
        norm_sh[1] = offd;
        mode_sh = mode;
        if (rank == 0) {
          UnitRec* r = P.recs + A.rec;
          r->px = px;
          r->qx = qx;
          r->offt = offt;
          r->offd = offd;
          r->mode = mode;
          r->rej = rejects ? 1 : 0;
        }
      }
    }
    __syncthreads();
    const float offt = norm_sh[0], offd = norm_sh[1];
    const int mode = mode_sh;
    if (rank == 0 && warp == 0 && has_prev) alpha_to_record(apar);

    // ---- pass 2, handing the slab over to the next unit item by item
    const uint8_t* nT = hasN ? N.gt + wl : nullptr;
    const uint8_t* nD = (hasN && N.pair) ? N.gd + wl : nullptr;
    float* const mrow = P.mass + static_cast<size_t>(A.rec) * kMassRowFloats;
    float aw;
    if (mode == kModeAlpha) aw = pass2(std::integral_constant<int, kModeAlpha>(), offt, offd, mrow, nT, nD);
    else if (mode == kModeFull) aw = pass2(std::integral_constant<int, kModeFull>(), offt, offd, mrow, nT, nD);
    else aw = pass2(std::integral_constant<int, kModeSingle>(), offt, offd, mrow, nT, nD);
    prev_aw = aw;
    prev_rec = A.rec;
    has_prev = true;
    if (!hasN) {
      // the last unit's alpha partials, in an exchange of their own (only rank 0 receives and waits)
      const int i = A.idx + 1, par = i & 1;
      if (rank == 0 && tid == 0) mbar_arrive_tx(smem_addr(&x1_bar[par]), static_cast<uint32_t>(nc) * 4u);
      if (lane == 0) apart_sh[warp] = prev_aw;
      __syncthreads();
      if (warp == 0) {
        const float Ac = cta_alpha();
        if (lane == 0)
          st_async_f32(peer_addr(smem_addr(&abox[par][rank]), 0), Ac, peer_addr(smem_addr(&x1_bar[par]), 0));
      }
      if (rank == 0) {
        if (tid == 0) wait_phase(smem_addr(&x1_bar[par]), (i >> 1) & 1);
        __syncthreads();
        if (warp == 0) alpha_to_record(par);
      }
    }
    A = N;
    hasA = hasN;
  }
  cp_async_wait<0>();                        // only empty groups remain; retire them before leaving
  // no CTA leaves while a store it sent into a peer (the last alpha partials) may be in flight;
  // every wait before this point is bounded, so every CTA of the cluster gets here
  cluster_sync();
}

}  // namespace sv

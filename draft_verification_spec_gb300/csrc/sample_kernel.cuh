// Sampling-path row kernel (T > 0): two streaming passes per (request, position) unit,
// software-pipelined across units.
//
// A thread-block cluster of C CTAs works on a sequence of units -- target row k and, for k < K,
// draft row k -- (persistent; units go round-robin to clusters, pairs first).  CTA r owns the
// vocabulary slice [r*slice, (r+1)*slice) of every row and walks it in items of kSampItemBytes per
// row; warp w owns bytes [w*kSampWarpBytes, (w+1)*kSampWarpBytes) of every item.  Every lane
// streams its own kSampPieces 16-byte pieces of each row with asynchronous copies (cp.async, L2
// only) into its own slots of the warp's ring of kSampStages stages in shared memory,
// kSampStages - 1 items ahead across steps, one commit group per item: the bytes in flight cost
// no registers and a wait is one cp.async.wait_group, no polling.  (Rows that do not start on
// 16-byte boundaries are read element-wise from global memory instead.)
//
// Step s of a CTA walks the items of two units at once: pass 1 of unit s (from HBM) and pass 2 of
// unit s - 1 (the same bytes it read one step earlier, now L2 hits), so the HBM stream never
// pauses for a second pass.
//   pass 1: per-lane online (max, sum of 2^((z - m) c)) of the target and draft rows -> warp
//     maximum and rescaled warp sum -> exchange #1 with st.async into every CTA of the cluster,
//     completing on its mbarrier -> the row normalisers of p and q, merged in one fixed order so
//     every warp of every CTA holds bitwise-identical values; p_k(x_k), q_k(x_k) and the accept
//     test, exactly as the cut kernel evaluates them afterwards
//   pass 2: per logit p = 2^(z c - offt), q = 2^(z c - offd).  A pair that passes the test and
//     needs no draw only needs alpha = sum 2^min(a, b) (one exp2 per logit pair); otherwise every
//     warp writes its (item, warp) masses of r = max(0, p - q) and of p to the row's mass table.
//     Every warp writes its alpha partial.  No second exchange: the chained cut kernel sums the
//     partials in one fixed order and makes the single draw each request needs (at its first
//     rejection, or the bonus) from the mass table, reloading only that one segment.
// A target row that no draw needs is skipped entirely.  DRAM reads each needed logit once while
// the bytes streamed between a logit's two reads fit in L2.
//
// Every wait is bounded by wall time.  A wait that runs out records SPEC_ERR_DEVICE_TIMEOUT and
// then waits once more with a long limit, so the exchange protocol stays consistent and no peer
// store lands in shared memory after the CTA has left.  Only if that second wait also runs out
// does the CTA stop waiting (abort mode; results unspecified).  Every phase a CTA arms it also
// waits for, so on the normal path no peer store can arrive after the CTA has exited.
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
// Logits 2i and 2i+1 of a lane's words as a packed pair (bf16 halves widen exactly).
template <bool BF16, int N>
__device__ __forceinline__ uint64_t pair_of(const uint32_t (&w)[N], int i) {
  if constexpr (BF16) return pk(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
  else return pk(__uint_as_float(w[2 * i]), __uint_as_float(w[2 * i + 1]));
}
// Largest logit of a lane's words.
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

// 16 read-only bytes from global memory, not kept in L1 (each byte is used once per pass).
__device__ __forceinline__ void ldg16(uint32_t* w, const uint8_t* p) {
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
               : "l"(p));
}

// 16-byte asynchronous copy global -> shared by this thread (cached in L2 only).
__device__ __forceinline__ void cp_async16(uint32_t dst, const uint8_t* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
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

// Pass-2 work of a unit.
enum : int { M2_ALPHA = 0, M2_FULL = 1, M2_SINGLE = 2 };

// A unit as a CTA walks it: its row slices, its record, its exchange buffers.
struct SampUnit {
  const uint8_t* gt;       // target row slice (this CTA's part)
  const uint8_t* gd;       // draft row slice (pairs)
  int b, k, rec, idx;      // request, position, record index, needed-unit ordinal of this CTA
  bool pair, pdraw;
  int x;                   // drafted token (lane 0; prefetched when the unit is taken)
  float uk;                // its accept uniform (prefetched)
  float ztx, zdx;          // target and draft logits at x (lane 0; loaded during pass 1)
};

template <bool BF16, bool ALIGNED>
__global__ void __launch_bounds__(kSampThreads, kSampMinBlocks) sample_kernel(const __grid_constant__ RowParams P) {
  using G = SampGeo<BF16>;
  constexpr int ESZ = G::ESZ, EPP = G::EPP, NPC = G::NPC, NWD = G::NWD;
  constexpr int IL = G::IL, WS = G::WS, PS = G::PS;
  constexpr int NWARP = kSampWarps;
  constexpr int IB = kSampItemBytes;
  constexpr int ENT = kMaxCluster * NWARP;         // exchange #1 entries per row: (CTA c, warp w) at c*NWARP + w
  constexpr int EPL = ENT / 32;
  constexpr int NQ = BF16 ? NWD : NWD / 2;         // logit pairs per lane per row per item
  constexpr uint32_t NEG = BF16 ? 0xff80ff80u : 0xff800000u;

  constexpr int S = kSampStages, WB = kSampWarpBytes;
  // warp w's ring: stage s, row slot r (0: pass-1 target, 1: pass-1 draft, 2: pass-2 target,
  // 3: pass-2 draft) at byte ((w * S + s) * 4 + r) * WB
  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(16) float4 mbox1[2][ENT];               // (m_t, s_t, m_d, s_d) per (CTA, warp)
  __shared__ __align__(8) uint64_t x1_bar[2];
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank(), C = cluster_ncta();
  const uint32_t cid = cluster_idx(), ncl = cluster_count();
  const int K = P.K, V = P.V;
  const int lo = static_cast<int>(rank) * P.slice;
  const int n = max(0, min(P.slice, V - lo));                  // this CTA's slice length
  const int nitems = (n + IL - 1) / IL;
  const bool need_draft = (P.flags & F_NEED_DRAFT) != 0;
  const bool stats_only = (P.flags & F_STATS_ONLY) != 0;
  const bool all_pdraws = (P.flags & F_ALL_PDRAWS) != 0;
  const float c = P.c;
  const int nent = static_cast<int>(C) * NWARP;
  const int nunits = static_cast<int>(cid) < P.total_units
                         ? (P.total_units - static_cast<int>(cid) + static_cast<int>(ncl) - 1) / static_cast<int>(ncl)
                         : 0;
  const int npairs = need_draft ? P.B * K : 0;   // units [0, npairs) are (target, draft) pairs
  // this lane's byte offset of piece j of item it: it * IB + wl + j * 512; its first logit: + el
  const int wl = warp * kSampWarpBytes + lane * 16;
  const int el = warp * WS + lane * EPP;

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
  __syncthreads();
  cluster_sync();   // every CTA's barriers exist before any peer sends into them
  // launched with programmatic serialization: the logits, tokens and records are touched only
  // once the preceding grid on the stream has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const long long wlimit = P.wait_limit;
  // A bounded wait on an exchange phase (completed by peers' stores; acquire at cluster scope).
  // On timeout record it, then wait with the long limit; if that also runs out, switch the CTA to
  // abort mode (no more waiting).  The common case reads no clock.
  auto wait_phase = [&](uint32_t bar, uint32_t parity) {
    if (wlimit > 0 && mbar_try_cluster(bar, parity)) return true;
    if (*static_cast<volatile int*>(&abort_flag)) return mbar_try_cluster(bar, parity);
    if (mbar_wait_for<true>(bar, parity, wlimit)) return true;
    atomicOr(P.status, kStatusTimeout);
    if (mbar_wait_for<true>(bar, parity, kDrainNs)) return true;
    *static_cast<volatile int*>(&abort_flag) = 1;
    return false;
  };

  // this lane's words of item `it` of a row (slice base g): NPC 16-byte pieces, -inf past the
  // slice end (only the last item can reach it)
  auto row_words = [&](uint32_t (&W)[NWD], const uint8_t* g, int it, bool last) {
#pragma unroll
    for (int j = 0; j < NPC; ++j) {
      if constexpr (ALIGNED) {
        if (!last || it * IL + el + j * PS < n) {
          ldg16(&W[4 * j], g + static_cast<size_t>(it) * IB + wl + j * 512);
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) W[4 * j + q] = NEG;
        }
      } else {
        const int o = it * IL + el + j * PS;     // first logit of the piece in the slice
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
  // A: in pass 1 during the current step.  B: in pass 2 during the current step.
  // The next needed unit at or after cursor `cur` (advanced past it), if any.
  auto next_needed = [&](int& cur, int& b, int& k, bool& pair, bool& pdraw) -> bool {
    for (; cur < nunits; ++cur) {
      unit_of(cur, b, k);
      pair = need_draft && k < K;
      pdraw = pdraw_row(b, k);
      if (pair || pdraw) {
        ++cur;
        return true;
      }
    }
    return false;
  };
  auto row_slice = [&](bool draft, int b, int k) {
    return draft ? static_cast<const uint8_t*>(P.draft) + ((static_cast<size_t>(b) * K + k) * static_cast<size_t>(V) + lo) * ESZ
                 : static_cast<const uint8_t*>(P.target) + ((static_cast<size_t>(b) * (K + 1) + k) * static_cast<size_t>(V) + lo) * ESZ;
  };

  // ---- this lane's copy ring, S - 1 items ahead of the consumer, across steps
  const uint32_t ring_w = smem_addr(ring) + static_cast<uint32_t>(warp * S * 4 * WB) + static_cast<uint32_t>(lane) * 16u;
  const int last_nval = nitems > 0 ? min(WS, max(0, n - (nitems - 1) * IL - warp * WS)) : 0;
  int icur = 0, iit = 0, istage = 0;
  bool ihA = false, ihB = false, iApair = false, iBpair = false;
  const uint8_t *iAt = nullptr, *iAd = nullptr, *iBt = nullptr, *iBd = nullptr;
  auto issue_take = [&]() {
    int b, k;
    bool pair, pdraw;
    ihA = next_needed(icur, b, k, pair, pdraw);
    if (ihA) {
      iApair = pair;
      iAt = row_slice(false, b, k) + wl;
      iAd = pair ? row_slice(true, b, k) + wl : iAt;
    }
  };
  if (ALIGNED && nitems > 0) issue_take();
  // every step of the sequence commits one group (possibly empty), so wait_group(S - 1)
  // always retires exactly the oldest item
  auto issue_next = [&]() {
    if (ihA || ihB) {
      const size_t off = static_cast<size_t>(iit) * IB;
      const uint32_t dst = ring_w + static_cast<uint32_t>(istage * 4 * WB);
      const bool full = iit != nitems - 1;
#pragma unroll
      for (int j = 0; j < NPC; ++j) {
        if (full || static_cast<int>(j * PS + lane * EPP) < last_nval) {
          if (ihA) {
            cp_async16(dst + j * 512, iAt + off + j * 512);
            if (iApair) cp_async16(dst + WB + j * 512, iAd + off + j * 512);
          }
          if (ihB) {
            cp_async16(dst + 2 * WB + j * 512, iBt + off + j * 512);
            if (iBpair) cp_async16(dst + 3 * WB + j * 512, iBd + off + j * 512);
          }
        }
      }
    }
    cp_async_commit();
    if (!(ihA || ihB)) return;
    istage = istage == S - 1 ? 0 : istage + 1;
    if (++iit == nitems) {                          // the next step: A moves to pass 2
      iit = 0;
      ihB = ihA;
      iBpair = iApair;
      iBt = iAt;
      iBd = iAd;
      issue_take();
    }
  };
  for (int q = 0; q < S - 1; ++q) issue_next();
  int cstage = 0;
  // the next item's stage: issue the one S - 1 further on (into the stage this lane finished
  // with last step), retire this one; returns this lane's address of row slot 0
  auto acquire = [&]() -> uint32_t {
    issue_next();
    cp_async_wait<S - 1>();
    const uint32_t base = ring_w + static_cast<uint32_t>(cstage * 4 * WB);
    cstage = cstage == S - 1 ? 0 : cstage + 1;
    return base;
  };
  // this lane's words of one row slot of the stage; -inf past the slice end on the last item
  auto slot_words = [&](uint32_t (&W)[NWD], uint32_t addr, bool last) {
#pragma unroll
    for (int j = 0; j < NPC; ++j) {
      asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(W[4 * j]), "=r"(W[4 * j + 1]), "=r"(W[4 * j + 2]), "=r"(W[4 * j + 3])
                   : "r"(addr + j * 512));
      if (last) {
#pragma unroll
        for (int e = 0; e < EPP; ++e) {
          if (j * PS + lane * EPP + e >= last_nval) {
            if constexpr (BF16) {
              uint32_t& w = W[4 * j + (e >> 1)];
              w = (e & 1) ? ((w & 0x0000ffffu) | 0xff800000u) : ((w & 0xffff0000u) | 0x0000ff80u);
            } else {
              W[4 * j + e] = NEG;
            }
          }
        }
      }
    }
  };

  int iu = 0;                                // next unit index to look at
  int taken = 0;                             // needed units taken so far
  auto take_unit = [&](SampUnit& U) -> bool {   // the next needed unit, if any
    int b, k;
    bool pair, pdraw;
    if (next_needed(iu, b, k, pair, pdraw)) {
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
      // the accept test's operands, fetched a step before they are needed
      const bool tested = !stats_only && k < K;
      U.x = (tested && lane == 0) ? __ldg(&P.tokens[static_cast<size_t>(b) * K + k]) : -1;
      U.uk = tested ? __ldg(&P.uniforms[static_cast<size_t>(b) * (K + 1) + k]) : 0.f;
      U.ztx = U.zdx = 0.f;
      return true;
    }
    return false;
  };
  // lane 0: the logits at the drafted token (issued once the token has had time to arrive)
  auto fetch_at_token = [&](SampUnit& U) {
    if (lane == 0 && U.x >= 0 && U.x < V) {
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

  SampUnit A = {}, B = {};
  bool hasA = take_unit(A), hasB = false;
  if (hasA && tid == 0) mbar_arrive_tx(smem_addr(&x1_bar[A.idx & 1]), static_cast<uint32_t>(nent) * 16u);
  // B's pass-2 parameters (set when it leaves pass 1)
  int modeB = kModeAlpha;
  float offtB = 0.f, offdB = 0.f;
  const int itmax = P.itmax;

  while (hasA || hasB) {
    // ---- the items of this step: pass 1 of A (HBM), pass 2 of B (L2)
    float mt = ninf(), st = 0.f, md = ninf(), sd = 0.f;
    uint64_t aacc = pk(0.f, 0.f), bacc = aacc;     // B in alpha mode
    float pw = 0.f, rw = 0.f;                      // B in full mode: the warp's totals (lanes 16 / 0)
    const uint64_t noff_t = pk(-offtB, -offtB), noff_d = pk(-offdB, -offdB);
    const uint64_t neg1 = pk(-1.f, -1.f);
    float* const mB = P.mass + static_cast<size_t>(B.rec) * kMassRowFloats;
    for (int it = 0; it < nitems; ++it) {
      const bool last = it == nitems - 1;
      uint32_t At[NWD], Ad[NWD], Bt[NWD], Bd[NWD];
      // every load of the step's item first, then the arithmetic
      if constexpr (ALIGNED) {
        const uint32_t base = acquire();
        const bool rag = last && last_nval < WS;
        if (hasA) {
          slot_words(At, base, rag);
          if (A.pair) slot_words(Ad, base + WB, rag);
        }
        if (hasB) {
          slot_words(Bt, base + 2 * WB, rag);
          if (modeB != kModeSingle) slot_words(Bd, base + 3 * WB, rag);
        }
      } else {
        if (hasA) {
          row_words(At, A.gt, it, last);
          if (A.pair) row_words(Ad, A.gd, it, last);
        }
        if (hasB) {
          row_words(Bt, B.gt, it, last);
          if (modeB != kModeSingle) row_words(Bd, B.gd, it, last);
        }
      }
      if (hasB) {
        if (modeB == kModeAlpha) {
#pragma unroll
          for (int q = 0; q < NQ; q += 2) {
            float a0, a1, b0, b1, a2, a3, b2, b3;
            upk(ffma2(pair_of<BF16>(Bt, q), c2, noff_t), a0, a1);
            upk(ffma2(pair_of<BF16>(Bd, q), c2, noff_d), b0, b1);
            upk(ffma2(pair_of<BF16>(Bt, q + 1), c2, noff_t), a2, a3);
            upk(ffma2(pair_of<BF16>(Bd, q + 1), c2, noff_d), b2, b3);
            aacc = fadd2(aacc, pk(ex2(fminf(a0, b0)), ex2(fminf(a1, b1))));
            bacc = fadd2(bacc, pk(ex2(fminf(a2, b2)), ex2(fminf(a3, b3))));
          }
        } else {
          uint64_t pacc = pk(0.f, 0.f), racc = pacc;
          if (modeB == kModeFull) {
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
              float a0, a1, b0, b1, d0, d1;
              upk(ffma2(pair_of<BF16>(Bt, q), c2, noff_t), a0, a1);
              const uint64_t p = pk(ex2(a0), ex2(a1));     // p of logits 2q, 2q+1
              pacc = fadd2(pacc, p);
              upk(ffma2(pair_of<BF16>(Bd, q), c2, noff_d), b0, b1);
              upk(ffma2(pk(ex2(b0), ex2(b1)), neg1, p), d0, d1);   // p - q
              racc = fadd2(racc, pk(fmaxf(d0, 0.f), fmaxf(d1, 0.f)));
            }
          } else {
#pragma unroll
            for (int q = 0; q < NQ; ++q) {
              float a0, a1;
              upk(ffma2(pair_of<BF16>(Bt, q), c2, noff_t), a0, a1);
              pacc = fadd2(pacc, pk(ex2(a0), ex2(a1)));
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
            mB[kMassAlphaFloats + ((static_cast<int>(rank) * itmax + it) * NWARP + warp) * 2 + (lane >> 4)] = keep;
            if (hi) pw += keep; else rw += keep;
          }
        }
      }
      if (hasA) {
        fold(At, mt, st);
        if (A.pair) fold(Ad, md, sd);
        if (it == 0) fetch_at_token(A);
      }
    }

    // ---- A: warp partials (warp maximum, then every lane's sum rescaled to it) -> exchange #1
    if (hasA) {
      const float wt = warp_max(mt), wd = warp_max(md);
      const float rt = wt == ninf() ? 0.f : wt, rd = wd == ninf() ? 0.f : wd;
      st = warp_sum(st * ex2((mt - rt) * c));
      sd = warp_sum(sd * ex2((md - rd) * c));
      if (lane < static_cast<int>(C)) {
        const uint32_t dst = smem_addr(&mbox1[A.idx & 1][rank * NWARP + warp]);
        st_async_v4(peer_addr(dst, lane), wt, st, wd, sd, peer_addr(smem_addr(&x1_bar[A.idx & 1]), lane));
      }
    }

    // ---- B: this warp's alpha partial into the row's mass table
    if (hasB) {
      float aw;
      if (modeB == kModeAlpha) {
        float a0, a1;
        upk(fadd2(aacc, bacc), a0, a1);
        aw = warp_sum(a0 + a1);
      } else {
        // sum p - R over this warp's items (lane 16 holds P, lane 0 holds R)
        aw = __shfl_sync(0xffffffffu, pw, 16) - __shfl_sync(0xffffffffu, rw, 0);
      }
      if (lane == 0) mB[static_cast<int>(rank) * NWARP + warp] = aw;
    }

    // ---- A leaves pass 1: normalisers and the accept test; it becomes B, the next unit A
    hasB = hasA;
    if (hasA) {
      const int apar = A.idx & 1;
      wait_phase(smem_addr(&x1_bar[apar]), (A.idx >> 1) & 1);
      float Mt = ninf(), Md = ninf();
#pragma unroll
      for (int q = 0; q < EPL; ++q) {
        const int e = lane * EPL + q;
        if (e < nent) {
          const float4 v = mbox1[apar][e];
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
            const float4 v = mbox1[apar][e];
            St += v.y * ex2((v.x - rt) * c);
            Sd += v.w * ex2((v.z - rd) * c);
          }
        }
      }
      St = warp_sum(St);
      Sd = warp_sum(Sd);
      // p_v = 2^(z c - offt), q_v = 2^(z c - offd): the normalisers folded into the exponent
      offtB = (Mt == ninf() ? 0.f : Mt * c) + lg2f(St);
      offdB = (Md == ninf() ? 0.f : Md * c) + lg2f(Sd);
      float px = 0.f, qx = 0.f;
      const bool xin = lane == 0 && A.x >= 0 && A.x < V;
      if (xin) {
        px = ex2(fmaf(A.ztx, c, -offtB));
        qx = ex2(fmaf(A.zdx, c, -offdB));
      }
      px = __shfl_sync(0xffffffffu, px, 0);
      qx = __shfl_sync(0xffffffffu, qx, 0);
      const bool xin_all = __shfl_sync(0xffffffffu, xin ? 1 : 0, 0) != 0;
      const bool rejects = !stats_only && A.k < K && !(xin_all && A.uk * qx < px);
      // a pair that passes the test and draws nothing needs only alpha = sum min(p, q), and
      // min(2^a, 2^b) = 2^min(a, b): one exp2 per logit pair and no mass table
      modeB = A.pair ? ((!rejects && !A.pdraw) ? kModeAlpha : kModeFull) : kModeSingle;
      if (rank == 0 && tid == 0) {
        UnitRec* r = P.recs + A.rec;
        r->px = px;
        r->qx = qx;
        r->offt = offtB;
        r->offd = offdB;
        r->mode = modeB;
      }
      B = A;
      hasA = take_unit(A);
      if (hasA && tid == 0) mbar_arrive_tx(smem_addr(&x1_bar[A.idx & 1]), static_cast<uint32_t>(nent) * 16u);
    }
  }
  cp_async_wait<0>();                        // only empty groups remain; retire them before leaving
}

}  // namespace sv

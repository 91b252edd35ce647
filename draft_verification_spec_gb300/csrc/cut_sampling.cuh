// The serial cut of one request on the sampling path (T > 0), run by one whole warp after the
// sampling row kernel: alpha from the row records, the accept test, the first rejection,
// and the one draw the request needs -- from norm(max(0, p - q)) at the first rejection, or from
// p at the verified depth -- located in the row's mass table and resolved by reloading the one
// segment of logits that owns it.
#pragma once

#include <cuda_bf16.h>

#include "spec_device.cuh"

namespace sv {

// Logit v of a row (element-wise read; bf16 widens exactly).
__device__ __forceinline__ float logit_at(const void* row, int v, bool bf16) {
  if (bf16) return __uint_as_float(static_cast<uint32_t>(__ldg(static_cast<const uint16_t*>(row) + v)) << 16);
  return __ldg(static_cast<const float*>(row) + v);
}

// First entry in vocabulary order (lane-major, E per lane) whose running prefix cum0 + sum
// crosses t, its lane-uniform result and the mass before it; -1 if none crosses.  *last_pos gets
// the last entry with positive mass (or keeps its value if none), *last_cum the mass before it.
template <int E>
__device__ __forceinline__ int cross_entry(const float (&m)[E], float cum0, float t, int lane, float* before,
                                           int* last_pos, float* last_cum, float* total) {
  float loc = 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) loc += m[i];
  const float incl = warp_incl_scan(loc, lane);
  float excl = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) excl = 0.f;
  int first = -1, lp = -1;
  float run = cum0 + excl, bf = 0.f, lb = 0.f;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    if (first < 0 && run + m[i] > t) { first = i; bf = run; }
    if (m[i] > 0.f) { lp = i; lb = run; }
    run += m[i];
  }
  *total = __shfl_sync(0xffffffffu, incl, 31);
  const unsigned pos = __ballot_sync(0xffffffffu, lp >= 0);
  if (pos) {
    const int l = 31 - __clz(pos);
    *last_pos = l * E + __shfl_sync(0xffffffffu, lp, l);
    *last_cum = __shfl_sync(0xffffffffu, lb, l);
  }
  const unsigned hit = __ballot_sync(0xffffffffu, first >= 0);
  if (!hit) return -1;
  const int l = __ffs(hit) - 1;
  *before = __shfl_sync(0xffffffffu, bf, l);
  return l * E + __shfl_sync(0xffffffffu, first, l);
}

// alpha_k of request b, as the row kernel summed and clamped it into the row's record.
__device__ __forceinline__ float alpha_of_row(const BudgetParams& P, int b, int k) {
  return __ldcg(&P.recs[static_cast<size_t>(b) * P.U + k].alpha);
}
// Lane k of the warp: alpha_k of request b (0 for k >= K); every row in parallel.
__device__ __forceinline__ float alpha_row_warp(const BudgetParams& P, int b, int lane) {
  return lane < P.K ? alpha_of_row(P, b, lane) : 0.f;
}

// The cut of request b at verified depth d (lane k <-> position k).  alpha_k may be given
// (alpha_given, lane k's value), and so may the accept test of every position (rej_tab: the [K, B]
// table of positions whose test fails, 1 byte each), as the budget kernel already computed them.
__device__ __forceinline__ void cut_sampling(const BudgetParams& P, int b, int d, int lane, bool alpha_given = false,
                                             float alpha_lane = 0.f, const uint8_t* rej_tab = nullptr) {
  const int K = P.K, U = P.U, V = P.V;
  const UnitRec* rb = P.recs + static_cast<size_t>(b) * U;
  const float a = alpha_given ? alpha_lane : alpha_row_warp(P, b, lane);
  write_stats(b, K, a, P.out_alpha, P.out_cum, P.out_E, lane);
  if (P.stats_only) return;

  const float uK = P.uniforms[static_cast<size_t>(b) * (K + 1) + K];   // the draw's uniform, loaded early
  // the serial accept test u_k q_k(x_k) < p_k(x_k) at positions k < d
  bool ok = true;
  int x = -1;
  if (lane < d) {
    x = P.tokens[static_cast<size_t>(b) * K + lane];
    if (rej_tab) {
      ok = rej_tab[lane * P.B + b] == 0;
    } else if (x < 0 || x >= V) {
      ok = false;
    } else {
      const float u = P.uniforms[static_cast<size_t>(b) * (K + 1) + lane];
      ok = u * __ldcg(&rb[lane].qx) < __ldcg(&rb[lane].px);
    }
  }
  const unsigned rej = __ballot_sync(0xffffffffu, lane < d && !ok);
  const int n = rej ? __ffs(rej) - 1 : d;

  // the draw at row n: the residual norm(max(0, p - q)) after a rejection (p when it is empty),
  // else p (the bonus)
  const float* mrow = P.mass + static_cast<size_t>(b * U + n) * kMassRowFloats;
  const int ncta = P.ncta, itmax = P.itmax, nseg = ncta * itmax;
  const int esz = P.bf16 ? 2 : 4;
  const int IL = kSampItemBytes / esz, WS = kSampWarpBytes / esz, EPP = 16 / esz, PS = 32 * EPP;
  const int nent = nseg * kSampWarps;
  // the row's (R, P) entries in (CTA, item, warp) order, 0 where CTA c's slice has no item it;
  // lane l holds entries base + l*8 .. base + l*8 + 7 of a 256-entry chunk (one chunk for most rows)
  auto load_chunk = [&](int base, float2 (&m)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = base + lane * 8 + i;
      m[i] = make_float2(0.f, 0.f);
      if (e < nent) {
        const int sg = e / kSampWarps, c = sg / itmax, it = sg - c * itmax;
        if (it * IL < min(P.slice, V - c * P.slice)) m[i] = __ldcg(reinterpret_cast<const float2*>(mrow) + e);
      }
    }
  };
  auto chunk_sums = [&](const float2 (&m)[8], float& r, float& p) {
    float lr = 0.f, lp = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      lr += m[i].x;
      lp += m[i].y;
    }
    r = __shfl_sync(0xffffffffu, warp_incl_scan(lr, lane), 31);
    p = __shfl_sync(0xffffffffu, warp_incl_scan(lp, lane), 31);
  };
  const UnitRec rn = rb[n];                // row n's normalisers, fetched with its mass table
  float2 m0[8];
  load_chunk(0, m0);
  float Rtot = 0.f, Ptot = 0.f;
  for (int base = 0; base < nent; base += 256) {
    float2 m[8];
    if (base == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) m[i] = m0[i];
    } else {
      load_chunk(base, m);
    }
    float r, p;
    chunk_sums(m, r, p);
    Rtot += r;
    Ptot += p;
  }
  const bool resid = n < d && Rtot > 0.f;
  const float total = resid ? Rtot : Ptot;
  const float t = uK * total;
  // the owner entry in (CTA, item, warp) order
  int owner = -1, lastpos = -1;
  float cum = 0.f, before = 0.f, lastcum = 0.f;
  for (int base = 0; base < nent && owner < 0; base += 256) {
    float2 mm[8];
    if (base == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) mm[i] = m0[i];
    } else {
      load_chunk(base, mm);
    }
    float m[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) m[i] = resid ? mm[i].x : mm[i].y;
    int lp = -1;
    float lc = 0.f, chunk = 0.f;
    const int hit = cross_entry<8>(m, cum, t, lane, &before, &lp, &lc, &chunk);
    if (lp >= 0) {
      lastpos = base + lp;
      lastcum = lc;
    }
    if (hit >= 0) owner = base + hit;
    cum += chunk;
  }
  if (owner < 0) {                         // rounding left no crossing: the last entry with mass
    owner = lastpos;
    before = lastcum;
  }
  int tok = -1;
  if (owner >= 0) {
    const int sg = owner / kSampWarps, w = owner % kSampWarps, c = sg / itmax, it = sg - c * itmax;
    const int nc = min(P.slice, V - c * P.slice);
    const int s0 = it * IL + w * WS;       // first logit of the segment in CTA c's slice
    const int v0 = c * P.slice + s0;       // ... in the row
    const void* trow = static_cast<const uint8_t*>(P.target) + (static_cast<size_t>(b) * (K + 1) + n) * V * esz;
    const void* drow = resid ? static_cast<const void*>(static_cast<const uint8_t*>(P.draft) +
                                                        (static_cast<size_t>(b) * K + n) * V * esz)
                             : nullptr;
    // this lane's logits of the segment: piece j covers [j*PS + l*EPP, +EPP) (16 bytes, one vector
    // load when rows are 16-byte aligned), with the draw's mass computed exactly as the row kernel did
    constexpr int NPC = kSampPieces;
    constexpr int MAXE = 8;                // logits per piece (bf16; fp32 uses the first 4)
    float zt[NPC][MAXE], zd[NPC][MAXE];
#pragma unroll
    for (int j = 0; j < NPC; ++j) {
      const int o = j * PS + lane * EPP;
      const bool in = s0 + o < nc;         // whole pieces lie inside or outside the slice when aligned
      if (P.aligned) {
        uint4 wt = make_uint4(0, 0, 0, 0), wd = wt;
        if (in) {
          wt = __ldcg(reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(trow) + static_cast<size_t>(v0 + o) * esz));
          if (resid) wd = __ldcg(reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(drow) + static_cast<size_t>(v0 + o) * esz));
        }
        const uint32_t tw[4] = {wt.x, wt.y, wt.z, wt.w}, dw[4] = {wd.x, wd.y, wd.z, wd.w};
#pragma unroll
        for (int e = 0; e < MAXE; ++e) {
          if (P.bf16) {
            zt[j][e] = __uint_as_float((e & 1) ? (tw[e >> 1] & 0xffff0000u) : (tw[e >> 1] << 16));
            zd[j][e] = __uint_as_float((e & 1) ? (dw[e >> 1] & 0xffff0000u) : (dw[e >> 1] << 16));
          } else {
            zt[j][e] = __uint_as_float(tw[e & 3]);
            zd[j][e] = __uint_as_float(dw[e & 3]);
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < MAXE; ++e) {
          const bool ok = e < EPP && s0 + o + e < nc;
          zt[j][e] = ok ? logit_at(trow, v0 + o + e, P.bf16) : 0.f;
          zd[j][e] = (ok && resid) ? logit_at(drow, v0 + o + e, P.bf16) : 0.f;
        }
      }
    }
    float me[NPC][MAXE];                   // this lane's masses, kept for the element walk
    float sj[NPC], tot[NPC];
#pragma unroll
    for (int j = 0; j < NPC; ++j) {
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < MAXE; ++e) {
        const int o = j * PS + lane * EPP + e;
        float m = 0.f;
        if (e < EPP && s0 + o < nc) {
          const float p = ex2(fmaf(zt[j][e], P.c, -rn.offt));
          m = resid ? fmaxf(p - ex2(fmaf(zd[j][e], P.c, -rn.offd)), 0.f) : p;
        }
        me[j][e] = m;
        s += m;
      }
      sj[j] = s;
      tot[j] = warp_sum(s);
    }
    // the piece, then the lane, then the element (each falling back to the last with mass)
    float run = before, cj = before;
    int js = -1;
#pragma unroll
    for (int j = 0; j < NPC; ++j) {
      if (js < 0 && run + tot[j] > t) { js = j; cj = run; }
      run += tot[j];
    }
    if (js < 0) {
      run = before;
#pragma unroll
      for (int j = 0; j < NPC; ++j) {
        if (tot[j] > 0.f) { js = j; cj = run; }
        run += tot[j];
      }
      if (js < 0) { js = 0; cj = before; }
    }
    float mine = 0.f;
#pragma unroll
    for (int j = 0; j < NPC; ++j) if (j == js) mine = sj[j];
    const float incl = warp_incl_scan(mine, lane);
    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0.f;
    const unsigned hit = __ballot_sync(0xffffffffu, cj + incl > t);
    const unsigned pos = __ballot_sync(0xffffffffu, mine > 0.f);
    const int l = hit ? __ffs(hit) - 1 : (pos ? 31 - __clz(pos) : 0);
    const float cl = cj + __shfl_sync(0xffffffffu, excl, l);
    int es = 0;
    if (lane == l) {
      float r = cl;
      int first = -1, lastp = -1;
#pragma unroll
      for (int j = 0; j < NPC; ++j) {
        if (j != js) continue;
#pragma unroll
        for (int e = 0; e < MAXE; ++e) {
          if (e >= EPP) break;
          r += me[j][e];
          if (first < 0 && r > t) first = e;
          if (me[j][e] > 0.f) lastp = e;
        }
      }
      es = first >= 0 ? first : (lastp >= 0 ? lastp : 0);
    }
    es = __shfl_sync(0xffffffffu, es, l);
    tok = v0 + js * PS + l * EPP + es;
  }
  if (lane < d && (x < 0 || x >= V)) atomicOr(P.status, kStatusTokenRange);   // (off the path to the draw)
  int32_t* ot = P.out_tokens + static_cast<size_t>(b) * (K + 1);
  for (int i = lane; i <= K; i += 32) ot[i] = (i < n) ? x : (i == n ? tok : -1);
  if (lane == 0) P.out_accepted[b] = n;
}

}  // namespace sv

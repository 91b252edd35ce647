// Row kernel: one thread-block cluster of C CTAs works on one (request, position) unit at a
// time -- the target row k and, for k < K, the draft row k -- and loops over units
// (persistent).  CTA r of the cluster owns the vocabulary slice [r*slice, (r+1)*slice) of every
// row.  Its slices are staged into a shared-memory ring by one-thread bulk copies issued
// `nstage` units ahead, so HBM keeps streaming while the CTA computes.
//
// Per unit (T > 0), in the order the verification rule needs them:
//   1. thread max -> warp max; e = 2^((z - m_w) c) kept in registers; warp sums s_w
//   2. CTA merge of (m_w, s_w) -> DSMEM exchange #1 -> (M, S) of p and q for the whole row;
//      per-CTA masses of p give the owner CTA of the bonus/p draw
//   3. r = max(0, p - q) summed from the registers -> DSMEM exchange #2 -> residual mass R;
//      alpha = sum p - R (= sum min(p, q))
//   4. the owner CTAs walk their warp / lane / element prefix sums to the inverse-CDF index
// The serial cut of each request runs in a separate small kernel chained with programmatic
// dependent launch (it waits for this grid's records, its launch overlaps this grid).
// T == 0: per-row argmax keys (value, lowest index) instead, one exchange.
#pragma once

#include <climits>

#include "spec_device.cuh"

namespace sv {

template <bool BF16>
__device__ __forceinline__ void chunk_from_smem(const uint8_t* row, int q, float (&f)[kChunk]) {
  if constexpr (BF16) {
    const uint4 v = *reinterpret_cast<const uint4*>(row + q * 16);
    f[0] = __uint_as_float(v.x << 16);
    f[1] = __uint_as_float(v.x & 0xffff0000u);
    f[2] = __uint_as_float(v.y << 16);
    f[3] = __uint_as_float(v.y & 0xffff0000u);
    f[4] = __uint_as_float(v.z << 16);
    f[5] = __uint_as_float(v.z & 0xffff0000u);
    f[6] = __uint_as_float(v.w << 16);
    f[7] = __uint_as_float(v.w & 0xffff0000u);
  } else {
    const float4 a = *reinterpret_cast<const float4*>(row + q * 32);
    const float4 b = *reinterpret_cast<const float4*>(row + q * 32 + 16);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
}

// Unaligned rows: element-wise loads straight from global memory.
template <bool BF16>
__device__ __forceinline__ void chunk_from_global(const void* row, int q, int nv,
                                                  float (&f)[kChunk]) {
#pragma unroll
  for (int e = 0; e < kChunk; ++e) {
    if (e < nv) {
      if constexpr (BF16) {
        const uint16_t h = reinterpret_cast<const uint16_t*>(row)[q * kChunk + e];
        f[e] = __uint_as_float(static_cast<uint32_t>(h) << 16);
      } else {
        f[e] = reinterpret_cast<const float*>(row)[q * kChunk + e];
      }
    }
  }
}

__device__ __forceinline__ void mask_chunk(float (&f)[kChunk], int nv) {
#pragma unroll
  for (int e = 0; e < kChunk; ++e)
    if (e >= nv) f[e] = ninf();
}

template <bool BF16, bool GREEDY, int NT>
__global__ void __launch_bounds__(NT, (NT <= 256) ? 2 : 1) row_kernel(const __grid_constant__ RowParams P) {
  constexpr int NW = NT / 32;
  constexpr int ESZ = BF16 ? 2 : 4;
  static_assert(NW <= 32, "one lane per warp in the CTA merge");

  extern __shared__ __align__(128) uint8_t ring[];
  // per-unit scratch, double-buffered by unit parity so no barrier is needed between units
  __shared__ __align__(16) float4 wred_[2][NW];                  // per-warp (m_t, s_t, m_d, s_d)
  __shared__ float wres_[2][NW];                                 // per-warp residual mass
  __shared__ __align__(16) float4 mbox1[2][kMaxCluster];         // DSMEM exchange #1
  __shared__ __align__(16) float4 mbox2[2][kMaxCluster];         // DSMEM exchange #2
  __shared__ float gstat_[2][8];                                 // row results for all warps
  __shared__ int gsel_[2][4];
  __shared__ __align__(8) uint64_t bars[4];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank(), C = cluster_ncta();
  const uint32_t cid = cluster_idx(), ncl = cluster_count();
  const int K = P.K, V = P.V, U = P.U;
  const int lo = static_cast<int>(rank) * P.slice;
  const int n = max(0, min(P.slice, V - lo));                     // this CTA's slice length
  const bool tma = (P.flags & F_TMA) != 0;
  const bool need_draft = (P.flags & F_NEED_DRAFT) != 0;
  const bool stats_only = (P.flags & F_STATS_ONLY) != 0;
  const float c = P.c;
  const int nstage = P.nstage;
  const uint32_t ring0 = smem_addr(ring);
  const uint32_t srb = static_cast<uint32_t>(P.stage_row_bytes);
  const uint32_t stage_bytes = (need_draft ? 2u : 1u) * srb;
  uint64_t policy = 0;

  // ---- staging ring: thread 0 owns the barriers and the copies
  uint32_t pending = 0, phase = 0;   // thread 0: stages with a copy in flight; parity bits
  bool aborted = false;              // this thread gave up on a wait
  auto issue = [&](int s, int u) {
    const int bb = u / U, kk = u - bb * U;
    const bool pr = need_draft && kk < K;
    const uint32_t bar = smem_addr(&bars[s]);
    const uint32_t bytes = static_cast<uint32_t>(n) * ESZ;
    mbar_arrive_tx(bar, bytes * (pr ? 2u : 1u));
    if (bytes) {
      const uint8_t* st = static_cast<const uint8_t*>(P.target) +
                          (static_cast<size_t>(bb) * (K + 1) + kk) * static_cast<size_t>(V) * ESZ +
                          static_cast<size_t>(lo) * ESZ;
      bulk_g2s(ring0 + s * stage_bytes, st, bytes, bar, policy);
      if (pr) {
        const uint8_t* sd = static_cast<const uint8_t*>(P.draft) +
                            (static_cast<size_t>(bb) * K + kk) * static_cast<size_t>(V) * ESZ +
                            static_cast<size_t>(lo) * ESZ;
        bulk_g2s(ring0 + s * stage_bytes + srb, sd, bytes, bar, policy);
      }
    }
    pending |= 1u << s;
  };

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tma && tid == 0) {
    policy = l2_evict_first_policy();
    for (int s = 0; s < nstage; ++s) mbar_init(smem_addr(&bars[s]), 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (tma && tid == 0) {
    for (int s = 0; s < nstage; ++s) {
      const long long u = cid + static_cast<long long>(s) * ncl;
      if (u < P.total_units) issue(s, static_cast<int>(u));
    }
  }

  int it = 0;
  for (int u = cid; u < P.total_units; u += ncl, ++it) {
    const int b = u / U, k = u - b * U;
    const bool pair = need_draft && k < K;
    const int par = it & 1;
    float4* wred = wred_[par];
    float* wres = wres_[par];
    float* gstat = gstat_[par];
    int* gsel = gsel_[par];
    const float uK = (GREEDY || stats_only) ? 0.f : P.uniforms[static_cast<size_t>(b) * (K + 1) + K];

    // rank 0 / thread 0 fetches the drafted token's logits early (T > 0, decisions wanted)
    float ztx = 0.f, zdx = 0.f;
    bool xin = false;
    if (!GREEDY && !stats_only && rank == 0 && tid == 0 && k < K) {
      const int x = P.tokens[static_cast<size_t>(b) * K + k];
      xin = (x >= 0 && x < V);
      if (xin) {
        const size_t rt = (static_cast<size_t>(b) * (K + 1) + k) * V + x;
        const size_t rd = (static_cast<size_t>(b) * K + k) * V + x;
        if constexpr (BF16) {
          ztx = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(P.target)[rt]) << 16);
          zdx = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(P.draft)[rd]) << 16);
        } else {
          ztx = reinterpret_cast<const float*>(P.target)[rt];
          zdx = reinterpret_cast<const float*>(P.draft)[rd];
        }
      }
    }

    // ---- 1. slice -> registers
    float xt[kNV][kChunk], xd[kNV][kChunk];
    const int s = tma ? it % nstage : 0;
    if (tma && !aborted) {
      const uint32_t parity = (it / nstage) & 1;
      if (!mbar_wait_bounded(smem_addr(&bars[s]), parity, P.wait_limit)) {
        aborted = true;
        atomicOr(P.status, kStatusTimeout);
      } else if (tid == 0) {
        pending &= ~(1u << s);
        phase ^= 1u << s;
      }
    }
    const uint8_t* st_t = ring + s * stage_bytes;
    const uint8_t* st_d = st_t + srb;
    const void* gt = static_cast<const uint8_t*>(P.target) +
                     ((static_cast<size_t>(b) * (K + 1) + k) * V + lo) * ESZ;
    const void* gd = pair ? static_cast<const void*>(static_cast<const uint8_t*>(P.draft) +
                                                     ((static_cast<size_t>(b) * K + k) * V + lo) * ESZ)
                          : nullptr;
#pragma unroll
    for (int j = 0; j < kNV; ++j) {
      const int q = (warp * kNV + j) * 32 + lane;
      const int nv = min(kChunk, max(0, n - q * kChunk));
      if (nv > 0 && !aborted) {
        if (tma) chunk_from_smem<BF16>(st_t, q, xt[j]);
        else chunk_from_global<BF16>(gt, q, nv, xt[j]);
      }
      if (nv < kChunk || aborted) mask_chunk(xt[j], aborted ? 0 : nv);
      if (pair) {
        if (nv > 0 && !aborted) {
          if (tma) chunk_from_smem<BF16>(st_d, q, xd[j]);
          else chunk_from_global<BF16>(gd, q, nv, xd[j]);
        }
        if (nv < kChunk || aborted) mask_chunk(xd[j], aborted ? 0 : nv);
      }
    }
    // stage s is refilled by thread 0 after the next CTA barrier (every thread has read it then)
    auto refill = [&]() {
      if (tma && tid == 0 && !aborted) {
        const long long un = u + static_cast<long long>(nstage) * ncl;
        if (un < P.total_units) issue(s, static_cast<int>(un));
      }
    };

    if constexpr (GREEDY) {
      // ---- argmax per row, lowest index on ties
      uint64_t kt = 0, kd = 0;
      {
        float bv = ninf();
        int bi = INT_MAX;
#pragma unroll
        for (int j = 0; j < kNV; ++j)
#pragma unroll
          for (int e = 0; e < kChunk; ++e)
            if (xt[j][e] > bv) { bv = xt[j][e]; bi = lo + ((warp * kNV + j) * 32 + lane) * kChunk + e; }
        const int q0 = (warp * kNV) * 32 + lane;
        if (bi == INT_MAX && n > q0 * kChunk && !aborted) bi = lo + q0 * kChunk;   // all -inf
        if (bi != INT_MAX) kt = argmax_key(bv, bi);
        kt = warp_max_u64(kt);
      }
      if (pair) {
        float bv = ninf();
        int bi = INT_MAX;
#pragma unroll
        for (int j = 0; j < kNV; ++j)
#pragma unroll
          for (int e = 0; e < kChunk; ++e)
            if (xd[j][e] > bv) { bv = xd[j][e]; bi = lo + ((warp * kNV + j) * 32 + lane) * kChunk + e; }
        const int q0 = (warp * kNV) * 32 + lane;
        if (bi == INT_MAX && n > q0 * kChunk && !aborted) bi = lo + q0 * kChunk;
        if (bi != INT_MAX) kd = argmax_key(bv, bi);
        kd = warp_max_u64(kd);
      }
      if (lane == 0)
        wred[warp] = make_float4(__uint_as_float(static_cast<uint32_t>(kt >> 32)),
                                 __uint_as_float(static_cast<uint32_t>(kt)),
                                 __uint_as_float(static_cast<uint32_t>(kd >> 32)),
                                 __uint_as_float(static_cast<uint32_t>(kd)));
      __syncthreads();
      refill();
      if (warp == 0) {
        uint64_t a = 0, d = 0;
        if (lane < NW) {
          const float4 v = wred[lane];
          a = (static_cast<uint64_t>(__float_as_uint(v.x)) << 32) | __float_as_uint(v.y);
          d = (static_cast<uint64_t>(__float_as_uint(v.z)) << 32) | __float_as_uint(v.w);
        }
        a = warp_max_u64(a);
        d = warp_max_u64(d);
        if (lane < static_cast<int>(C))
          st_peer_v4u(peer_addr(smem_addr(&mbox1[par][rank]), lane), static_cast<uint32_t>(a >> 32),
                      static_cast<uint32_t>(a), static_cast<uint32_t>(d >> 32), static_cast<uint32_t>(d));
      }
      cluster_sync();
      if (rank == 0 && warp == 0) {
        uint64_t a = 0, d = 0;
        if (lane < static_cast<int>(C)) {
          const float4 v = mbox1[par][lane];
          a = (static_cast<uint64_t>(__float_as_uint(v.x)) << 32) | __float_as_uint(v.y);
          d = (static_cast<uint64_t>(__float_as_uint(v.z)) << 32) | __float_as_uint(v.w);
        }
        a = warp_max_u64(a);
        d = warp_max_u64(d);
        if (lane == 0) {
          UnitRec* r = P.recs + u;
          const int g = a ? key_index(a) : 0;
          const int gdd = pair ? (d ? key_index(d) : 0) : -1;
          r->g = g;
          r->gd = gdd;
          r->alpha = (pair && g == gdd) ? 1.f : 0.f;
          r->R = 0.f;
        }
      }
    } else {
      // ---- 1b. exponentials relative to the warp max, kept in registers
      float mt = ninf(), md = ninf();
#pragma unroll
      for (int j = 0; j < kNV; ++j)
#pragma unroll
        for (int e = 0; e < kChunk; ++e) mt = fmaxf(mt, xt[j][e]);
      mt = warp_max(mt);
      float st = 0.f, sd = 0.f;
      {
        const float ref = (mt == ninf()) ? 0.f : mt * c;
#pragma unroll
        for (int j = 0; j < kNV; ++j)
#pragma unroll
          for (int e = 0; e < kChunk; ++e) {
            const float v = ex2(fmaf(xt[j][e], c, -ref));
            xt[j][e] = v;
            st += v;
          }
        st = warp_sum(st);
      }
      if (pair) {
#pragma unroll
        for (int j = 0; j < kNV; ++j)
#pragma unroll
          for (int e = 0; e < kChunk; ++e) md = fmaxf(md, xd[j][e]);
        md = warp_max(md);
        const float ref = (md == ninf()) ? 0.f : md * c;
#pragma unroll
        for (int j = 0; j < kNV; ++j)
#pragma unroll
          for (int e = 0; e < kChunk; ++e) {
            const float v = ex2(fmaf(xd[j][e], c, -ref));
            xd[j][e] = v;
            sd += v;
          }
        sd = warp_sum(sd);
      }
      if (lane == 0) wred[warp] = make_float4(mt, st, md, sd);
      __syncthreads();
      refill();

      // ---- 2. CTA merge, exchange #1
      if (warp == 0) {
        float m1 = ninf(), s1 = 0.f, m2 = ninf(), s2 = 0.f;
        if (lane < NW) {
          const float4 v = wred[lane];
          m1 = v.x; s1 = v.y; m2 = v.z; s2 = v.w;
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const float om1 = __shfl_xor_sync(0xffffffffu, m1, o), os1 = __shfl_xor_sync(0xffffffffu, s1, o);
          const float om2 = __shfl_xor_sync(0xffffffffu, m2, o), os2 = __shfl_xor_sync(0xffffffffu, s2, o);
          ms_merge(m1, s1, om1, os1, c);
          ms_merge(m2, s2, om2, os2, c);
        }
        if (lane < static_cast<int>(C)) st_peer_v4(peer_addr(smem_addr(&mbox1[par][rank]), lane), m1, s1, m2, s2);
      }
      cluster_sync();
      if (warp == 0) {
        float Mc = ninf(), Sc = 0.f, m2 = ninf(), s2 = 0.f;
        if (lane < static_cast<int>(C)) {
          const float4 v = mbox1[par][lane];
          Mc = v.x; Sc = v.y; m2 = v.z; s2 = v.w;
        }
        float M = Mc, S = Sc;
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const float om1 = __shfl_xor_sync(0xffffffffu, M, o), os1 = __shfl_xor_sync(0xffffffffu, S, o);
          const float om2 = __shfl_xor_sync(0xffffffffu, m2, o), os2 = __shfl_xor_sync(0xffffffffu, s2, o);
          ms_merge(M, S, om1, os1, c);
          ms_merge(m2, s2, om2, os2, c);
        }
        // p mass of each CTA slice, its prefix, the owner of the p draw
        const float Pc = (lane < static_cast<int>(C)) ? Sc * ex2((Mc - M) * c) / S : 0.f;
        const float Ptot = __shfl_sync(0xffffffffu, warp_incl_scan(Pc, lane), 31);
        float cum = 0.f;
        const int own = stats_only ? -1 : select_lane(Pc, 0.f, uK * Ptot, lane < static_cast<int>(C), lane, &cum);
        if (lane == 0) {
          gstat[0] = M; gstat[1] = S; gstat[2] = m2; gstat[3] = s2;
          gstat[4] = Ptot; gstat[5] = cum;
          gsel[0] = own;
        }
      }
      __syncthreads();
      const float Mt = gstat[0], St = gstat[1], Md = gstat[2], Sd = gstat[3], Ptot = gstat[4];
      const float at = ex2((mt - Mt) * c) / St;      // p_v = e_v * at for this warp's elements
      const float ad = pair ? ex2((md - Md) * c) / Sd : 0.f;

      // ---- 3. residual mass, exchange #2
      float Rtot = 0.f;
      if (pair) {
        float r = 0.f;
#pragma unroll
        for (int j = 0; j < kNV; ++j)
#pragma unroll
          for (int e = 0; e < kChunk; ++e) r += fmaxf(fmaf(xt[j][e], at, -xd[j][e] * ad), 0.f);
        r = warp_sum(r);
        if (lane == 0) wres[warp] = r;
        __syncthreads();
        if (warp == 0) {
          const float rc = warp_sum(lane < NW ? wres[lane] : 0.f);
          if (lane < static_cast<int>(C)) st_peer_v4(peer_addr(smem_addr(&mbox2[par][rank]), lane), rc, 0.f, 0.f, 0.f);
        }
        cluster_sync();
        if (warp == 0) {
          const float Rc = (lane < static_cast<int>(C)) ? mbox2[par][lane].x : 0.f;
          const float Rt = __shfl_sync(0xffffffffu, warp_incl_scan(Rc, lane), 31);
          float cum = 0.f;
          const int own = stats_only ? -1 : select_lane(Rc, 0.f, uK * Rt, lane < static_cast<int>(C), lane, &cum);
          if (lane == 0) {
            gstat[6] = Rt;
            gstat[7] = cum;
            gsel[1] = own;
          }
        }
        __syncthreads();
        Rtot = gstat[6];
      }

      // ---- 4. row record and inverse-CDF draws
      if (rank == 0 && tid == 0) {
        UnitRec* r = P.recs + u;
        const float px = xin ? ex2(fmaf(ztx, c, -Mt * c)) / St : 0.f;
        const float qx = xin ? ex2(fmaf(zdx, c, -Md * c)) / Sd : 0.f;
        r->px = px;
        r->qx = qx;
        r->alpha = pair ? fminf(fmaxf(Ptot - Rtot, 0.f), 1.f) : 0.f;
        r->R = Rtot;
        if (!stats_only) {
          if (gsel[0] < 0) r->ps = -1;
          if (!pair || gsel[1] < 0) r->rs = -1;
        }
      }
      if (!stats_only) {
        // draw from p (bonus candidate) by the owner CTA
        if (gsel[0] == static_cast<int>(rank)) {
          const float tP = uK * Ptot;
          float wm = 0.f;
          if (lane < NW) {
            const float4 v = wred[lane];
            wm = v.y * ex2((v.x - Mt) * c) / St;
          }
          float cw = 0.f;
          const int w = select_lane(wm, gstat[5], tP, lane < NW, lane, &cw);
          if (w == warp) {
            float sj[kNV];
#pragma unroll
            for (int j = 0; j < kNV; ++j) {
              float a = 0.f;
#pragma unroll
              for (int e = 0; e < kChunk; ++e) a += xt[j][e] * at;
              sj[j] = a;
            }
            // slot, lane, element
            float cum = cw;
            int js = -1;
            float cumj = cw;
#pragma unroll
            for (int j = 0; j < kNV; ++j) {
              const float tot = warp_sum(sj[j]);
              if (js < 0 && cum + tot > tP) { js = j; cumj = cum; }
              cum += tot;
            }
            if (js < 0) {
#pragma unroll
              for (int j = kNV - 1; j >= 0; --j)
                if (js < 0 && __ballot_sync(0xffffffffu, sj[j] > 0.f)) js = j;
              if (js < 0) js = 0;
              cumj = cw;
#pragma unroll
              for (int j = 0; j < kNV; ++j) if (j < js) cumj += warp_sum(sj[j]);
            }
            float mys = 0.f;
#pragma unroll
            for (int j = 0; j < kNV; ++j) if (j == js) mys = sj[j];
            float cl = 0.f;
            const int l = select_lane(mys, cumj, tP, true, lane, &cl);
            if (lane == (l < 0 ? 0 : l)) {
              float me[kChunk];
#pragma unroll
              for (int j = 0; j < kNV; ++j)
                if (j == js)
#pragma unroll
                  for (int e = 0; e < kChunk; ++e) me[e] = xt[j][e] * at;
              int es = -1, lastpos = -1;
              float run = cl;
#pragma unroll
              for (int e = 0; e < kChunk; ++e) {
                run += me[e];
                if (es < 0 && run > tP) es = e;
                if (me[e] > 0.f) lastpos = e;
              }
              if (es < 0) es = lastpos < 0 ? 0 : lastpos;
              P.recs[u].ps = lo + ((warp * kNV + js) * 32 + (l < 0 ? 0 : l)) * kChunk + es;
            }
          }
        }
        // residual draw by its owner CTA
        if (pair && gsel[1] == static_cast<int>(rank)) {
          const float tR = uK * Rtot;
          float cw = 0.f;
          const int w = select_lane(lane < NW ? wres[lane] : 0.f, gstat[7], tR, lane < NW, lane, &cw);
          if (w == warp) {
            float sj[kNV];
#pragma unroll
            for (int j = 0; j < kNV; ++j) {
              float a = 0.f;
#pragma unroll
              for (int e = 0; e < kChunk; ++e) a += fmaxf(fmaf(xt[j][e], at, -xd[j][e] * ad), 0.f);
              sj[j] = a;
            }
            float cum = cw;
            int js = -1;
            float cumj = cw;
#pragma unroll
            for (int j = 0; j < kNV; ++j) {
              const float tot = warp_sum(sj[j]);
              if (js < 0 && cum + tot > tR) { js = j; cumj = cum; }
              cum += tot;
            }
            if (js < 0) {
#pragma unroll
              for (int j = kNV - 1; j >= 0; --j)
                if (js < 0 && __ballot_sync(0xffffffffu, sj[j] > 0.f)) js = j;
              if (js < 0) js = 0;
              cumj = cw;
#pragma unroll
              for (int j = 0; j < kNV; ++j) if (j < js) cumj += warp_sum(sj[j]);
            }
            float mys = 0.f;
#pragma unroll
            for (int j = 0; j < kNV; ++j) if (j == js) mys = sj[j];
            float cl = 0.f;
            const int l = select_lane(mys, cumj, tR, true, lane, &cl);
            if (lane == (l < 0 ? 0 : l)) {
              float me[kChunk];
#pragma unroll
              for (int j = 0; j < kNV; ++j)
                if (j == js)
#pragma unroll
                  for (int e = 0; e < kChunk; ++e) me[e] = fmaxf(fmaf(xt[j][e], at, -xd[j][e] * ad), 0.f);
              int es = -1, lastpos = -1;
              float run = cl;
#pragma unroll
              for (int e = 0; e < kChunk; ++e) {
                run += me[e];
                if (es < 0 && run > tR) es = e;
                if (me[e] > 0.f) lastpos = e;
              }
              if (es < 0) es = lastpos < 0 ? 0 : lastpos;
              P.recs[u].rs = lo + ((warp * kNV + js) * 32 + (l < 0 ? 0 : l)) * kChunk + es;
            }
          }
        }
      }
    }

  }

  // ---- drain copies still in flight (only after a wait gave up)
  if (tma && tid == 0) {
    for (int s = 0; s < nstage; ++s)
      if (pending & (1u << s)) {
        if (!mbar_wait_bounded(smem_addr(&bars[s]), (phase >> s) & 1u, 1ll << 26)) atomicOr(P.status, kStatusTimeout);
      }
  }
}

}  // namespace sv

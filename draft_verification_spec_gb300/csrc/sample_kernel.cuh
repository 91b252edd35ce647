// Sampling-path row kernel (T > 0).  A thread-block cluster of C CTAs works on one
// (request, position) unit at a time -- target row k and, for k < K, draft row k -- and loops
// over units (persistent).  CTA r owns the vocabulary slice [r*slice, (r+1)*slice) of every row;
// inside it, warp w owns a contiguous range of 32*kNV*8 logits, lane-interleaved in 16-byte
// chunks.  Slices are staged into a shared-memory ring by one-thread bulk copies issued `nstage`
// units ahead.
//
// Per unit:
//   1. chunks -> registers; warp max m_w; e = 2^((z - m_w) c) kept in registers; warp sum s_w
//   2. every warp sends (m_w, s_w) of both rows to every CTA of the cluster with st.async; the
//      copies complete on the receiver's mbarrier (no cluster barrier, no fence).  Each warp then
//      merges the C*NW entries into the row's (M, S) of p and q, in one fixed order, so all warps
//      of all CTAs hold bitwise-identical normalisers and p-mass prefix sums.
//   3. r = max(0, p - q) summed per warp -> second st.async exchange -> residual mass R per row,
//      alpha = sum p - R (= sum min(p, q)).
//   4. the warp that owns the inverse-CDF threshold (by the exchanged per-warp masses, in
//      vocabulary order) walks slot / lane / element prefix sums in its registers.
// The serial cut runs afterwards in a small kernel chained with programmatic dependent launch.
#pragma once

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
__device__ __forceinline__ void chunk_from_global(const void* row, int q, int nv, float (&f)[kChunk]) {
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

// Inverse-CDF walk inside one warp's range: masses come from registers via `mass(j, e)`; the
// warp's prefix before its range is cum0.  Returns the element offset inside the slice.
template <typename MassFn>
__device__ __forceinline__ int warp_draw(MassFn mass, float cum0, float t, int warp, int lane) {
  float sj[kNV];
#pragma unroll
  for (int j = 0; j < kNV; ++j) {
    float a = 0.f;
#pragma unroll
    for (int e = 0; e < kChunk; ++e) a += mass(j, e);
    sj[j] = a;
  }
  // slot j covers chunks (warp*kNV + j)*32 + lane for lanes 0..31: slots are in vocabulary order
  float cum = cum0, cumj = cum0;
  int js = -1;
  float tot[kNV];
#pragma unroll
  for (int j = 0; j < kNV; ++j) {
    tot[j] = warp_sum(sj[j]);
    if (js < 0 && cum + tot[j] > t) { js = j; cumj = cum; }
    cum += tot[j];
  }
  if (js < 0) {   // rounding: take the last slot with mass
    cum = cum0;
#pragma unroll
    for (int j = 0; j < kNV; ++j) {
      if (tot[j] > 0.f) { js = j; cumj = cum; }
      cum += tot[j];
    }
    if (js < 0) { js = 0; cumj = cum0; }
  }
  float mine = 0.f;
#pragma unroll
  for (int j = 0; j < kNV; ++j) if (j == js) mine = sj[j];
  float m1[1] = {mine};
  float cl = cumj;
  int l = select_entry<1>(m1, cumj, t, lane, &cl);
  if (l < 0) l = 0;
  int es = 0;
  if (lane == l) {
    float run = cl;
    int first = -1, lastpos = -1;
#pragma unroll
    for (int j = 0; j < kNV; ++j) {
      if (j == js) {
#pragma unroll
        for (int e = 0; e < kChunk; ++e) {
          const float me = mass(j, e);
          run += me;
          if (first < 0 && run > t) first = e;
          if (me > 0.f) lastpos = e;
        }
      }
    }
    es = first >= 0 ? first : (lastpos >= 0 ? lastpos : 0);
  }
  es = __shfl_sync(0xffffffffu, es, l);
  return ((warp * kNV + js) * 32 + l) * kChunk + es;
}

// lane 0 of each warp loads the drafted token; every lane needs to know whether it was in range
__device__ __forceinline__ bool xin_all(bool xin_lane0) {
  return __shfl_sync(0xffffffffu, xin_lane0 ? 1 : 0, 0) != 0;
}

template <bool BF16, int NT>
__global__ void __launch_bounds__(NT, (NT <= 256) ? 2 : 1) sample_kernel(const __grid_constant__ RowParams P) {
  constexpr int NW = NT / 32;
  constexpr int ESZ = BF16 ? 2 : 4;
  constexpr int ENT = kMaxCluster * NW;   // exchanged entries per row: (CTA c, warp w) at c*NW + w
  constexpr int EPL = ENT / 32;           // entries per lane in the merges
  static_assert(ENT % 32 == 0, "entries per lane");

  extern __shared__ __align__(128) uint8_t ring[];
  __shared__ __align__(16) float4 mbox1[2][ENT];   // (m_t, s_t, m_d, s_d) per (CTA, warp)
  __shared__ __align__(16) float mbox2[2][ENT];    // residual mass per (CTA, warp)
  __shared__ __align__(8) uint64_t full_bar[4];
  __shared__ __align__(8) uint64_t x1_bar[2];
  __shared__ __align__(8) uint64_t x2_bar[2];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank(), C = cluster_ncta();
  const uint32_t cid = cluster_idx(), ncl = cluster_count();
  const int K = P.K, V = P.V, U = P.U;
  const int lo = static_cast<int>(rank) * P.slice;
  const int n = max(0, min(P.slice, V - lo));
  const bool tma = (P.flags & F_TMA) != 0;
  const bool need_draft = (P.flags & F_NEED_DRAFT) != 0;
  const bool stats_only = (P.flags & F_STATS_ONLY) != 0;
  const float c = P.c;
  const int nstage = P.nstage;
  const uint32_t ring0 = smem_addr(ring);
  const uint32_t srb = static_cast<uint32_t>(P.stage_row_bytes);
  const uint32_t stage_bytes = (need_draft ? 2u : 1u) * srb;
  const int nent = static_cast<int>(C) * NW;
  uint64_t policy = 0;

  uint32_t pending = 0, phase = 0;   // thread 0: stages with a copy in flight; their parities
  auto issue = [&](int s, int u) {
    const int bb = u / U, kk = u - bb * U;
    const bool pr = need_draft && kk < K;
    const uint32_t bar = smem_addr(&full_bar[s]);
    const uint32_t bytes = static_cast<uint32_t>(n) * ESZ;
    mbar_arrive_tx(bar, bytes * (pr ? 2u : 1u));
    if (bytes) {
      const uint8_t* st = static_cast<const uint8_t*>(P.target) +
                          ((static_cast<size_t>(bb) * (K + 1) + kk) * static_cast<size_t>(V) + lo) * ESZ;
      bulk_g2s(ring0 + s * stage_bytes, st, bytes, bar, policy);
      if (pr) {
        const uint8_t* sd = static_cast<const uint8_t*>(P.draft) +
                            ((static_cast<size_t>(bb) * K + kk) * static_cast<size_t>(V) + lo) * ESZ;
        bulk_g2s(ring0 + s * stage_bytes + srb, sd, bytes, bar, policy);
      }
    }
    pending |= 1u << s;
  };

  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (tid == 0) {
    if (tma) {
      policy = l2_evict_first_policy();
      for (int s = 0; s < nstage; ++s) mbar_init(smem_addr(&full_bar[s]), 1);
    }
    for (int p = 0; p < 2; ++p) {
      mbar_init(smem_addr(&x1_bar[p]), 1);
      mbar_init(smem_addr(&x2_bar[p]), 1);
    }
    mbar_fence_init();
  }
  __syncthreads();
  cluster_sync();   // every CTA's barriers exist before any peer sends into them
  if (tma && tid == 0) {
    for (int s = 0; s < nstage; ++s) {
      const long long u = cid + static_cast<long long>(s) * ncl;
      if (u < P.total_units) issue(s, static_cast<int>(u));
    }
  }

  uint32_t x2ph = 0;     // parity of the next phase of x2_bar[0], x2_bar[1] (used by pair units only)
  bool tabort = false;   // gave up waiting for staged data (test hook or a lost copy)
  bool xabort = false;   // gave up waiting for an exchange
  const long long xlimit = 1ll << 24;
  int it = 0;
  for (int u = cid; u < P.total_units; u += ncl, ++it) {
    const int b = u / U, k = u - b * U;
    const bool pair = need_draft && k < K;
    const int par = it & 1;
    const uint32_t xpar = (it >> 1) & 1;
    const uint32_t x1 = smem_addr(&x1_bar[par]), x2 = smem_addr(&x2_bar[par]);
    if (tid == 0) {   // arm this unit's exchanges (their previous phases completed two units ago)
      mbar_arrive_tx(x1, static_cast<uint32_t>(nent) * 16u);
      if (pair) mbar_arrive_tx(x2, static_cast<uint32_t>(nent) * 4u);
    }
    // the draws this unit may need: the bonus draw from p only at the request's verified depth
    // (or at every row when the depth is chosen after this kernel); the residual only where the
    // accept test fails (decided below from the merged normalisers, as the cut kernel will)
    const float uK = stats_only ? 0.f : P.uniforms[static_cast<size_t>(b) * (K + 1) + K];
    const float uk = (stats_only || k >= K) ? 0.f : P.uniforms[static_cast<size_t>(b) * (K + 1) + k];
    const int dep = P.depth ? min(max(P.depth[b], 0), K) : K;
    const bool pdraw_here = !stats_only && ((P.flags & F_ALL_PDRAWS) != 0 || k == dep);
    float ztx = 0.f, zdx = 0.f;
    bool xin = false;
    if (!stats_only && k < K && lane == 0) {
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
    if (tma && !tabort) {
      if (!mbar_wait_bounded(smem_addr(&full_bar[s]), (it / nstage) & 1, P.wait_limit)) {
        tabort = true;
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
      const int nv = tabort ? 0 : min(kChunk, max(0, n - q * kChunk));
      if (nv > 0) {
        if (tma) chunk_from_smem<BF16>(st_t, q, xt[j]);
        else chunk_from_global<BF16>(gt, q, nv, xt[j]);
      }
      if (nv < kChunk) mask_chunk(xt[j], nv);
      if (pair) {
        if (nv > 0) {
          if (tma) chunk_from_smem<BF16>(st_d, q, xd[j]);
          else chunk_from_global<BF16>(gd, q, nv, xd[j]);
        }
        if (nv < kChunk) mask_chunk(xd[j], nv);
      }
    }

    // ---- exponentials relative to the warp max, kept in registers
    float mt = ninf(), md = ninf(), st = 0.f, sd = 0.f;
#pragma unroll
    for (int j = 0; j < kNV; ++j)
#pragma unroll
      for (int e = 0; e < kChunk; ++e) mt = fmaxf(mt, xt[j][e]);
    mt = warp_max(mt);
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

    // ---- 2. exchange #1: (m_w, s_w) of this warp to every CTA of the cluster
    if (lane < static_cast<int>(C)) {
      const uint32_t slot = smem_addr(&mbox1[par][rank * NW + warp]);
      st_async_v4(peer_addr(slot, lane), mt, st, md, sd, peer_addr(x1, lane));
    }
    if (!xabort && !mbar_wait_cluster_bounded(x1, xpar, xlimit)) {
      xabort = true;
      atomicOr(P.status, kStatusTimeout);
    }
    // every warp of this CTA has sent, hence read its stage: refill it
    if (tma && tid == 0 && !tabort) {
      const long long un = u + static_cast<long long>(nstage) * ncl;
      if (un < P.total_units) issue(s, static_cast<int>(un));
    }
    float em_t[EPL], es_t[EPL], em_d[EPL], es_d[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane * EPL + i;
      if (e < nent) {
        const float4 v = mbox1[par][e];
        em_t[i] = v.x; es_t[i] = v.y; em_d[i] = v.z; es_d[i] = v.w;
      } else {
        em_t[i] = ninf(); es_t[i] = 0.f; em_d[i] = ninf(); es_d[i] = 0.f;
      }
    }
    float Mt = ninf(), Md = ninf();
#pragma unroll
    for (int i = 0; i < EPL; ++i) { Mt = fmaxf(Mt, em_t[i]); Md = fmaxf(Md, em_d[i]); }
    Mt = warp_max(Mt);
    Md = warp_max(Md);
    float St = 0.f, Sd = 0.f, wp[EPL];
    {
      const float rt = (Mt == ninf()) ? 0.f : Mt;
      const float rd = (Md == ninf()) ? 0.f : Md;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        wp[i] = es_t[i] * ex2((em_t[i] - rt) * c);
        St += wp[i];
        Sd += es_d[i] * ex2((em_d[i] - rd) * c);
      }
    }
    St = warp_sum(St);
    Sd = warp_sum(Sd);
    const float inv_St = 1.f / St;
    float Ptot = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      wp[i] *= inv_St;   // p mass of entry (CTA, warp)
      Ptot += wp[i];
    }
    Ptot = warp_sum(Ptot);
    const float at = ex2((mt - Mt) * c) * inv_St;       // p_v = e_v * at for this warp's logits
    const float ad = pair ? ex2((md - Md) * c) / Sd : 0.f;
    // p_k(x_k), q_k(x_k) and the accept test, bitwise as the cut kernel will evaluate it
    float px = 0.f, qx = 0.f;
    if (lane == 0 && xin) {
      px = ex2(fmaf(ztx, c, -Mt * c)) * inv_St;
      qx = ex2(fmaf(zdx, c, -Md * c)) / Sd;
    }
    px = __shfl_sync(0xffffffffu, px, 0);
    qx = __shfl_sync(0xffffffffu, qx, 0);
    const bool rejects = !stats_only && k < K && !(xin_all(xin) && uk * qx < px);

    // ---- 3. exchange #2: residual mass per warp
    float Rtot = 0.f, wr[EPL];
#pragma unroll
    for (int i = 0; i < EPL; ++i) wr[i] = 0.f;
    if (pair) {
      float r = 0.f;
#pragma unroll
      for (int j = 0; j < kNV; ++j)
#pragma unroll
        for (int e = 0; e < kChunk; ++e) r += fmaxf(fmaf(xt[j][e], at, -xd[j][e] * ad), 0.f);
      r = warp_sum(r);
      if (lane < static_cast<int>(C)) {
        const uint32_t slot = smem_addr(&mbox2[par][rank * NW + warp]);
        st_async_f32(peer_addr(slot, lane), r, peer_addr(x2, lane));
      }
      if (!xabort && !mbar_wait_cluster_bounded(x2, (x2ph >> par) & 1u, xlimit)) {
        xabort = true;
        atomicOr(P.status, kStatusTimeout);
      }
      x2ph ^= 1u << par;
#pragma unroll
      for (int i = 0; i < EPL; ++i) {
        const int e = lane * EPL + i;
        wr[i] = e < nent ? mbox2[par][e] : 0.f;
        Rtot += wr[i];
      }
      Rtot = warp_sum(Rtot);
    }

    // ---- 4. row record and inverse-CDF draws
    const bool need_r = pair && rejects && Rtot > 0.f;
    const bool need_p = pdraw_here || (rejects && !(Rtot > 0.f));   // p == q: the residual is empty
    int own_p = -1, own_r = -1;
    float cum_p = 0.f, cum_r = 0.f;
    if (need_p) own_p = select_entry<EPL>(wp, 0.f, uK * Ptot, lane, &cum_p);
    if (need_r) own_r = select_entry<EPL>(wr, 0.f, uK * Rtot, lane, &cum_r);
    if (rank == 0 && tid == 0) {
      UnitRec* r = P.recs + u;
      r->px = px;
      r->qx = qx;
      r->alpha = pair ? fminf(fmaxf(Ptot - Rtot, 0.f), 1.f) : 0.f;
      r->R = Rtot;
      if (own_p < 0) r->ps = -1;
      if (own_r < 0) r->rs = -1;
    }
    const int me = static_cast<int>(rank) * NW + warp;
    if (need_p && own_p == me) {
      const int off = warp_draw([&](int j, int e) { return xt[j][e] * at; }, cum_p, uK * Ptot, warp, lane);
      if (lane == 0) P.recs[u].ps = lo + off;
    }
    if (need_r && own_r == me) {
      const int off = warp_draw([&](int j, int e) { return fmaxf(fmaf(xt[j][e], at, -xd[j][e] * ad), 0.f); },
                                cum_r, uK * Rtot, warp, lane);
      if (lane == 0) P.recs[u].rs = lo + off;
    }
  }

  // ---- drain copies still in flight (only after a wait gave up)
  if (tma && tid == 0) {
    for (int s = 0; s < nstage; ++s)
      if (pending & (1u << s)) {
        if (!mbar_wait_bounded(smem_addr(&full_bar[s]), (phase >> s) & 1u, 1ll << 26)) atomicOr(P.status, kStatusTimeout);
      }
  }
  // no CTA leaves while a peer may still write into its shared memory
  cluster_sync_relaxed();
}

}  // namespace sv

// Draft-side statistics for the confidence budget chosen before the target forward (the AngelSpec
// page's runtime section: what to verify is decided from the draft model's output distribution).
//
// One CTA per (draft row, part of the vocabulary): a single streaming pass that keeps, per lane,
// the running maximum and the sum of 2^((z - max) c) -- or, at T = 0, the maximum and the first
// index that holds it -- then reduces them over the CTA into one float4 (max, sum, first argmax
// index, 0).  The budget kernel merges a row's parts in part order into
// q_k(x_k) = 2^((z_x - M) c) / S, or [x_k == argmax] at T = 0.  Each logit is read once, with
// evict-first loads; nothing is staged in shared memory.
#include <climits>

#include "packed_math.cuh"
#include "spec_device.cuh"

namespace sv {

__device__ __forceinline__ unsigned warp_min_u32(unsigned v) {
  unsigned r;
  asm volatile("redux.sync.min.u32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}

template <bool BF16, bool GREEDY, bool ALIGNED>
__global__ void __launch_bounds__(kDraftStatsThreads) draft_stats_kernel(const __grid_constant__ DraftStatsParams P) {
  constexpr int ESZ = BF16 ? 2 : 4, EPP = 16 / ESZ;
  constexpr int NT = kDraftStatsThreads, NW = NT / 32;
  constexpr int U = 4;                                   // 16-byte pieces in flight per lane
  constexpr uint32_t NEG = BF16 ? 0xff80ff80u : 0xff800000u;
  __shared__ float sm_m[NW], sm_s[NW];
  __shared__ unsigned sm_i[NW];

  // the budget kernel chained after this one may start (it reads only the caller's inputs
  // before it waits for this grid)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int part = blockIdx.x, row = blockIdx.y;
  const int lo = part * P.part_len, hi = min(P.V, lo + P.part_len);
  const uint8_t* g = static_cast<const uint8_t*>(P.draft) + static_cast<size_t>(row) * P.V * ESZ;
  const float c = P.c;
  float m = ninf(), s = 0.f;
  unsigned idx = UINT_MAX;

  if constexpr (ALIGNED) {
    // piece i holds logits [lo + i*EPP, +EPP); rows and parts start on 16-byte boundaries and
    // the row length is a multiple of EPP, so every piece lies wholly inside [lo, hi)
    const int npieces = (hi - lo) / EPP;
    const uint64_t c2 = pk(c, c);
    for (int i0 = tid; i0 < npieces; i0 += NT * U) {
      uint32_t w[U][4];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * NT;
        if (i < npieces) {
          const uint4 v = __ldcs(reinterpret_cast<const uint4*>(g + static_cast<size_t>(lo + i * EPP) * ESZ));
          w[u][0] = v.x;
          w[u][1] = v.y;
          w[u][2] = v.z;
          w[u][3] = v.w;
        } else {
#pragma unroll
          for (int q = 0; q < 4; ++q) w[u][q] = NEG;
        }
      }
      if constexpr (GREEDY) {
        // pieces in increasing index order: a strictly larger value moves the index, a tie keeps
        // the earlier one
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const float pm = words_max<BF16>(w[u]);
          if (pm > m) {
            m = pm;
            const int base = lo + (i0 + u * NT) * EPP;
            int first = EPP - 1;
#pragma unroll
            for (int e = EPP - 1; e >= 0; --e) {
              float z;
              if constexpr (BF16) z = __uint_as_float((e & 1) ? (w[u][e >> 1] & 0xffff0000u) : (w[u][e >> 1] << 16));
              else z = __uint_as_float(w[u][e]);
              if (z == pm) first = e;
            }
            idx = static_cast<unsigned>(base + first);
          }
        }
      } else {
        // online (max, sum) over the group: the sum is rescaled to the new maximum (reference 0
        // while every logit so far is -inf)
        float gm = ninf();
#pragma unroll
        for (int u = 0; u < U; ++u) gm = fmaxf(gm, words_max<BF16>(w[u]));
        const float nm = fmaxf(m, gm);
        const float ref = nm == ninf() ? 0.f : nm;
        s *= ex2((m - ref) * c);
        const uint64_t nref = pk(-ref * c, -ref * c);
        uint64_t acc = pk(0.f, 0.f);
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
          for (int q = 0; q < (BF16 ? 4 : 2); ++q) {
            float x0, x1;
            upk(ffma2(pair_of<BF16>(w[u], q), c2, nref), x0, x1);
            acc = fadd2(acc, pk(ex2(x0), ex2(x1)));
          }
        }
        float a0, a1;
        upk(acc, a0, a1);
        s += a0 + a1;
        m = nm;
      }
    }
  } else {
    // rows not on 16-byte boundaries: element by element, in increasing index order per lane
    for (int v = lo + tid; v < hi; v += NT) {
      const float z = BF16 ? __uint_as_float(static_cast<uint32_t>(__ldcs(reinterpret_cast<const uint16_t*>(g) + v)) << 16)
                           : __ldcs(reinterpret_cast<const float*>(g) + v);
      if constexpr (GREEDY) {
        if (z > m) {
          m = z;
          idx = static_cast<unsigned>(v);
        }
      } else if (z != ninf()) {
        if (z > m) {
          s = s * ex2((m - z) * c) + 1.f;
          m = z;
        } else {
          s += ex2((z - m) * c);
        }
      }
    }
  }

  // the CTA's (max, sum) or (max, first index), merged in one fixed order
  const float wm = warp_maxf(m);
  if constexpr (GREEDY) {
    const unsigned wi = warp_min_u32(m == wm ? idx : UINT_MAX);
    if (lane == 0) {
      sm_m[warp] = wm;
      sm_i[warp] = wi;
    }
  } else {
    const float ref = wm == ninf() ? 0.f : wm;
    const float ws = warp_sum(s * ex2((m - ref) * c));
    if (lane == 0) {
      sm_m[warp] = wm;
      sm_s[warp] = ws;
    }
  }
  __syncthreads();
  if (warp == 0) {
    const float mm = lane < NW ? sm_m[lane] : ninf();
    const float M = warp_maxf(mm);
    float4 r;
    if constexpr (GREEDY) {
      const unsigned I = warp_min_u32(lane < NW && mm == M ? sm_i[lane] : UINT_MAX);
      r = make_float4(M, 0.f, __uint_as_float(I), 0.f);
    } else {
      const float ref = M == ninf() ? 0.f : M;
      const float S = warp_sum(lane < NW ? sm_s[lane] * ex2((mm - ref) * c) : 0.f);
      r = make_float4(M, S, 0.f, 0.f);
    }
    if (lane == 0) P.out[static_cast<size_t>(row) * P.nparts + part] = r;
  }
}

cudaError_t launch_draft_stats(bool bf16, bool greedy, bool aligned, const DraftStatsParams& p, cudaStream_t stream) {
  const void* fn;
  if (bf16) {
    if (greedy) fn = aligned ? reinterpret_cast<const void*>(&draft_stats_kernel<true, true, true>)
                             : reinterpret_cast<const void*>(&draft_stats_kernel<true, true, false>);
    else fn = aligned ? reinterpret_cast<const void*>(&draft_stats_kernel<true, false, true>)
                      : reinterpret_cast<const void*>(&draft_stats_kernel<true, false, false>);
  } else {
    if (greedy) fn = aligned ? reinterpret_cast<const void*>(&draft_stats_kernel<false, true, true>)
                             : reinterpret_cast<const void*>(&draft_stats_kernel<false, true, false>);
    else fn = aligned ? reinterpret_cast<const void*>(&draft_stats_kernel<false, false, true>)
                      : reinterpret_cast<const void*>(&draft_stats_kernel<false, false, false>);
  }
  DraftStatsParams q = p;
  void* args[] = {&q};
  return cudaLaunchKernel(fn, dim3(p.nparts, p.rows, 1), dim3(kDraftStatsThreads, 1, 1), args, 0, stream);
}

}  // namespace sv

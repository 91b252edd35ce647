// Device helpers shared by every kernel: exp2, warp reductions, argmax keys, and the
// per-request cut.  The cluster / DSMEM / mbarrier wrappers live in spec_async.cuh.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "spec_internal.h"

namespace sv {

__device__ __forceinline__ float ninf() { return __int_as_float(0xff800000); }

// 2^x with the hardware approximation (MUFU.EX2); flushes denormal results to 0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- warp helpers
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// Butterfly sum: every lane ends with the same value (fp add is commutative).
// Largest value across the warp in one instruction (-inf if every lane holds -inf).
__device__ __forceinline__ float warp_maxf(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_sum_int(int v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_incl_scan(float v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    float t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}
__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    uint64_t t = __shfl_xor_sync(0xffffffffu, v, o);
    v = t > v ? t : v;
  }
  return v;
}

// Merge two (max, sum of 2^((x - max) c)) pairs; symmetric in its arguments.
__device__ __forceinline__ void ms_merge(float& m, float& s, float m2, float s2, float c) {
  const float mn = fmaxf(m, m2);
  const float ref = (mn == ninf()) ? 0.f : mn;
  s = s * ex2((m - ref) * c) + s2 * ex2((m2 - ref) * c);
  m = mn;
}

// Order-preserving map of a float to uint32 (-0 folded into +0).
__device__ __forceinline__ uint32_t ord_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
// Argmax key: larger value wins, then the smaller index; 0 means "no element".
__device__ __forceinline__ uint64_t argmax_key(float v, int idx) {
  return (static_cast<uint64_t>(ord_key(v)) << 32) | static_cast<uint32_t>(0x7fffffff - idx);
}
__device__ __forceinline__ int key_index(uint64_t key) {
  return 0x7fffffff - static_cast<int>(static_cast<uint32_t>(key & 0xffffffffu));
}

// First lane (among `valid` lanes) whose running prefix cum0 + incl crosses t; if rounding
// leaves none, the last valid lane with positive mass; -1 if no lane has mass.  Uniform.
__device__ __forceinline__ int select_lane(float mass, float cum0, float t, bool valid, int lane,
                                           float* cum_before) {
  const float m = valid ? mass : 0.f;
  const float incl = warp_incl_scan(m, lane);
  float excl = __shfl_up_sync(0xffffffffu, incl, 1);
  if (lane == 0) excl = 0.f;
  const unsigned hit = __ballot_sync(0xffffffffu, valid && (cum0 + incl > t));
  int sel;
  if (hit) {
    sel = __ffs(hit) - 1;
  } else {
    const unsigned pos = __ballot_sync(0xffffffffu, valid && m > 0.f);
    sel = pos ? 31 - __clz(pos) : -1;
  }
  const float eb = __shfl_sync(0xffffffffu, excl, sel < 0 ? 0 : sel);
  *cum_before = cum0 + eb;
  return sel;
}

__device__ __forceinline__ float ldcg_f(const float* p) { return __ldcg(p); }
__device__ __forceinline__ int ldcg_i(const int32_t* p) { return __ldcg(p); }

// Alpha, prefix confidences and expected length of one request from this lane's alpha (lane k
// holds alpha_k, k < K): left-to-right fp32 products, written where requested.
__device__ __forceinline__ void write_stats(int b, int K, float a, float* out_alpha, float* out_cum,
                                            float* out_E, int lane) {
  if (out_alpha && lane < K) out_alpha[static_cast<size_t>(b) * K + lane] = a;
  if (out_cum || out_E) {
    float cprod = 1.f, esum = 0.f, mine = 0.f;
    for (int m = 0; m < K; ++m) {
      cprod *= __shfl_sync(0xffffffffu, a, m);
      esum += cprod;
      if (lane == m) mine = cprod;
    }
    if (out_cum && lane < K) out_cum[static_cast<size_t>(b) * K + lane] = mine;
    if (out_E && lane == 0) out_E[b] = esum;
  }
}

// Greedy serial-acceptance cut of one request, run by one whole warp (lane k <-> position k):
// resolves the argmax keys (and clears them for the next call when `clear_keys`).  d = verified
// depth in [0, K].
__device__ __forceinline__ void cut_request(int b, int d, bool stats_only, uint64_t* keys, bool draft_keys,
                                            bool clear_keys, int U, int K, int V, const int32_t* tokens,
                                            int32_t* out_tokens, int32_t* out_accepted, float* out_alpha,
                                            float* out_cum, float* out_E, int32_t* status, int lane) {
  uint64_t* kb = keys + static_cast<size_t>(b) * (K + 1) * 2;
  // argmax of the target row at this lane's position (and of the draft row)
  int g = -1, gd = -2;
  if (lane < U) {
    g = key_index(__ldcg(reinterpret_cast<const unsigned long long*>(kb) + 2 * lane));
    if (draft_keys && lane < K) gd = key_index(__ldcg(reinterpret_cast<const unsigned long long*>(kb) + 2 * lane + 1));
  }
  // the one-hot alpha: 1 where the target and draft argmaxes agree
  const float a = (lane < K && draft_keys && g == gd) ? 1.f : 0.f;
  write_stats(b, K, a, out_alpha, out_cum, out_E, lane);
  if (!stats_only) {
    bool ok = true;
    int x = -1;
    if (lane < d) {
      x = tokens[static_cast<size_t>(b) * K + lane];
      if (x < 0 || x >= V) {
        ok = false;
        atomicOr(status, kStatusTokenRange);
      } else {
        ok = (x == g);
      }
    }
    const unsigned rej = __ballot_sync(0xffffffffu, lane < d && !ok);
    const int n = rej ? __ffs(rej) - 1 : d;
    const int tok = __shfl_sync(0xffffffffu, g, n);
    int32_t* ot = out_tokens + static_cast<size_t>(b) * (K + 1);
    for (int i = lane; i <= K; i += 32) ot[i] = (i < n) ? x : (i == n ? tok : -1);
    if (lane == 0) out_accepted[b] = n;
  }
  if (clear_keys && lane < U) {
    kb[2 * lane] = 0ull;
    kb[2 * lane + 1] = 0ull;
  }
}

}  // namespace sv

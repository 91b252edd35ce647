// Greedy-path row kernel (T == 0): argmax of every target row (and of the draft rows when the
// one-hot alpha is wanted), lowest index on ties, fused with the serial cut.
//
// The rows are cut into warp tiles (2048 bf16 / 1024 fp32 logits in 16-byte chunks), ordered request by
// request; each warp takes one contiguous run of tiles and streams it with 16-byte loads (the
// other resident warps cover their latency).  Per tile: packed bf16 max (HMNMX2) per lane, warp max,
// then only lanes holding the maximum look for its first index.  Keys (value, lowest index) of
// one row are folded in registers and published with one atomicMax per row segment; a
// release-add per request segment counts finished tiles, and the warp that completes a request
// runs its cut and clears the request's slots and counter for the next call.  No CTA barrier.
#pragma once

#include <climits>
#include <cuda_bf16.h>

#include "spec_device.cuh"

namespace sv {

// Tile geometry: bf16 lanes hold 8 chunks of 8 logits (one 16-byte load each), fp32 lanes 4
// chunks of 8 logits (two 16-byte loads each); a warp tile is 32 lanes of that.
template <bool BF16> struct Geo {
  static constexpr int kChunks = BF16 ? 8 : 4;          // chunks per lane
  static constexpr int kWords = BF16 ? 8 : 8;           // uint4 per lane
  static constexpr int kTile = 32 * kChunks * kChunk;   // logits per warp tile (2048 / 1024)
};

template <bool BF16>
struct TileRegs {
  uint4 w[Geo<BF16>::kWords];
};

__device__ __forceinline__ __nv_bfloat162 as_bf2(uint32_t u) {
  __nv_bfloat162 r;
  memcpy(&r, &u, sizeof(r));
  return r;
}

template <bool BF16>
__device__ __forceinline__ float tile_elem(const TileRegs<BF16>& r, int j, int e) {
  if constexpr (BF16) {
    const uint4 v = r.w[j];
    const uint32_t word = (e < 2) ? v.x : (e < 4) ? v.y : (e < 6) ? v.z : v.w;
    return __uint_as_float((e & 1) ? (word & 0xffff0000u) : (word << 16));
  } else {
    const uint4 v = r.w[2 * j + (e >> 2)];
    const uint32_t word = ((e & 3) == 0) ? v.x : ((e & 3) == 1) ? v.y : ((e & 3) == 2) ? v.z : v.w;
    return __uint_as_float(word);
  }
}

// Load one tile; chunks past the row end read as -inf (their logits do not exist).
template <bool BF16>
__device__ __forceinline__ void load_tile(TileRegs<BF16>& r, const uint8_t* row, int base, int V, int lane) {
  constexpr int ESZ = BF16 ? 2 : 4;
  constexpr uint32_t NEG = BF16 ? 0xff80ff80u : 0xff800000u;
#pragma unroll
  for (int j = 0; j < Geo<BF16>::kChunks; ++j) {
    const int e0 = base + (j * 32 + lane) * kChunk;
    const uint4* p = reinterpret_cast<const uint4*>(row + static_cast<size_t>(e0) * ESZ);
    if (e0 + kChunk <= V) {
      if constexpr (BF16) {
        r.w[j] = __ldcs(p);
      } else {
        r.w[2 * j] = __ldcs(p);
        r.w[2 * j + 1] = __ldcs(p + 1);
      }
    } else {
      uint32_t v[kChunk * ESZ / 4];
#pragma unroll
      for (int i = 0; i < kChunk * ESZ / 4; ++i) v[i] = NEG;
#pragma unroll
      for (int e = 0; e < kChunk; ++e) {
        if (e0 + e < V) {
          if constexpr (BF16) {
            const uint32_t h = reinterpret_cast<const uint16_t*>(row)[e0 + e];
            v[e >> 1] = (e & 1) ? ((v[e >> 1] & 0x0000ffffu) | (h << 16)) : ((v[e >> 1] & 0xffff0000u) | h);
          } else {
            v[e] = reinterpret_cast<const uint32_t*>(row)[e0 + e];
          }
        }
      }
      if constexpr (BF16) {
        r.w[j] = make_uint4(v[0], v[1], v[2], v[3]);
      } else {
        r.w[2 * j] = make_uint4(v[0], v[1], v[2], v[3]);
        r.w[2 * j + 1] = make_uint4(v[4], v[5], v[6], v[7]);
      }
    }
  }
}

// Warp argmax key of a tile in registers: per-chunk maxima, lane max, warp max; then only lanes
// holding the maximum find its first chunk and the first logit in it (lowest index wins).
template <bool BF16>
__device__ __forceinline__ uint64_t tile_key_regs(const TileRegs<BF16>& r, int base, int lane) {
  constexpr int NC = Geo<BF16>::kChunks;
  float cm[NC];
  if constexpr (BF16) {
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      const __nv_bfloat162 m = __hmax2(__hmax2(as_bf2(r.w[j].x), as_bf2(r.w[j].y)),
                                       __hmax2(as_bf2(r.w[j].z), as_bf2(r.w[j].w)));
      cm[j] = fmaxf(__low2float(m), __high2float(m));
    }
  } else {
#pragma unroll
    for (int j = 0; j < NC; ++j) {
      float a = fmaxf(tile_elem<false>(r, j, 0), tile_elem<false>(r, j, 1));
      float b = fmaxf(tile_elem<false>(r, j, 2), tile_elem<false>(r, j, 3));
      float c = fmaxf(tile_elem<false>(r, j, 4), tile_elem<false>(r, j, 5));
      float d = fmaxf(tile_elem<false>(r, j, 6), tile_elem<false>(r, j, 7));
      cm[j] = fmaxf(fmaxf(a, b), fmaxf(c, d));
    }
  }
  float lm = cm[0];
#pragma unroll
  for (int j = 1; j < NC; ++j) lm = fmaxf(lm, cm[j]);
  const float wm = warp_max(lm);
  int idx = INT_MAX;
  if (lm == wm) {   // usually one lane
    int jf = NC - 1;
#pragma unroll
    for (int j = NC - 1; j >= 0; --j)
      if (cm[j] == wm) jf = j;
    int ef = kChunk - 1;
#pragma unroll
    for (int j = 0; j < NC; ++j)
      if (j == jf) {
#pragma unroll
        for (int e = kChunk - 1; e >= 0; --e)
          if (tile_elem<BF16>(r, j, e) == wm) ef = e;
      }
    idx = base + (jf * 32 + lane) * kChunk + ef;
  }
  idx = __reduce_min_sync(0xffffffffu, idx);
  if (idx == INT_MAX) idx = base;   // NaN maximum: unspecified, keep the index in range
  return argmax_key(wm, idx);
}

// Partial or unaligned tile: element-wise loads with bounds checks.
template <bool BF16>
__device__ __forceinline__ uint64_t tile_key_scalar(const uint8_t* row, int base, int V, int lane) {
  float best = ninf();
  int bi = INT_MAX;
#pragma unroll
  for (int j = 0; j < Geo<BF16>::kChunks; ++j) {
    const int e0 = base + (j * 32 + lane) * kChunk;
#pragma unroll
    for (int e = 0; e < kChunk; ++e) {
      if (e0 + e < V) {
        float x;
        if constexpr (BF16) {
          x = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(row)[e0 + e]) << 16);
        } else {
          x = reinterpret_cast<const float*>(row)[e0 + e];
        }
        if (bi == INT_MAX) bi = e0 + e;     // the first logit this lane sees (covers all -inf)
        if (x > best) { best = x; bi = e0 + e; }
      }
    }
  }
  uint64_t key = bi == INT_MAX ? 0ull : argmax_key(best, bi);
  return warp_max_u64(key);
}

// Position of a tile in the request-major tile order, advanced without divisions.
struct TileCursor {
  const uint8_t* row;
  int base, q, req, slot;
};

template <bool BF16>
__global__ void __launch_bounds__(256, BF16 ? 4 : 2) argmax_kernel(const __grid_constant__ ArgmaxParams P) {
  constexpr int ESZ = BF16 ? 2 : 4;
  constexpr int NWARP = 8;
  constexpr int kTile = Geo<BF16>::kTile;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int K = P.K, V = P.V, tpr = P.tpr;
  const int rows_req = P.rows_t + P.drows;            // rows per request: target, then draft
  const int tiles_req = rows_req * tpr;
  const int total = static_cast<int>(P.total_tiles);  // < 2^31 (checked by the host)
  // this warp's contiguous run of tiles
  const long long gw = static_cast<long long>(blockIdx.x) * NWARP + warp, nw = static_cast<long long>(gridDim.x) * NWARP;
  const int t0 = static_cast<int>(gw * total / nw), t1 = static_cast<int>((gw + 1) * total / nw);
  if (t0 >= t1) return;

  auto set_row = [&](TileCursor& c) {
    if (c.q < P.rows_t) {
      c.row = static_cast<const uint8_t*>(P.target) + ((static_cast<size_t>(c.req) * (K + 1) + c.q) * V) * ESZ;
      c.slot = (c.req * (K + 1) + c.q) * 2;
    } else {
      const int k = c.q - P.rows_t;
      c.row = static_cast<const uint8_t*>(P.draft) + ((static_cast<size_t>(c.req) * K + k) * V) * ESZ;
      c.slot = (c.req * (K + 1) + k) * 2 + 1;
    }
  };
  auto step = [&](TileCursor& c) {
    c.base += kTile;
    if (c.base >= V) {
      c.base = 0;
      if (++c.q == rows_req) { c.q = 0; ++c.req; }
      set_row(c);
    }
  };
  TileCursor cur;
  {
    const int rg = t0 / tpr;
    cur.base = (t0 - rg * tpr) * kTile;
    cur.req = rg / rows_req;
    cur.q = rg - cur.req * rows_req;
    set_row(cur);
  }

  // publish a row's folded key; count a request's finished tiles, the last warp runs the cut
  auto flush_key = [&](int slot, uint64_t key) {
    if (lane == 0 && key) atomicMax(reinterpret_cast<unsigned long long*>(P.keys) + slot, key);
  };
  auto flush_count = [&](int req, int cnt) {
    if (!P.fused_cut) return;
    int old = 0;
    if (lane == 0) {   // release: this lane's key updates precede the count; acquire: others' too
      asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], %2;" : "=r"(old) : "l"(P.counters + req), "r"(cnt) : "memory");
    }
    old = __shfl_sync(0xffffffffu, old, 0);
    if (old + cnt == tiles_req) {                      // this warp finished request `req`
      __syncwarp();   // lane 0's acquire, then the warp barrier: every lane's loads see the keys
      const int d = P.depth ? min(max(P.depth[req], 0), K) : K;
      cut_request(req, d, P.stats_only != 0, P.keys, P.drows > 0, true, P.rows_t, K, V, P.tokens,
                  P.out_tokens, P.out_accepted, P.out_alpha, P.out_cum, P.out_E, P.status, lane);
      if (lane == 0) P.counters[req] = 0;
    }
  };

  // launched with programmatic serialization: everything above is index arithmetic; the logits,
  // keys and counters are touched only once the preceding grid has completed and flushed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int acc_slot = cur.slot, acc_req = cur.req, acc_cnt = 0;
  uint64_t acc_key = 0;
  for (int t = t0; t < t1; ++t) {
    uint64_t key;
    if (P.aligned) {                                   // 16-byte loads; the other resident warps hide them
      TileRegs<BF16> a;
      load_tile<BF16>(a, cur.row, cur.base, V, lane);
      key = tile_key_regs<BF16>(a, cur.base, lane);
    } else {
      key = tile_key_scalar<BF16>(cur.row, cur.base, V, lane);
    }
    if (cur.slot != acc_slot) {
      flush_key(acc_slot, acc_key);
      acc_slot = cur.slot;
      acc_key = key;
    } else {
      acc_key = key > acc_key ? key : acc_key;
    }
    if (cur.req != acc_req) {
      flush_count(acc_req, acc_cnt);
      acc_req = cur.req;
      acc_cnt = 1;
    } else {
      ++acc_cnt;
    }
    step(cur);
  }
  flush_key(acc_slot, acc_key);
  flush_count(acc_req, acc_cnt);
}

}  // namespace sv

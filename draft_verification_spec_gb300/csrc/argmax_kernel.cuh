// Greedy-path row kernel (T == 0): argmax of every target row (and of the draft rows when the
// one-hot alpha is wanted), lowest index on ties.  No cross-CTA dependency: each warp scans
// 1024-logit tiles (grid-stride over all rows' tiles) with 16-byte loads prefetched one tile
// ahead in registers, reduces a 64-bit (value, lowest index) key over the warp and folds it into
// the row's slot with atomicMax.  The cut kernel resolves and clears the slots.
#pragma once

#include <climits>

#include "spec_device.cuh"

namespace sv {

constexpr int kTile = kTileLogits;   // logits per warp tile (1024)

template <bool BF16>
struct TileRegs {
  static constexpr int kWords = BF16 ? kNV : 2 * kNV;   // uint4 per lane per tile
  uint4 w[kWords];
};

template <bool BF16>
__device__ __forceinline__ void load_tile(TileRegs<BF16>& r, const uint8_t* row, int base, int V, int lane) {
  constexpr int ESZ = BF16 ? 2 : 4;
#pragma unroll
  for (int j = 0; j < kNV; ++j) {
    const int e0 = base + (j * 32 + lane) * kChunk;
    if (e0 + kChunk <= V) {
      const uint4* p = reinterpret_cast<const uint4*>(row + static_cast<size_t>(e0) * ESZ);
      if constexpr (BF16) {
        r.w[j] = __ldcs(p);
      } else {
        r.w[2 * j] = __ldcs(p);
        r.w[2 * j + 1] = __ldcs(p + 1);
      }
    }
  }
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

// Scan one tile (aligned rows: from prefetched registers; otherwise element-wise loads).
template <bool BF16>
__device__ __forceinline__ uint64_t tile_key(const TileRegs<BF16>& r, const uint8_t* row, int base, int V,
                                             int lane, bool aligned) {
  constexpr int ESZ = BF16 ? 2 : 4;
  float best = ninf();
  int bi = INT_MAX;
#pragma unroll
  for (int j = 0; j < kNV; ++j) {
    const int e0 = base + (j * 32 + lane) * kChunk;
    if (aligned && e0 + kChunk <= V) {
      if (bi == INT_MAX) bi = e0;            // first logit this lane sees (covers all -inf)
#pragma unroll
      for (int e = 0; e < kChunk; ++e) {
        const float x = tile_elem<BF16>(r, j, e);
        if (x > best) { best = x; bi = e0 + e; }
      }
    } else {
#pragma unroll
      for (int e = 0; e < kChunk; ++e) {
        if (e0 + e < V) {
          float x;
          if constexpr (BF16) {
            x = __uint_as_float(static_cast<uint32_t>(reinterpret_cast<const uint16_t*>(row)[e0 + e]) << 16);
          } else {
            x = reinterpret_cast<const float*>(row)[e0 + e];
          }
          if (bi == INT_MAX) bi = e0 + e;
          if (x > best) { best = x; bi = e0 + e; }
        }
      }
    }
  }
  (void)ESZ;
  return bi == INT_MAX ? 0ull : argmax_key(best, bi);
}

template <bool BF16>
__global__ void __launch_bounds__(256) argmax_kernel(const __grid_constant__ ArgmaxParams P) {
  constexpr int ESZ = BF16 ? 2 : 4;
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const long long gw = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
  const long long trows = static_cast<long long>(P.B) * P.rows_t;
  const int K = P.K, V = P.V, tpr = P.tpr;

  auto locate = [&](long long t, const uint8_t*& row, int& base, size_t& slot) {
    const long long r = t / tpr;
    base = static_cast<int>(t - r * tpr) * kTile;
    if (r < trows) {
      const long long b = r / P.rows_t, k = r - b * P.rows_t;
      row = static_cast<const uint8_t*>(P.target) + ((b * (K + 1) + k) * static_cast<size_t>(V)) * ESZ;
      slot = static_cast<size_t>(b * (K + 1) + k) * 2;
    } else {
      const long long rr = r - trows, b = rr / K, k = rr - b * K;
      row = static_cast<const uint8_t*>(P.draft) + ((b * K + k) * static_cast<size_t>(V)) * ESZ;
      slot = static_cast<size_t>(b * (K + 1) + k) * 2 + 1;
    }
  };

  TileRegs<BF16> cur, nxt;
  const uint8_t* row = nullptr;
  int base = 0;
  size_t slot = 0;
  long long t = gw;
  if (t < P.total_tiles) {
    locate(t, row, base, slot);
    if (P.aligned) load_tile<BF16>(cur, row, base, V, lane);
  }
  while (t < P.total_tiles) {
    const long long tn = t + nwarps;
    const uint8_t* nrow = nullptr;
    int nbase = 0;
    size_t nslot = 0;
    if (tn < P.total_tiles) {                  // prefetch the next tile while this one is scanned
      locate(tn, nrow, nbase, nslot);
      if (P.aligned) load_tile<BF16>(nxt, nrow, nbase, V, lane);
    }
    uint64_t key = tile_key<BF16>(cur, row, base, V, lane, P.aligned != 0);
    key = warp_max_u64(key);
    if (lane == 0 && key) atomicMax(reinterpret_cast<unsigned long long*>(P.keys) + slot, key);
    cur = nxt;
    row = nrow;
    base = nbase;
    slot = nslot;
    t = tn;
  }
}

}  // namespace sv

// Packed-fp32 arithmetic and logit-word helpers shared by the kernels that scan logit rows: bf16
// words widen exactly to fp32 pairs, and Blackwell's paired fp32 FMA / add work on the pairs.
#pragma once

#include <cstdint>
#include <cstring>

#include <cuda_bf16.h>

namespace sv {

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

}  // namespace sv

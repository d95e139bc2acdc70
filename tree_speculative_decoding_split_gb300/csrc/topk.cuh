// Order keys for the top-k selections of the Medusa and EAGLE tree expansions (sm_103a).
#pragma once

#include "common.cuh"

namespace spectree {

// ---- order keys (top-k) -------------------------------------------------------------------
// A 64-bit key orders candidates best first: the upper half maps the value monotonically
// (-0 = +0; NaN maps to 0, below -inf), the lower half breaks ties by the lower id; key 0 means
// "no candidate".

__device__ __forceinline__ uint32_t order_u(float f) {
  if (f != f) return 0u;
  const uint32_t b = __float_as_uint(f == 0.f ? 0.f : f);
  const uint32_t u = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
  return u == 0u ? 1u : u;  // keep 0 for NaN
}
__device__ __forceinline__ float order_value(uint32_t u) {  // the value order_u maps to u (u >= 1)
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}
__device__ __forceinline__ unsigned long long order_key(uint32_t u, int id) {
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)id);
}
__device__ __forceinline__ int key_token(unsigned long long k) {
  return (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull));
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, o);
    x = y > x ? y : x;
  }
  return x;
}
// Largest of the warp's keys strictly below `below` (0 when there is none); every lane gets it.
template <int N>
__device__ __forceinline__ unsigned long long warp_max_below(const unsigned long long (&keys)[N],
                                                             unsigned long long below) {
  unsigned long long m = 0ull;
#pragma unroll
  for (int e = 0; e < N; ++e)
    if (keys[e] < below && keys[e] > m) m = keys[e];
  return warp_max_u64(m);
}

}  // namespace spectree

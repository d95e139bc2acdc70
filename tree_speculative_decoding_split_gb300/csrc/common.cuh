// Device-side helpers shared by the tree-verification kernels (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "spectree.h"

namespace spectree {

constexpr int kMaxNodes = SPEC_MAX_NODES;
constexpr int kAncWords = (kMaxNodes + 31) / 32;  // 8 words of ancestor bits per node
constexpr float kMargin = 1e-4f;                  // decision margin band
constexpr unsigned long long kWaitLimitNs = 1000000000ull;  // bounded waits: 1 s

// ---- status ---------------------------------------------------------------------------------

__device__ __forceinline__ void set_status(int32_t* st, int32_t code) {
  if (st) atomicCAS(st, SPEC_OK, code);
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- warp reductions ------------------------------------------------------------------------

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---- row statistics record ------------------------------------------------------------------
// Partial softmax statistics of one logit row over a slice of the vocabulary, at y = z / tau:
//   m = max y, s = sum exp(y - m), t = sum exp(y - m) * y, y2 = second largest y,
//   idx = lowest vocabulary index attaining m.
struct RowPart {
  float m, s, t, y2;
  int idx;
};

__device__ __forceinline__ RowPart rowpart_empty() {
  RowPart r;
  r.m = -INFINITY; r.s = 0.f; r.t = 0.f; r.y2 = -INFINITY; r.idx = 0x7fffffff;
  return r;
}

// Merge two partials of disjoint vocabulary slices (order-independent tie-break: lowest idx).
__device__ __forceinline__ RowPart rowpart_merge(const RowPart& a, const RowPart& b) {
  RowPart r;
  const bool take_b = (b.m > a.m) || (b.m == a.m && b.idx < a.idx);
  r.m = fmaxf(a.m, b.m);
  r.idx = take_b ? b.idx : a.idx;
  r.y2 = fmaxf(fminf(a.m, b.m), fmaxf(a.y2, b.y2));
  if (r.m == -INFINITY) {
    r.s = 0.f; r.t = 0.f;
  } else {
    const float fa = (a.s > 0.f) ? expf(a.m - r.m) : 0.f;
    const float fb = (b.s > 0.f) ? expf(b.m - r.m) : 0.f;
    r.s = a.s * fa + b.s * fb;
    r.t = a.t * fa + b.t * fb;
  }
  return r;
}

// ---- Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11) --------------------------------------
// Round: products of counter words 0 and 2 with two odd multipliers; high halves are xored
// with counter words 1 / 3 and the round key; the key is bumped by two Weyl increments.
__device__ __forceinline__ uint32_t philox_x0(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                             uint32_t k0, uint32_t k1) {
  const uint32_t kMulA = 0xD2511F53u, kMulB = 0xCD9E8D57u;
  const uint32_t kWeylA = 0x9E3779B9u, kWeylB = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = kMulA * c0, hi0 = __umulhi(kMulA, c0);
    const uint32_t lo1 = kMulB * c2, hi1 = __umulhi(kMulB, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
    k0 += kWeylA; k1 += kWeylB;
  }
  return c0;
}

// U(seed, request, node, purpose) in (0, 1), exact in float32.
__device__ __forceinline__ float accept_uniform(uint64_t seed, uint32_t request, uint32_t node,
                                                uint32_t purpose) {
  const uint32_t x0 = philox_x0(request, node, purpose, 0u, (uint32_t)seed, (uint32_t)(seed >> 32));
  return (float)((x0 >> 9) * 2u + 1u) * 5.9604644775390625e-08f;  // 2^-24
}

// ---- shared memory / mbarrier / TMA (sm_90+ async proxy) ------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe: has the phase of parity `parity` completed?  (try_wait may suspend the
// thread for a while when the phase is incomplete; test_wait never does.)
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of parity `parity` to complete.  Gives up after kWaitLimitNs, or as soon
// as *abort becomes non-zero; returns false in both cases.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (abort && *abort) return false;
    if ((it & 255u) == 0u && globaltimer_ns() - t0 > kWaitLimitNs) return false;
  }
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, uint64_t* bar, int x,
                                            int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x,
                                            int y, int z, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "l"(policy)
      : "memory");
}
// Tiled TMA loads without an L2 cache hint (the operands' default policy).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y, int z,
                                            int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}
// Prefetch one 4-D box into L2 (no shared-memory destination, no barrier).
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap* map, int x, int y, int z, int w) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(map), "r"(x), "r"(y),
               "r"(z), "r"(w)
               : "memory");
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 2^x with the special-function unit's approximation (PTX ex2.approx.ftz: about 2 ulp; results
// below the normal range flush to 0).  The attention kernels round P to bf16 right after, so this
// is ample there.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- bf16 helpers ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

}  // namespace spectree

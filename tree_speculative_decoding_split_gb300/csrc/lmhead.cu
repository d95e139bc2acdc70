// K2: LM head z = W h for every tree node, fused with per-row softmax statistics.
// K2f: fp32 variant (SIMT).
//
// The LM head is a linear layer followed by softmax (tech-tldr "多トークン予測（Medusa・EAGLE）",
// section "Medusa"; jisaku glossary "Medusa", architecture table: hidden_dim x vocab_size).  It
// is the one dense contraction of the verification step: [rows x hidden] . [hidden x vocab].
//
// bf16 kernel (tcgen05).  The vocabulary sits on the MMA M dimension (tiles of 128 rows of W)
// and the tree rows on N (BN = 32..256 per tile), so a batch of 63 nodes still fills a full
// M = 128 instruction.  A persistent grid walks (vocab tile, row chunk) units; warp 0 issues
// TMA loads of W and hidden-state tiles (128-byte swizzle) into a shared-memory ring, warp 1
// issues tcgen05.mma (kind::f16, bf16 in, fp32 accumulators in tensor memory, double-buffered
// across units), warps 2..5 drain the accumulators with tcgen05.ld and reduce every node's
// column over the 128 vocabulary rows with warp shuffles into {max, sum exp, sum exp*y, second
// max, argmax} at y = z / tau.  Each CTA owns one chunk of rows and a strided set of vocabulary
// tiles, and keeps one running record per row in shared memory across its tiles, so it writes
// one record per row at the end (about 150 records per row in total, merged by the row
// finalisation kernel).  Full fp32 logits go to HBM only when the caller needs them (rejection
// sampling), written once from the same epilogue.  Larger batches put the tree rows on M instead:
// 128 rows per CTA (65..128 rows), or 256 rows per MMA over a pair of CTAs (more than 128 rows).

#include "common.cuh"
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace spectree {

namespace {

constexpr int kBM = 128;  // vocabulary rows per tile (MMA M)
constexpr int kBK = 64;   // hidden elements per stage (one 128-byte swizzle atom of bf16)
constexpr int kLmThreads = 192;

// Shared-memory descriptor of a K-major tile written by TMA with 128-byte swizzle: 128-byte rows,
// 8-row groups 1024 bytes apart (the leading byte offset is unused for this layout).
__device__ __forceinline__ uint64_t sdesc_k(uint32_t saddr) { return sdesc_sw128(saddr, 16, 1024); }

// Vocabulary-on-M kernel: four 64-element k atoms per pipeline stage, so that every W row is read
// 512 contiguous bytes at a time (measured on the 63-row, 128256 x 4096 head: 177.4 us with one
// atom and 8 stages, 174.6 us with two atoms and 4 stages, 173.4 us with four atoms and 2).
template <int BN>
struct LmCfg {
  static constexpr int kAtoms = 4;
  static constexpr int kAtomA = kBM * kBK * 2;
  static constexpr int kAtomB = BN * kBK * 2;
  static constexpr int kStageA = kAtomA * kAtoms;
  static constexpr int kStageB = kAtomB * kAtoms;
  static constexpr int kStage = kStageA + kStageB;
  static constexpr int kStages = 2;
  static constexpr uint32_t kTmemCols = (2 * BN <= 32) ? 32 : (2 * BN <= 64 ? 64 : (2 * BN <= 128 ? 128 : (2 * BN <= 256 ? 256 : 512)));
  static constexpr int kEpiBytes = 5 * BN * (int)sizeof(float4) + 5 * BN * (int)sizeof(int);
  static constexpr int kSmem = 1024 + kStages * kStage + kEpiBytes + 256;
};

}  // namespace

template <int BN>
__global__ void __launch_bounds__(kLmThreads, 1)
    lmhead_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH,
                     const LmParams p) {
  using C = LmCfg<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + C::kStages * C::kStageA;
  float4* sEpi = reinterpret_cast<float4*>(base + C::kStages * C::kStage);  // [4][BN] per-warp records
  float4* sRun = sEpi + 4 * BN;                                               // [BN] running records
  int* sEpiIdx = reinterpret_cast<int*>(sRun + BN);
  int* sRunIdx = sEpiIdx + 4 * BN;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sRunIdx + BN);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::kStages;
  uint64_t* tfull = empty + C::kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drained = tempty + 2;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ uint32_t s_issued, s_consumed;
  __shared__ int s_epi_fail;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_atoms = p.Hd / kBK;
  const int n_kb = (n_atoms + C::kAtoms - 1) / C::kAtoms;  // stages per tile
  // CTA c owns row chunk nc = c % n_nc and vocabulary tiles slot, slot + cpc, ...
  const int nc = blockIdx.x % p.n_nc, slot = blockIdx.x / p.n_nc;
  if (blockIdx.x == 0 && threadIdx.x < 32)
    for (int i = threadIdx.x; i < p.n_counters; i += 32) p.counters[i] = 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(drained, 1);
    s_abort = 0;
    s_epi_fail = 0;
    s_issued = 0;
    s_consumed = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem;

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer ----
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_h = l2_policy_evict_last();
      uint32_t it = 0;
      bool ok = true;
      for (int vt = slot; vt < p.n_vt && ok; vt += p.cpc) {
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int st = it % C::kStages;
          if (!mbar_wait_bounded(&empty[st], ((it / C::kStages) & 1) ^ 1, &s_abort)) {
            ok = false;
            break;
          }
          const int na = min(C::kAtoms, n_atoms - kb * C::kAtoms);
          mbar_arrive_expect_tx(&full[st], na * (C::kAtomA + C::kAtomB));
          for (int at = 0; at < na; ++at) {
            const int x = (kb * C::kAtoms + at) * kBK;
            tma_load_2d(sA + st * C::kStageA + at * C::kAtomA, &tmW, &full[st], x, vt * kBM, pol_w);
            tma_load_2d(sB + st * C::kStageB + at * C::kAtomB, &tmH, &full[st], x, nc * BN, pol_h);
          }
          s_issued = it + 1;
        }
      }
      if (!ok) {
        s_abort = 1;
        set_status(p.dev_status, SPEC_ERR_TIMEOUT);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer ----
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN, 0);
      uint32_t it = 0;
      int lu = 0;
      bool ok = true;
      for (int vt = slot; vt < p.n_vt && ok; vt += p.cpc, ++lu) {
        const int a = lu & 1;
        if (!mbar_wait_bounded(&tempty[a], ((lu >> 1) & 1) ^ 1, &s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(a * BN);
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int st = it % C::kStages;
          if (!mbar_wait_bounded(&full[st], (it / C::kStages) & 1, &s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int na = min(C::kAtoms, n_atoms - kb * C::kAtoms);
          for (int at = 0; at < na; ++at) {
            const uint64_t ad = sdesc_k(smem_u32(sA + st * C::kStageA + at * C::kAtomA));
            const uint64_t bd = sdesc_k(smem_u32(sB + st * C::kStageB + at * C::kAtomB));
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk)
              umma_bf16(d_tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, (kb | at | kk) != 0);
          }
          umma_commit(&empty[st]);
          s_consumed = it + 1;
        }
        if (ok) umma_commit(&tfull[a]);
      }
      if (!ok) {
        s_abort = 1;
        set_status(p.dev_status, SPEC_ERR_TIMEOUT);
      }
      // Every MMA issued by this thread has finished once `drained` completes.
      umma_commit(drained);
      mbar_wait_bounded(drained, 0, nullptr);
    }
  } else {
    // ---- epilogue: warps 2..5, TMEM lane quarter q = warp % 4 ----
    const int q = warp & 3;
    const int etid = (warp - 2) * 32 + lane;
    int lu = 0;
    for (int j = etid; j < BN; j += 128) {
      sRun[j] = make_float4(-INFINITY, 0.f, 0.f, -INFINITY);
      sRunIdx[j] = 0x7fffffff;
    }
    for (int vt = slot; vt < p.n_vt; vt += p.cpc, ++lu) {
      const int a = lu & 1;
      // The four epilogue warps agree on the outcome of the wait before going on, so that
      // none of them can be left alone at a named barrier.
      if (!mbar_wait_bounded(&tfull[a], (lu >> 1) & 1, &s_abort) && lane == 0) s_epi_fail = 1;
      named_bar_sync(1, 128);
      if (s_epi_fail) {
        if (etid == 0) {
          s_abort = 1;
          set_status(p.dev_status, SPEC_ERR_TIMEOUT);
        }
        break;
      }
      tc_fence_after();
      const int v = vt * kBM + q * 32 + lane;
      const bool vvalid = v < p.V;
#pragma unroll 1
      for (int cc = 0; cc < BN / 32; ++cc) {
        uint32_t r[32];
        tmem_ld_x32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * BN + cc * 32), r);
        tmem_ld_wait();
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int j = cc * 32 + jj;
          const int n = nc * BN + j;
          const float z = __uint_as_float(r[jj]);
          if (p.logits && vvalid && n < p.R) p.logits[(size_t)n * p.V + v] = z;
          const float y = vvalid ? z * p.inv_tau : -INFINITY;
          const float m = warp_max(y);
          const unsigned bal = __ballot_sync(0xffffffffu, y == m);
          const int first = __ffs(bal) - 1;
          const float y2 = warp_max(lane == first ? -INFINITY : y);
          const float e = (y > -INFINITY) ? expf(y - m) : 0.f;
          const float s = warp_sum(e);
          const float t = warp_sum(e > 0.f ? e * y : 0.f);
          if (lane == jj) {
            sEpi[q * BN + j] = make_float4(m, s, t, y2);
            sEpiIdx[q * BN + j] = (m > -INFINITY) ? vt * kBM + q * 32 + first : 0x7fffffff;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[a]);
      named_bar_sync(1, 128);
      for (int j = etid; j < BN; j += 128) {
        RowPart acc;
        const float4 r0 = sRun[j];
        acc.m = r0.x; acc.s = r0.y; acc.t = r0.z; acc.y2 = r0.w; acc.idx = sRunIdx[j];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const float4 f = sEpi[qq * BN + j];
          RowPart o;
          o.m = f.x; o.s = f.y; o.t = f.z; o.y2 = f.w; o.idx = sEpiIdx[qq * BN + j];
          acc = rowpart_merge(acc, o);
        }
        sRun[j] = make_float4(acc.m, acc.s, acc.t, acc.y2);
        sRunIdx[j] = acc.idx;
      }
      named_bar_sync(1, 128);
    }
    if (!s_epi_fail) {
      for (int j = etid; j < BN; j += 128) {
        const int n = nc * BN + j;
        if (n < p.R) {
          p.part[(size_t)slot * p.R + n] = sRun[j];
          p.part_idx[(size_t)slot * p.R + n] = sRunIdx[j];
        }
      }
    }
  }

  __syncthreads();
  if (threadIdx.x == 0 && s_abort) {
    // Let the copies still in flight land before shared memory is released.
    for (uint32_t it = s_consumed; it < s_issued; ++it)
      mbar_wait_bounded(&full[it % C::kStages], (it / C::kStages) & 1, nullptr);
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::kTmemCols);
}

// ---- rows-on-M orientation (128 tree rows per MMA tile, vocabulary on N) --------------------
// Used when there are at least 128 tree rows: the epilogue thread that owns TMEM lane r owns
// tree row r of the chunk, so the softmax statistics of a row are a running, per-thread
// reduction over the vocabulary columns (no cross-lane shuffles), carried in registers across
// all vocabulary tiles of the CTA.  CTA c owns row chunk rc = c % n_nc and vocabulary tiles
// slot, slot + cpc, ... of BNV entries each.

template <int BNV>
struct LmRowsCfg {
  static constexpr int kStageA = kBM * kBK * 2;   // 128 tree rows x 64 hidden
  static constexpr int kStageB = BNV * kBK * 2;   // BNV vocabulary rows x 64 hidden
  static constexpr int kStage = kStageA + kStageB;
  static constexpr int kStages = (BNV >= 256) ? 4 : 6;
  static constexpr uint32_t kTmemCols = 2 * BNV;  // double-buffered accumulators
  static constexpr int kSmem = 1024 + kStages * kStage + 256;
};

template <int BNV>
__global__ void __launch_bounds__(kLmThreads, 1)
    lmhead_tc_rows_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH,
                          const LmParams p) {
  using C = LmRowsCfg<BNV>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + C::kStages * C::kStageA;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::kStages * C::kStage);
  uint64_t* full = bars;
  uint64_t* empty = bars + C::kStages;
  uint64_t* tfull = empty + C::kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drained = tempty + 2;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ uint32_t s_issued, s_consumed;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_kb = p.Hd / kBK;
  const int rc = blockIdx.x % p.n_nc, slot = blockIdx.x / p.n_nc;
  const int n_vt = (p.V + BNV - 1) / BNV;
  if (blockIdx.x == 0 && threadIdx.x < 32)
    for (int i = threadIdx.x; i < p.n_counters; i += 32) p.counters[i] = 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(drained, 1);
    s_abort = 0;
    s_issued = 0;
    s_consumed = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = s_tmem;

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer: tree rows (re-read from L2 per tile), vocabulary rows of W ----
      const uint64_t pol_h = l2_policy_evict_last();
      const uint64_t pol_w = (p.n_nc > 1) ? l2_policy_evict_last() : l2_policy_evict_first();
      uint32_t it = 0;
      bool ok = true;
      for (int vt = slot; vt < n_vt && ok; vt += p.cpc) {
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int st = it % C::kStages;
          if (!mbar_wait_bounded(&empty[st], ((it / C::kStages) & 1) ^ 1, &s_abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[st], C::kStage);
          tma_load_2d(sA + st * C::kStageA, &tmH, &full[st], kb * kBK, rc * kBM, pol_h);
          tma_load_2d(sB + st * C::kStageB, &tmW, &full[st], kb * kBK, vt * BNV, pol_w);
          s_issued = it + 1;
        }
      }
      if (!ok) {
        s_abort = 1;
        set_status(p.dev_status, SPEC_ERR_TIMEOUT);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer ----
      constexpr uint32_t idesc = idesc_bf16_f32(kBM, BNV, 0);
      uint32_t it = 0;
      int lu = 0;
      bool ok = true;
      for (int vt = slot; vt < n_vt && ok; vt += p.cpc, ++lu) {
        const int a = lu & 1;
        if (!mbar_wait_bounded(&tempty[a], ((lu >> 1) & 1) ^ 1, &s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(a * BNV);
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int st = it % C::kStages;
          if (!mbar_wait_bounded(&full[st], (it / C::kStages) & 1, &s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_k(smem_u32(sA + st * C::kStageA));
          const uint64_t bd = sdesc_k(smem_u32(sB + st * C::kStageB));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16(d_tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, (kb | kk) != 0);
          umma_commit(&empty[st]);
          s_consumed = it + 1;
        }
        if (ok) umma_commit(&tfull[a]);
      }
      if (!ok) {
        s_abort = 1;
        set_status(p.dev_status, SPEC_ERR_TIMEOUT);
      }
      umma_commit(drained);
      mbar_wait_bounded(drained, 0, nullptr);
    }
  } else {
    // ---- epilogue: warps 2..5; thread (q, lane) owns tree row rc*128 + 32q + lane ----
    const int q = warp & 3;
    const int n = rc * kBM + q * 32 + lane;
    const bool nvalid = n < p.R;
    constexpr float kLog2e = 1.4426950408889634f;
    float m1 = -INFINITY, m2 = -INFINITY, s = 0.f, t = 0.f;
    int i1 = 0x7fffffff;
    bool failed = false;
    int lu = 0;
    for (int vt = slot; vt < n_vt; vt += p.cpc, ++lu) {
      const int a = lu & 1;
      // every lane waits on the barrier itself; a timeout is the same verdict in all four warps
      if (!mbar_wait_bounded(&tfull[a], (lu >> 1) & 1, &s_abort)) {
        failed = true;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int cc = 0; cc < BNV / 32; ++cc) {
        uint32_t r[32];
        tmem_ld_x32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * BNV + cc * 32), r);
        tmem_ld_wait();
        const int vbase = vt * BNV + cc * 32;
        if (p.logits && nvalid) {
          float* dst = p.logits + (size_t)n * p.V + vbase;
          if (vbase + 32 <= p.V && ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0)) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(dst + j) = make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                                                __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
          } else {
            for (int j = 0; j < 32; ++j)
              if (vbase + j < p.V) dst[j] = __uint_as_float(r[j]);
          }
        }
        const float m_prev = m1;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float y = (vbase + j < p.V) ? __uint_as_float(r[j]) * p.inv_tau : -INFINITY;
          if (y > m1) {
            m2 = m1;
            m1 = y;
            i1 = vbase + j;
          } else if (y > m2) {
            m2 = y;
          }
        }
        if (m1 > -INFINITY) {
          const float scale = (m_prev > -INFINITY) ? exp2f((m_prev - m1) * kLog2e) : 0.f;
          s *= scale;
          t *= scale;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (vbase + j < p.V) {  // entries past the vocabulary contribute nothing (0 * -inf is NaN)
              const float y = __uint_as_float(r[j]) * p.inv_tau;
              const float e = exp2f((y - m1) * kLog2e);
              s += e;
              t = fmaf(e, y, t);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[a]);
    }
    if (failed) {
      if (lane == 0) {
        s_abort = 1;
        set_status(p.dev_status, SPEC_ERR_TIMEOUT);
      }
    } else if (nvalid) {
      p.part[(size_t)slot * p.R + n] = make_float4(m1, s, t, m2);
      p.part_idx[(size_t)slot * p.R + n] = i1;
    }
  }

  __syncthreads();
  if (threadIdx.x == 0 && s_abort) {
    for (uint32_t it = s_consumed; it < s_issued; ++it)
      mbar_wait_bounded(&full[it % C::kStages], (it / C::kStages) & 1, nullptr);
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem_base, C::kTmemCols);
}

// ---- CTA-pair orientation (cta_group::2): 256 tree rows per MMA over two SMs ---------------------
// Used above 128 tree rows.  A cluster of two CTAs computes 256-row x 256-vocabulary tiles with one
// pair MMA: each CTA stages its own 128 tree rows and its half (128 entries) of the vocabulary tile,
// so a 64-wide k stage is 32 KB per SM instead of 48 KB and six stages fit where four did.  The
// even CTA's MMA warp issues the MMAs and multicasts each commit to both CTAs' barriers; both
// CTAs' TMA loads count on the even CTA's stage barrier; each CTA's epilogue drains its own tensor
// memory (its 128 rows) as in the rows-on-M kernel and signals the even CTA when a buffer is free.
// Cluster c owns row pair rc = c % n_nc and vocabulary tiles slot, slot + cpc, ... (slot = c / n_nc).
struct LmPairCfg {
  static constexpr int kN = 256;                  // vocabulary entries per pair tile (MMA N)
  static constexpr int kStageA = kBM * kBK * 2;   // this CTA's 128 tree rows x 64 hidden
  static constexpr int kStageB = (kN / 2) * kBK * 2;  // this CTA's half of the vocabulary tile
  static constexpr int kStage = kStageA + kStageB;
  static constexpr int kStages = 6;
  static constexpr uint32_t kTmemCols = 2 * kN;   // double-buffered accumulators
  static constexpr int kSmem = 1024 + kStages * kStage + 256;
};

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kLmThreads, 1)
    lmhead_tc_pair_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH,
                          const LmParams p) {
  using C = LmPairCfg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sA = base;
  uint8_t* sB = base + C::kStages * C::kStageA;
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + C::kStages * C::kStage);
  uint64_t* full = bars;                  // [stage] both CTAs' tiles landed (used in the even CTA)
  uint64_t* empty = bars + C::kStages;    // [stage] the pair MMA consumed the stage (each CTA)
  uint64_t* tfull = empty + C::kStages;   // [buffer] accumulator ready (each CTA)
  uint64_t* tempty = tfull + 2;           // [buffer] both CTAs drained it (used in the even CTA)
  uint64_t* drained = tempty + 2;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int n_kb = p.Hd / kBK;
  const int cl = blockIdx.x >> 1;
  const int rc = cl % p.n_nc, slot = cl / p.n_nc;
  const int n_vt = (p.V + C::kN - 1) / C::kN;
  if (blockIdx.x == 0 && threadIdx.x < 32)
    for (int i = threadIdx.x; i < p.n_counters; i += 32) p.counters[i] = 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8);  // four epilogue warps in each CTA
    }
    mbar_init(drained, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(&s_tmem, C::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync_all();  // both CTAs' barriers exist before any remote arrival or completion
  tc_fence_after();
  const uint32_t tmem_base = s_tmem;

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer (both CTAs): this CTA's tree rows and half vocabulary tile ----
      const uint64_t pol_h = l2_policy_evict_last();
      const uint64_t pol_w = (p.n_nc > 1) ? l2_policy_evict_last() : l2_policy_evict_first();
      uint32_t it = 0;
      bool ok = true;
      for (int vt = slot; vt < n_vt && ok; vt += p.cpc) {
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int st = it % C::kStages;
          if (!mbar_wait_bounded(&empty[st], ((it / C::kStages) & 1) ^ 1, &s_abort)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full[st], 2 * C::kStage);  // both CTAs' bytes
          const uint32_t fb = cluster_addr(&full[st], 0);
          tma_load_2d_pair(sA + st * C::kStageA, &tmH, fb, kb * kBK, rc * 2 * kBM + (int)rank * kBM, pol_h);
          tma_load_2d_pair(sB + st * C::kStageB, &tmW, fb, kb * kBK, vt * C::kN + (int)rank * (C::kN / 2), pol_w);
        }
      }
      if (!ok) {
        s_abort = 1;
        set_status(p.dev_status, SPEC_ERR_TIMEOUT);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---- MMA issuer (even CTA): 256 x 256 x 16 pair MMAs ----
      constexpr uint32_t idesc = idesc_bf16_f32(2 * kBM, C::kN, 0);
      uint32_t it = 0;
      int lu = 0;
      bool ok = true;
      for (int vt = slot; vt < n_vt && ok; vt += p.cpc, ++lu) {
        const int a = lu & 1;
        if (!mbar_wait_bounded(&tempty[a], ((lu >> 1) & 1) ^ 1, &s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(a * C::kN);
        for (int kb = 0; kb < n_kb; ++kb, ++it) {
          const int st = it % C::kStages;
          if (!mbar_wait_bounded(&full[st], (it / C::kStages) & 1, &s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_k(smem_u32(sA + st * C::kStageA));
          const uint64_t bd = sdesc_k(smem_u32(sB + st * C::kStageB));
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk)
            umma_bf16_pair(d_tmem, ad + (uint64_t)(kk * 2), bd + (uint64_t)(kk * 2), idesc, (kb | kk) != 0);
          umma_commit_pair(&empty[st], 3);  // the stage is free in both CTAs
        }
        if (ok) umma_commit_pair(&tfull[a], 3);
      }
      if (!ok) {
        s_abort = 1;
        set_status(p.dev_status, SPEC_ERR_TIMEOUT);
      }
      umma_commit_pair(drained, 1);
      mbar_wait_bounded(drained, 0, nullptr);
    }
  } else {
    // ---- epilogue (both CTAs): thread (q, lane) owns tree row 256 rc + 128 rank + 32 q + lane ----
    const int q = warp & 3;
    const int n = rc * 2 * kBM + (int)rank * kBM + q * 32 + lane;
    const bool nvalid = n < p.R;
    constexpr float kLog2e = 1.4426950408889634f;
    float m1 = -INFINITY, m2 = -INFINITY, s = 0.f, t = 0.f;
    int i1 = 0x7fffffff;
    bool failed = false;
    int lu = 0;
    for (int vt = slot; vt < n_vt; vt += p.cpc, ++lu) {
      const int a = lu & 1;
      if (!mbar_wait_bounded(&tfull[a], (lu >> 1) & 1, &s_abort)) {
        failed = true;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int cc = 0; cc < C::kN / 32; ++cc) {
        uint32_t r[32];
        tmem_ld_x32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(a * C::kN + cc * 32), r);
        tmem_ld_wait();
        const int vbase = vt * C::kN + cc * 32;
        if (p.logits && nvalid) {
          float* dst = p.logits + (size_t)n * p.V + vbase;
          if (vbase + 32 <= p.V && ((reinterpret_cast<uintptr_t>(dst) & 15u) == 0)) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(dst + j) = make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                                                __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
          } else {
            for (int j = 0; j < 32; ++j)
              if (vbase + j < p.V) dst[j] = __uint_as_float(r[j]);
          }
        }
        const float m_prev = m1;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float y = (vbase + j < p.V) ? __uint_as_float(r[j]) * p.inv_tau : -INFINITY;
          if (y > m1) {
            m2 = m1;
            m1 = y;
            i1 = vbase + j;
          } else if (y > m2) {
            m2 = y;
          }
        }
        if (m1 > -INFINITY) {
          const float scale = (m_prev > -INFINITY) ? exp2f((m_prev - m1) * kLog2e) : 0.f;
          s *= scale;
          t *= scale;
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            if (vbase + j < p.V) {  // entries past the vocabulary contribute nothing (0 * -inf is NaN)
              const float y = __uint_as_float(r[j]) * p.inv_tau;
              const float e = exp2f((y - m1) * kLog2e);
              s += e;
              t = fmaf(e, y, t);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(cluster_addr(&tempty[a], 0));
    }
    if (failed) {
      if (lane == 0) {
        s_abort = 1;
        set_status(p.dev_status, SPEC_ERR_TIMEOUT);
      }
    } else if (nvalid) {
      p.part[(size_t)slot * p.R + n] = make_float4(m1, s, t, m2);
      p.part_idx[(size_t)slot * p.R + n] = i1;
    }
  }

  __syncthreads();
  // Both CTAs finish here together: every remote arrival has landed and the even CTA's MMAs have
  // completed before either releases shared or tensor memory.  (After a timeout the copies still in
  // flight land within the bounded waits of the peer's producer or issuer.)
  cluster_sync_all();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem_base, C::kTmemCols);
}

// ---- fp32 path ------------------------------------------------------------------------------

// logits[R][V] = H[R][Hd] . W[V][Hd]^T, 64 x 64 output tile per CTA, 4 x 4 per thread.
__global__ void __launch_bounds__(256) lmhead_f32_kernel(const float* __restrict__ H, const float* __restrict__ W,
                                                         float* __restrict__ logits, int R, int V, int Hd) {
  __shared__ float sH[16][64 + 1];
  __shared__ float sW[16][64 + 1];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int r0 = blockIdx.y * 64, v0 = blockIdx.x * 64;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < Hd; k0 += 16) {
    for (int e = threadIdx.x; e < 16 * 64; e += 256) {
      const int kk = e & 15, rr = e >> 4;
      sH[kk][rr] = (r0 + rr < R && k0 + kk < Hd) ? H[(size_t)(r0 + rr) * Hd + k0 + kk] : 0.f;
      sW[kk][rr] = (v0 + rr < V && k0 + kk < Hd) ? W[(size_t)(v0 + rr) * Hd + k0 + kk] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < 16; ++kk) {
      float a[4], bw[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) { a[i] = sH[kk][ty * 4 + i]; bw[i] = sW[kk][tx * 4 + i]; }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bw[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int r = r0 + ty * 4 + i, v = v0 + tx * 4 + j;
      if (r < R && v < V) logits[(size_t)r * V + v] = acc[i][j];
    }
}

// Partial statistics of logits[row][vt*128 .. +128): one warp per (tile, row).  Records are laid
// out [tile][row] like the tensor-core kernel's [slot][row], with one slot per tile.
__global__ void __launch_bounds__(256) stats_from_logits_kernel(const float* __restrict__ logits, int R, int V,
                                                                int n_vt, float inv_tau, float4* __restrict__ part,
                                                                int* __restrict__ part_idx) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t id = (size_t)blockIdx.x * 8 + warp;
  if (id >= (size_t)n_vt * R) return;
  const int vt = (int)(id / R), n = (int)(id % R);
  RowPart acc = rowpart_empty();
  for (int k = 0; k < 4; ++k) {
    const int v = vt * kBM + k * 32 + lane;
    const float y = (v < V) ? logits[(size_t)n * V + v] * inv_tau : -INFINITY;
    const float m = warp_max(y);
    const unsigned bal = __ballot_sync(0xffffffffu, y == m);
    const int first = __ffs(bal) - 1;
    const float y2 = warp_max(lane == first ? -INFINITY : y);
    const float e = (y > -INFINITY) ? expf(y - m) : 0.f;
    RowPart o;
    o.m = m; o.y2 = y2;
    o.s = warp_sum(e);
    o.t = warp_sum(e > 0.f ? e * y : 0.f);
    o.idx = (m > -INFINITY) ? vt * kBM + k * 32 + first : 0x7fffffff;
    acc = rowpart_merge(acc, o);
  }
  if (lane == 0) {
    part[id] = make_float4(acc.m, acc.s, acc.t, acc.y2);
    part_idx[id] = acc.idx;
  }
}

// ---- host side ------------------------------------------------------------------------------

int lmhead_pick_bn(int R) {
  if (R <= 32) return 32;
  if (R <= 64) return 64;
  return 128;  // 128 tree rows per chunk: the rows-on-M kernel
}

size_t lmhead_smem_bytes(int BN) {
  switch (BN) {
    case 32: return LmCfg<32>::kSmem;
    case 64: return LmCfg<64>::kSmem;
    default: return LmRowsCfg<256>::kSmem;
  }
}

int lmhead_rows_bnv(int n_nc, int num_sms) {
  // vocabulary entries per tile: 256 once every SM has a row chunk's worth of tiles to stream
  return (n_nc >= 4 || num_sms <= 0) ? 256 : 128;
}

template <int BN>
static cudaError_t launch_lm(const CUtensorMap* tmW, const CUtensorMap* tmH, const LmParams& p, int num_sms,
                             cudaStream_t stream) {
  const int smem = LmCfg<BN>::kSmem;
  cudaError_t err = cudaFuncSetAttribute(lmhead_tc_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  lmhead_tc_kernel<BN><<<p.cpc * p.n_nc, kLmThreads, smem, stream>>>(*tmW, *tmH, p);
  return cudaGetLastError();
}

template <int BNV>
static cudaError_t launch_lm_rows(const CUtensorMap* tmW, const CUtensorMap* tmH, const LmParams& p,
                                  cudaStream_t stream) {
  const int smem = LmRowsCfg<BNV>::kSmem;
  cudaError_t err =
      cudaFuncSetAttribute(lmhead_tc_rows_kernel<BNV>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  lmhead_tc_rows_kernel<BNV><<<p.cpc * p.n_nc, kLmThreads, smem, stream>>>(*tmW, *tmH, p);
  return cudaGetLastError();
}

static cudaError_t launch_lm_pair(const CUtensorMap* tmW, const CUtensorMap* tmH, const LmParams& p,
                                  cudaStream_t stream) {
  const int smem = LmPairCfg::kSmem;
  cudaError_t err = cudaFuncSetAttribute(lmhead_tc_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  lmhead_tc_pair_kernel<<<2 * p.cpc * p.n_nc, kLmThreads, smem, stream>>>(*tmW, *tmH, p);
  return cudaGetLastError();
}

cudaError_t launch_lmhead_bf16(const CUtensorMap* tmW, const CUtensorMap* tmH, const LmParams& p, int num_sms,
                               cudaStream_t stream) {
  if (p.pair) return launch_lm_pair(tmW, tmH, p, stream);
  switch (p.BN) {
    case 32: return launch_lm<32>(tmW, tmH, p, num_sms, stream);
    case 64: return launch_lm<64>(tmW, tmH, p, num_sms, stream);
    default:
      return (p.BNV == 256) ? launch_lm_rows<256>(tmW, tmH, p, stream) : launch_lm_rows<128>(tmW, tmH, p, stream);
  }
}

void launch_lmhead_f32(const float* H, const float* W, const LmParams& p, cudaStream_t stream) {
  const dim3 grid((p.V + 63) / 64, (p.R + 63) / 64);
  lmhead_f32_kernel<<<grid, 256, 0, stream>>>(H, W, p.logits, p.R, p.V, p.Hd);
  const size_t units = (size_t)p.n_vt * p.R;
  stats_from_logits_kernel<<<(unsigned)((units + 7) / 8), 256, 0, stream>>>(p.logits, p.R, p.V, p.n_vt, p.inv_tau,
                                                                            p.part, p.part_idx);
}


}  // namespace spectree

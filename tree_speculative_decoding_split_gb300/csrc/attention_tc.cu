// K1 (bf16): split-KV tree attention on tcgen05 tensor cores.
//
// Parallel verification scores every candidate in one forward pass over the KV cache (qiita
// "EAGLE-3とMedusaで実装するSpeculative Decoding実践ガイド", section "並列検証"); each tree node
// attends only to its ancestors and itself (tech-tldr "多トークン予測（Medusa・EAGLE）", section
// "ツリー検証"; qiita, section "Tree Attention").
//
// One CTA owns (request b, KV head g, key split, group of 128 rows); a row is a (tree node i,
// GQA head j) pair r = i * G + j, so the 128 rows fill the M = 128 side of every MMA and all query
// heads sharing KV head g and all tree nodes read each K/V tile once.  Roles (192 threads):
//   warp 0     TMA producer: 64-key K and V tiles (128-byte swizzle) into a 3-stage ring;
//   warp 1     MMA issuer: S = Q K^T into one of two TMEM buffers, then O += P V into a TMEM
//              accumulator once the softmax has written P; V is consumed MN-major, so no
//              transpose is needed;
//   warps 2-5  softmax: the thread owning TMEM lane r owns row r -- it loads its S row, applies
//              the tree mask (ancestor bits, tail split only) and the online softmax in the log2
//              domain, and writes the bf16 P row to shared memory.  O is rescaled in TMEM only
//              when a row's running maximum grows by more than 2^8 (exact: P and the running sum
//              use the same stale maximum).
// Every CTA validates the tree; the tail CTA builds the ancestor bits by pointer jumping.  Each
// split writes a normalised partial (o, running max, sum), merged by the merge kernel.

#include "common.cuh"
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace spectree {

namespace {

constexpr int kKT = 64;         // keys per tile (MMA N of S, K of P V)
constexpr int kStages = 3;      // K/V ring depth
constexpr int kRows = 128;      // rows per CTA (MMA M)
constexpr int kTcThreads = 192;
constexpr float kRescaleLog2 = 8.f;

template <int D>
struct AttnTcCfg {
  static constexpr int kQ = kRows * D * 2;      // Q tile bytes
  static constexpr int kTile = kKT * D * 2;     // K (or V) tile bytes
  static constexpr int kP = kRows * kKT * 2;    // P tile bytes
  static constexpr int kSmem = 1024 + kQ + 2 * kStages * kTile + 2 * kP + kRows * kAncWords * 4 + 32 * 8;
  static constexpr uint32_t kTmemCols = (2 * kKT + D <= 256) ? 256 : 512;  // S x 2 + O
};

__device__ __forceinline__ uint32_t sw128_off(int r, int ch, int rows) {
  return (uint32_t)((ch >> 3) * rows * 128 + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void tma_load_3d_plain(void* dst, const CUtensorMap* map, uint64_t* bar, int x, int y,
                                                  int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const AttnParams p) {
  using C = AttnTcCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;
  uint8_t* sK = sQ + C::kQ;
  uint8_t* sV = sK + kStages * C::kTile;
  uint8_t* sP = sV + kStages * C::kTile;
  uint32_t* sAnc = reinterpret_cast<uint32_t*>(sP + 2 * C::kP);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sAnc + kRows * kAncWords);
  uint64_t* full = bars;                 // [3] K/V landed
  uint64_t* empty = full + kStages;      // [3] K/V consumed
  uint64_t* sfull = empty + kStages;     // [2] S computed
  uint64_t* sfree = sfull + 2;           // [2] S read by the softmax
  uint64_t* pfull = sfree + 2;           // [2] P written
  uint64_t* pfree = pfull + 2;           // [2] P consumed
  uint64_t* ofull = pfree + 2;           // O updated (one phase per tile)
  uint64_t* drained = ofull + 1;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_issued, s_consumed;
  __shared__ int s_par[kMaxNodes];
  __shared__ int s_jmp[kMaxNodes];
  __shared__ uint32_t s_nanc[kMaxNodes][kAncWords];

  const int rg = blockIdx.x, split = blockIdx.y, bg = blockIdx.z;
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long L = p.prefix_len[b];
  const int n = p.n_nodes[b];
  const bool tail = (split == p.n_prefix);
  const int rows_total = p.N * p.G;
  const int row0 = rg * kRows;

  // ---- tree checks, done by every CTA of the request (same verdict everywhere) ----
  int bad_tree = (n < 1 || n > p.N) ? 1 : 0, bad_cap = 0;
  if (!bad_tree) {
    bad_cap = (L < 0 || L + n > p.L_cap) ? 1 : 0;
    for (int c = tid; c < n; c += kTcThreads) {
      const int par = p.parent[(size_t)b * p.N + c];
      s_par[c] = par;
      if (c == 0 ? par != -1 : (par < 0 || par >= c)) bad_tree = 1;
    }
  }
  bad_tree = __syncthreads_or(bad_tree);
  bad_cap = __syncthreads_or(bad_cap);
  const int err = bad_tree ? SPEC_ERR_BAD_TREE : (bad_cap ? SPEC_ERR_CAPACITY : 0);
  if (err) {  // the merge kernel zeroes this request's outputs
    if (tid == 0 && rg == 0 && split == 0 && g == 0) set_status(p.dev_status, err);
    return;
  }
  long long kb, ke;
  if (!tail) {
    kb = (long long)split * p.chunk;
    ke = kb + p.chunk < L ? kb + p.chunk : L;
  } else {
    kb = L;
    ke = L + n;
  }
  const int T = ke > kb ? (int)((ke - kb + kKT - 1) / kKT) : 0;
  if (T == 0) {  // no keys here: the merge skips this split
    if (tid < kRows && row0 + tid < rows_total) {
      const int row = row0 + tid, i = row / p.G, h = g * p.G + row % p.G;
      const size_t orow = ((size_t)b * p.N + i) * p.Hq + h;
      p.part_ml[orow * p.n_split + split] = make_float2(-INFINITY, 0.f);
    }
    return;
  }

  // ---- ancestor bits of this CTA's rows (tail split) ----
  if (tail) {
    // pointer jumping: s_nanc[c] = nodes from c up to, not including, s_jmp[c]
    for (int c = tid; c < n; c += kTcThreads) {
#pragma unroll
      for (int w = 0; w < kAncWords; ++w) s_nanc[c][w] = 0u;
      s_nanc[c][c >> 5] = 1u << (c & 31);
      s_jmp[c] = (c == 0) ? -1 : s_par[c];
    }
    __syncthreads();
    for (int round = 0; round < 8; ++round) {
      int jj[2] = {-1, -1}, nj[2] = {-1, -1};
      uint32_t up[2][kAncWords];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int c = tid + k * kTcThreads;
        if (c < n) {
          jj[k] = s_jmp[c];
          if (jj[k] >= 0) {
            nj[k] = s_jmp[jj[k]];
#pragma unroll
            for (int w = 0; w < kAncWords; ++w) up[k][w] = s_nanc[jj[k]][w];
          }
        }
      }
      __syncthreads();
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int c = tid + k * kTcThreads;
        if (c < n && jj[k] >= 0) {
#pragma unroll
          for (int w = 0; w < kAncWords; ++w) s_nanc[c][w] |= up[k][w];
          s_jmp[c] = nj[k];
        }
      }
      __syncthreads();
    }
    for (int c = tid; c < kRows * kAncWords; c += kTcThreads) {
      const int r = c / kAncWords, w = c % kAncWords, row = row0 + r;
      uint32_t word = 0;
      if (row < rows_total) {
        const int i = row / p.G;
        if (i < n) word = s_nanc[i][w];
      }
      sAnc[c] = word;
    }
  }

  // ---- Q rows -> shared memory in the K-major 128-byte-swizzle layout of the MMA A operand ----
  constexpr int NCH = D / 8;
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
  for (int c = tid; c < kRows * NCH; c += kTcThreads) {
    const int r = c / NCH, ch = c % NCH, row = row0 + r;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (row < rows_total) {
      const int i = row / p.G, j = row % p.G;
      val = *reinterpret_cast<const uint4*>(q + (((size_t)b * p.N + i) * p.Hq + g * p.G + j) * D + ch * 8);
    }
    *reinterpret_cast<uint4*>(sQ + sw128_off(r, ch, kRows)) = val;
  }
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sfull[a], 1);
      mbar_init(&sfree[a], 4);
      mbar_init(&pfull[a], 4);
      mbar_init(&pfree[a], 1);
    }
    mbar_init(ofull, 1);
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
  fence_proxy_async_smem();  // Q (generic stores) becomes visible to the tensor cores
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t tmem_o = tmem + 2 * kKT;

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer ----
      bool ok = true;
      for (int t = 0; t < T && ok; ++t) {
        const int st = t % kStages;
        if (!mbar_wait_bounded(&empty[st], ((t / kStages) & 1) ^ 1, &s_abort)) {
          ok = false;
          break;
        }
        const int key = (int)(kb + (long long)t * kKT);
        mbar_arrive_expect_tx(&full[st], 2 * C::kTile);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d_plain(sK + st * C::kTile + c * kKT * 128, &tmK, &full[st], c * 64, key, bg);
          tma_load_3d_plain(sV + st * C::kTile + c * kKT * 128, &tmV, &full[st], c * 64, key, bg);
        }
        s_issued = t + 1;
      }
      if (!ok) {
        s_abort = 1;
        set_status(p.dev_status, SPEC_ERR_TIMEOUT);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMA issuer ----
      constexpr uint32_t idS = idesc_bf16_f32(kRows, kKT, 0);
      constexpr uint32_t idP = idesc_bf16_f32(kRows, D, 1);
      bool ok = true;
      auto issue_s = [&](int t) -> bool {
        const int st = t % kStages, sb = t & 1;
        if (!mbar_wait_bounded(&full[st], (t / kStages) & 1, &s_abort)) return false;
        if (!mbar_wait_bounded(&sfree[sb], ((t >> 1) & 1) ^ 1, &s_abort)) return false;
        tc_fence_after();
        const uint32_t qa = smem_u32(sQ), ka = smem_u32(sK + st * C::kTile);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(qa + (kk >> 2) * (kRows * 128) + (kk & 3) * 32, 0, 1024);
          const uint64_t bd = sdesc_sw128(ka + (kk >> 2) * (kKT * 128) + (kk & 3) * 32, 0, 1024);
          umma_bf16(tmem + sb * kKT, ad, bd, idS, kk > 0);
        }
        umma_commit(&sfull[sb]);
        return true;
      };
      ok = issue_s(0);
      for (int t = 0; t < T && ok; ++t) {
        if (t + 1 < T && !issue_s(t + 1)) {
          ok = false;
          break;
        }
        const int pb = t & 1, st = t % kStages;
        if (!mbar_wait_bounded(&pfull[pb], (t >> 1) & 1, &s_abort)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t pa = smem_u32(sP + pb * C::kP), va = smem_u32(sV + st * C::kTile);
#pragma unroll
        for (int kk = 0; kk < kKT / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(pa + kk * 32, 0, 1024);
          const uint64_t bd = sdesc_sw128(va + kk * 16 * 128, kKT * 128, 1024);
          umma_bf16(tmem_o, ad, bd, idP, (t > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&empty[st]);
        umma_commit(&pfree[pb]);
        umma_commit(ofull);
        s_consumed = t + 1;
      }
      if (!ok) {
        s_abort = 1;
        set_status(p.dev_status, SPEC_ERR_TIMEOUT);
      }
      umma_commit(drained);
      mbar_wait_bounded(drained, 0, nullptr);
    }
  } else {
    // ---- softmax: warps 2..5, TMEM lane quarter q, row r = 32 q + lane ----
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const int row = row0 + r;
    float m_run = -INFINITY, l_run = 0.f;
    uint32_t anc[kAncWords];
#pragma unroll
    for (int w = 0; w < kAncWords; ++w) anc[w] = tail ? sAnc[r * kAncWords + w] : 0u;
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      const int sb = t & 1;
      if (!mbar_wait_bounded(&sfull[sb], (t >> 1) & 1, &s_abort)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t s0[32], s1[32];
      tmem_ld_x32(tmem + lane_off + sb * kKT, s0);
      tmem_ld_x32(tmem + lane_off + sb * kKT + 32, s1);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sfree[sb]);
      float v[kKT];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        v[j] = __uint_as_float(s0[j]) * p.scale_log2;
        v[j + 32] = __uint_as_float(s1[j]) * p.scale_log2;
      }
      const long long kbase = kb + (long long)t * kKT;
      if (tail || kbase + kKT > ke) {
#pragma unroll
        for (int j = 0; j < kKT; ++j) {
          const long long kidx = kbase + j;
          bool keep = kidx < ke;
          if (tail && keep) {
            const int jj = (int)(kidx - kb);
            keep = (anc[jj >> 5] >> (jj & 31)) & 1u;
          }
          if (!keep) v[j] = -INFINITY;
        }
      }
      float tmax = v[0];
#pragma unroll
      for (int j = 1; j < kKT; ++j) tmax = fmaxf(tmax, v[j]);
      const float m_new = fmaxf(m_run, tmax);
      const bool need = m_new > m_run + kRescaleLog2;  // includes the first finite maximum
      if (__any_sync(0xffffffffu, need)) {
        const float f = need ? exp2f(m_run - m_new) : 1.f;  // 0 when m_run is -inf
        if (t > 0) {
          // O holds the previous tiles: wait for their last P V, then rescale in place
          if (!mbar_wait_bounded(ofull, (t - 1) & 1, &s_abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld_x32(tmem_o + lane_off + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
            tmem_st_x32(tmem_o + lane_off + c * 32, o);
          }
          tmem_st_wait();
        }
        if (need) {
          l_run *= f;
          m_run = m_new;
        }
      }
      const float mu = (m_run == -INFINITY) ? 0.f : m_run;
      float psum = 0.f;
      uint32_t pk[kKT / 2];
#pragma unroll
      for (int j = 0; j < kKT; j += 2) {
        const float p0 = exp2f(v[j] - mu), p1 = exp2f(v[j + 1] - mu);
        psum += p0 + p1;
        pk[j / 2] = pack_bf16x2(p0, p1);
      }
      l_run += psum;
      if (!mbar_wait_bounded(&pfree[sb], ((t >> 1) & 1) ^ 1, &s_abort)) {
        ok = false;
        break;
      }
      uint8_t* prow = sP + sb * C::kP;
#pragma unroll
      for (int ch = 0; ch < kKT / 8; ++ch)
        *reinterpret_cast<uint4*>(prow + sw128_off(r, ch, kRows)) =
            make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pfull[sb]);
    }
    if (ok && mbar_wait_bounded(ofull, (T - 1) & 1, &s_abort)) {
      tc_fence_after();
      const bool valid = row < rows_total;
      size_t orow = 0;
      if (valid) {
        const int i = row / p.G, h = g * p.G + row % p.G;
        orow = ((size_t)b * p.N + i) * p.Hq + h;
        p.part_ml[orow * p.n_split + split] = make_float2(m_run, l_run);
      }
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld_x32(tmem_o + lane_off + c * 32, o);
        tmem_ld_wait();
        if (valid) {
          float* dst = p.part_o + (orow * p.n_split + split) * D + c * 32;
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(dst + j) =
                make_float4(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv,
                            __uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv);
        }
      }
    } else {
      if (lane == 0) {
        s_abort = 1;
        set_status(p.dev_status, SPEC_ERR_TIMEOUT);
      }
      if (row < rows_total) {  // the merge skips this split
        const int i = row / p.G, h = g * p.G + row % p.G;
        p.part_ml[(((size_t)b * p.N + i) * p.Hq + h) * p.n_split + split] = make_float2(-INFINITY, 0.f);
      }
    }
  }

  __syncthreads();
  if (tid == 0 && s_abort) {
    // let the copies still in flight land before shared memory is released
    for (int u = s_consumed; u < s_issued; ++u)
      mbar_wait_bounded(&full[u % kStages], (uint32_t)((u / kStages) & 1), nullptr);
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

size_t attention_tc_smem_bytes(int d) { return d == 128 ? AttnTcCfg<128>::kSmem : AttnTcCfg<64>::kSmem; }

cudaError_t launch_attention_tc(const CUtensorMap* tmK, const CUtensorMap* tmV, const AttnParams& p,
                                cudaStream_t stream) {
  const dim3 grid(p.n_rg, p.n_split, p.B * p.Hkv);
  cudaError_t err;
  if (p.d == 128) {
    const int smem = AttnTcCfg<128>::kSmem;
    err = cudaFuncSetAttribute(attn_tc_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    attn_tc_kernel<128><<<grid, kTcThreads, smem, stream>>>(*tmK, *tmV, p);
  } else {
    const int smem = AttnTcCfg<64>::kSmem;
    err = cudaFuncSetAttribute(attn_tc_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    attn_tc_kernel<64><<<grid, kTcThreads, smem, stream>>>(*tmK, *tmV, p);
  }
  return cudaGetLastError();
}

}  // namespace spectree

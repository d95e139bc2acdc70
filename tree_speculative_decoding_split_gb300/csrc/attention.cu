// K1: split-KV tree attention, K1m: merge of the splits, K1f: fp32 exact variant.
//
// Parallel verification scores every candidate in one forward pass over the KV cache (qiita
// "EAGLE-3とMedusaで実装するSpeculative Decoding実践ガイド", section "並列検証"); each tree node
// attends only to its ancestors and itself (tech-tldr "多トークン予測（Medusa・EAGLE）", section
// "ツリー検証"; qiita, section "Tree Attention").
//
// bf16 kernel layout.  One CTA owns (request b, KV head g, key split, row group of 128 rows);
// its rows are (node i, GQA head j) pairs r = i * G + j, so all query heads that share KV head
// g and all tree nodes read every K/V tile from shared memory once.  K/V tiles of 64 keys are
// brought in by TMA (128-byte swizzle, 3-stage ring, mbarrier completion).  Each of the eight
// warps holds 16 rows; S = Q K^T and O += P V run on mma.sync m16n8k16 (bf16 in, fp32 out) with
// an online softmax in the log2 domain.  The prefix splits are unmasked except for their
// ragged end; the last split covers the tree slots [L_b, L_b + n_b) and applies the ancestor
// mask from a bit matrix (one 32-bit word per 32 nodes) that the CTA builds in shared memory by
// pointer jumping over the parent array.  Every CTA validates the tree itself.  Each split
// writes a normalised partial (o, running max, sum); the merge kernel combines the splits per
// row with warp shuffles and writes O and the natural-log LSE.

#include "common.cuh"
#include "kernels.cuh"

namespace spectree {

namespace {

constexpr int kKT = 64;        // keys per tile
constexpr int kStages = 3;     // TMA ring depth
constexpr int kRows = 128;     // rows (node x GQA head) per CTA
constexpr int kThreads = 256;  // 8 warps x 16 rows

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void mma_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void tma_load_3d_nohint(void* dst, const CUtensorMap* map, uint64_t* bar,
                                                   int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(map), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}

// Byte offset of 16-byte chunk `ch` of row `r` in a tile whose rows are split into 128-byte
// swizzle atoms of 8 chunks (TMA SWIZZLE_128B layout, atoms of `rows` rows stacked per 64
// columns).
__device__ __forceinline__ uint32_t sw128(int r, int ch, int rows) {
  return (uint32_t)((ch >> 3) * rows * 128 + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_splitkv_bf16_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                             const AttnParams p) {
  constexpr int TILE = kKT * D * 2;  // bytes of a K (or V) tile
  constexpr int NCH = D / 8;         // 16-byte chunks per row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sK = base;
  uint8_t* sV = base + kStages * TILE;
  uint8_t* sQ = base + 2 * kStages * TILE;
  uint32_t* sAnc = reinterpret_cast<uint32_t*>(sQ + kRows * D * 2);  // ancestor words of this CTA's rows
  uint64_t* full = reinterpret_cast<uint64_t*>(sAnc + kRows * kAncWords);
  __shared__ int s_abort;
  __shared__ int s_issued;
  __shared__ int s_par[kMaxNodes];
  __shared__ int s_jmp[kMaxNodes];
  __shared__ uint32_t s_nanc[kMaxNodes][kAncWords];  // ancestor-or-self words of every node

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
    for (int c = tid; c < n; c += kThreads) {
      const int par = p.parent[(size_t)b * p.N + c];
      s_par[c] = par;
      if (c == 0 ? par != -1 : (par < 0 || par >= c)) bad_tree = 1;
    }
  }
  bad_tree = __syncthreads_or(bad_tree);
  bad_cap = __syncthreads_or(bad_cap);
  const int err = bad_tree ? SPEC_ERR_BAD_TREE : (bad_cap ? SPEC_ERR_CAPACITY : 0);

  if (!err) {
    long long kb, ke;
    if (!tail) {
      kb = (long long)split * p.chunk;
      ke = kb + p.chunk < L ? kb + p.chunk : L;
    } else {
      kb = L;
      ke = L + n;
    }
    const int ntiles = ke > kb ? (int)((ke - kb + kKT - 1) / kKT) : 0;
    bool wrote = false;
    if (ntiles > 0) {
      if (tail) {
        // Ancestor-or-self sets by pointer jumping (one node per thread, 8 rounds cover 255
        // levels): s_nanc[c] = nodes from c up to, not including, s_jmp[c].
        if (tid < n) {
#pragma unroll
          for (int w = 0; w < kAncWords; ++w) s_nanc[tid][w] = 0u;
          s_nanc[tid][tid >> 5] = 1u << (tid & 31);
          s_jmp[tid] = (tid == 0) ? -1 : s_par[tid];
        }
        __syncthreads();
        for (int round = 0; round < 8; ++round) {
          int j = -1, nj = -1;
          uint32_t up[kAncWords];
          if (tid < n) {
            j = s_jmp[tid];
            if (j >= 0) {
              nj = s_jmp[j];
#pragma unroll
              for (int w = 0; w < kAncWords; ++w) up[w] = s_nanc[j][w];
            }
          }
          __syncthreads();
          if (tid < n && j >= 0) {
#pragma unroll
            for (int w = 0; w < kAncWords; ++w) s_nanc[tid][w] |= up[w];
            s_jmp[tid] = nj;
          }
          __syncthreads();
        }
      }
    if (tid == 0) {
      for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
      s_abort = 0;
      fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int t) {
      const int st = t % kStages;
      const int key = (int)(kb + (long long)t * kKT);
      mbar_arrive_expect_tx(&full[st], 2 * TILE);
  #pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        tma_load_3d_nohint(sK + st * TILE + c * kKT * 128, &tmK, &full[st], c * 64, key, bg);
        tma_load_3d_nohint(sV + st * TILE + c * kKT * 128, &tmV, &full[st], c * 64, key, bg);
      }
    };
    if (tid == 0) {
      const int pro = ntiles < kStages ? ntiles : kStages;
      for (int t = 0; t < pro; ++t) issue(t);
      s_issued = pro;
    }

    // Q rows -> shared memory (swizzled like the K/V tiles so ldmatrix is conflict-free).
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
    for (int c = tid; c < kRows * NCH; c += kThreads) {
      const int r = c / NCH, ch = c % NCH, row = row0 + r;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (row < rows_total) {
        const int i = row / p.G, j = row % p.G;
        val = *reinterpret_cast<const uint4*>(q + (((size_t)b * p.N + i) * p.Hq + g * p.G + j) * D + ch * 8);
      }
      *reinterpret_cast<uint4*>(sQ + sw128(r, ch, kRows)) = val;
    }
    if (tail) {
      for (int c = tid; c < kRows * kAncWords; c += kThreads) {
        const int r = c / kAncWords, w = c % kAncWords, row = row0 + r;
        uint32_t word = 0;
        if (row < rows_total) {
          const int i = row / p.G;
          if (i < n) word = s_nanc[i][w];
        }
        sAnc[c] = word;
      }
    }
    __syncthreads();

    uint32_t qf[D / 16][4];
  #pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      const int r = warp * 16 + (lane & 15), ch = kk * 2 + (lane >> 4);
      ldsm_x4(qf[kk], sQ + sw128(r, ch, kRows));
    }

    float o[D / 8][4];
  #pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
    const int rA = warp * 16 + (lane >> 2);  // CTA-local rows of this thread: rA and rA + 8

    int t = 0;
    for (; t < ntiles; ++t) {
      const int st = t % kStages;
      if (!mbar_wait_bounded(&full[st], (uint32_t)((t / kStages) & 1), &s_abort)) {
        s_abort = 1;
        set_status(p.dev_status, SPEC_ERR_TIMEOUT);
        break;
      }
      const uint8_t* tK = sK + st * TILE;
      const uint8_t* tV = sV + st * TILE;
      float s[8][4];
  #pragma unroll
      for (int nt = 0; nt < 8; ++nt) s[nt][0] = s[nt][1] = s[nt][2] = s[nt][3] = 0.f;
  #pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
  #pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t bf[4];
          const int key = np * 16 + (lane & 7) + ((lane >> 4) << 3);
          const int ch = kk * 2 + ((lane >> 3) & 1);
          ldsm_x4(bf, tK + sw128(key, ch, kKT));
          mma_16816(s[2 * np], qf[kk], bf[0], bf[1]);
          mma_16816(s[2 * np + 1], qf[kk], bf[2], bf[3]);
        }
      }
      const long long kbase = kb + (long long)t * kKT;
      const bool need_mask = tail || (kbase + kKT > ke);
  #pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
  #pragma unroll
        for (int e = 0; e < 4; ++e) {
          float v = s[nt][e] * p.scale_log2;
          if (need_mask) {
            const int col = nt * 8 + (lane & 3) * 2 + (e & 1);
            const long long kidx = kbase + col;
            bool ok = kidx < ke;
            if (tail && ok) {
              const int jj = (int)(kidx - kb);
              const int r = (e < 2) ? rA : rA + 8;
              ok = (sAnc[r * kAncWords + (jj >> 5)] >> (jj & 31)) & 1u;
            }
            if (!ok) v = -INFINITY;
          }
          s[nt][e] = v;
        }
      }
      float mx[2] = {m_run[0], m_run[1]};
  #pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        mx[0] = fmaxf(mx[0], fmaxf(s[nt][0], s[nt][1]));
        mx[1] = fmaxf(mx[1], fmaxf(s[nt][2], s[nt][3]));
      }
  #pragma unroll
      for (int r = 0; r < 2; ++r) {
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
        mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
      }
      float mu[2], alpha[2], psum[2] = {0.f, 0.f};
  #pragma unroll
      for (int r = 0; r < 2; ++r) {
        mu[r] = (mx[r] == -INFINITY) ? 0.f : mx[r];
        alpha[r] = exp2f(m_run[r] - mu[r]);
        m_run[r] = mx[r];
      }
  #pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        s[nt][0] = exp2f(s[nt][0] - mu[0]);
        s[nt][1] = exp2f(s[nt][1] - mu[0]);
        s[nt][2] = exp2f(s[nt][2] - mu[1]);
        s[nt][3] = exp2f(s[nt][3] - mu[1]);
        psum[0] += s[nt][0] + s[nt][1];
        psum[1] += s[nt][2] + s[nt][3];
      }
      l_run[0] = l_run[0] * alpha[0] + psum[0];
      l_run[1] = l_run[1] * alpha[1] + psum[1];
  #pragma unroll
      for (int dt = 0; dt < D / 8; ++dt) {
        o[dt][0] *= alpha[0]; o[dt][1] *= alpha[0];
        o[dt][2] *= alpha[1]; o[dt][3] *= alpha[1];
      }
  #pragma unroll
      for (int k2 = 0; k2 < 4; ++k2) {
        uint32_t a[4];
        a[0] = pack_bf16x2(s[2 * k2][0], s[2 * k2][1]);
        a[1] = pack_bf16x2(s[2 * k2][2], s[2 * k2][3]);
        a[2] = pack_bf16x2(s[2 * k2 + 1][0], s[2 * k2 + 1][1]);
        a[3] = pack_bf16x2(s[2 * k2 + 1][2], s[2 * k2 + 1][3]);
  #pragma unroll
        for (int dp = 0; dp < D / 16; ++dp) {
          uint32_t bv[4];
          const int key = k2 * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
          const int ch = dp * 2 + (lane >> 4);
          ldsm_x4_t(bv, tV + sw128(key, ch, kKT));
          mma_16816(o[2 * dp], a, bv[0], bv[1]);
          mma_16816(o[2 * dp + 1], a, bv[2], bv[3]);
        }
      }
      __syncthreads();  // every warp is done with stage st
      if (tid == 0 && t + kStages < ntiles && !s_abort) {
        issue(t + kStages);
        s_issued = t + kStages + 1;
      }
    }

      if (s_abort) {
        // Let the copies still in flight land before the CTA's shared memory is released.
        __syncthreads();
        if (tid == 0)
          for (int u = t; u < s_issued; ++u)
            mbar_wait_bounded(&full[u % kStages], (uint32_t)((u / kStages) & 1), nullptr);
        __syncthreads();
      } else {
  #pragma unroll
    for (int r = 0; r < 2; ++r) {
      l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
      l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
    }
  #pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int row = row0 + rA + r * 8;
      if (row >= rows_total) continue;
      const int i = row / p.G, h = g * p.G + row % p.G;
      const size_t orow = ((size_t)b * p.N + i) * p.Hq + h;
      if ((lane & 3) == 0) p.part_ml[orow * p.n_split + split] = make_float2(m_run[r], l_run[r]);
      const float inv = l_run[r] > 0.f ? 1.f / l_run[r] : 0.f;
      float* dst = p.part_o + (orow * p.n_split + split) * D + (lane & 3) * 2;
  #pragma unroll
      for (int dt = 0; dt < D / 8; ++dt)
        *reinterpret_cast<float2*>(dst + dt * 8) = make_float2(o[dt][2 * r] * inv, o[dt][2 * r + 1] * inv);
    }

        wrote = true;
      }
    }
    if (!wrote) {  // no keys in this split (or a timed-out wait): the merge skips it
      if (tid < kRows && row0 + tid < rows_total) {
        const int row = row0 + tid, i = row / p.G, h = g * p.G + row % p.G;
        const size_t orow = ((size_t)b * p.N + i) * p.Hq + h;
        p.part_ml[orow * p.n_split + split] = make_float2(-INFINITY, 0.f);
      }
    }
  }

  // the first CTA of each request reports a bad tree; the merge kernel zeroes its outputs
  if (err && tid == 0 && blockIdx.x == 0 && split == 0 && g == 0) set_status(p.dev_status, err);
}

// K1m: merge of the splits, one warp per output row (b, i, h); lane s holds split s.  Requests
// with an invalid tree (checked again here: a handful of loads per warp) get zero outputs.
template <int D>
__global__ void __launch_bounds__(256) attn_merge_bf16_kernel(const AttnParams p) {
  constexpr int EPL = D / 32;  // elements per lane, contiguous
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t orow = (size_t)blockIdx.x * 8 + warp;
  const size_t total = (size_t)p.B * p.N * p.Hq;
  if (orow >= total) return;
  const int b = (int)(orow / ((size_t)p.N * p.Hq));
  const int i = (int)((orow / p.Hq) % p.N);
  const int n = p.n_nodes[b];
  const long long L = p.prefix_len[b];
  bool zero = n < 1 || n > p.N || i >= n || L < 0 || L + n > p.L_cap;
  if (!zero) {
    bool bad = false;
    for (int c = lane; c < n; c += 32) {
      const int par = p.parent[(size_t)b * p.N + c];
      bad |= (c == 0) ? par != -1 : (par < 0 || par >= c);
    }
    zero = __any_sync(0xffffffffu, bad);
  }
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + orow * D + lane * EPL;
  if (zero) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) out[e] = __float2bfloat16(0.f);
    if (p.lse && lane == 0) p.lse[orow] = 0.f;
    return;
  }
  float2 ml = make_float2(-INFINITY, 0.f);
  if (lane < p.n_split) ml = p.part_ml[orow * p.n_split + lane];
  const float M = warp_max(ml.y > 0.f ? ml.x : -INFINITY);
  const float w = (ml.y > 0.f) ? ml.y * exp2f(ml.x - M) : 0.f;
  const float wsum = warp_sum(w);
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  for (int s = 0; s < p.n_split; ++s) {
    const float ws = __shfl_sync(0xffffffffu, w, s);
    if (ws > 0.f) {
      const float* src = p.part_o + (orow * p.n_split + s) * D + lane * EPL;
      if constexpr (EPL == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        acc[0] += ws * v.x; acc[1] += ws * v.y; acc[2] += ws * v.z; acc[3] += ws * v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        acc[0] += ws * v.x; acc[1] += ws * v.y;
      }
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
  for (int e = 0; e < EPL; ++e) out[e] = __float2bfloat16(acc[e] * inv);
  if (p.lse && lane == 0) p.lse[orow] = (M + log2f(wsum)) * 0.69314718055994531f;
}

// K1f: fp32 tree attention, one warp per output row; keys visited one by one (prefix, then the
// ancestor bits of the node), online softmax in natural-exp form.
template <int D>
__global__ void __launch_bounds__(128) attn_rows_f32_kernel(const AttnParams p) {
  constexpr int EPL = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t orow = (size_t)blockIdx.x * 4 + warp;
  const size_t total = (size_t)p.B * p.N * p.Hq;
  if (orow >= total) return;
  const int b = (int)(orow / ((size_t)p.N * p.Hq));
  const int i = (int)((orow / p.Hq) % p.N);
  const int h = (int)(orow % p.Hq);
  float* out = static_cast<float*>(p.out) + orow * D;
  if (p.bad[b] || i >= p.n_nodes[b]) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) out[lane + 32 * e] = 0.f;
    if (p.lse && lane == 0) p.lse[orow] = 0.f;
    return;
  }
  const int g = h / p.G;
  const long long L = p.prefix_len[b];
  const float* qrow = static_cast<const float*>(p.q) + orow * D;
  float qv[EPL], acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) { qv[e] = qrow[lane + 32 * e]; acc[e] = 0.f; }
  const size_t head = ((size_t)b * p.Hkv + g) * (size_t)p.L_cap;
  float m = -INFINITY, l = 0.f;
  auto visit = [&](long long slot) {
    const float* kr = p.k32 + (head + slot) * D;
    const float* vr = p.v32 + (head + slot) * D;
    float dot = 0.f;
#pragma unroll
    for (int e = 0; e < EPL; ++e) dot = fmaf(qv[e], kr[lane + 32 * e], dot);
    dot = warp_sum(dot) * p.scale;
    const float mn = fmaxf(m, dot);
    const float corr = expf(m - mn);
    const float pe = expf(dot - mn);
    l = l * corr + pe;
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = acc[e] * corr + pe * vr[lane + 32 * e];
    m = mn;
  };
  for (long long s = 0; s < L; ++s) visit(s);
  for (int w = 0; w < p.W; ++w) {
    uint32_t bits = p.anc[((size_t)b * p.N + i) * p.W + w];
    while (bits) {
      const int jj = w * 32 + __ffs(bits) - 1;
      bits &= bits - 1;
      visit(L + jj);
    }
  }
  const float inv = 1.f / l;
#pragma unroll
  for (int e = 0; e < EPL; ++e) out[lane + 32 * e] = acc[e] * inv;
  if (p.lse && lane == 0) p.lse[orow] = m + logf(l);
}

// ---- host side ------------------------------------------------------------------------------

AttnPlan plan_attention(int B, int N, int G, int Hkv, long long L_cap, int num_sms) {
  AttnPlan pl;
  pl.n_rg = (N * G + kRows - 1) / kRows;
  const long long base = (long long)B * Hkv * pl.n_rg;
  long long want = (2LL * num_sms + base - 1) / base;  // about two CTAs per SM
  if (want < 1) want = 1;
  if (want > 31) want = 31;
  long long chunk = (L_cap + want - 1) / want;
  chunk = (chunk + kKT - 1) / kKT * kKT;
  if (chunk < 4 * kKT) chunk = 4 * kKT;
  long long np = (L_cap + chunk - 1) / chunk;
  if (np < 1) np = 1;
  while (np > 31) {  // keep n_split within a warp for the merge
    chunk *= 2;
    np = (L_cap + chunk - 1) / chunk;
  }
  pl.chunk = (int)chunk;
  pl.n_prefix = (int)np;
  pl.n_split = pl.n_prefix + 1;
  return pl;
}

size_t attention_smem_bytes(int d) {
  return 1024 + 2 * kStages * (size_t)kKT * d * 2 + (size_t)kRows * d * 2 + kRows * kAncWords * 4 +
         kStages * 8;
}

cudaError_t launch_attention_bf16(const CUtensorMap* tmK, const CUtensorMap* tmV, const AttnParams& p,
                                  cudaStream_t stream) {
  const dim3 grid(p.n_rg, p.n_split, p.B * p.Hkv);
  const size_t smem = attention_smem_bytes(p.d);
  cudaError_t err;
  if (p.d == 128) {
    err = cudaFuncSetAttribute(attn_splitkv_bf16_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    attn_splitkv_bf16_kernel<128><<<grid, kThreads, smem, stream>>>(*tmK, *tmV, p);
  } else {
    err = cudaFuncSetAttribute(attn_splitkv_bf16_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (err != cudaSuccess) return err;
    attn_splitkv_bf16_kernel<64><<<grid, kThreads, smem, stream>>>(*tmK, *tmV, p);
  }
  return cudaGetLastError();
}

void launch_attention_merge_bf16(const AttnParams& p, cudaStream_t stream) {
  const size_t total = (size_t)p.B * p.N * p.Hq;
  const unsigned blocks = (unsigned)((total + 7) / 8);
  if (p.d == 128)
    attn_merge_bf16_kernel<128><<<blocks, 256, 0, stream>>>(p);
  else
    attn_merge_bf16_kernel<64><<<blocks, 256, 0, stream>>>(p);
}

void launch_attention_f32(const AttnParams& p, cudaStream_t stream) {
  const size_t total = (size_t)p.B * p.N * p.Hq;
  const unsigned blocks = (unsigned)((total + 3) / 4);
  if (p.d == 128)
    attn_rows_f32_kernel<128><<<blocks, 128, 0, stream>>>(p);
  else
    attn_rows_f32_kernel<64><<<blocks, 128, 0, stream>>>(p);
}

}  // namespace spectree

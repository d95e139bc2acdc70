// K1m: merge of the split-KV partials of tree attention; K1f: fp32 exact tree attention; and
// the split plan shared by the bf16 kernel (attention_tc.cu).
//
// Parallel verification scores every candidate in one forward pass over the KV cache (qiita
// "EAGLE-3とMedusaで実装するSpeculative Decoding実践ガイド", section "並列検証"); each tree node
// attends only to its ancestors and itself (tech-tldr "多トークン予測（Medusa・EAGLE）", section
// "ツリー検証"; qiita, section "Tree Attention").  Each split of the bf16 kernel writes a normalised
// partial (bf16 o, running max in log2 units, sum); the merge kernel combines them per output row
// with warp shuffles and writes O and the natural-log LSE.

#include "common.cuh"
#include "kernels.cuh"

namespace spectree {

namespace {

constexpr int kKT = 64;    // keys per tile of the bf16 kernel (split sizes are multiples of it)

}  // namespace

// K1m: merge of the splits, one warp per output row (b, i, h); lane s holds split s.  Requests
// whose tree, capacity or block table the attention kernel found invalid get zero outputs.
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
  const bool zero = n < 1 || n > p.N || i >= n || L < 0 || L + n > p.L_cap || p.tree_bad[b] ||
                    (p.table && p.req_bad[b]);
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
  // Partials are loaded in batches of 8 so that the loads overlap; splits of zero weight (no key
  // of this row, or past the request's last key) are not read.
  constexpr int kBatch = 8;
  for (int s0 = 0; s0 < p.n_split; s0 += kBatch) {
    float v[kBatch][EPL];
    float ws[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int s = s0 + k;
      ws[k] = __shfl_sync(0xffffffffu, w, s & 31);
      if (s < p.n_split && ws[k] > 0.f) {
        const uint16_t* src = p.part_o + (orow * p.n_split + s) * D + lane * EPL;
        if constexpr (EPL == 4) {
          const uint2 t = __ldcg(reinterpret_cast<const uint2*>(src));
          const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&t.x));
          const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&t.y));
          v[k][0] = a.x; v[k][1] = a.y; v[k][2] = b.x; v[k][3] = b.y;
        } else {
          const uint32_t t = __ldcg(reinterpret_cast<const unsigned int*>(src));
          const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&t));
          v[k][0] = a.x; v[k][1] = a.y;
        }
      } else {
        ws[k] = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) v[k][e] = 0.f;
      }
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k)
      if (ws[k] > 0.f) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = fmaf(ws[k], v[k][e], acc[e]);
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
  // Two 128-row groups per CTA (ping-pong) when that still gives every SM work before any key
  // splitting; small problems keep one group so that there are more, shorter CTAs.
  const long long units2 = (long long)B * Hkv * ((N * G + attention_tc_rows_per_cta(2) - 1) / attention_tc_rows_per_cta(2));
  pl.groups = (units2 * 2 >= num_sms) ? 2 : 1;
  const int rows_cta = attention_tc_rows_per_cta(pl.groups);  // (node, GQA head) rows per bf16 CTA
  pl.n_rg = (N * G + rows_cta - 1) / rows_cta;
  const long long base = (long long)B * Hkv * pl.n_rg;
  // Key splits.  A CTA costs about kFixedTiles key tiles of fixed work (tree checks, prologue,
  // epilogue) plus its key tiles, and the CTAs run one per SM in rounds; more than one split adds
  // the merge kernel, about kMergeTiles.  Prefix lengths are only known on the device, so the
  // estimate takes every request at L_cap.  Among chunks of 4 or more key tiles (at most 16K
  // keys, at most 31 splits) take the one with the smallest estimated time, preferring grids that
  // fill at least one round; a grid that leaves SMs idle in its only round wins only when its
  // estimate is lower by more than 15 % (requests shorter than L_cap shrink the filling grids'
  // real time, not its).  When the pick takes at most two rounds, take the most splits (up to
  // twice as many) whose estimate is within 10 %: with few rounds, requests shorter than L_cap
  // would leave SMs idle unless the work is cut finer.
  constexpr long long kFixedTiles = 7, kMergeTiles = 4;
  struct Cand {
    long long chunk, np, cost, rounds;
    bool fills;
  };
  Cand cand[32];
  int nc = 0;
  for (long long s = 1; s <= 31; ++s) {
    long long chunk = (L_cap + s - 1) / s;
    chunk = (chunk + kKT - 1) / kKT * kKT;
    if (chunk < 4 * kKT) chunk = 4 * kKT;
    if (chunk > 16384) continue;
    const long long np = (L_cap + chunk - 1) / chunk;
    const long long ctas = base * np;
    const long long rounds = (ctas + num_sms - 1) / num_sms;
    const Cand c = {chunk, np, rounds * (kFixedTiles + chunk / kKT) + (np > 1 ? kMergeTiles : 0), rounds,
                    ctas >= num_sms};
    if (nc > 0 && cand[nc - 1].np == np)
      cand[nc - 1] = c;  // same split count with a smaller chunk
    else
      cand[nc++] = c;
  }
  long long best_chunk = -1, best_np = 0;
  if (nc > 0) {
    int bf = -1, bn = -1;  // cheapest filling grid, cheapest other grid
    for (int i = 0; i < nc; ++i) {
      int& bx = cand[i].fills ? bf : bn;
      if (bx < 0 || cand[i].cost < cand[bx].cost) bx = i;
    }
    const int bi = (bf < 0 || (bn >= 0 && cand[bn].cost * 115 < cand[bf].cost * 100)) ? bn : bf;
    int pick = bi;
    if (cand[bi].rounds <= 2)
      for (int i = 0; i < nc; ++i)
        if (cand[i].fills == cand[bi].fills && cand[i].np <= 2 * cand[bi].np && cand[i].np > cand[pick].np &&
            cand[i].cost * 10 <= cand[bi].cost * 11)
          pick = i;
    best_chunk = cand[pick].chunk;
    best_np = cand[pick].np;
  } else {  // very long prefixes: 16K-key chunks, doubled until 31 splits cover L_cap
    best_chunk = 16384;
    best_np = (L_cap + best_chunk - 1) / best_chunk;
    while (best_np > 31) {
      best_chunk *= 2;
      best_np = (L_cap + best_chunk - 1) / best_chunk;
    }
  }
  pl.chunk = (int)best_chunk;
  pl.n_split = (int)(best_np < 1 ? 1 : best_np);
  return pl;
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

// Static Medusa tree expansion: the top-k tokens of every Medusa head, placed on a fixed tree
// topology.  jisaku glossary "Medusa", section "ツリー構造の候補構築": the candidate tree is
// built from combinations of each head's top candidates (head 0's top-3 x head 1's top-3 x head
// 2's top-2 = 18 paths) along a predefined topology ("Medusa Tree", 63 / 127 / 255 nodes).  A
// node at depth d >= 1 with rank r carries the r-th best token of head d - 1.
//
// K5a: per (request, head, vocabulary chunk) top-k over 64-bit order keys (value, then the lower
// token id) held in registers: every warp takes its own top-k by k rounds of a warp-wide maximum
// below the previous winner, then one warp merges the warps' candidates the same way.  K5b: per request, the chunk
// candidates of every head merge into the head's top-k (one warp per head, the heads side by
// side), the topology is validated and every node's token is looked up.

#include "common.cuh"
#include "kernels.cuh"

namespace spectree {

namespace {

constexpr int kMxThreads = 256;
constexpr int kMxEpt = 16;  // vocabulary entries per thread in K5a (chunk <= 4096)

// Order key: larger is better.  Values order as floats (-0 = +0, NaN below -inf); equal values
// order by the lower token id.
__device__ __forceinline__ unsigned long long topk_key(float f, int v) {
  uint32_t u;
  if (f != f) {
    u = 0u;
  } else {
    const uint32_t b = __float_as_uint(f == 0.f ? 0.f : f);
    u = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    if (u == 0u) u = 1u;  // keep 0 for NaN
  }
  return ((unsigned long long)u << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)v);
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

// Largest of `n` keys below `below` over the warp (0 when there is none); every lane gets it.
__device__ __forceinline__ unsigned long long warp_max_below(const unsigned long long* keys, int n,
                                                             unsigned long long below) {
  unsigned long long m = 0ull;
  for (int e = 0; e < n; ++e)
    if (keys[e] < below && keys[e] > m) m = keys[e];
  return warp_max_u64(m);
}

}  // namespace

// K5a: grid (n_chunks, B * K).  Writes k keys per (row, chunk), best first (0 = none).
__global__ void __launch_bounds__(kMxThreads) medusa_chunk_topk_kernel(const MedusaParams p) {
  constexpr int kWarps = kMxThreads / 32;
  __shared__ unsigned long long s_cand[kWarps * kMaxTopk];  // [warp][rank]
  const int chunk = blockIdx.x, row = blockIdx.y;  // row = b * K + head
  const int v0 = chunk * p.chunk;
  const int v1 = min(p.V, v0 + p.chunk);
  unsigned long long keys[kMxEpt];
#pragma unroll
  for (int e = 0; e < kMxEpt; ++e) {
    const int v = v0 + e * kMxThreads + (int)threadIdx.x;
    float f = 0.f;
    bool in = v < v1;
    if (in) {
      if (p.is_bf16)
        f = __bfloat162float(static_cast<const __nv_bfloat16*>(p.logits)[(size_t)row * p.V + v]);
      else
        f = static_cast<const float*>(p.logits)[(size_t)row * p.V + v];
    }
    keys[e] = in ? topk_key(f, v) : 0ull;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  unsigned long long below = ~0ull;
  for (int r = 0; r < p.k; ++r) {  // this warp's top-k
    below = warp_max_below(keys, kMxEpt, below);
    if (lane == 0) s_cand[warp * kMaxTopk + r] = below;  // 0 once the warp's keys are exhausted
  }
  __syncthreads();
  if (warp == 0) {  // the chunk's top-k among the warps' candidates (kWarps * k <= 256)
    constexpr int kPer = kWarps * kMaxTopk / 32;
    unsigned long long c[kPer];
#pragma unroll
    for (int e = 0; e < kPer; ++e) {
      const int j = lane + 32 * e, w = j / kMaxTopk, r = j % kMaxTopk;
      c[e] = (r < p.k) ? s_cand[w * kMaxTopk + r] : 0ull;
    }
    unsigned long long* out = p.cand + ((size_t)row * p.n_chunks + chunk) * p.k;
    below = ~0ull;
    for (int r = 0; r < p.k; ++r) {
      below = warp_max_below(c, kPer, below);
      if (lane == 0) out[r] = below;  // 0 once the chunk is exhausted
    }
  }
}

// K5b: one CTA per request.
__global__ void __launch_bounds__(kMxThreads, 1) medusa_expand_kernel(const MedusaParams p) {
  __shared__ int s_top[kMaxHeads * kMaxTopk];
  __shared__ int s_par[kMaxNodes];
  __shared__ int s_depth[kMaxNodes];
  const int b = blockIdx.x, tid = threadIdx.x;
  // topology: parent[0] = -1, 0 <= parent[i] < i, depth(i) <= K heads, rank(i) < k
  int bad = 0;
  for (int i = tid; i < p.N; i += kMxThreads) {
    const int pa = p.topo_parent[i];
    s_par[i] = pa;
    if (i == 0 ? pa != -1 : (pa < 0 || pa >= i)) bad = 1;
    if (i > 0) {
      const int r = p.topo_rank[i];
      if (r < 0 || r >= p.k) bad = 1;
    }
  }
  bad = __syncthreads_or(bad);
  if (!bad) {  // depth by walking at most K + 1 parents (parents precede their children)
    for (int i = tid; i < p.N; i += kMxThreads) {
      int j = i, d = 0;
      while (j > 0 && d <= p.K) {
        j = s_par[j];
        ++d;
      }
      s_depth[i] = d;
      if (j != 0 || d > p.K) bad = 1;  // deeper than the heads reach
    }
  }
  bad = __syncthreads_or(bad);
  // every head's top-k from its chunk candidates: one warp per head, k rounds of a warp-wide
  // maximum below the previous winner (the candidates are re-read from L1 each round), so the
  // heads proceed side by side with no block barrier
  const int nc = p.n_chunks * p.k;
  const int warp = tid >> 5, lane = tid & 31;
  for (int h = warp; h < p.K; h += kMxThreads / 32) {
    const unsigned long long* c = p.cand + (size_t)(b * p.K + h) * nc;
    unsigned long long below = ~0ull;
    for (int r = 0; r < p.k; ++r) {
      unsigned long long m = 0ull;
      for (int j = lane; j < nc; j += 32) {
        const unsigned long long x = c[j];
        if (x < below && x > m) m = x;
      }
      below = warp_max_u64(m);
      if (lane == 0) {
        const int tok = below ? key_token(below) : -1;
        s_top[h * kMaxTopk + r] = tok;
        if (p.topk_index) p.topk_index[((size_t)b * p.K + h) * p.k + r] = tok;
      }
    }
  }
  __syncthreads();
  if (bad && tid == 0) set_status(p.dev_status, SPEC_ERR_BAD_TREE);
  for (int i = tid; i < p.N; i += kMxThreads) {
    int tok = 0;
    if (i == 0)
      tok = p.root_token ? p.root_token[b] : 0;
    else if (!bad)
      tok = s_top[(s_depth[i] - 1) * kMaxTopk + p.topo_rank[i]];
    p.tokens[(size_t)b * p.N + i] = bad ? 0 : tok;
    if (p.parent_out) p.parent_out[(size_t)b * p.N + i] = p.topo_parent[i];
  }
  if (tid == 0 && p.n_nodes_out) p.n_nodes_out[b] = p.N;
}

// Vocabulary chunks per head: about two CTAs per SM in all, at least one entry per thread, at
// most 4096 entries per chunk, and at most 2048 candidates (chunks x k) for the merge; 0 when
// the vocabulary needs more chunks than the merge holds.
int medusa_chunks(int B, int K, int V, int k, int num_sms) {
  const int min_chunks = (V + kMxThreads * kMxEpt - 1) / (kMxThreads * kMxEpt);
  const int cap = kMedusaMergeCands / k;
  if (min_chunks > cap) return 0;
  int want = (2 * num_sms + B * K - 1) / (B * K);
  const int max_chunks = (V + kMxThreads - 1) / kMxThreads;
  if (want > max_chunks) want = max_chunks;
  if (want > cap) want = cap;
  if (want < min_chunks) want = min_chunks;
  return want < 1 ? 1 : want;
}

void launch_row_topk_chunks(const MedusaParams& p, cudaStream_t stream) {
  medusa_chunk_topk_kernel<<<dim3(p.n_chunks, p.B * p.K), kMxThreads, 0, stream>>>(p);
}

void launch_medusa(const MedusaParams& p, cudaStream_t stream) {
  medusa_chunk_topk_kernel<<<dim3(p.n_chunks, p.B * p.K), kMxThreads, 0, stream>>>(p);
  medusa_expand_kernel<<<p.B, kMxThreads, 0, stream>>>(p);
}

}  // namespace spectree

// Dynamic (context-aware) draft tree construction in the EAGLE-2 manner: tech-tldr
// "多トークン予測（Medusa・EAGLE）", section "ツリー検証" (EAGLE-2's dynamic tree adapts the tree's
// shape to the context's confidence); jisaku glossary "Medusa", section "EAGLE: Medusaの発展形"
// (context-aware tree construction).  A node's value is the cumulative log-probability of its
// path under the draft model.
//
// K6a: one expansion layer.  Every frontier node's top-k draft tokens (the chunked top-k of K5a
// over its log-probability row, merged here by one warp per frontier row); a candidate scores its
// parent's score + log p(token) in float32; warp 0 keeps the best F' candidates as the next
// frontier.  K6b: the tree: the root plus the N - 1 best candidates of all layers (bitonic sort
// of 64-bit score keys in shared memory), numbered breadth-first by a block prefix sum.

#include "common.cuh"
#include "kernels.cuh"
#include "pdl.cuh"
#include "topk.cuh"

namespace spectree {

namespace {

constexpr int kEgThreads = 256;
constexpr int kEgPerLane = 8;           // candidate keys per lane in the warp merges (<= 256)
constexpr int kEgTreeThreads = 512;

// score key: better score first, equal scores by the lower candidate id; 0 = absent
__device__ __forceinline__ unsigned long long score_key(float s, int c) {
  return s > -INFINITY ? order_key(order_u(s), c) : 0ull;
}

}  // namespace

// K6a merge: one CTA per request.
__global__ void __launch_bounds__(kEgThreads) eagle_expand_kernel(const EagleExpandParams p) {
  __shared__ unsigned long long s_key[kEgPerLane * 32];
  const int b = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int C = p.F * p.k;
  const int nc = p.n_chunks * p.k;  // chunk candidates per frontier row (<= 256)
  const size_t ob = (size_t)b * p.cand_stride;
  pdl_wait();  // the chunk candidates of the kernel before are complete
  for (int f = warp; f < p.F; f += kEgThreads / 32) {
    const bool valid = !p.frontier_valid || p.frontier_valid[(size_t)b * p.F + f] != 0;
    const unsigned long long* cand = p.chunk_keys + (size_t)(b * p.F + f) * nc;
    unsigned long long keys[kEgPerLane];
#pragma unroll
    for (int e = 0; e < kEgPerLane; ++e) {
      const int j = lane + 32 * e;
      keys[e] = (valid && j < nc) ? cand[j] : 0ull;
    }
    const float fs = p.frontier_score[(size_t)b * p.F + f];
    const int par = p.frontier_cand ? p.frontier_cand[(size_t)b * p.F + f] : -1;
    unsigned long long below = ~0ull;
    for (int r = 0; r < p.k; ++r) {
      below = warp_max_below(keys, below);
      const int c = f * p.k + r;
      if (lane == 0) {
        int tok = -1;
        float sc = -INFINITY;
        if (valid && below) {
          tok = (int)(0xFFFFFFFFu - (uint32_t)(below & 0xFFFFFFFFull));
          sc = fs + order_value((uint32_t)(below >> 32));  // one float32 rounding
        }
        p.cand_token[ob + c] = tok;
        p.cand_score[ob + c] = sc;
        p.cand_parent[ob + c] = (tok >= 0) ? par : -1;
        s_key[c] = score_key(sc, c);
      }
    }
  }
  __syncthreads();
  if (warp == 0) {  // next frontier: the best next_k of the C <= 256 candidates
    unsigned long long keys[kEgPerLane];
#pragma unroll
    for (int e = 0; e < kEgPerLane; ++e) {
      const int j = lane + 32 * e;
      keys[e] = j < C ? s_key[j] : 0ull;
    }
    unsigned long long below = ~0ull;
    for (int r = 0; r < p.next_k; ++r) {
      below = warp_max_below(keys, below);
      if (lane == 0) {
        const int c = below ? (int)(0xFFFFFFFFu - (uint32_t)(below & 0xFFFFFFFFull)) : -1;
        p.next_index[(size_t)b * p.next_k + r] = c;
        p.next_score[(size_t)b * p.next_k + r] = c >= 0 ? order_value((uint32_t)(below >> 32)) : -INFINITY;
      }
    }
  }
}

// K6b: one CTA per request.
__global__ void __launch_bounds__(kEgTreeThreads) eagle_tree_kernel(const EagleTreeParams p) {
  __shared__ unsigned long long s_key[kEagleMaxCands];
  __shared__ int s_node[kEagleMaxCands];  // node index of each kept candidate, 0 if not kept
  __shared__ int s_warp[kEgTreeThreads / 32];
  const int b = blockIdx.x, tid = threadIdx.x;
  const int total = p.D * p.C;
  int P = 1;
  while (P < total) P <<= 1;
  const size_t cb = (size_t)b * total;
  for (int c = tid; c < P; c += kEgTreeThreads) {
    unsigned long long key = 0ull;
    if (c < total) {
      const int l = c / p.C;
      const bool present = l == 0 || p.parent[cb + c] >= 0;
      key = present ? score_key(p.score[cb + c], c) : 0ull;
    }
    s_key[c] = key;
  }
  __syncthreads();
  // bitonic sort, descending
  for (int size = 2; size <= P; size <<= 1)
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < P; i += kEgTreeThreads) {
        const int j = i ^ stride;
        if (j > i) {
          const bool desc = (i & size) == 0;
          const unsigned long long a = s_key[i], c2 = s_key[j];
          if (desc ? a < c2 : a > c2) {
            s_key[i] = c2;
            s_key[j] = a;
          }
        }
      }
      __syncthreads();
    }
  // kept candidates: the first min(N - 1, present) keys
  for (int c = tid; c < total; c += kEgTreeThreads) s_node[c] = 0;
  __syncthreads();
  const int want = p.N - 1;
  for (int r = tid; r < want && r < P; r += kEgTreeThreads) {
    const unsigned long long key = s_key[r];
    if (key) s_node[(int)(0xFFFFFFFFu - (uint32_t)(key & 0xFFFFFFFFull))] = 1;
  }
  __syncthreads();
  // breadth-first numbering: exclusive prefix sum of the flags in candidate order (layer, index);
  // thread t owns the contiguous run [t * per, t * per + per)
  const int per = (total + kEgTreeThreads - 1) / kEgTreeThreads;
  const int c0 = tid * per, c1 = min(total, c0 + per);
  int cnt = 0;
  for (int c = c0; c < c1; ++c) cnt += s_node[c];
  const int lane = tid & 31, warp = tid >> 5;
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  int base = 0, kept = 0;
  for (int w = 0; w < kEgTreeThreads / 32; ++w) {
    if (w < warp) base += s_warp[w];
    kept += s_warp[w];
  }
  int run = base + incl - cnt;
  for (int c = c0; c < c1; ++c)
    if (s_node[c]) s_node[c] = 1 + run++;
  __syncthreads();
  // closure (every kept candidate's parent kept) and token range
  int bad_tree = 0, bad_tok = 0;
  for (int c = tid; c < total; c += kEgTreeThreads) {
    if (!s_node[c]) continue;
    const int l = c / p.C;
    if (l > 0) {
      const int pc = p.parent[cb + c];
      if (pc < 0 || pc >= p.C || !s_node[(l - 1) * p.C + pc]) bad_tree = 1;
    }
    const int t = p.token[cb + c];
    if (p.d2t && (t < 0 || t >= p.Vd)) bad_tok = 1;
  }
  bad_tree = __syncthreads_or(bad_tree);
  bad_tok = __syncthreads_or(bad_tok);
  const size_t ob = (size_t)b * p.N;
  const bool bad = bad_tree || bad_tok;
  if (bad && tid == 0) set_status(p.dev_status, bad_tree ? SPEC_ERR_BAD_TREE : SPEC_ERR_BAD_TOKEN);
  for (int i = tid; i < p.N; i += kEgTreeThreads) {  // root and padding
    const bool pad = bad ? i > 0 : i > kept;
    if (i == 0 || pad) {
      p.tree_parent[ob + i] = -1;
      p.tree_token[ob + i] = (i == 0 && p.root_token) ? p.root_token[b] : 0;
      if (p.node_cand) p.node_cand[ob + i] = -1;
    }
  }
  if (tid == 0 && p.n_nodes) p.n_nodes[b] = bad ? 1 : 1 + kept;
  if (bad) return;
  for (int c = tid; c < total; c += kEgTreeThreads) {
    const int node = s_node[c];
    if (!node) continue;
    const int l = c / p.C;
    p.tree_parent[ob + node] = (l == 0) ? 0 : s_node[(l - 1) * p.C + p.parent[cb + c]];
    const int t = p.token[cb + c];
    p.tree_token[ob + node] = p.d2t ? p.d2t[t] : t;
    if (p.node_cand) p.node_cand[ob + node] = c;
  }
}

void launch_eagle_expand(const EagleExpandParams& p, const MedusaParams& chunks, cudaStream_t stream) {
  launch_row_topk_chunks(chunks, stream);
  launch_dependent(eagle_expand_kernel, dim3(p.B), dim3(kEgThreads), 0, stream, p);
}

void launch_eagle_tree(const EagleTreeParams& p, cudaStream_t stream) {
  eagle_tree_kernel<<<p.B, kEgTreeThreads, 0, stream>>>(p);
}

}  // namespace spectree

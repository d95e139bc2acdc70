// K0: tree preparation.
//
// The tree attention mask lets every draft-tree node see only its ancestors (tech-tldr
// "多トークン予測（Medusa・EAGLE）", section "ツリー検証"; qiita "EAGLE-3とMedusaで実装する
// Speculative Decoding実践ガイド", section "Tree Attention").  This kernel turns a parent array
// into the ancestor-or-self bit matrix (one 32-bit word per 32 nodes) and node depths, and
// validates the tree, the KV capacity and the tokens.  One CTA per request.

#include "common.cuh"
#include "kernels.cuh"

namespace spectree {

__global__ void __launch_bounds__(256) tree_prep_kernel(
    const int32_t* __restrict__ parent, const int32_t* __restrict__ n_nodes,
    const int32_t* __restrict__ prefix_len, long long kv_capacity, const int32_t* __restrict__ tokens,
    int vocab, int N, int W, int32_t* __restrict__ depth_out, uint32_t* __restrict__ anc_out,
    int32_t* __restrict__ bad_out, int32_t* dev_status) {
  __shared__ int s_parent[kMaxNodes];
  __shared__ uint32_t s_anc[kMaxNodes][kAncWords];
  __shared__ int s_err;
  const int b = blockIdx.x, tid = threadIdx.x;
  const int n = n_nodes[b];
  if (tid == 0) {
    int err = 0;
    if (n < 1 || n > N) err = SPEC_ERR_BAD_TREE;
    if (!err && prefix_len) {
      const long long L = prefix_len[b];
      if (L < 0 || L + n > kv_capacity) err = SPEC_ERR_CAPACITY;
    }
    s_err = err;
  }
  __syncthreads();
  for (int i = tid; i < N; i += blockDim.x) {
    const int p = parent[(size_t)b * N + i];
    s_parent[i] = p;
    if (i < n && s_err == 0) {
      const bool ok = (i == 0) ? (p == -1) : (p >= 0 && p < i);
      if (!ok) atomicCAS(&s_err, 0, SPEC_ERR_BAD_TREE);
      if (tokens && i > 0) {
        const int t = tokens[(size_t)b * N + i];
        if (t < 0 || t >= vocab) atomicCAS(&s_err, 0, SPEC_ERR_BAD_TOKEN);
      }
    }
  }
  __syncthreads();
  const int err = s_err;
  if (err) {
    if (tid == 0) {
      bad_out[b] = err;
      set_status(dev_status, err);
    }
    for (int i = tid; i < N; i += blockDim.x) {
      depth_out[(size_t)b * N + i] = -1;
      for (int w = 0; w < W; ++w) anc_out[((size_t)b * N + i) * W + w] = 0u;
    }
    return;
  }
  // Ancestor-or-self words, in topological order: lane w owns word w of every row, so each
  // row only reads words this lane wrote for an earlier row.
  if (tid < 32) {
    const int w = tid;
    if (w < W) {
      for (int i = 0; i < n; ++i) {
        uint32_t word = (i > 0) ? s_anc[s_parent[i]][w] : 0u;
        if ((i >> 5) == w) word |= 1u << (i & 31);
        s_anc[i][w] = word;
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < N; i += blockDim.x) {
    int dep = -1;
    if (i < n) {
      int cnt = 0;
      for (int w = 0; w < W; ++w) cnt += __popc(s_anc[i][w]);
      dep = cnt - 1;
    }
    depth_out[(size_t)b * N + i] = dep;
    for (int w = 0; w < W; ++w) anc_out[((size_t)b * N + i) * W + w] = (i < n) ? s_anc[i][w] : 0u;
  }
  if (tid == 0) bad_out[b] = 0;
}

void launch_tree_prep(const int32_t* parent, const int32_t* n_nodes, const int32_t* prefix_len,
                      long long kv_capacity, const int32_t* tokens, int vocab, int B, int N,
                      int32_t* depth, uint32_t* anc, int32_t* bad, int32_t* dev_status,
                      cudaStream_t stream) {
  const int W = (N + 31) / 32;
  tree_prep_kernel<<<B, 256, 0, stream>>>(parent, n_nodes, prefix_len, kv_capacity, tokens, vocab, N,
                                          W, depth, anc, bad, dev_status);
}

}  // namespace spectree

// C ABI of the static Medusa tree expansion (see include/spectree.h): argument checks, the
// workspace, the launch, and the host-side builder of the pruned Cartesian topology (jisaku
// glossary "Medusa", section "ツリー構造の候補構築").

#include <algorithm>
#include <vector>

#include "common.cuh"
#include "kernels.cuh"

namespace {

int num_sms_here() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
  return n;
}

spec_status check_medusa(const spec_medusa_args* a, int* n_chunks) {
  if (!a) return SPEC_ERR_INVALID_ARGUMENT;
  if (a->batch < 1 || a->num_heads < 1 || a->vocab < 1 || a->n_nodes < 1 || a->topk < 1)
    return SPEC_ERR_INVALID_ARGUMENT;
  if (a->dtype != SPEC_DTYPE_F32 && a->dtype != SPEC_DTYPE_BF16) return SPEC_ERR_UNSUPPORTED;
  if (a->num_heads > spectree::kMaxHeads || a->topk > spectree::kMaxTopk || a->n_nodes > SPEC_MAX_NODES)
    return SPEC_ERR_UNSUPPORTED;
  if (a->topk > a->vocab) return SPEC_ERR_INVALID_ARGUMENT;
  const int nc = spectree::medusa_chunks(a->batch, a->num_heads, a->vocab, a->topk, 1);
  if (nc == 0) return SPEC_ERR_UNSUPPORTED;
  if (n_chunks) *n_chunks = nc;
  return SPEC_OK;
}

}  // namespace

extern "C" {

size_t spec_medusa_expand_workspace(const spec_medusa_args* a) {
  int nc = 0;
  if (check_medusa(a, &nc) != SPEC_OK) return 0;
  nc = spectree::medusa_chunks(a->batch, a->num_heads, a->vocab, a->topk, num_sms_here());
  return (size_t)a->batch * a->num_heads * nc * a->topk * sizeof(unsigned long long);
}

spec_status spec_medusa_expand(const spec_medusa_args* a, void* workspace, size_t workspace_bytes,
                               int32_t* dev_status, void* stream) {
  spec_status st = check_medusa(a, nullptr);
  if (st != SPEC_OK) return st;
  if (!a->head_logits || !a->topo_parent || !a->topo_rank || !a->tokens) return SPEC_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(a->head_logits) & 15u) != 0) return SPEC_ERR_INVALID_ARGUMENT;
  if (!workspace) return SPEC_ERR_INVALID_ARGUMENT;
  spectree::MedusaParams p = {};
  p.B = a->batch; p.K = a->num_heads; p.V = a->vocab; p.N = a->n_nodes; p.k = a->topk;
  p.is_bf16 = a->dtype == SPEC_DTYPE_BF16;
  p.n_chunks = spectree::medusa_chunks(p.B, p.K, p.V, p.k, num_sms_here());
  p.chunk = spectree::topk_chunk_len(p.V, p.n_chunks);
  const size_t need = (size_t)p.B * p.K * p.n_chunks * p.k * sizeof(unsigned long long);
  if (workspace_bytes < need) return SPEC_ERR_WORKSPACE_TOO_SMALL;
  p.logits = a->head_logits;
  p.topo_parent = a->topo_parent;
  p.topo_rank = a->topo_rank;
  p.root_token = a->root_token;
  p.cand = static_cast<unsigned long long*>(workspace);
  p.tokens = a->tokens;
  p.parent_out = a->parent_out;
  p.n_nodes_out = a->n_nodes_out;
  p.topk_index = a->topk_index;
  p.dev_status = dev_status;
  spectree::launch_medusa(p, static_cast<cudaStream_t>(stream));
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status spec_medusa_topology(const int32_t* topk, int32_t K, int32_t n_nodes, int32_t* parent, int32_t* rank) {
  if (!topk || !parent || !rank || K < 1 || n_nodes < 1) return SPEC_ERR_INVALID_ARGUMENT;
  if (K > spectree::kMaxHeads || n_nodes > SPEC_MAX_NODES) return SPEC_ERR_UNSUPPORTED;
  long long total = 0, level = 1, max_sum = 0;
  for (int j = 0; j < K; ++j) {
    if (topk[j] < 1) return SPEC_ERR_INVALID_ARGUMENT;
    level = std::min<long long>(level * topk[j], 1LL << 40);
    total = std::min<long long>(total + level, 1LL << 40);
    max_sum += topk[j] - 1;
  }
  if (n_nodes - 1 > total) return SPEC_ERR_INVALID_ARGUMENT;
  // every tuple with rank sum <= S, for the smallest S that yields n_nodes - 1 of them
  using Tuple = std::vector<int>;
  std::vector<Tuple> tuples;
  for (long long S = 0;; ++S) {
    tuples.clear();
    Tuple t;
    // depth-first over tuples whose rank sum stays <= S
    struct Rec {
      static void go(const int32_t* topk, int K, long long S, long long sum, Tuple& t, std::vector<Tuple>& out) {
        if (!t.empty()) out.push_back(t);
        const int d = (int)t.size();
        if (d == K) return;
        for (int r = 0; r < topk[d] && sum + r <= S; ++r) {
          t.push_back(r);
          go(topk, K, S, sum + r, t, out);
          t.pop_back();
        }
      }
    };
    Rec::go(topk, K, S, 0, t, tuples);
    if ((long long)tuples.size() >= n_nodes - 1 || S >= max_sum) break;
  }
  auto sum_of = [](const Tuple& t) {
    long long s = 0;
    for (int r : t) s += r;
    return s;
  };
  std::sort(tuples.begin(), tuples.end(), [&](const Tuple& x, const Tuple& y) {
    const long long sx = sum_of(x), sy = sum_of(y);
    if (sx != sy) return sx < sy;
    if (x.size() != y.size()) return x.size() < y.size();
    return x < y;
  });
  tuples.resize(n_nodes - 1);
  std::sort(tuples.begin(), tuples.end(), [](const Tuple& x, const Tuple& y) {
    if (x.size() != y.size()) return x.size() < y.size();
    return x < y;
  });
  parent[0] = -1;
  rank[0] = 0;
  for (int i = 0; i < n_nodes - 1; ++i) {
    const Tuple& t = tuples[i];
    int pi = 0;
    if (t.size() > 1) {
      const Tuple pre(t.begin(), t.end() - 1);
      // the prefix is kept and precedes t in breadth-first order
      pi = 1 + (int)(std::lower_bound(tuples.begin(), tuples.begin() + i, pre,
                                      [](const Tuple& x, const Tuple& y) {
                                        if (x.size() != y.size()) return x.size() < y.size();
                                        return x < y;
                                      }) -
                     tuples.begin());
    }
    parent[i + 1] = pi;
    rank[i + 1] = t.back();
  }
  return SPEC_OK;
}

}  // extern "C"

// C ABI of the layered dynamic draft tree (see include/spectree.h): argument checks, workspace
// and launches.

#include "common.cuh"
#include "kernels.cuh"

namespace {

int eagle_chunks(int Vd) { return (Vd + 4095) / 4096; }  // K5a chunks of <= 4096 entries

spec_status check_expand(const spec_eagle_expand_args* a) {
  if (!a) return SPEC_ERR_INVALID_ARGUMENT;
  if (a->batch < 1 || a->frontier < 1 || a->draft_vocab < 1 || a->topk < 1 || a->next_k < 1 || a->reserved0 != 0)
    return SPEC_ERR_INVALID_ARGUMENT;
  if (a->frontier > 32 || a->topk > 16 || a->frontier * a->topk > 256 || a->next_k > a->frontier * a->topk)
    return SPEC_ERR_UNSUPPORTED;
  if (a->topk > a->draft_vocab) return SPEC_ERR_INVALID_ARGUMENT;
  if (eagle_chunks(a->draft_vocab) * a->topk > 256) return SPEC_ERR_UNSUPPORTED;
  if (a->cand_stride != 0 && a->cand_stride < (int64_t)a->frontier * a->topk) return SPEC_ERR_INVALID_ARGUMENT;
  return SPEC_OK;
}

}  // namespace

extern "C" {

size_t spec_eagle_expand_workspace(const spec_eagle_expand_args* a) {
  if (check_expand(a) != SPEC_OK) return 0;
  return (size_t)a->batch * a->frontier * eagle_chunks(a->draft_vocab) * a->topk * sizeof(unsigned long long);
}

spec_status spec_eagle_expand(const spec_eagle_expand_args* a, void* workspace, size_t workspace_bytes,
                              int32_t* dev_status, void* stream) {
  const spec_status st = check_expand(a);
  if (st != SPEC_OK) return st;
  if (!a->logp || !a->frontier_score || !a->cand_token || !a->cand_score || !a->cand_parent || !a->next_index ||
      !a->next_score || !workspace)
    return SPEC_ERR_INVALID_ARGUMENT;
  if ((reinterpret_cast<uintptr_t>(a->logp) & 15u) != 0) return SPEC_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < spec_eagle_expand_workspace(a)) return SPEC_ERR_WORKSPACE_TOO_SMALL;
  spectree::MedusaParams m = {};
  m.B = a->batch; m.K = a->frontier; m.V = a->draft_vocab; m.N = 1; m.k = a->topk;
  m.is_bf16 = 0;
  m.n_chunks = eagle_chunks(a->draft_vocab);
  m.chunk = spectree::topk_chunk_len(a->draft_vocab, m.n_chunks);
  m.logits = a->logp;
  m.cand = static_cast<unsigned long long*>(workspace);
  m.dev_status = dev_status;
  spectree::EagleExpandParams p = {};
  p.B = a->batch; p.F = a->frontier; p.k = a->topk; p.next_k = a->next_k; p.n_chunks = m.n_chunks;
  p.cand_stride = a->cand_stride ? (size_t)a->cand_stride : (size_t)a->frontier * a->topk;
  p.chunk_keys = m.cand;
  p.frontier_score = a->frontier_score;
  p.frontier_valid = a->frontier_valid;
  p.frontier_cand = a->frontier_cand;
  p.cand_token = a->cand_token; p.cand_score = a->cand_score; p.cand_parent = a->cand_parent;
  p.next_index = a->next_index; p.next_score = a->next_score;
  spectree::launch_eagle_expand(p, m, static_cast<cudaStream_t>(stream));
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status spec_eagle_tree(const spec_eagle_tree_args* a, int32_t* dev_status, void* stream) {
  if (!a) return SPEC_ERR_INVALID_ARGUMENT;
  if (a->batch < 1 || a->layers < 1 || a->cands < 1 || a->n_max < 1 || a->reserved0 != 0)
    return SPEC_ERR_INVALID_ARGUMENT;
  if ((long long)a->layers * a->cands > spectree::kEagleMaxCands || a->n_max > SPEC_MAX_NODES)
    return SPEC_ERR_UNSUPPORTED;
  if (!a->score || !a->token || !a->parent || !a->tree_parent || !a->tree_token) return SPEC_ERR_INVALID_ARGUMENT;
  if (a->draft_to_target && a->draft_vocab < 1) return SPEC_ERR_INVALID_ARGUMENT;
  spectree::EagleTreeParams p = {};
  p.B = a->batch; p.D = a->layers; p.C = a->cands; p.N = a->n_max; p.Vd = a->draft_vocab;
  p.score = a->score; p.token = a->token; p.parent = a->parent;
  p.d2t = a->draft_to_target; p.root_token = a->root_token;
  p.tree_parent = a->tree_parent; p.tree_token = a->tree_token; p.n_nodes = a->n_nodes; p.node_cand = a->node_cand;
  p.dev_status = dev_status;
  spectree::launch_eagle_tree(p, static_cast<cudaStream_t>(stream));
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // extern "C"

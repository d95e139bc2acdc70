// One verification round (tree attention, LM head + acceptance, KV compaction) captured into a
// CUDA graph, so that a serving loop enqueues the whole round with one launch.  The round's
// steps are those of parallel tree verification (qiita "EAGLE-3とMedusaで実装するSpeculative
// Decoding実践ガイド", sections "並列検証" and "棄却サンプリング"); the graph only removes the
// per-call host work and launch gaps between its short kernels.

#include <new>

#include "common.cuh"
#include "kernels.cuh"

struct spec_round {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
};

extern "C" spec_status spec_round_create(const spec_attn_args* attn, void* attn_workspace,
                                         size_t attn_workspace_bytes, const spec_verify_args* verify,
                                         void* verify_workspace, size_t verify_workspace_bytes,
                                         const spec_compact_args* compact, int32_t* dev_status,
                                         spec_round** out) {
  if (!out) return SPEC_ERR_INVALID_ARGUMENT;
  *out = nullptr;
  if (!attn && !verify && !compact) return SPEC_ERR_INVALID_ARGUMENT;
  // lazily initialised launch state is set up outside the capture
  if (verify && verify->rule == SPEC_RULE_REJECTION) spectree::prepare_rejection_launch();

  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return SPEC_ERR_CUDA;
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    cudaStreamDestroy(s);
    cudaGetLastError();
    return SPEC_ERR_CUDA;
  }
  spec_status st = SPEC_OK;
  if (attn) st = spec_tree_attention(attn, attn_workspace, attn_workspace_bytes, dev_status, s);
  if (st == SPEC_OK && verify) st = spec_verify_accept(verify, verify_workspace, verify_workspace_bytes, dev_status, s);
  if (st == SPEC_OK && compact) st = spec_compact_kv(compact, dev_status, s);
  cudaGraph_t graph = nullptr;
  const cudaError_t end = cudaStreamEndCapture(s, &graph);  // always ends the capture
  cudaStreamDestroy(s);
  if (st != SPEC_OK || end != cudaSuccess || !graph) {
    if (graph) cudaGraphDestroy(graph);
    cudaGetLastError();
    return st != SPEC_OK ? st : SPEC_ERR_CUDA;
  }
  cudaGraphExec_t exec = nullptr;
  if (cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) {
    cudaGraphDestroy(graph);
    cudaGetLastError();
    return SPEC_ERR_CUDA;
  }
  spec_round* r = new (std::nothrow) spec_round{graph, exec};
  if (!r) {
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(graph);
    return SPEC_ERR_CUDA;
  }
  *out = r;
  return SPEC_OK;
}

extern "C" spec_status spec_round_launch(const spec_round* round, void* stream) {
  if (!round) return SPEC_ERR_INVALID_ARGUMENT;
  return cudaGraphLaunch(round->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

extern "C" void spec_round_destroy(spec_round* round) {
  if (!round) return;
  cudaGraphExecDestroy(round->exec);
  cudaGraphDestroy(round->graph);
  delete round;
}

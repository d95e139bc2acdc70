// One verification round (tree attention, LM head + acceptance, KV compaction) captured into a
// CUDA graph, so that a serving loop enqueues the whole round with one launch.  The round's
// steps are those of parallel tree verification (qiita "EAGLE-3とMedusaで実装するSpeculative
// Decoding実践ガイド", sections "並列検証" and "棄却サンプリング"); the graph only removes the
// per-call host work and launch gaps between its short kernels.

#include <new>

#include <algorithm>

#include "common.cuh"
#include "kernels.cuh"

struct spec_round {
  cudaGraph_t graph;
  cudaGraphExec_t exec;
  // Host-buffer launches: the three calls also as graphs of their own, so that the copies that
  // feed only the verification run on `side` beside the attention (null when the round lacks
  // the attention or the verification, or when they could not be made).
  cudaGraph_t g_part[3];
  cudaGraphExec_t x_part[3];  // attention, verification, compaction (or null)
  cudaStream_t side;
  cudaEvent_t e_fork, e_join;
  cudaEvent_t e_vin, e_ain;   // the first / the second group of input copies is done
  bool verify_first;          // the verification is the longer branch: it is issued first
  uintptr_t vonly[6][2];      // [lo, hi) of the buffers only the verification reads (but draft_probs)
  int n_vonly;
  uintptr_t vshared[2][2];    // [lo, hi) of the verification's parent and n_nodes (the attention reads them too)
  // Rejection with draft distributions: their copies run on `side_d` beside the LM head, and
  // the verification is issued as direct calls whose rejection walk waits for e_draft (a wait
  // with well-defined host-order semantics, recorded afresh every launch).
  bool direct_verify;
  spec_verify_args vargs;     // the round's verification arguments, draft_ready = e_draft
  void* vws;
  size_t vws_bytes;
  int32_t* dev_status;
  cudaStream_t side_d;
  cudaEvent_t e_draft;
  uintptr_t draft[2];
};

namespace {

// One call captured into a graph of its own (null exec on failure).
template <typename F>
void capture_part(F call, cudaGraph_t* g, cudaGraphExec_t* x) {
  *g = nullptr;
  *x = nullptr;
  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) return;
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) == cudaSuccess) {
    const spec_status st = call(s);
    cudaGraph_t graph = nullptr;
    if (cudaStreamEndCapture(s, &graph) == cudaSuccess && graph && st == SPEC_OK &&
        cudaGraphInstantiate(x, graph, 0) == cudaSuccess) {
      *g = graph;
    } else {
      if (graph) cudaGraphDestroy(graph);
      *x = nullptr;
    }
  }
  cudaStreamDestroy(s);
  cudaGetLastError();
}

void release_parts(spec_round* r) {
  for (int i = 0; i < 3; ++i) {
    if (r->x_part[i]) cudaGraphExecDestroy(r->x_part[i]);
    if (r->g_part[i]) cudaGraphDestroy(r->g_part[i]);
    r->x_part[i] = nullptr;
    r->g_part[i] = nullptr;
  }
  if (r->side) cudaStreamDestroy(r->side);
  if (r->side_d) cudaStreamDestroy(r->side_d);
  if (r->e_fork) cudaEventDestroy(r->e_fork);
  if (r->e_join) cudaEventDestroy(r->e_join);
  if (r->e_draft) cudaEventDestroy(r->e_draft);
  if (r->e_vin) cudaEventDestroy(r->e_vin);
  if (r->e_ain) cudaEventDestroy(r->e_ain);
  r->side = r->side_d = nullptr;
  r->e_fork = r->e_join = r->e_draft = r->e_vin = r->e_ain = nullptr;
  r->direct_verify = false;
}

// The split launch state for a round with attention and verification; left empty (the host
// launch then copies everything before the round's graph) if any part cannot be made.
void make_parts(spec_round* r, const spec_attn_args* attn, void* attn_ws, size_t attn_ws_bytes,
                const spec_verify_args* verify, void* verify_ws, size_t verify_ws_bytes,
                const spec_compact_args* compact, int32_t* dev_status) {
  capture_part([&](cudaStream_t s) { return spec_tree_attention(attn, attn_ws, attn_ws_bytes, dev_status, s); },
               &r->g_part[0], &r->x_part[0]);
  capture_part([&](cudaStream_t s) { return spec_verify_accept(verify, verify_ws, verify_ws_bytes, dev_status, s); },
               &r->g_part[1], &r->x_part[1]);
  if (compact)
    capture_part([&](cudaStream_t s) { return spec_compact_kv(compact, dev_status, s); }, &r->g_part[2],
                 &r->x_part[2]);
  bool ok = r->x_part[0] && r->x_part[1] && (!compact || r->x_part[2]) &&
            cudaStreamCreateWithFlags(&r->side, cudaStreamNonBlocking) == cudaSuccess &&
            cudaEventCreateWithFlags(&r->e_fork, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&r->e_join, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&r->e_vin, cudaEventDisableTiming) == cudaSuccess &&
            cudaEventCreateWithFlags(&r->e_ain, cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    release_parts(r);
    cudaGetLastError();
    return;
  }
  const size_t es = verify->dtype == SPEC_DTYPE_BF16 ? 2 : 4;
  const size_t rows = (size_t)verify->batch * verify->n_max;
  auto add = [&](const void* p, size_t bytes) {
    if (!p || !bytes) return;
    r->vonly[r->n_vonly][0] = reinterpret_cast<uintptr_t>(p);
    r->vonly[r->n_vonly][1] = reinterpret_cast<uintptr_t>(p) + bytes;
    ++r->n_vonly;
  };
  r->vshared[0][0] = reinterpret_cast<uintptr_t>(verify->parent);
  r->vshared[0][1] = r->vshared[0][0] + rows * sizeof(int32_t);
  r->vshared[1][0] = reinterpret_cast<uintptr_t>(verify->n_nodes);
  r->vshared[1][1] = r->vshared[1][0] + (size_t)verify->batch * sizeof(int32_t);
  add(verify->hidden_states, rows * verify->hidden * es);
  add(verify->tokens, rows * sizeof(int32_t));
  add(verify->lm_head_weight, (size_t)verify->vocab * verify->hidden * es);
  const bool compact_draft = verify->rule == SPEC_RULE_REJECTION && verify->draft_rows;
  if (compact_draft) add(verify->draft_rows, rows * sizeof(int32_t));
  if (verify->rule == SPEC_RULE_REJECTION) add(verify->draft_to_target, (size_t)verify->draft_vocab * sizeof(int32_t));
  const size_t draft_bytes = (compact_draft ? (size_t)verify->n_draft_rows : rows) * verify->draft_vocab * sizeof(float);
  if (verify->rule == SPEC_RULE_REJECTION && verify->draft_probs && !verify->draft_ready &&
      cudaStreamCreateWithFlags(&r->side_d, cudaStreamNonBlocking) == cudaSuccess &&
      cudaEventCreateWithFlags(&r->e_draft, cudaEventDisableTiming) == cudaSuccess) {
    r->direct_verify = true;
    r->vargs = *verify;
    r->vargs.draft_ready = r->e_draft;
    r->vws = verify_ws;
    r->vws_bytes = verify_ws_bytes;
    r->dev_status = dev_status;
    r->draft[0] = reinterpret_cast<uintptr_t>(verify->draft_probs);
    r->draft[1] = r->draft[0] + draft_bytes;
  } else if (verify->rule == SPEC_RULE_REJECTION && verify->draft_probs) {
    add(verify->draft_probs, draft_bytes);
  }
  cudaGetLastError();
}

// Rough device time of each branch from its shapes, for the order of the branches only: the
// larger of its FLOPs at the tensor rate and its bytes at HBM bandwidth (nominal GB300 figures;
// only the comparison matters).  The attention's keys are taken at the cache capacity.
double attention_seconds(const spec_attn_args* a) {
  const double rows = (double)a->batch * a->n_max * a->num_q_heads;
  const double flops = 4.0 * a->head_dim * rows * (double)a->kv_capacity;
  const double es = a->dtype == SPEC_DTYPE_BF16 ? 2.0 : 4.0;
  const double bytes = 2.0 * es * a->batch * a->num_kv_heads * (double)a->kv_capacity * a->head_dim;
  return std::max(flops / 2.0e15, bytes / 7.0e12);
}
double verification_seconds(const spec_verify_args* v) {
  const double es = v->dtype == SPEC_DTYPE_BF16 ? 2.0 : 4.0;
  const double flops = 2.0 * v->batch * v->n_max * (double)v->hidden * v->vocab;
  const double bytes = es * (double)v->vocab * v->hidden;
  return std::max(flops / 2.0e15, bytes / 7.0e12);
}

}  // namespace

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

  // Tree attention and the verification read disjoint inputs, so with both present they are
  // captured as parallel branches (a second stream forked from and joined back into the capture):
  // the LM head then runs beside the split merge and fills SMs as the attention's last CTAs
  // drain.  The compaction rewrites K/V rows the attention reads, so it follows both branches and
  // is folded into the acceptance kernels only when the round has no attention call.
  const bool branch = attn && verify;
  cudaStream_t s = nullptr, s2 = nullptr;
  cudaEvent_t e_fork = nullptr, e_join = nullptr;
  auto release = [&]() {
    if (s) cudaStreamDestroy(s);
    if (s2) cudaStreamDestroy(s2);
    if (e_fork) cudaEventDestroy(e_fork);
    if (e_join) cudaEventDestroy(e_join);
  };
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess ||
      (branch && (cudaStreamCreateWithFlags(&s2, cudaStreamNonBlocking) != cudaSuccess ||
                  cudaEventCreateWithFlags(&e_fork, cudaEventDisableTiming) != cudaSuccess ||
                  cudaEventCreateWithFlags(&e_join, cudaEventDisableTiming) != cudaSuccess))) {
    release();
    cudaGetLastError();
    return SPEC_ERR_CUDA;
  }
  if (cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess) {
    release();
    cudaGetLastError();
    return SPEC_ERR_CUDA;
  }
  spec_status st = SPEC_OK;
  if (branch && (cudaEventRecord(e_fork, s) != cudaSuccess || cudaStreamWaitEvent(s2, e_fork, 0) != cudaSuccess))
    st = SPEC_ERR_CUDA;
  // The longer branch is captured (and so launched) first: its kernels take the SMs and the
  // shorter branch fills those left over, rather than the long one waiting for them.
  const bool verify_first = branch && verification_seconds(verify) >= attention_seconds(attn);
  if (st == SPEC_OK && verify_first)
    st = spec_verify_accept(verify, verify_workspace, verify_workspace_bytes, dev_status, s2);
  if (st == SPEC_OK && attn) st = spec_tree_attention(attn, attn_workspace, attn_workspace_bytes, dev_status, s);
  // a compaction of the verification's own outputs is folded into the acceptance kernels
  const bool fuse = !branch && verify && compact && compact->path == verify->path &&
                    compact->accept_len == verify->accept_len && compact->path_cap == verify->path_cap &&
                    compact->batch == verify->batch;
  if (st == SPEC_OK && fuse)
    st = spec_verify_accept_compact(verify, verify_workspace, verify_workspace_bytes, compact, dev_status, s);
  else if (st == SPEC_OK && verify && !verify_first)
    st = spec_verify_accept(verify, verify_workspace, verify_workspace_bytes, dev_status, branch ? s2 : s);
  // the join is captured even after a failure, so that the capture ends cleanly
  if (branch && (cudaEventRecord(e_join, s2) != cudaSuccess || cudaStreamWaitEvent(s, e_join, 0) != cudaSuccess) &&
      st == SPEC_OK)
    st = SPEC_ERR_CUDA;
  if (st == SPEC_OK && compact && !fuse) st = spec_compact_kv(compact, dev_status, s);
  cudaGraph_t graph = nullptr;
  const cudaError_t end = cudaStreamEndCapture(s, &graph);  // always ends the capture
  release();
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
  spec_round* r = new (std::nothrow) spec_round{};
  if (!r) {
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(graph);
    return SPEC_ERR_CUDA;
  }
  r->graph = graph;
  r->exec = exec;
  r->verify_first = verify_first;
  if (branch)
    make_parts(r, attn, attn_workspace, attn_workspace_bytes, verify, verify_workspace, verify_workspace_bytes,
               compact, dev_status);
  *out = r;
  return SPEC_OK;
}

extern "C" spec_status spec_round_launch(const spec_round* round, void* stream) {
  if (!round) return SPEC_ERR_INVALID_ARGUMENT;
  return cudaGraphLaunch(round->exec, static_cast<cudaStream_t>(stream)) == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

namespace {

spec_status check_copies(const spec_host_copy* c, int32_t n) {
  if (n < 0 || (n > 0 && !c)) return SPEC_ERR_INVALID_ARGUMENT;
  for (int32_t i = 0; i < n; ++i) {
    if (c[i].row_bytes == 0 || c[i].rows == 0) continue;  // nothing to copy
    if (!c[i].host || !c[i].device) return SPEC_ERR_INVALID_ARGUMENT;
    if (c[i].rows > 1 && (c[i].host_pitch < c[i].row_bytes || c[i].device_pitch < c[i].row_bytes))
      return SPEC_ERR_INVALID_ARGUMENT;
  }
  return SPEC_OK;
}

cudaError_t enqueue_copy(const spec_host_copy& c, bool to_device, cudaStream_t s) {
  if (c.row_bytes == 0 || c.rows == 0) return cudaSuccess;
  if (c.rows == 1)
    return to_device ? cudaMemcpyAsync(c.device, c.host, c.row_bytes, cudaMemcpyHostToDevice, s)
                     : cudaMemcpyAsync(c.host, c.device, c.row_bytes, cudaMemcpyDeviceToHost, s);
  return to_device ? cudaMemcpy2DAsync(c.device, c.device_pitch, c.host, c.host_pitch, c.row_bytes, c.rows,
                                       cudaMemcpyHostToDevice, s)
                   : cudaMemcpy2DAsync(c.host, c.host_pitch, c.device, c.device_pitch, c.row_bytes, c.rows,
                                       cudaMemcpyDeviceToHost, s);
}

}  // namespace

extern "C" spec_status spec_round_launch_host(const spec_round* round, const spec_host_copy* inputs,
                                              int32_t n_inputs, const spec_host_copy* outputs, int32_t n_outputs,
                                              void* stream) {
  spec_status st = check_copies(inputs, n_inputs);
  if (st == SPEC_OK) st = check_copies(outputs, n_outputs);
  if (st != SPEC_OK) return st;
  if (!round) return SPEC_ERR_INVALID_ARGUMENT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (round->x_part[0]) {
    // Copies into buffers that only the verification reads go on the side stream, which then
    // runs the verification beside the attention; the compaction and the result copies follow
    // both.  The side stream starts after everything enqueued on `s` so far (the previous
    // round included), so no copy overwrites a buffer still being read.
    // The copy groups take the host link one after another rather than sharing it, so that each
    // consumer starts as early as it can: the longer branch's inputs first (that branch is
    // issued first and holds the SMs it needs; the other fills the rest), then the other
    // branch's, then the draft distributions, which only the rejection walk at the end of the
    // verification reads.
    auto extent = [](const spec_host_copy& c, uintptr_t& lo, uintptr_t& hi) {
      lo = reinterpret_cast<uintptr_t>(c.device);
      hi = lo + (c.rows > 1 ? (size_t)(c.rows - 1) * c.device_pitch : 0) + c.row_bytes;
    };
    // 0: the caller's stream; 1: the verification's stream; 2: the draft distributions' stream.
    // Inputs both branches read go with the first group, which the other branch's stream waits
    // for: with the verification first, its parent and n_nodes are copied on its own stream.
    auto route = [&](const spec_host_copy& c) {
      uintptr_t lo, hi;
      extent(c, lo, hi);
      if (round->direct_verify && lo >= round->draft[0] && hi <= round->draft[1]) return 2;
      for (int k = 0; k < round->n_vonly; ++k)
        if (lo >= round->vonly[k][0] && hi <= round->vonly[k][1]) return 1;
      if (round->verify_first)
        for (int k = 0; k < 2; ++k)
          if (hi > round->vshared[k][0] && lo < round->vshared[k][1]) return 1;
      return 0;
    };
    if (cudaEventRecord(round->e_fork, s) != cudaSuccess || cudaStreamWaitEvent(round->side, round->e_fork, 0) != cudaSuccess)
      return SPEC_ERR_CUDA;
    auto copies = [&](int group, cudaStream_t on) {
      for (int32_t i = 0; i < n_inputs; ++i)
        if (route(inputs[i]) == group && enqueue_copy(inputs[i], true, on) != cudaSuccess) return false;
      return true;
    };
    const int first = round->verify_first ? 1 : 0, second = 1 - first;
    cudaStream_t on[2] = {s, round->side};
    if (!copies(first, on[first]) || cudaEventRecord(round->e_vin, on[first]) != cudaSuccess ||
        cudaStreamWaitEvent(on[second], round->e_vin, 0) != cudaSuccess || !copies(second, on[second]))
      return SPEC_ERR_CUDA;
    if (round->direct_verify &&
        (cudaEventRecord(round->e_ain, on[second]) != cudaSuccess ||
         cudaStreamWaitEvent(round->side_d, round->e_ain, 0) != cudaSuccess || !copies(2, round->side_d)))
      return SPEC_ERR_CUDA;
    // the draft distributions are complete once e_draft (recorded after their copies, before the
    // walk's wait is enqueued) completes
    if (round->direct_verify && cudaEventRecord(round->e_draft, round->side_d) != cudaSuccess) return SPEC_ERR_CUDA;
    if (!round->verify_first && cudaGraphLaunch(round->x_part[0], s) != cudaSuccess) return SPEC_ERR_CUDA;
    if (round->direct_verify) {
      const spec_status vs = spec_verify_accept(&round->vargs, round->vws, round->vws_bytes, round->dev_status, round->side);
      if (vs != SPEC_OK) return vs;
    } else if (cudaGraphLaunch(round->x_part[1], round->side) != cudaSuccess) {
      return SPEC_ERR_CUDA;
    }
    if (round->verify_first && cudaGraphLaunch(round->x_part[0], s) != cudaSuccess) return SPEC_ERR_CUDA;
    if (cudaEventRecord(round->e_join, round->side) != cudaSuccess || cudaStreamWaitEvent(s, round->e_join, 0) != cudaSuccess)
      return SPEC_ERR_CUDA;
    if (round->x_part[2] && cudaGraphLaunch(round->x_part[2], s) != cudaSuccess) return SPEC_ERR_CUDA;
  } else {
    for (int32_t i = 0; i < n_inputs; ++i)
      if (enqueue_copy(inputs[i], true, s) != cudaSuccess) return SPEC_ERR_CUDA;
    if (cudaGraphLaunch(round->exec, s) != cudaSuccess) return SPEC_ERR_CUDA;
  }
  for (int32_t i = 0; i < n_outputs; ++i)
    if (enqueue_copy(outputs[i], false, s) != cudaSuccess) return SPEC_ERR_CUDA;
  return SPEC_OK;
}

extern "C" void spec_round_destroy(spec_round* round) {
  if (!round) return;
  release_parts(round);
  cudaGraphExecDestroy(round->exec);
  cudaGraphDestroy(round->graph);
  delete round;
}

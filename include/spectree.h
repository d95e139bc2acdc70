/*
 * spectree.h -- tree verification for Medusa/EAGLE-style speculative decoding on one GB300
 * (sm_103a).  C ABI of libspectree.so.
 *
 * What the three calls compute (sources are cited by page title and section):
 *
 *   spec_tree_attention  One target-model attention layer over a draft tree.  Every tree node
 *       attends to the request's KV-cache prefix plus only its own ancestors and itself
 *       (tech-tldr "多トークン予測（Medusa・EAGLE）", section "ツリー検証"; qiita "EAGLE-3と
 *       Medusaで実装するSpeculative Decoding実践ガイド", sections "並列検証" and "Tree Attention").
 *   spec_verify_accept   The LM head z = W h at every node (tech-tldr, section "Medusa": linear
 *       layer + softmax), then per-node acceptance by one of three rules -- greedy argmax match;
 *       typical acceptance (jisaku glossary "Medusa", section "Medusa-1: 典型的採択");
 *       rejection sampling with min(1, T[x]/D[x]) and resampling from norm(relu(T - D)) (qiita,
 *       section "棄却サンプリング") -- and the longest accepted root path plus a bonus token.
 *   spec_compact_kv      Keeps the accepted path's K/V entries right after the prefix (qiita,
 *       section "棄却サンプリング": everything after a rejection is discarded).
 *   spec_medusa_expand   Builds the draft tree the verification consumes from the top-k of
 *       every Medusa head along a static topology (jisaku glossary "Medusa", section
 *       "ツリー構造の候補構築").
 *   spec_eagle_expand / spec_eagle_tree  Build a dynamic draft tree layer by layer from the
 *       draft model's log-probabilities, EAGLE-2 style (tech-tldr, section "ツリー検証").
 *
 * Conventions shared by every call
 *   - Node 0 of a tree is its root (the last accepted token); parent[0] = -1 and
 *     0 <= parent[i] < i for 0 < i < n_nodes[b], so nodes are in topological order and siblings
 *     are ordered by index.  Entries at i >= n_nodes[b] are padding and are ignored.
 *   - KV cache layout [B][Hkv][L_cap][head_dim]: request b's prefix occupies slots
 *     [0, prefix_len[b]); tree node i occupies slot prefix_len[b] + i.
 *   - All array arguments are caller-owned, contiguous, row-major DEVICE memory with 16-byte
 *     aligned base addresses.  The three calls never allocate: scratch space is the caller's
 *     `workspace`, sized by the matching *_workspace() query, and every call may be issued from
 *     any host thread.  (spec_round_create, below, has the driver build a CUDA graph.)
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *   - Errors found on the host (NULL pointer, unsupported size or dtype, short workspace) are
 *     returned before anything is launched.  Errors that depend on device data (a bad parent
 *     array, prefix_len + n_nodes > L_cap, a token outside the vocabulary, an accepted path
 *     longer than path_cap) are written to *dev_status with first-error-wins semantics
 *     (atomicCAS from SPEC_OK); the offending request's outputs are zeroed (attention rows 0;
 *     accept_len 0, path {0, -1, ...}, bonus -1).  The caller zeroes *dev_status before the
 *     calls it wants checked and reads it after synchronising.  No kernel traps; every wait
 *     inside a kernel is bounded and reports SPEC_ERR_TIMEOUT instead of hanging.
 */
#ifndef SPECTREE_H_
#define SPECTREE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t spec_status;

#define SPEC_OK 0
#define SPEC_ERR_INVALID_ARGUMENT 1   /* host: NULL pointer, non-positive or inconsistent size */
#define SPEC_ERR_UNSUPPORTED 2        /* host: dtype / head_dim / size outside what is built */
#define SPEC_ERR_WORKSPACE_TOO_SMALL 3 /* host: workspace_bytes below the *_workspace() query */
#define SPEC_ERR_BAD_TREE 4           /* device: parent array is not a valid rooted tree */
#define SPEC_ERR_CUDA 5               /* host: a CUDA runtime call failed (launch, attribute) */
#define SPEC_ERR_BAD_TOKEN 6          /* device: token or draft map entry outside the vocabulary,
                                         or a node with children without a draft row */
#define SPEC_ERR_CAPACITY 7           /* device: prefix_len + n_nodes > L_cap, or a path longer
                                         than path_cap */
#define SPEC_ERR_TIMEOUT 8            /* device: a bounded wait in a kernel ran out */

#define SPEC_DTYPE_F32 0   /* float32 tensors (exact path; SIMT kernels) */
#define SPEC_DTYPE_BF16 1  /* bfloat16 tensors, float32 accumulation (tensor-core kernels) */

#define SPEC_RULE_GREEDY 0
#define SPEC_RULE_TYPICAL 1
#define SPEC_RULE_REJECTION 2

#define SPEC_MAX_NODES 255 /* n_max limit (the largest Medusa tree named on the pages) */

/* ---------------------------------------------------------------------------------------
 * Tree attention.
 *
 * For request b, query head h, node i < n_nodes[b], with G = Hq / Hkv and KV head g = h / G:
 *   visible(i) = prefix slots [0, L_b)  +  tree slots {L_b + a : a ancestor of i, or a = i}
 *   out[b][i][h] = sum_j softmax_j(scale * q[b][i][h] . k[b][g][j]) v[b][g][j]   (j visible)
 *   lse[b][i][h] = ln sum_j exp(scale * q[b][i][h] . k[b][g][j])
 * Padded nodes (i >= n_nodes[b]) get out = 0 and lse = 0.
 * ------------------------------------------------------------------------------------- */
typedef struct spec_attn_args {
  int32_t dtype;          /* SPEC_DTYPE_F32 or SPEC_DTYPE_BF16 (q, caches and out) */
  int32_t batch;          /* B >= 1 */
  int32_t n_max;          /* N, padded nodes per request incl. root, 1..SPEC_MAX_NODES */
  int32_t num_q_heads;    /* Hq, a multiple of num_kv_heads */
  int32_t num_kv_heads;   /* Hkv >= 1 */
  int32_t head_dim;       /* d: 64 or 128 */
  int64_t kv_capacity;    /* L_cap, slots per (request, KV head) in the caches */
  float scale;            /* softmax scale; <= 0 selects 1/sqrt(head_dim) */
  int32_t schedule;       /* SPEC_ATTN_SPLIT_KV (0) or SPEC_ATTN_STREAM_K (1), see below */
  const void* q;          /* [B][N][Hq][d] */
  const void* k_cache;    /* [B][Hkv][L_cap][d] */
  const void* v_cache;    /* [B][Hkv][L_cap][d] */
  const int32_t* prefix_len; /* [B], L_b >= 0 */
  const int32_t* n_nodes;    /* [B], 1 <= n_b <= N */
  const int32_t* parent;     /* [B][N] */
  void* out;              /* [B][N][Hq][d], same dtype as q */
  float* lse;             /* [B][N][Hq] natural-log LSE, or NULL */
  void* timing_begin;     /* optional cudaEvent_t recorded on `stream` right before the split-KV
                             attention kernel (bf16) or the fp32 attention kernel; NULL = none */
  void* timing_end;       /* optional cudaEvent_t recorded right after that kernel */
  /* Paged KV cache (block_table != NULL; bf16 only).  k_cache / v_cache are then pools
   * [num_blocks][Hkv][block_size][d], and request b's logical slot s (prefix at [0, L_b), tree
   * node i at L_b + i, as above) is row s % block_size of block block_table[b][s / block_size].
   * kv_capacity must equal max_blocks * block_size.  A table entry outside [0, num_blocks) among
   * the blocks covering [0, L_b + n_b) sets SPEC_ERR_CAPACITY and zeroes that request's outputs
   * (nothing outside the pools is read).  Blocks may be shared between requests (read only). */
  const int32_t* block_table; /* [B][max_blocks], or NULL for the contiguous layout above */
  int32_t block_size;     /* 16, 32, 64, 128 or 256 */
  int32_t max_blocks;     /* table entries per request */
  int32_t num_blocks;     /* blocks per pool; num_blocks * Hkv < 2^31 */
  int32_t reserved1;      /* must be 0 */
} spec_attn_args;

/* Work schedules of the bf16 kernels (the results are the same up to rounding):
 *   SPEC_ATTN_SPLIT_KV  one CTA per (request, KV head, key split, 256 rows), the key splits chosen
 *                       on the host from kv_capacity and merged by a second kernel when there
 *                       are several.  Every layout and size.
 *   SPEC_ATTN_STREAM_K  a persistent kernel, one CTA per SM, each taking an equal share of all
 *                       key tiles; partially covered (request, KV head, row block) segments are
 *                       merged by the last CTA to finish one.  Contiguous bf16 caches, Hq / Hkv
 *                       dividing 128, batch <= 1024; SPEC_ERR_UNSUPPORTED otherwise.  Balances
 *                       batches of very uneven prefixes without a host-side plan, but pays at
 *                       every segment boundary for partial stores and reloads, which the split
 *                       kernel does not. */
#define SPEC_ATTN_SPLIT_KV 0
#define SPEC_ATTN_STREAM_K 1

/* Bytes of workspace spec_tree_attention needs for these shapes (0 on invalid args).  The
 * workspace (device memory, 16-byte aligned: the split partials are written there by bulk
 * copies; SPEC_ERR_INVALID_ARGUMENT otherwise) holds the per-split partial outputs. */
size_t spec_tree_attention_workspace(const spec_attn_args* args);

spec_status spec_tree_attention(const spec_attn_args* args, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------------------------
 * LM head, acceptance, longest accepted path, bonus token.
 *
 * z[b][i] = lm_head_weight . hidden_states[b][i] (no bias), for every real node.  Node c != 0
 * carries tokens[b][c] and is judged with the distribution at its parent p = parent[b][c]:
 *   GREEDY     accept iff tokens[c] == argmax_v z[p][v] (lowest index on ties).
 *   TYPICAL    p_p = softmax(z[p] / temperature), H = -sum p_p ln p_p (nats);
 *              accept iff p_p(x) >= min(eps, delta * exp(-H)).
 *   REJECTION  walk from the root: R = softmax(z[e] / temperature); for each child c of e in
 *              index order, u = U(seed, b, c, 0): accept iff u < min(1, R[x] / D_e[x]) (ratio 1
 *              when D_e[x] = 0 < R[x], 0 when both are 0); on acceptance e = c and R restarts
 *              from e's distribution; on rejection R = relu(R - D_e) / sum (kept if the sum is 0).
 *              D_e = draft_probs[b][e], scattered into the target vocabulary by
 *              draft_to_target (zero outside the map).
 * Path: greedy/typical take the deepest node whose whole root chain is accepted (lowest index
 * on ties); rejection takes the walk's last node e.  accept_len = depth(e); path = root..e.
 * Bonus token: argmax z[e] (greedy/typical); for rejection the inverse-CDF sample of R at
 * u' = U(seed, b, e, 1) -- the smallest j with sum_{v<=j} R[v] > u' sum R.
 * U(seed, b, node, purpose) = (2 * (x0 >> 9) + 1) * 2^-24 where x0 is the first output word of
 * Philox4x32-10 (Salmon et al., SC'11) with key (seed & 0xffffffff, seed >> 32) and counter
 * (b, node, purpose, 0).
 * Margin cases -- decisions within 1e-4 of their threshold (greedy: top-2 logit gap; typical:
 * |ln p(x) - ln thr|; rejection: |u - min(1, R[x]/D[x])|) among the decisions the walk
 * evaluates -- are counted in margin_count; bonus_margin flags a bonus decision within 1e-4
 * (greedy/typical: top-2 gap of z[e]; rejection: u' sum R within 1e-4 sum R of a cumulative
 * boundary).
 * ------------------------------------------------------------------------------------- */
typedef struct spec_verify_args {
  int32_t dtype;          /* dtype of hidden_states and lm_head_weight */
  int32_t batch;          /* B >= 1 */
  int32_t n_max;          /* N, 1..SPEC_MAX_NODES */
  int32_t hidden;         /* Hd: a multiple of 64 for BF16, of 4 for F32 */
  int32_t vocab;          /* V >= 2 */
  int32_t rule;           /* SPEC_RULE_* */
  float temperature;      /* tau > 0 for TYPICAL / REJECTION; ignored by GREEDY */
  float eps;              /* TYPICAL: epsilon */
  float delta;            /* TYPICAL: delta */
  int32_t draft_vocab;    /* REJECTION: Vd (= vocab when draft_to_target is NULL) */
  int32_t path_cap;       /* entries per request in `path`: >= deepest accepted depth + 1 */
  int32_t reserved0;      /* must be 0 */
  uint64_t seed;          /* key of the acceptance uniforms */
  const void* hidden_states;      /* [B][N][Hd] */
  const void* lm_head_weight;     /* [V][Hd] (each vocab row contiguous in Hd) */
  const int32_t* tokens;          /* [B][N] target-vocab ids (entry 0 unused) */
  const int32_t* parent;          /* [B][N] */
  const int32_t* n_nodes;         /* [B] */
  const float* draft_probs;       /* REJECTION: [B][N][Vd]; row e = distribution of e's children
                                     (compact [n_draft_rows][Vd] with draft_rows, below) */
  const int32_t* draft_to_target; /* REJECTION: [Vd] injective map into [0, V), or NULL */
  int32_t* accept_len;            /* out [B] */
  int32_t* path;                  /* out [B][path_cap], -1 padded */
  int32_t* bonus_token;           /* out [B] */
  int32_t* margin_count;          /* out [B] or NULL */
  int32_t* bonus_margin;          /* out [B] (0/1) or NULL */
  float* row_max;                 /* optional out [B][N]: max_v z/tau (z for GREEDY) */
  float* row_lse;                 /* optional out [B][N]: ln sum exp(z/tau) */
  float* row_entropy;             /* optional out [B][N]: H in nats */
  int32_t* row_argmax;            /* optional out [B][N]: argmax_v z */
  void* timing_begin;             /* optional cudaEvent_t recorded on `stream` right before the
                                     LM-head kernel; NULL = none */
  void* timing_end;               /* optional cudaEvent_t recorded right after it */
  void* draft_ready;              /* REJECTION, optional cudaEvent_t: the rejection walk (the only
                                     reader of draft_probs) waits for it, so the distributions may
                                     still be arriving while the LM head runs; NULL = none.  Inside
                                     a stream capture the wait is captured as an external one. */
  const int32_t* draft_rows;      /* REJECTION, optional [B][N]: with it, draft_probs is a compact
                                     [n_draft_rows][Vd] array and node e's distribution is row
                                     draft_rows[b][e]; nodes without children may hold -1.  A
                                     dynamic tree expands only some of its nodes (the EAGLE-2
                                     reading of tech-tldr, section "ツリー検証"), so only their rows
                                     need to exist and travel.  NULL = draft_probs is [B][N][Vd]. */
  int32_t n_draft_rows;           /* rows of draft_probs when draft_rows != NULL (>= 1) */
  int32_t reserved1;              /* must be 0 */
} spec_verify_args;

/* Bytes of workspace spec_verify_accept needs for these shapes (0 on invalid args).  The
 * workspace (device memory, 16-byte aligned: statistics records and fp32 logits are stored there
 * as 16-byte vectors; SPEC_ERR_INVALID_ARGUMENT otherwise) holds the LM head's per-row records,
 * the row statistics and, for rejection sampling, the fp32 logits. */
size_t spec_verify_accept_workspace(const spec_verify_args* args);

spec_status spec_verify_accept(const spec_verify_args* args, void* workspace,
                               size_t workspace_bytes, int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------------------------
 * KV compaction (in place).  For j = 0..accept_len[b]:
 *   K/V[b][g][L_b + j] <- K/V[b][g][L_b + path[b][j]] for every KV head g (reads see the
 *   cache as it was before the call), src_slot[b][j] = L_b + path[b][j] (-1 beyond),
 *   new_len[b] = L_b + 1 + accept_len[b].
 * A path that is not a root path of increasing node indices, or that leaves the cache, sets
 * SPEC_ERR_BAD_TREE / SPEC_ERR_CAPACITY and leaves that request's cache untouched.
 * ------------------------------------------------------------------------------------- */
typedef struct spec_compact_args {
  int32_t dtype;          /* element type of the caches */
  int32_t batch;
  int32_t num_kv_heads;
  int32_t head_dim;       /* 64 or 128 */
  int64_t kv_capacity;    /* L_cap */
  int32_t path_cap;
  int32_t reserved0;      /* must be 0 */
  void* k_cache;          /* [B][Hkv][L_cap][d], updated in place */
  void* v_cache;
  const int32_t* prefix_len;  /* [B] */
  const int32_t* path;        /* [B][path_cap] */
  const int32_t* accept_len;  /* [B] */
  int32_t* src_slot;          /* out [B][path_cap] or NULL (logical slots) */
  int32_t* new_len;           /* out [B] or NULL */
  /* Paged KV cache, as in spec_attn_args (either dtype): slots are logical, moved between the
   * physical rows the table maps them to; a table entry outside [0, num_blocks) among the
   * blocks the request's moves touch sets SPEC_ERR_CAPACITY and moves nothing for it.  Requests
   * must not share the blocks that hold their tree slots. */
  const int32_t* block_table; /* [B][max_blocks] or NULL */
  int32_t block_size;         /* 16, 32, 64, 128 or 256 */
  int32_t max_blocks;
  int32_t num_blocks;
  int32_t reserved1;          /* must be 0 */
} spec_compact_args;

spec_status spec_compact_kv(const spec_compact_args* args, int32_t* dev_status, void* stream);

/* spec_verify_accept followed by spec_compact_kv of its own outputs, with the compaction folded
 * into the kernel that decides each request (the last row-statistics block of the request for
 * greedy / typical acceptance, the end of the rejection walk), so the round has one launch less.
 * (qiita, section "棄却サンプリング": the accepted prefix is kept, everything after a rejection is
 * discarded; which kernel performs the move is not part of the method.)
 * `compact` must name the verification's outputs: compact->path == verify->path,
 * compact->accept_len == verify->accept_len, equal path_cap and batch; SPEC_ERR_INVALID_ARGUMENT
 * otherwise.  Results (accept_len, path, bonus, margins, the caches, src_slot, new_len, device
 * status codes) are exactly those of the two calls in sequence.  Workspace: as
 * spec_verify_accept_workspace(verify). */
spec_status spec_verify_accept_compact(const spec_verify_args* verify, void* workspace, size_t workspace_bytes,
                                       const spec_compact_args* compact, int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------------------------
 * spec_verify_accept without a caller workspace.  (The pages have no counterpart: this is a
 * deployment convenience, not part of the method.)
 *
 * For callers that cannot allocate device memory themselves -- for example code running inside
 * a host framework's callback or plugin that has no access to the framework's allocator, or a
 * latency-critical loop where cudaMalloc would synchronise the device -- this entry point runs
 * exactly spec_verify_accept, but takes its scratch space from a fixed array of
 * SPEC_NOALLOC_SCRATCH_BYTES bytes that lives in device memory for as long as the library is
 * loaded (every GPU that loads the library holds it until process exit).  It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *   - Inputs and outputs are the caller's device memory, as for spec_verify_accept.
 *   - Shapes whose spec_verify_accept_workspace() exceeds SPEC_NOALLOC_SCRATCH_BYTES are
 *     rejected with SPEC_ERR_WORKSPACE_TOO_SMALL before anything is launched (at a 128256-token
 *     vocabulary this fits greedy / typical verification of up to a few hundred tree rows;
 *     rejection sampling keeps fp32 logits and fits only small rows x vocabulary products).
 *   - Calls look up the array's device address on the current device (a cheap runtime query)
 *     and remember it per device.  While `stream` is being captured the remembered address is
 *     used instead, so make one call on the device before any stream capture.  A device reset
 *     (cudaDeviceReset) invalidates the remembered address; the next call outside a capture
 *     looks it up again.
 *   - All calls on a device share the one array and it keeps the last call's contents; every
 *     call overwrites what it reads.  Calls whose kernels overlap on the GPU (different streams,
 *     or different host threads without ordering) race on the array and must not be issued.
 * Other errors are those of spec_verify_accept. */
#define SPEC_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

spec_status spec_verify_accept_noalloc(const spec_verify_args* args, int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------------------------
 * Static Medusa tree expansion (jisaku glossary "Medusa", section "ツリー構造の候補構築": the
 * candidate tree combines the top candidates of every Medusa head -- head 0's top-3 x head 1's
 * top-3 x head 2's top-2 gives 18 paths -- along a predefined topology of 63 / 127 / 255 nodes).
 *
 * Head j (0 <= j < K) predicts the token j + 1 steps ahead.  Its candidates are its top-k
 * logits, best first, equal logits ordered by the lower token id (-0 = +0; NaN ranks below
 * -inf).  A topology node i >= 1 at depth d(i) (edges from the root) with rank r(i) carries
 * head d(i) - 1's candidate r(i):
 *   tokens[b][i] = topk(head_logits[b][d(i) - 1])[r(i)],   tokens[b][0] = root_token[b] (or 0)
 * and parent_out[b][i] = topo_parent[i], so the outputs feed spec_verify_accept directly.
 * The topology is shared by every request: topo_parent[0] = -1, 0 <= topo_parent[i] < i,
 * 1 <= d(i) <= K and 0 <= topo_rank[i] < topk for i >= 1; a topology that breaks this sets
 * SPEC_ERR_BAD_TREE and writes tokens 0.  (spec_medusa_topology builds the pruned Cartesian
 * topology on the host.)
 * Host errors: SPEC_ERR_INVALID_ARGUMENT (sizes < 1, NULL logits / topology / tokens, topk > V,
 * unaligned logits), SPEC_ERR_UNSUPPORTED (K > 16, topk > 32, N > 255, or
 * V > 4096 * floor(2048 / topk)), SPEC_ERR_WORKSPACE_TOO_SMALL. */
typedef struct spec_medusa_args {
  int32_t dtype;              /* head logits: SPEC_DTYPE_F32 or SPEC_DTYPE_BF16 */
  int32_t batch;              /* B */
  int32_t num_heads;          /* K, 1..16 */
  int32_t vocab;              /* V */
  int32_t n_nodes;            /* N, topology nodes including the root, 1..255 */
  int32_t topk;               /* candidates per head, 1..32 */
  const void* head_logits;    /* [B][K][V] */
  const int32_t* topo_parent; /* [N] */
  const int32_t* topo_rank;   /* [N] (entry 0 unused) */
  const int32_t* root_token;  /* [B] or NULL */
  int32_t* tokens;            /* out [B][N] */
  int32_t* parent_out;        /* out [B][N] or NULL */
  int32_t* n_nodes_out;       /* out [B] (all N) or NULL */
  int32_t* topk_index;        /* out [B][K][topk] or NULL: every head's candidates, best first */
} spec_medusa_args;

size_t spec_medusa_expand_workspace(const spec_medusa_args* args);
spec_status spec_medusa_expand(const spec_medusa_args* args, void* workspace, size_t workspace_bytes,
                               int32_t* dev_status, void* stream);

/* Host-side helper (no GPU): the Cartesian topology of per-head candidate counts topk[0..K-1],
 * pruned to n_nodes nodes.  Nodes are rank tuples (r_0, ..., r_{d-1}), r_j < topk[j]; the kept
 * ones are the first n_nodes - 1 in the order (sum of ranks, depth, tuple), which keeps every
 * prefix of a kept tuple; they are numbered breadth-first (depth, then tuple) after the root, so
 * siblings are contiguous and ordered by rank.  Writes HOST arrays parent[n_nodes] and
 * rank[n_nodes] (rank[0] = 0).  SPEC_ERR_INVALID_ARGUMENT for K < 1, a count < 1, n_nodes < 1 or
 * beyond 1 + the number of tuples, or NULL outputs; SPEC_ERR_UNSUPPORTED beyond 255 nodes or
 * 16 heads. */
spec_status spec_medusa_topology(const int32_t* topk, int32_t num_heads, int32_t n_nodes, int32_t* parent,
                                 int32_t* rank);

/* ---------------------------------------------------------------------------------------
 * Dynamic (context-aware) draft tree, layer by layer, in the EAGLE-2 manner (tech-tldr
 * "多トークン予測（Medusa・EAGLE）", section "ツリー検証": EAGLE-2's dynamic tree shapes the tree
 * by the context's confidence; jisaku glossary "Medusa", section "EAGLE: Medusaの発展形").  A
 * node's value is the cumulative log-probability of its path under the draft model.  The draft
 * model itself runs between the layers, outside this library.
 *
 * spec_eagle_expand, one layer: frontier node f of request b (F per request) proposes its topk
 * best draft tokens by logp[b][f][:] (equal log-probabilities by the lower token id).  Candidate
 * c = f * topk + r gets token = the r-th token, score = frontier_score[b][f] + logp (one float32
 * addition), parent = frontier_cand[b][f] (-1 when frontier_cand is NULL); a frontier row with
 * frontier_valid 0 gives token -1, score -inf, parent -1.  The next frontier is the next_k best
 * candidates (score, then lower c), -1 / -inf padded; candidates with score -inf or NaN are
 * never chosen.  Candidate rows of request b start at element b * cand_stride (0 = F * topk), so
 * a caller can write every layer into one [B][layers][cands] array.
 * Host errors: SPEC_ERR_INVALID_ARGUMENT (sizes, NULL pointers, topk > draft_vocab,
 * cand_stride < F * topk), SPEC_ERR_UNSUPPORTED (F > 32, topk > 16, F * topk > 256, next_k >
 * F * topk, draft_vocab > 4096 * floor(256 / topk)), SPEC_ERR_WORKSPACE_TOO_SMALL. */
typedef struct spec_eagle_expand_args {
  int32_t batch;                  /* B */
  int32_t frontier;               /* F */
  int32_t draft_vocab;            /* Vd */
  int32_t topk;                   /* children per frontier node */
  int32_t next_k;                 /* frontier size of the next layer */
  int32_t reserved0;              /* must be 0 */
  int64_t cand_stride;            /* elements between requests' candidate rows; 0 = F * topk */
  const float* logp;              /* [B][F][Vd] draft log-probabilities */
  const float* frontier_score;    /* [B][F] */
  const int32_t* frontier_valid;  /* [B][F] or NULL (all valid) */
  const int32_t* frontier_cand;   /* [B][F] or NULL: each frontier node's candidate index in the previous layer */
  int32_t* cand_token;            /* out [B][stride] */
  float* cand_score;              /* out [B][stride] */
  int32_t* cand_parent;           /* out [B][stride] */
  int32_t* next_index;            /* out [B][next_k] candidate indices, best first */
  float* next_score;              /* out [B][next_k] */
} spec_eagle_expand_args;

size_t spec_eagle_expand_workspace(const spec_eagle_expand_args* args);
spec_status spec_eagle_expand(const spec_eagle_expand_args* args, void* workspace, size_t workspace_bytes,
                              int32_t* dev_status, void* stream);

/* spec_eagle_tree: the draft tree of each request from all layers' candidates, stacked as
 * [B][layers][cands] (candidate (l, j); on layer l > 0, parent = its candidate index on layer
 * l - 1, -1 = absent; a score of -inf or NaN = absent).  The tree is the root plus the n_max - 1
 * best present candidates (score, then lower (l, j)), numbered breadth-first by (l, j) after the
 * root: tree_parent[0] = -1, tree_token[0] = root_token[b] (0 if NULL), tokens mapped through
 * draft_to_target when given; padding nodes get parent -1, token 0; node_cand = l * cands + j
 * (-1 for the root and padding).  Outputs feed spec_verify_accept (n_nodes, parent, tokens).
 * Scores must not increase from a candidate to its child (true for cumulative log-probabilities);
 * a kept candidate whose parent is not kept sets SPEC_ERR_BAD_TREE, a token outside
 * [0, draft_vocab) with a map SPEC_ERR_BAD_TOKEN; either leaves the request a lone root.
 * Host errors: SPEC_ERR_INVALID_ARGUMENT, SPEC_ERR_UNSUPPORTED (layers * cands > 2048,
 * n_max > 255). */
typedef struct spec_eagle_tree_args {
  int32_t batch;
  int32_t layers;                 /* D */
  int32_t cands;                  /* C, candidates per layer */
  int32_t n_max;                  /* N, tree nodes including the root */
  int32_t draft_vocab;            /* Vd (range of tokens when draft_to_target is given) */
  int32_t reserved0;              /* must be 0 */
  const float* score;             /* [B][D][C] */
  const int32_t* token;           /* [B][D][C] draft-vocabulary ids */
  const int32_t* parent;          /* [B][D][C] */
  const int32_t* draft_to_target; /* [Vd] or NULL */
  const int32_t* root_token;      /* [B] or NULL */
  int32_t* tree_parent;           /* out [B][N] */
  int32_t* tree_token;            /* out [B][N] */
  int32_t* n_nodes;               /* out [B] */
  int32_t* node_cand;             /* out [B][N] or NULL */
} spec_eagle_tree_args;

spec_status spec_eagle_tree(const spec_eagle_tree_args* args, int32_t* dev_status, void* stream);

/* ---------------------------------------------------------------------------------------
 * One verification round as a single CUDA-graph launch.  (Deployment convenience: the pages
 * describe the round's steps -- parallel tree verification, acceptance, keeping the accepted
 * prefix -- not how they are launched.  At batch 1 the round is a handful of short kernels
 * around the LM head, so per-call host work and launch gaps are a visible share of it.)
 *
 * spec_round_create captures spec_tree_attention(attn, attn_workspace), spec_verify_accept(verify,
 * verify_workspace) and spec_compact_kv(compact) into a CUDA graph and instantiates it.  With
 * both `attn` and `verify` given, the two run as parallel branches of the graph (they read
 * disjoint inputs), the one that the shapes make longer (FLOPs at the tensor rate against bytes
 * at HBM bandwidth, keys taken at kv_capacity) captured first so that its kernels take the SMs
 * and the other fills those left over; the compaction follows both, since it rewrites K/V rows
 * the attention reads.  Without `attn`,
 * a `compact` that names the verification's outputs (same path, accept_len, path_cap and batch)
 * is captured with it as spec_verify_accept_compact.  Any of the three may be NULL to leave that
 * call out; at least one must be given.  Because of the branches, `attn` and `verify` must not
 * share output or workspace buffers, and the attention's out / lse must not alias the
 * verification's inputs.
 *   - Everything in the argument structs is frozen at creation: device pointers, shapes,
 *     scalars (rule, temperature, eps, delta, seed), dev_status and the optional timing events.
 *     The CONTENTS of the device buffers are read when the round runs, so a serving loop refills
 *     q / hidden_states / tokens / parent / n_nodes / prefix_len / draft_probs / the caches in
 *     place and launches again.  The argument structs themselves may be freed after creation.
 *   - Host-side validation runs at creation: the status of the first call that rejects its
 *     arguments is returned, and no round is made (*out = NULL).
 *   - The workspaces and every buffer named in the arguments must stay allocated until
 *     spec_round_destroy, and must not be used by other work that overlaps a running round.
 *   - spec_round_launch enqueues the whole round on `stream` (one cudaGraphLaunch).  Device-side
 *     errors reach dev_status exactly as for the individual calls.  Rounds of one spec_round
 *     must not overlap each other on the GPU (they share the workspaces).
 *   - Creation captures a private stream in thread-local mode; do not call it while the calling
 *     thread is capturing another stream.
 * Errors: SPEC_ERR_INVALID_ARGUMENT (no call given, or out == NULL / round == NULL),
 * SPEC_ERR_CUDA (capture, instantiation or launch failed), or a captured call's host-side
 * status.  spec_round_destroy(NULL) does nothing. */
typedef struct spec_round spec_round;

spec_status spec_round_create(const spec_attn_args* attn, void* attn_workspace, size_t attn_workspace_bytes,
                              const spec_verify_args* verify, void* verify_workspace,
                              size_t verify_workspace_bytes, const spec_compact_args* compact,
                              int32_t* dev_status, spec_round** out);
spec_status spec_round_launch(const spec_round* round, void* stream);
void spec_round_destroy(spec_round* round);

/* One round end to end from host memory: the step's inputs are copied in, the round runs, and
 * its results are copied out, all enqueued by one call and complete in `stream` order.
 * (Deployment convenience, like the round itself: the pages describe what a round computes, not
 * where its inputs come from.)  When the round has both tree attention and verification, a copy
 * whose destination lies wholly inside a buffer only the verification reads (hidden_states,
 * tokens, lm_head_weight, draft_probs, draft_rows, draft_to_target) goes to a stream of the
 * round's own: it starts after everything already enqueued on `stream`, carries the verification
 * beside the attention, and rejoins `stream` before the compaction and the result copies.  When
 * the verification is the longer branch, so do the copies that touch its parent or n_nodes
 * (read by both branches; the attention's stream waits for that group).  Every other input copy,
 * and every output copy, is on `stream`.  Those verification-only buffers must therefore not
 * overlap any buffer the attention reads.  The input copies run group after group, each with the
 * whole host link: the longer branch's first (that branch is also issued first, as in the
 * graph), then the other's, then the draft distributions (and with draft_rows, the compact rows),
 * which only the rejection walk at the end of the verification reads.
 *
 * Each spec_host_copy moves `rows` rows of `row_bytes` bytes; row r starts at
 * host + r * host_pitch and at device + r * device_pitch (pitches are ignored when rows == 1).
 * A strided destination lets one copy place, say, a request's new tree K rows of every KV head
 * into the cache slots [prefix_len, prefix_len + n) of a [Hkv][L_cap][d] block.  The device
 * pointers are normally buffers the round was created on (q, hidden_states, tokens, parent,
 * n_nodes, prefix_len, draft_probs, cache slots; accept_len, path, bonus_token, new_len, ...).
 *   - Host memory should be page-locked (cudaHostAlloc / cudaHostRegister); with pageable memory
 *     the copies are staged by the driver and the call returns only after they are done.
 *   - The call returns once everything is enqueued: synchronise `stream` before reading the
 *     outputs on the host or refilling the input buffers.
 *   - A copy with row_bytes == 0 or rows == 0 is skipped.
 * Errors: SPEC_ERR_INVALID_ARGUMENT (round == NULL, a negative count, NULL arrays with a positive
 * count, a NULL pointer in a non-empty copy, a pitch below row_bytes with rows > 1),
 * SPEC_ERR_CUDA (a copy or the graph launch could not be enqueued). */
typedef struct spec_host_copy {
  void* host;             /* host memory */
  void* device;           /* device memory */
  size_t row_bytes;       /* bytes per row */
  size_t rows;            /* rows (1 = one contiguous block of row_bytes) */
  size_t host_pitch;      /* bytes between rows on the host (rows > 1) */
  size_t device_pitch;    /* bytes between rows on the device (rows > 1) */
} spec_host_copy;

spec_status spec_round_launch_host(const spec_round* round, const spec_host_copy* inputs, int32_t n_inputs,
                                   const spec_host_copy* outputs, int32_t n_outputs, void* stream);

/* Static English description of a status code (never NULL). */
const char* spec_status_string(spec_status status);

#ifdef __cplusplus
}
#endif

#endif /* SPECTREE_H_ */

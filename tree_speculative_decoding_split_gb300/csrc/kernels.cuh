// Host-side launchers of the tree-verification kernels (internal to libspectree.so).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace spectree {

// ---- K0: tree preparation -------------------------------------------------------------------
// Validates each request's tree (and optionally its KV capacity and tokens) and builds
// depth [B][N] and the ancestor-or-self bit matrix anc [B][N][W] (W = ceil(N / 32) words).
// bad[b] receives the request's error code (0 = fine).
void launch_tree_prep(const int32_t* parent, const int32_t* n_nodes, const int32_t* prefix_len,
                      long long kv_capacity, const int32_t* tokens, int vocab, int B, int N,
                      int32_t* depth, uint32_t* anc, int32_t* bad, int32_t* dev_status,
                      cudaStream_t stream);

// ---- K1: tree attention ---------------------------------------------------------------------
struct AttnParams {
  const void* q;
  void* out;
  float* lse;
  const float* k32;  // fp32 path only (raw cache pointers)
  const float* v32;
  const int32_t* prefix_len;
  const int32_t* n_nodes;
  const uint32_t* anc;      // fp32 path: ancestor bits from the tree-prep kernel
  const int32_t* bad;       // fp32 path: per-request verdict of the tree-prep kernel
  const int32_t* parent;    // [B][N]
  uint16_t* part_o;  // [B*N*Hq][n_split][d] normalised partial rows, bf16 bits
  float2* part_ml;   // [B*N*Hq][n_split] (running max in log2 units, sum)
  int B, N, Hq, Hkv, G, W, d;
  long long L_cap;
  int chunk;         // keys per split (a multiple of 64)
  int n_split;       // key splits; the one holding slot prefix_len also takes the tree keys
  int n_rg;          // row groups of (node, head) rows per KV head (one bf16 CTA each)
  int groups;        // 128-row groups per bf16 CTA (1 or 2)
  float scale;
  float scale_log2;
  int32_t* dev_status;
  // paged KV (bf16): pools [num_blocks][Hkv][bs][d]; table [B][max_blocks]; nullptr = contiguous
  const int32_t* table;
  int bs, bs_shift, max_blocks, num_blocks;
  int32_t* req_bad;  // [B] written by the tree-split CTAs: the request's table has an entry out of range
  int32_t* tree_bad; // [B] bf16: written by CTA (split 0, row group 0, KV head 0) of each request --
                     // the request's tree or capacity check failed (the merge zeroes its rows)
  int q_tma;         // bf16: Q rows arrive by TMA through the (d, Hq, N, B) map (128 % G == 0)
  int v_rows;        // bf16: V tile layout [64 / v_rows][d / 64][v_rows][128 B]; 64 = one block of
                     // rows per d/64 chunk; a paged block size below 64 when its V rows arrive as
                     // one (64, block, d / 64) box per block
  int direct;        // bf16, one split: the kernel writes out / lse itself and no merge runs
  // persistent stream-K kernel (n_rg then counts 256-row blocks)
  float* sk_o;       // [grid][2][256][d] normalised partial outputs of the CTAs' partial pieces
  float2* sk_ml;     // [grid][2][256] (running max in log2 units, sum) of those partials
  int32_t* sk_cnt;   // [B * Hkv * n_rg][2] arrival counters, zeroed before each launch
};

struct AttnPlan {
  int n_rg, chunk, n_split, groups;
  int sk;            // 1: the persistent stream-K kernel (attention_sk.cu) runs instead
  int sk_grid;       // its CTAs (one per SM)
};
constexpr int kSkMaxBatch = 1024;  // requests the stream-K kernel schedules in shared memory
constexpr int kSkRows = 256;       // (node, GQA head) rows per stream-K segment
cudaError_t launch_attention_sk(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                                const AttnParams& p, int grid, cudaStream_t stream);
AttnPlan plan_attention(int B, int N, int G, int Hkv, long long L_cap, int num_sms);
void launch_attention_merge_bf16(const AttnParams& p, cudaStream_t stream);
int attention_tc_rows_per_cta(int groups);
cudaError_t launch_attention_tc(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                                const AttnParams& p, cudaStream_t stream);
void launch_attention_f32(const AttnParams& p, cudaStream_t stream);

// ---- K2: LM head + row statistics -----------------------------------------------------------
struct LmParams {
  int R;           // rows (B * N)
  int V, Hd;
  int n_vt;        // vocabulary tiles of 128
  int n_nc;        // node chunks of BN rows
  int BN;
  int cpc;         // CTAs per node chunk (grid = cpc * n_nc); records per row of the tc kernel
  int BNV;         // rows-on-M kernel (BN == 128): vocabulary entries per tile (128 or 256)
  int pair;        // CTA-pair kernel: n_nc counts 256-row pairs, cpc clusters per pair, 256-entry tiles
  float inv_tau;
  float4* part;    // [slot][R] {max, sumexp, sumexp*y, second max}
  int* part_idx;   // [slot][R] argmax
  float* logits;   // [R][V] raw z, or nullptr
  int32_t* counters;  // zeroed by the kernel (per-request arrival counters of the finalisation)
  int n_counters;
  int32_t* dev_status;
};
int lmhead_pick_bn(int R);
int lmhead_rows_bnv(int n_nc, int num_sms);
// The CTA-pair kernel takes more than this many tree rows (bf16).
constexpr int kLmPairMinRows = 128;
size_t lmhead_smem_bytes(int BN);
cudaError_t launch_lmhead_bf16(const CUtensorMap* tmW, const CUtensorMap* tmH, const LmParams& p,
                               int num_sms, cudaStream_t stream);
void launch_lmhead_f32(const float* H, const float* W, const LmParams& p, cudaStream_t stream);

// ---- K4: KV compaction ----------------------------------------------------------------------
struct PagedKV {
  const int32_t* table;  // [B][max_blocks], nullptr = contiguous caches
  int bs, bs_shift, max_blocks, num_blocks;
};
struct CompactParams {
  uint8_t* k;                // caches (or pools), updated in place
  uint8_t* v;
  int row_bytes;             // bytes of one K (or V) row: head_dim x element size
  const int32_t* prefix_len; // [B]
  int Hkv;
  long long L_cap;
  int path_cap;
  int32_t* src_slot;         // [B][path_cap] or nullptr
  int32_t* new_len;          // [B] or nullptr
  int32_t* dev_status;
  PagedKV pg;
};
// ---- K3: acceptance + longest path ----------------------------------------------------------
struct AcceptParams {
  int B, N, V, Vd, rule, path_cap;
  float inv_tau, log_eps, log_delta;
  unsigned long long seed;
  const int32_t* tokens;
  const int32_t* parent;
  const int32_t* n_nodes;
  const float* rmax; const float* rlse; const float* rent; const float* rgap;
  const int32_t* rarg; const float* clog;
  const float* logits;         // [R][V] (rejection)
  const float4* part;          // [n_parts][R] LM-head records {max, sumexp, ...} of z / tau (rejection)
  int n_parts, R;
  const float* draft;          // [B][N][Vd], or [n_draft_rows][Vd] with draft_rows (rejection)
  const int32_t* draft_rows;   // [B][N] node -> row of draft, or nullptr (row b * N + e)
  int n_draft_rows;
  const int32_t* inv_map;      // [V] target -> draft index, -1 if unmapped; nullptr = identity
  const int32_t* map_bad;      // non-zero when the draft map is invalid
  float* rbuf;                 // [B][2][V] residual buffers (rejection)
  int32_t* accept_len; int32_t* path; int32_t* bonus; int32_t* margin_count; int32_t* bonus_margin;
  int32_t* dev_status;
  int fuse_compact;            // compact the accepted path's K/V at the end of the decision
  CompactParams cp;            // (its path and length are this call's outputs)
};

// K2r: per-row statistics from the LM-head records, the child logit of each node, and (greedy /
// typical) the acceptance of a request by the last of its rows to finish.
struct FinalizeParams {
  const float4* part;
  const int* part_idx;
  int n_parts;             // records per row
  const float* logits;     // [R][V] or nullptr
  const void* hidden;      // [R][Hd]
  const void* weight;      // [V][Hd]
  int is_bf16;
  int B, N, R, V, Hd;
  float* rmax; float* rlse; float* rent; float* rgap; int32_t* rarg; float* clog;
  float* hook_max; float* hook_lse; float* hook_ent; int32_t* hook_arg;
  int fuse_accept;         // greedy / typical: accept in the last CTA of each request
  int32_t* counters;       // [B], zero on entry
  AcceptParams acc;
};
void launch_row_finalize(const FinalizeParams& p, cudaStream_t stream);

void launch_build_inverse_map(const int32_t* map, int Vd, int V, int32_t* inv, int32_t* map_bad,
                              int32_t* dev_status, cudaStream_t stream);
cudaError_t launch_accept(const AcceptParams& p, cudaStream_t stream);
// True when the rejection walk runs on a thread-block cluster (R held on chip, no R buffer).
bool rejection_uses_cluster(int V);
// Sets up the rejection walk's per-device launch state (shared-memory attribute, cluster
// occupancy) ahead of a stream capture.
void prepare_rejection_launch();

// ---- K5: static Medusa tree expansion -------------------------------------------------------
constexpr int kMaxHeads = 16;          // Medusa heads
constexpr int kMaxTopk = 32;           // candidates per head
constexpr int kMedusaMergeCands = 2048;  // chunk candidates per head the merge holds

struct MedusaParams {
  int B, K, V, N, k;
  int is_bf16;
  int n_chunks, chunk;                 // vocabulary chunks per head and their length
  const void* logits;                  // [B][K][V]
  const int32_t* topo_parent;          // [N]
  const int32_t* topo_rank;            // [N]
  const int32_t* root_token;           // [B] or nullptr
  unsigned long long* cand;            // workspace [B*K][n_chunks][k] order keys
  int32_t* tokens;                     // [B][N]
  int32_t* parent_out;                 // [B][N] or nullptr
  int32_t* n_nodes_out;                // [B] or nullptr
  int32_t* topk_index;                 // [B][K][k] or nullptr
  int32_t* dev_status;
};
int medusa_chunks(int B, int K, int V, int k, int num_sms);
int topk_chunk_len(int V, int n_chunks);
void launch_medusa(const MedusaParams& p, cudaStream_t stream);
// K5a alone: per-row chunk top-k keys of p.logits [p.B * p.K][p.V] into p.cand.
void launch_row_topk_chunks(const MedusaParams& p, cudaStream_t stream);

// ---- K6: layered dynamic draft tree (EAGLE-2 reading) --------------------------------------
constexpr int kEagleMaxCands = 2048;   // candidates of all layers per request (tree selection)

struct EagleExpandParams {
  int B, F, k, next_k, n_chunks;
  size_t cand_stride;                  // elements between requests' candidate rows
  const unsigned long long* chunk_keys;  // [B*F][n_chunks][k] from K5a
  const float* frontier_score;         // [B][F]
  const int32_t* frontier_valid;       // [B][F] or nullptr
  const int32_t* frontier_cand;        // [B][F] or nullptr
  int32_t* cand_token; float* cand_score; int32_t* cand_parent;  // [B][stride], F*k used
  int32_t* next_index; float* next_score;                        // [B][next_k]
};
void launch_eagle_expand(const EagleExpandParams& p, const MedusaParams& chunks, cudaStream_t stream);

struct EagleTreeParams {
  int B, D, C, N, Vd;
  const float* score; const int32_t* token; const int32_t* parent;  // [B][D][C]
  const int32_t* d2t;                  // [Vd] or nullptr
  const int32_t* root_token;           // [B] or nullptr
  int32_t* tree_parent; int32_t* tree_token; int32_t* n_nodes; int32_t* node_cand;
  int32_t* dev_status;
};
void launch_eagle_tree(const EagleTreeParams& p, cudaStream_t stream);

constexpr int kCompactBufChunks = 2048;  // 32 KB of staged rows (64 bf16 rows of d = 128, K and V)
void launch_compact_kv(const CompactParams& c, const int32_t* path, const int32_t* accept_len, int B,
                       cudaStream_t stream);

}  // namespace spectree

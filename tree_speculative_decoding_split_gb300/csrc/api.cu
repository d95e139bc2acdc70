// C ABI of libspectree.so: argument checks, workspace carving, tensor maps and launch order.
// The functions are declared, with their contracts, in include/spectree.h.

#include <cmath>
#include <cstring>

#include "common.cuh"
#include "kernels.cuh"

using namespace spectree;

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Sequential carve-out of a caller-provided workspace (or a pure size count when base is null).
struct Carver {
  char* base;
  size_t off = 0;
  explicit Carver(void* b) : base(static_cast<char*>(b)) {}
  template <typename T>
  T* take(size_t count) {
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += align_up(count * sizeof(T));
    return p;
  }
};

int num_sms_current() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) return 148;
  return sms;
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver entry point is looked up once per process (immutable after the first call).
EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// bf16 tensor map with 128-byte swizzle.  dims/box are innermost first; strides (bytes) are for
// dims 1.. (rank - 1).
bool make_map_bf16(CUtensorMap* m, const void* ptr, int rank, const cuuint64_t* dims, const cuuint64_t* strides,
                   const cuuint32_t* box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  if (rank < 1 || rank > 5) return false;
  std::memset(m, 0, sizeof(*m));
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Records an optional caller-owned event (cudaEvent_t) on the stream.
void record(void* event, cudaStream_t stream) {
  if (event) cudaEventRecord(static_cast<cudaEvent_t>(event), stream);
}

// ---- attention ------------------------------------------------------------------------------

// Paged KV: block size a power of two in [16, 256], kv_capacity = max_blocks * block_size, and
// pool coordinates that fit the tensor map.
spec_status check_paged(int bs, int max_blocks, int num_blocks, int Hkv, long long L_cap) {
  if (bs != 16 && bs != 32 && bs != 64 && bs != 128 && bs != 256) return SPEC_ERR_UNSUPPORTED;
  if (max_blocks < 1 || num_blocks < 1) return SPEC_ERR_INVALID_ARGUMENT;
  if ((long long)max_blocks * bs != L_cap) return SPEC_ERR_INVALID_ARGUMENT;
  if ((long long)num_blocks * Hkv >= 0x7fffffffLL) return SPEC_ERR_UNSUPPORTED;
  return SPEC_OK;
}

int log2_of(int x) {
  int s = 0;
  while ((1 << s) < x) ++s;
  return s;
}

spec_status check_attn(const spec_attn_args* a) {
  if (!a) return SPEC_ERR_INVALID_ARGUMENT;
  if (a->dtype != SPEC_DTYPE_F32 && a->dtype != SPEC_DTYPE_BF16) return SPEC_ERR_UNSUPPORTED;
  if (a->head_dim != 64 && a->head_dim != 128) return SPEC_ERR_UNSUPPORTED;
  if (a->batch < 1 || a->n_max < 1 || a->num_q_heads < 1 || a->num_kv_heads < 1 || a->kv_capacity < 1 ||
      (a->schedule != SPEC_ATTN_SPLIT_KV && a->schedule != SPEC_ATTN_STREAM_K))
    return SPEC_ERR_INVALID_ARGUMENT;
  if (a->n_max > SPEC_MAX_NODES) return SPEC_ERR_UNSUPPORTED;
  if (a->num_q_heads % a->num_kv_heads) return SPEC_ERR_INVALID_ARGUMENT;
  if (a->kv_capacity > 0x7fffffffLL) return SPEC_ERR_UNSUPPORTED;
  if ((long long)a->batch * a->num_kv_heads > 65535) return SPEC_ERR_UNSUPPORTED;  // grid.z
  if (!a->q || !a->k_cache || !a->v_cache || !a->prefix_len || !a->n_nodes || !a->parent || !a->out)
    return SPEC_ERR_INVALID_ARGUMENT;
  if (!aligned16(a->q) || !aligned16(a->k_cache) || !aligned16(a->v_cache) || !aligned16(a->out))
    return SPEC_ERR_INVALID_ARGUMENT;
  if (a->reserved1 != 0) return SPEC_ERR_INVALID_ARGUMENT;
  if (a->block_table) {
    if (a->dtype != SPEC_DTYPE_BF16) return SPEC_ERR_UNSUPPORTED;
    const spec_status ps = check_paged(a->block_size, a->max_blocks, a->num_blocks, a->num_kv_heads, a->kv_capacity);
    if (ps != SPEC_OK) return ps;
  }
  if (a->schedule == SPEC_ATTN_STREAM_K) {
    const int G = a->num_q_heads / a->num_kv_heads;
    if (a->dtype != SPEC_DTYPE_BF16 || a->block_table || G > 128 || 128 % G != 0 || a->batch > kSkMaxBatch)
      return SPEC_ERR_UNSUPPORTED;
    const long long blocks = ((long long)a->n_max * G + kSkRows - 1) / kSkRows;
    if ((a->kv_capacity + 63) / 64 * a->batch * a->num_kv_heads * blocks >= 0x7fffffffLL)
      return SPEC_ERR_UNSUPPORTED;  // the kernel indexes tiles with 32-bit integers
  }
  return SPEC_OK;
}

struct AttnLayout {
  int32_t* depth; uint32_t* anc; int32_t* bad; int32_t* tree_bad; uint16_t* part_o; float2* part_ml;
  float* sk_o; float2* sk_ml; int32_t* sk_cnt;
  AttnPlan plan;
  size_t bytes;
};

AttnLayout layout_attn(const spec_attn_args* a, void* ws) {
  AttnLayout l;
  const int B = a->batch, N = a->n_max, W = (N + 31) / 32;
  const int G = a->num_q_heads / a->num_kv_heads;
  const int sms = num_sms_current();
  l.plan = plan_attention(B, N, G, a->num_kv_heads, a->kv_capacity, sms);
  l.plan.sk = a->schedule == SPEC_ATTN_STREAM_K ? 1 : 0;
  l.plan.sk_grid = sms;
  Carver c(ws);
  l.depth = c.take<int32_t>((size_t)B * N);
  l.anc = c.take<uint32_t>((size_t)B * N * W);
  l.bad = c.take<int32_t>(B);
  l.tree_bad = c.take<int32_t>(B);
  l.part_o = nullptr;
  l.part_ml = nullptr;
  l.sk_o = nullptr;
  l.sk_ml = nullptr;
  l.sk_cnt = nullptr;
  if (l.plan.sk) {
    l.plan.n_rg = (N * G + kSkRows - 1) / kSkRows;
    l.sk_cnt = c.take<int32_t>((size_t)B * a->num_kv_heads * l.plan.n_rg * 2);
    l.sk_ml = c.take<float2>((size_t)sms * 2 * kSkRows);
    l.sk_o = c.take<float>((size_t)sms * 2 * kSkRows * a->head_dim);
  } else if (a->dtype == SPEC_DTYPE_BF16) {
    const size_t rows = (size_t)B * N * a->num_q_heads;
    l.part_o = c.take<uint16_t>(rows * l.plan.n_split * a->head_dim);
    l.part_ml = c.take<float2>(rows * l.plan.n_split);
  }
  l.bytes = c.off;
  return l;
}

// ---- verify ---------------------------------------------------------------------------------

spec_status check_verify(const spec_verify_args* a) {
  if (!a) return SPEC_ERR_INVALID_ARGUMENT;
  if (a->dtype != SPEC_DTYPE_F32 && a->dtype != SPEC_DTYPE_BF16) return SPEC_ERR_UNSUPPORTED;
  if (a->batch < 1 || a->n_max < 1 || a->hidden < 1 || a->vocab < 2 || a->path_cap < 1 || a->reserved0 != 0 ||
      a->reserved1 != 0)
    return SPEC_ERR_INVALID_ARGUMENT;
  if (a->n_max > SPEC_MAX_NODES) return SPEC_ERR_UNSUPPORTED;
  if (a->dtype == SPEC_DTYPE_BF16 && a->hidden % 64) return SPEC_ERR_UNSUPPORTED;
  if (a->dtype == SPEC_DTYPE_F32 && a->hidden % 4) return SPEC_ERR_UNSUPPORTED;
  if (a->rule != SPEC_RULE_GREEDY && a->rule != SPEC_RULE_TYPICAL && a->rule != SPEC_RULE_REJECTION)
    return SPEC_ERR_INVALID_ARGUMENT;
  if (a->rule != SPEC_RULE_GREEDY && !(a->temperature > 0.f && std::isfinite(a->temperature)))
    return SPEC_ERR_INVALID_ARGUMENT;
  if (a->rule == SPEC_RULE_TYPICAL && (!(a->eps >= 0.f) || !(a->delta >= 0.f))) return SPEC_ERR_INVALID_ARGUMENT;
  if (!a->hidden_states || !a->lm_head_weight || !a->tokens || !a->parent || !a->n_nodes || !a->accept_len ||
      !a->path || !a->bonus_token)
    return SPEC_ERR_INVALID_ARGUMENT;
  if (!aligned16(a->hidden_states) || !aligned16(a->lm_head_weight)) return SPEC_ERR_INVALID_ARGUMENT;
  if (a->rule == SPEC_RULE_REJECTION) {
    if (!a->draft_probs || a->draft_vocab < 1) return SPEC_ERR_INVALID_ARGUMENT;
    if (!a->draft_to_target && a->draft_vocab != a->vocab) return SPEC_ERR_INVALID_ARGUMENT;
    if (a->draft_vocab > a->vocab) return SPEC_ERR_INVALID_ARGUMENT;
    if (a->draft_rows && a->n_draft_rows < 1) return SPEC_ERR_INVALID_ARGUMENT;
  }
  const long long R = (long long)a->batch * a->n_max;
  if (R > 0x7fffffffLL / 2 || (long long)a->vocab * R > (1LL << 40)) return SPEC_ERR_UNSUPPORTED;
  return SPEC_OK;
}

struct VerifyLayout {
  float4* part; int* part_idx;
  float *rmax, *rlse, *rent, *rgap, *clog; int32_t* rarg;
  float* logits; float* rbuf; int32_t* inv; int32_t* map_bad; int32_t* counters;
  int R, n_vt, BN, BNV, n_nc, cpc, n_parts, pair;
  size_t bytes;
};

VerifyLayout layout_verify(const spec_verify_args* a, void* ws) {
  VerifyLayout l;
  const int B = a->batch, N = a->n_max;
  l.R = B * N;
  l.n_vt = (a->vocab + 127) / 128;
  l.BN = lmhead_pick_bn(l.R);
  l.n_nc = (l.R + l.BN - 1) / l.BN;
  const int sms = num_sms_current();
  // BN == 128: tree rows on the MMA M side, BNV vocabulary entries per tile; else vocabulary
  // on M in tiles of 128 and BN tree rows on N.  Above 128 rows (bf16) CTA pairs take 256 rows per
  // MMA, 256 vocabulary entries per tile, cpc clusters per row pair.
  l.pair = (a->dtype == SPEC_DTYPE_BF16 && l.BN == 128 && l.R > kLmPairMinRows) ? 1 : 0;
  int tiles;
  if (l.pair) {
    l.n_nc = (l.R + 255) / 256;
    l.BNV = 256;
    tiles = (a->vocab + 255) / 256;
    l.cpc = (sms / 2) / l.n_nc;
  } else {
    l.BNV = (l.BN == 128) ? lmhead_rows_bnv(l.n_nc, sms) : 128;
    tiles = (a->vocab + l.BNV - 1) / l.BNV;
    l.cpc = sms / l.n_nc;
  }
  if (l.cpc < 1) l.cpc = 1;
  if (l.cpc > tiles) l.cpc = tiles;
  // statistics records per row: one per CTA of the row's chunk (bf16), one per tile (fp32)
  l.n_parts = (a->dtype == SPEC_DTYPE_BF16) ? l.cpc : l.n_vt;
  Carver c(ws);
  l.part = c.take<float4>((size_t)l.n_parts * l.R);
  l.part_idx = c.take<int>((size_t)l.n_parts * l.R);
  l.rmax = c.take<float>(l.R);
  l.rlse = c.take<float>(l.R);
  l.rent = c.take<float>(l.R);
  l.rgap = c.take<float>(l.R);
  l.clog = c.take<float>(l.R);
  l.rarg = c.take<int32_t>(l.R);
  l.counters = c.take<int32_t>(B);
  const bool need_logits = a->rule == SPEC_RULE_REJECTION || a->dtype == SPEC_DTYPE_F32;
  l.logits = need_logits ? c.take<float>((size_t)l.R * a->vocab) : nullptr;
  l.rbuf = nullptr;
  l.inv = nullptr;
  l.map_bad = nullptr;
  if (a->rule == SPEC_RULE_REJECTION) {
    if (!rejection_uses_cluster(a->vocab)) l.rbuf = c.take<float>((size_t)B * 2 * a->vocab);
    if (a->draft_to_target) {
      l.inv = c.take<int32_t>(a->vocab);
      l.map_bad = c.take<int32_t>(1);
    }
  }
  l.bytes = c.off;
  return l;
}

spec_status check_compact(const spec_compact_args* a) {
  if (!a) return SPEC_ERR_INVALID_ARGUMENT;
  if (a->dtype != SPEC_DTYPE_F32 && a->dtype != SPEC_DTYPE_BF16) return SPEC_ERR_UNSUPPORTED;
  if (a->head_dim != 64 && a->head_dim != 128) return SPEC_ERR_UNSUPPORTED;
  if (a->batch < 1 || a->num_kv_heads < 1 || a->kv_capacity < 1 || a->path_cap < 1 || a->reserved0 != 0)
    return SPEC_ERR_INVALID_ARGUMENT;
  if (!a->k_cache || !a->v_cache || !a->prefix_len || !a->path || !a->accept_len) return SPEC_ERR_INVALID_ARGUMENT;
  if (!aligned16(a->k_cache) || !aligned16(a->v_cache)) return SPEC_ERR_INVALID_ARGUMENT;
  if ((long long)a->batch * a->num_kv_heads > 0x7fffffffLL) return SPEC_ERR_UNSUPPORTED;
  if (a->reserved1 != 0) return SPEC_ERR_INVALID_ARGUMENT;
  if (a->block_table) {
    const spec_status ps = check_paged(a->block_size, a->max_blocks, a->num_blocks, a->num_kv_heads, a->kv_capacity);
    if (ps != SPEC_OK) return ps;
  }
  return SPEC_OK;
}

CompactParams compact_params(const spec_compact_args* a, int32_t* dev_status) {
  CompactParams c;
  std::memset(&c, 0, sizeof(c));
  c.k = static_cast<uint8_t*>(a->k_cache);
  c.v = static_cast<uint8_t*>(a->v_cache);
  c.row_bytes = a->head_dim * (a->dtype == SPEC_DTYPE_BF16 ? 2 : 4);
  c.prefix_len = a->prefix_len;
  c.Hkv = a->num_kv_heads;
  c.L_cap = a->kv_capacity;
  c.path_cap = a->path_cap;
  c.src_slot = a->src_slot;
  c.new_len = a->new_len;
  c.dev_status = dev_status;
  if (a->block_table) {
    c.pg.table = a->block_table;
    c.pg.bs = a->block_size;
    c.pg.bs_shift = log2_of(a->block_size);
    c.pg.max_blocks = a->max_blocks;
    c.pg.num_blocks = a->num_blocks;
  }
  return c;
}

}  // namespace

extern "C" {

size_t spec_tree_attention_workspace(const spec_attn_args* a) {
  if (check_attn(a) != SPEC_OK) return 0;
  return layout_attn(a, nullptr).bytes;
}

spec_status spec_tree_attention(const spec_attn_args* a, void* workspace, size_t workspace_bytes,
                                int32_t* dev_status, void* stream_ptr) {
  spec_status st = check_attn(a);
  if (st != SPEC_OK) return st;
  if (!workspace || !aligned16(workspace)) return SPEC_ERR_INVALID_ARGUMENT;
  const AttnLayout need = layout_attn(a, nullptr);
  if (workspace_bytes < need.bytes) return SPEC_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const AttnLayout l = layout_attn(a, workspace);
  const int B = a->batch, N = a->n_max, Hq = a->num_q_heads, Hkv = a->num_kv_heads, d = a->head_dim;
  if (a->dtype == SPEC_DTYPE_F32)
    launch_tree_prep(a->parent, a->n_nodes, a->prefix_len, a->kv_capacity, nullptr, 0, B, N, l.depth, l.anc, l.bad,
                     dev_status, stream);
  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = a->q;
  p.out = a->out;
  p.lse = a->lse;
  p.prefix_len = a->prefix_len;
  p.n_nodes = a->n_nodes;
  p.anc = l.anc;
  p.bad = l.bad;
  p.tree_bad = l.tree_bad;
  p.parent = a->parent;
  p.part_o = l.part_o;
  p.part_ml = l.part_ml;
  p.B = B; p.N = N; p.Hq = Hq; p.Hkv = Hkv; p.G = Hq / Hkv; p.W = (N + 31) / 32; p.d = d;
  p.L_cap = a->kv_capacity;
  p.chunk = l.plan.chunk;
  p.n_split = l.plan.n_split;
  p.n_rg = l.plan.n_rg;
  p.groups = l.plan.groups;
  p.scale = a->scale > 0.f ? a->scale : 1.f / std::sqrt((float)d);
  p.scale_log2 = p.scale * 1.4426950408889634f;
  p.dev_status = dev_status;
  if (a->block_table) {
    p.table = a->block_table;
    p.bs = a->block_size;
    p.bs_shift = log2_of(a->block_size);
    p.max_blocks = a->max_blocks;
    p.num_blocks = a->num_blocks;
    p.req_bad = l.bad;
  }
  if (a->dtype == SPEC_DTYPE_F32) {
    p.k32 = static_cast<const float*>(a->k_cache);
    p.v32 = static_cast<const float*>(a->v_cache);
    record(a->timing_begin, stream);
    launch_attention_f32(p, stream);
    record(a->timing_end, stream);
  } else {
    CUtensorMap tmK, tmV;
    // contiguous: (d, L_cap, B*Hkv), 64-slot boxes; paged pools: (d, block, num_blocks*Hkv),
    // boxes of min(block, 64) slots
    const bool paged = a->block_table != nullptr;
    const long long rows = paged ? a->block_size : a->kv_capacity;
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows,
                                paged ? (cuuint64_t)a->num_blocks * Hkv : (cuuint64_t)B * Hkv};
    const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)rows * d * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)(paged && a->block_size < 64 ? a->block_size : 64), 1};
    if (!make_map_bf16(&tmK, a->k_cache, 3, dims, strides, box) ||
        !make_map_bf16(&tmV, a->v_cache, 3, dims, strides, box))
      return SPEC_ERR_CUDA;
    p.v_rows = 64;
    if (paged && a->block_size < 64 && d == 128 && !l.plan.sk) {
      // a pool block's V rows as one box of both 64-column halves: (64, block, d / 64 with a
      // 128-byte stride, num_blocks*Hkv), landing as [half][block rows][128 B] -- the layout the
      // P V MMA then reads with a block-sized stride between the halves
      const cuuint64_t vd[4] = {64, (cuuint64_t)a->block_size, 2, (cuuint64_t)a->num_blocks * Hkv};
      const cuuint64_t vs[3] = {(cuuint64_t)d * 2, 128, (cuuint64_t)a->block_size * d * 2};
      const cuuint32_t vb[4] = {64, (cuuint32_t)a->block_size, 2, 1};
      CUtensorMap tmV4;
      if (make_map_bf16(&tmV4, a->v_cache, 4, vd, vs, vb)) {
        tmV = tmV4;
        p.v_rows = a->block_size;
      }
    }
    // Q as (d, Hq, N, B): one box of (64, G, 128 / G, 1) is a 128-row group of (node, head) rows
    // of one KV head.  Other G stage Q through registers.
    CUtensorMap tmQ;
    std::memset(&tmQ, 0, sizeof(tmQ));
    if (p.G <= 128 && 128 % p.G == 0) {
      const cuuint64_t qd[4] = {(cuuint64_t)d, (cuuint64_t)Hq, (cuuint64_t)N, (cuuint64_t)B};
      const cuuint64_t qs[3] = {(cuuint64_t)d * 2, (cuuint64_t)Hq * d * 2, (cuuint64_t)N * Hq * d * 2};
      const cuuint32_t qb[4] = {64, (cuuint32_t)p.G, (cuuint32_t)(128 / p.G), 1};
      if (!make_map_bf16(&tmQ, a->q, 4, qd, qs, qb)) return SPEC_ERR_CUDA;
      p.q_tma = 1;
    }
    if (l.plan.sk) {
      p.sk_o = l.sk_o;
      p.sk_ml = l.sk_ml;
      p.sk_cnt = l.sk_cnt;
      const size_t cnt_bytes = (size_t)B * Hkv * l.plan.n_rg * 2 * sizeof(int32_t);
      if (cudaMemsetAsync(l.sk_cnt, 0, cnt_bytes, stream) != cudaSuccess) return SPEC_ERR_CUDA;
      record(a->timing_begin, stream);
      if (launch_attention_sk(&tmQ, &tmK, &tmV, p, l.plan.sk_grid, stream) != cudaSuccess) return SPEC_ERR_CUDA;
      record(a->timing_end, stream);
      return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
    }
    p.direct = p.n_split == 1 ? 1 : 0;
    record(a->timing_begin, stream);
    if (launch_attention_tc(&tmQ, &tmK, &tmV, p, stream) != cudaSuccess) return SPEC_ERR_CUDA;
    record(a->timing_end, stream);
    if (!p.direct) launch_attention_merge_bf16(p, stream);
  }
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

size_t spec_verify_accept_workspace(const spec_verify_args* a) {
  if (check_verify(a) != SPEC_OK) return 0;
  return layout_verify(a, nullptr).bytes;
}

}  // extern "C"

namespace {

// spec_verify_accept, and with `cmp` non-null the compaction of each request's accepted path,
// folded into the tail of the kernel that decides the request.
spec_status verify_accept_impl(const spec_verify_args* a, void* workspace, size_t workspace_bytes,
                               const spec_compact_args* cmp, int32_t* dev_status, void* stream_ptr) {
  spec_status st = check_verify(a);
  if (st != SPEC_OK) return st;
  if (!workspace || !aligned16(workspace)) return SPEC_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < layout_verify(a, nullptr).bytes) return SPEC_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  const VerifyLayout l = layout_verify(a, workspace);
  const int B = a->batch, N = a->n_max, V = a->vocab, Hd = a->hidden;
  if (a->rule == SPEC_RULE_REJECTION && a->draft_to_target)
    launch_build_inverse_map(a->draft_to_target, a->draft_vocab, V, l.inv, l.map_bad, dev_status, stream);
  const float inv_tau = (a->rule == SPEC_RULE_GREEDY) ? 1.f : 1.f / a->temperature;

  LmParams lp;
  std::memset(&lp, 0, sizeof(lp));
  lp.R = l.R; lp.V = V; lp.Hd = Hd; lp.n_vt = l.n_vt; lp.n_nc = l.n_nc; lp.BN = l.BN; lp.BNV = l.BNV; lp.cpc = l.cpc;
  lp.pair = l.pair;
  lp.inv_tau = inv_tau;
  lp.part = l.part;
  lp.part_idx = l.part_idx;
  lp.logits = l.logits;
  lp.counters = l.counters;
  lp.n_counters = B;
  lp.dev_status = dev_status;
  if (a->dtype == SPEC_DTYPE_BF16) {
    CUtensorMap tmW, tmH;
    const cuuint64_t dW[2] = {(cuuint64_t)Hd, (cuuint64_t)V};
    const cuuint64_t dH[2] = {(cuuint64_t)Hd, (cuuint64_t)l.R};
    const cuuint64_t str[1] = {(cuuint64_t)Hd * 2};
    const cuuint32_t bW[2] = {64, (cuuint32_t)(l.pair ? l.BNV / 2 : l.BNV)};  // a pair CTA loads half a tile
    const cuuint32_t bH[2] = {64, (cuuint32_t)l.BN};
    if (!make_map_bf16(&tmW, a->lm_head_weight, 2, dW, str, bW) ||
        !make_map_bf16(&tmH, a->hidden_states, 2, dH, str, bH))
      return SPEC_ERR_CUDA;
    const int sms = num_sms_current();
    record(a->timing_begin, stream);
    if (launch_lmhead_bf16(&tmW, &tmH, lp, sms, stream) != cudaSuccess) return SPEC_ERR_CUDA;
    record(a->timing_end, stream);
  } else {
    if (cudaMemsetAsync(l.counters, 0, (size_t)B * sizeof(int32_t), stream) != cudaSuccess) return SPEC_ERR_CUDA;
    record(a->timing_begin, stream);
    launch_lmhead_f32(static_cast<const float*>(a->hidden_states), static_cast<const float*>(a->lm_head_weight), lp,
                      stream);
    record(a->timing_end, stream);
  }

  AcceptParams ap;
  std::memset(&ap, 0, sizeof(ap));
  ap.B = B; ap.N = N; ap.V = V; ap.Vd = a->draft_vocab; ap.rule = a->rule; ap.path_cap = a->path_cap;
  ap.inv_tau = inv_tau;
  ap.log_eps = (a->eps > 0.f) ? logf(a->eps) : -INFINITY;
  ap.log_delta = (a->delta > 0.f) ? logf(a->delta) : -INFINITY;
  ap.seed = a->seed;
  ap.tokens = a->tokens; ap.parent = a->parent; ap.n_nodes = a->n_nodes;
  ap.rmax = l.rmax; ap.rlse = l.rlse; ap.rent = l.rent; ap.rgap = l.rgap; ap.rarg = l.rarg; ap.clog = l.clog;
  ap.logits = l.logits; ap.draft = a->draft_probs; ap.inv_map = l.inv; ap.map_bad = l.map_bad; ap.rbuf = l.rbuf;
  ap.part = l.part; ap.n_parts = l.n_parts; ap.R = l.R;
  if (a->rule == SPEC_RULE_REJECTION && a->draft_rows) {
    ap.draft_rows = a->draft_rows;
    ap.n_draft_rows = a->n_draft_rows;
  }
  ap.accept_len = a->accept_len; ap.path = a->path; ap.bonus = a->bonus_token;
  ap.margin_count = a->margin_count; ap.bonus_margin = a->bonus_margin;
  ap.dev_status = dev_status;
  if (cmp) {
    ap.fuse_compact = 1;
    ap.cp = compact_params(cmp, dev_status);
  }

  FinalizeParams fp;
  std::memset(&fp, 0, sizeof(fp));
  fp.part = l.part; fp.part_idx = l.part_idx; fp.n_parts = l.n_parts; fp.logits = l.logits;
  fp.hidden = a->hidden_states; fp.weight = a->lm_head_weight; fp.is_bf16 = a->dtype == SPEC_DTYPE_BF16;
  fp.B = B; fp.N = N; fp.R = l.R; fp.V = V; fp.Hd = Hd;
  fp.rmax = l.rmax; fp.rlse = l.rlse; fp.rent = l.rent; fp.rgap = l.rgap; fp.rarg = l.rarg; fp.clog = l.clog;
  fp.hook_max = a->row_max; fp.hook_lse = a->row_lse; fp.hook_ent = a->row_entropy; fp.hook_arg = a->row_argmax;
  fp.fuse_accept = a->rule != SPEC_RULE_REJECTION;
  fp.counters = l.counters;
  fp.acc = ap;
  // Rejection sampling reads only the visited rows' LSE, which the walk merges from the records
  // itself; the row finalisation then runs only for the optional per-row outputs.
  const bool hooks = a->row_max || a->row_lse || a->row_entropy || a->row_argmax;
  if (a->rule != SPEC_RULE_REJECTION || hooks) launch_row_finalize(fp, stream);
  if (a->rule == SPEC_RULE_REJECTION && a->draft_ready) {  // the walk is the first reader of draft_probs
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return SPEC_ERR_CUDA;
    if (cudaStreamWaitEvent(stream, static_cast<cudaEvent_t>(a->draft_ready),
                            cs == cudaStreamCaptureStatusActive ? cudaEventWaitExternal : 0) != cudaSuccess)
      return SPEC_ERR_CUDA;
  }
  if (a->rule == SPEC_RULE_REJECTION && launch_accept(ap, stream) != cudaSuccess) return SPEC_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // namespace

extern "C" {

spec_status spec_verify_accept(const spec_verify_args* a, void* workspace, size_t workspace_bytes,
                               int32_t* dev_status, void* stream_ptr) {
  return verify_accept_impl(a, workspace, workspace_bytes, nullptr, dev_status, stream_ptr);
}

spec_status spec_verify_accept_compact(const spec_verify_args* a, void* workspace, size_t workspace_bytes,
                                       const spec_compact_args* c, int32_t* dev_status, void* stream_ptr) {
  spec_status st = check_verify(a);
  if (st != SPEC_OK) return st;
  st = check_compact(c);
  if (st != SPEC_OK) return st;
  if (c->path != a->path || c->accept_len != a->accept_len || c->path_cap != a->path_cap || c->batch != a->batch)
    return SPEC_ERR_INVALID_ARGUMENT;
  return verify_accept_impl(a, workspace, workspace_bytes, c, dev_status, stream_ptr);
}

spec_status spec_compact_kv(const spec_compact_args* a, int32_t* dev_status, void* stream_ptr) {
  spec_status st = check_compact(a);
  if (st != SPEC_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  launch_compact_kv(compact_params(a, dev_status), a->path, a->accept_len, a->batch, stream);
  return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

const char* spec_status_string(spec_status s) {
  switch (s) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARGUMENT: return "invalid argument (null pointer, bad size or misaligned buffer)";
    case SPEC_ERR_UNSUPPORTED: return "unsupported dtype, head_dim or size";
    case SPEC_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than the *_workspace() query";
    case SPEC_ERR_BAD_TREE: return "parent array is not a valid rooted, topologically ordered tree";
    case SPEC_ERR_CUDA: return "CUDA runtime error";
    case SPEC_ERR_BAD_TOKEN: return "token or draft-map entry outside the vocabulary, or a missing draft row";
    case SPEC_ERR_CAPACITY: return "KV capacity or path capacity exceeded";
    case SPEC_ERR_TIMEOUT: return "a bounded wait inside a kernel ran out";
    default: return "unknown status";
  }
}

}  // extern "C"

// Static Medusa tree expansion: the top-k tokens of every Medusa head, placed on a fixed tree
// topology.  jisaku glossary "Medusa", section "ツリー構造の候補構築": the candidate tree is
// built from combinations of each head's top candidates (head 0's top-3 x head 1's top-3 x head
// 2's top-2 = 18 paths) along a predefined topology ("Medusa Tree", 63 / 127 / 255 nodes).  A
// node at depth d >= 1 with rank r carries the r-th best token of head d - 1.
//
// K5a: per (request, head, vocabulary chunk) top-k over 64-bit order keys (value, then the lower
// token id) held in registers: a threshold taken from the threads' own maxima narrows the chunk
// to a few candidates, whose top-k one warp takes by k rounds of a warp-wide maximum below the
// previous winner.  K5b: per request, the chunk candidates of every head merge into the head's
// top-k (one warp per head, the heads side by side), the topology is validated and every node's
// token is looked up.

#include "common.cuh"
#include "kernels.cuh"
#include "pdl.cuh"
#include "topk.cuh"

namespace spectree {

namespace {

constexpr int kMxThreads = 256;
constexpr int kMxEpt = 16;  // vocabulary entries per thread in K5a (chunk <= 4096)

// Where this thread's entries lie in its chunk: with rows and chunk starts on 16-byte boundaries
// a thread reads 16-byte vectors (8 bf16 or 4 fp32 neighbours each), the threads side by side;
// otherwise single entries.  Entry e of thread t is token v0 + entry_offset(mode, t, e).
enum { kLoadScalar = 0, kLoadVec4 = 4, kLoadVec8 = 8 };
__device__ __forceinline__ int load_mode(const MedusaParams& p) {
  const bool aligned = (reinterpret_cast<uintptr_t>(p.logits) & 15u) == 0;
  if (p.is_bf16 && aligned && (p.V & 7) == 0 && (p.chunk & 7) == 0) return kLoadVec8;
  if (!p.is_bf16 && aligned && (p.V & 3) == 0 && (p.chunk & 3) == 0) return kLoadVec4;
  return kLoadScalar;
}
__device__ __forceinline__ int entry_offset(int mode, int t, int e) {
  if (mode == kLoadVec8) return ((e >> 3) * kMxThreads + t) * 8 + (e & 7);
  if (mode == kLoadVec4) return ((e >> 2) * kMxThreads + t) * 4 + (e & 3);
  return e * kMxThreads + t;
}

// The values of this thread's kMxEpt entries in the chunk [v0, v1) of logits row `row`, as
// floats; NaN for entries past the chunk (callers tell them from NaN logits by the token).
__device__ __forceinline__ void load_vals(const MedusaParams& p, int mode, int row, int v0, int v1,
                                          float (&x)[kMxEpt]) {
  const int tid = threadIdx.x;
  const size_t rb = (size_t)row * p.V;
  const float nan = __uint_as_float(0x7FFFFFFFu);
  if (mode == kLoadVec8) {
    const __nv_bfloat16* src = static_cast<const __nv_bfloat16*>(p.logits) + rb;
#pragma unroll
    for (int h = 0; h < kMxEpt / 8; ++h) {
      const int base = v0 + entry_offset(mode, tid, h * 8);
      uint4 w = make_uint4(0x7FFF7FFFu, 0x7FFF7FFFu, 0x7FFF7FFFu, 0x7FFF7FFFu);  // bf16 NaNs
      if (base + 8 <= v1) w = *reinterpret_cast<const uint4*>(src + base);  // v1 is a multiple of 8 here
      const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
        x[h * 8 + i] = __uint_as_float((i & 1) ? (q[i >> 1] & 0xFFFF0000u) : (q[i >> 1] << 16));
    }
    return;
  }
  if (mode == kLoadVec4) {
    const float* src = static_cast<const float*>(p.logits) + rb;
#pragma unroll
    for (int h = 0; h < kMxEpt / 4; ++h) {
      const int base = v0 + entry_offset(mode, tid, h * 4);
      float4 w = make_float4(nan, nan, nan, nan);
      if (base + 4 <= v1) w = *reinterpret_cast<const float4*>(src + base);  // v1 is a multiple of 4 here
      x[h * 4 + 0] = w.x;
      x[h * 4 + 1] = w.y;
      x[h * 4 + 2] = w.z;
      x[h * 4 + 3] = w.w;
    }
    return;
  }
#pragma unroll
  for (int e = 0; e < kMxEpt; ++e) {
    const int v = v0 + entry_offset(mode, tid, e);
    x[e] = nan;
    if (v < v1)
      x[e] = p.is_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(p.logits)[rb + v])
                       : static_cast<const float*>(p.logits)[rb + v];
  }
}

}  // namespace

// K5a: grid (n_chunks, B * K).  Writes k keys per (row, chunk), best first (0 = none).
// The chunk's top k by a threshold T on the order values with at least k entries at or above it,
// so that the chunk's top k all reach it.  With j = ceil(k / 8), every warp finds the j-th
// largest of its threads' maxima (counting repeats: a warp-wide maximum and a ballot per round),
// and T is the ceil(k / j)-th largest of those eight, so that ceil(k / j) warps hold j entries
// each at or above it.  The entries that reach T -- a few times k of them on the benchmark's rows
// -- become 64-bit keys in shared memory and each finds its rank by counting the larger ones;
// ranks below k are the result.  When more than kMxThreads entries reach T (a chunk of many
// equal values) every warp instead takes its own top k from registers by k rounds of a
// warp-wide maximum below the previous winner, and warp 0 merges the warps' candidates.  Either
// way the result is the top k of one strict order (value, then the lower token id).
__global__ void __launch_bounds__(kMxThreads) medusa_chunk_topk_kernel(const MedusaParams p) {
  constexpr int kWarps = kMxThreads / 32;
  __shared__ unsigned long long s_keys[kMxThreads];         // the candidates
  __shared__ uint32_t s_wv[kWarps];
  __shared__ unsigned long long s_cand[kWarps * kMaxTopk];  // fallback: [warp][rank]
  __shared__ int s_n;
  const int chunk = blockIdx.x, row = blockIdx.y;  // row = b * K + head
  const int v0 = chunk * p.chunk;
  const int v1 = min(p.V, v0 + p.chunk);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  pdl_launch_dependents();  // the merge may launch now; it waits for this grid before reading
  const int mode = load_mode(p);
  float x[kMxEpt];
  load_vals(p, mode, row, v0, v1, x);
  float xm = x[0];
#pragma unroll
  for (int e = 1; e < kMxEpt; ++e) xm = fmaxf(xm, x[e]);  // NaN only if every entry is NaN
  const uint32_t um = order_u(xm);
  // the warp's j-th largest thread maximum, repeats counted (0 once the maxima run out)
  const int j = (p.k + kWarps - 1) / kWarps;
  uint32_t wv = 0u, prev = 0xFFFFFFFFu;
  for (int have = 0, r = 0; r < j && have < j; ++r) {
    const uint32_t m = __reduce_max_sync(0xffffffffu, um < prev ? um : 0u);
    have += __popc(__ballot_sync(0xffffffffu, um == m));
    wv = m;
    prev = m;
    if (m == 0u) break;
  }
  if (lane == 0) s_wv[warp] = wv;
  if (tid == 0) s_n = 0;
  __syncthreads();
  // T: the largest warp value with at least ceil(k / j) of the eight at or above it
  const int need = (p.k + j - 1) / j;
  uint32_t thr = 0u;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) {
    const uint32_t w = s_wv[i];
    int ge = 0;
#pragma unroll
    for (int q = 0; q < kWarps; ++q) ge += s_wv[q] >= w;
    if (ge >= need && w > thr) thr = w;
  }
  // order_u(x) >= thr exactly when x >= the value thr stands for (x not NaN); at thr = 0 every
  // entry of the chunk, NaN included, is a candidate
  const bool all = thr == 0u;
  const float tf = order_value(thr);
#pragma unroll
  for (int e = 0; e < kMxEpt; ++e) {
    const int v = v0 + entry_offset(mode, tid, e);
    if (v < v1 && (all || x[e] >= tf)) {
      const int i = atomicAdd(&s_n, 1);
      if (i < kMxThreads) s_keys[i] = order_key(order_u(x[e]), v);
    }
  }
  __syncthreads();
  const int n = s_n;
  unsigned long long* out = p.cand + ((size_t)row * p.n_chunks + chunk) * p.k;
  if (n <= kMxThreads) {
    if (tid < n) {  // keys are distinct, so the ranks are
      const unsigned long long c = s_keys[tid];
      int rank = 0;
      for (int q = 0; q < n; ++q) rank += s_keys[q] > c;
      if (rank < p.k) out[rank] = c;
    } else if (tid < p.k) {
      out[tid] = 0ull;  // fewer than k entries in the chunk
    }
    return;
  }
  // many entries tie at the threshold: per-warp top k from registers, then warp 0 merges
  unsigned long long keys[kMxEpt];
#pragma unroll
  for (int e = 0; e < kMxEpt; ++e) {
    const int v = v0 + entry_offset(mode, tid, e);
    keys[e] = v < v1 ? order_key(order_u(x[e]), v) : 0ull;
  }
  unsigned long long below = ~0ull;
  for (int r = 0; r < p.k; ++r) {
    below = warp_max_below(keys, below);
    if (lane == 0) s_cand[warp * kMaxTopk + r] = below;  // 0 once the warp's keys are exhausted
  }
  __syncthreads();
  if (warp == 0) {  // the chunk's top-k among the warps' candidates (kWarps * k <= 256)
    constexpr int kPerC = kWarps * kMaxTopk / 32;
    unsigned long long c[kPerC];
#pragma unroll
    for (int e = 0; e < kPerC; ++e) {
      const int q = lane + 32 * e, w = q / kMaxTopk, r = q % kMaxTopk;
      c[e] = (r < p.k) ? s_cand[w * kMaxTopk + r] : 0ull;
    }
    below = ~0ull;
    for (int r = 0; r < p.k; ++r) {
      below = warp_max_below(c, below);
      if (lane == 0) out[r] = below;
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
  pdl_wait();  // the chunk candidates are complete (the topology above is an input of its own)
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

// Entries per chunk for n_chunks chunks of a V-entry row: rounded up to 8 entries so that chunk
// starts stay on 16-byte boundaries (vector loads); at most kMxThreads * kMxEpt whenever n_chunks
// covers the row at that length.  Trailing chunks may be short or empty.
int topk_chunk_len(int V, int n_chunks) {
  const int len = (V + n_chunks - 1) / n_chunks;
  return (len + 7) & ~7;
}

void launch_row_topk_chunks(const MedusaParams& p, cudaStream_t stream) {
  medusa_chunk_topk_kernel<<<dim3(p.n_chunks, p.B * p.K), kMxThreads, 0, stream>>>(p);
}

void launch_medusa(const MedusaParams& p, cudaStream_t stream) {
  medusa_chunk_topk_kernel<<<dim3(p.n_chunks, p.B * p.K), kMxThreads, 0, stream>>>(p);
  launch_dependent(medusa_expand_kernel, dim3(p.B), dim3(kMxThreads), 0, stream, p);
}

}  // namespace spectree

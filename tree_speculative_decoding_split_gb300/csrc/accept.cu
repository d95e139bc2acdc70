// K3: per-node acceptance, longest accepted root path and the bonus token.  One CTA per request.
//
// Rules: greedy argmax match (temperature 0, qiita "EAGLE-3とMedusaで実装するSpeculative Decoding
// 実践ガイド", section "結論・成果"); typical acceptance, p(x) >= min(eps, delta * exp(-H))
// (jisaku glossary "Medusa", section "Medusa-1: 典型的採択", which states only an entropy-based
// threshold; the formula is the Medusa-1 reading); rejection sampling, accept with
// min(1, T[x]/D[x]) and on rejection continue from norm(relu(T - D)) (qiita, section
// "棄却サンプリング：出力品質を保証する").  Every candidate after a rejection is discarded, and
// the path that passes acceptance furthest is kept (same section; tech-tldr
// "多トークン予測（Medusa・EAGLE）", section "ツリー検証").
//
// Greedy / typical: every child decision is independent, so each thread decides one node; the
// reachable set is built level by level over tree depth (a barrier per level, at most the tree
// depth), and the deepest reachable node with the lowest index is found by a block reduction.
// Rejection: the walk is sequential over siblings; each rejected sibling costs one pass over the
// vocabulary (R <- relu(R - D_e) and its sum) by all 1024 threads, and the bonus token is an
// inverse-CDF search (per-thread chunk sums, a block scan, then one chunk).

#include "common.cuh"
#include "kernels.cuh"

namespace spectree {

namespace {

__device__ __forceinline__ void zero_outputs(const AcceptParams& p, int b, int tid, int nthreads) {
  for (int j = tid; j < p.path_cap; j += nthreads) p.path[(size_t)b * p.path_cap + j] = (j == 0) ? 0 : -1;
  if (tid == 0) {
    p.accept_len[b] = 0;
    p.bonus[b] = -1;
    if (p.margin_count) p.margin_count[b] = 0;
    if (p.bonus_margin) p.bonus_margin[b] = 0;
  }
}

// Writes path = root .. e (depth(e) + 1 entries) and pads with -1.
__device__ void write_path(const AcceptParams& p, int b, int e, int dep, const int* s_parent, int tid,
                           int nthreads) {
  int32_t* out = p.path + (size_t)b * p.path_cap;
  for (int j = tid; j < p.path_cap; j += nthreads)
    if (j > dep) out[j] = -1;
  if (tid == 0) {
    int node = e;
    for (int j = dep; j >= 0; --j) {
      out[j] = node;
      node = (node > 0) ? s_parent[node] : -1;
    }
  }
}

}  // namespace

// ---- greedy / typical -----------------------------------------------------------------------

__global__ void __launch_bounds__(256) accept_tree_kernel(const AcceptParams p) {
  __shared__ int s_parent[kMaxNodes];
  __shared__ int s_depth[kMaxNodes];
  __shared__ unsigned char s_acc[kMaxNodes];
  __shared__ unsigned char s_ok[kMaxNodes];
  __shared__ unsigned char s_mg[kMaxNodes];
  __shared__ int s_red[8];
  __shared__ int s_red2[8];
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (p.bad[b]) {
    zero_outputs(p, b, tid, blockDim.x);
    return;
  }
  const int n = p.n_nodes[b];
  const size_t rb = (size_t)b * p.N;
  int maxdep = 0;
  for (int c = tid; c < n; c += blockDim.x) {
    const int par = p.parent[rb + c];
    const int dep = p.depth[rb + c];
    s_parent[c] = par;
    s_depth[c] = dep;
    maxdep = max(maxdep, dep);
    unsigned char acc = 1, mg = 0;
    if (c > 0) {
      const size_t pr = rb + par;
      if (p.rule == SPEC_RULE_GREEDY) {
        acc = p.tokens[rb + c] == p.rarg[pr];
        mg = p.rgap[pr] < kMargin;
      } else {
        const float lp = p.clog[rb + c] * p.inv_tau - p.rlse[pr];
        const float lthr = fminf(p.log_eps, p.log_delta - p.rent[pr]);
        acc = lp >= lthr;
        mg = (lthr > -INFINITY) && fabsf(lp - lthr) < kMargin;
      }
    }
    s_acc[c] = acc;
    s_mg[c] = mg;
    s_ok[c] = (c == 0);
  }
  // block max of depth
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) maxdep = max(maxdep, __shfl_xor_sync(0xffffffffu, maxdep, o));
  if (lane == 0) s_red[warp] = maxdep;
  __syncthreads();
  maxdep = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) maxdep = max(maxdep, s_red[w]);
  for (int d = 1; d <= maxdep; ++d) {
    for (int c = tid; c < n; c += blockDim.x)
      if (s_depth[c] == d) s_ok[c] = s_acc[c] && s_ok[s_parent[c]];
    __syncthreads();
  }
  // deepest reachable node, lowest index on ties; margins of the evaluated decisions
  int key = -1, mcount = 0;
  for (int c = tid; c < n; c += blockDim.x) {
    if (s_ok[c]) key = max(key, (s_depth[c] << 16) | (0xFFFF - c));
    if (c > 0 && s_ok[s_parent[c]] && s_mg[c]) ++mcount;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    key = max(key, __shfl_xor_sync(0xffffffffu, key, o));
    mcount += __shfl_xor_sync(0xffffffffu, mcount, o);
  }
  __syncthreads();
  if (lane == 0) {
    s_red[warp] = key;
    s_red2[warp] = mcount;
  }
  __syncthreads();
  key = -1;
  mcount = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) {
    key = max(key, s_red[w]);
    mcount += s_red2[w];
  }
  const int e = 0xFFFF - (key & 0xFFFF);
  const int dep = key >> 16;
  if (dep + 1 > p.path_cap) {
    if (tid == 0) set_status(p.dev_status, SPEC_ERR_CAPACITY);
    zero_outputs(p, b, tid, blockDim.x);
    return;
  }
  write_path(p, b, e, dep, s_parent, tid, blockDim.x);
  if (tid == 0) {
    p.accept_len[b] = dep;
    p.bonus[b] = p.rarg[rb + e];
    if (p.margin_count) p.margin_count[b] = mcount;
    if (p.bonus_margin) p.bonus_margin[b] = p.rgap[rb + e] < kMargin;
  }
}

// ---- rejection sampling ---------------------------------------------------------------------

namespace {

constexpr int kRejThreads = 1024;

__device__ __forceinline__ float block_sum_f(float v, float* s_tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) s_tmp[warp] = v;
  __syncthreads();
  float t = (lane < (int)(blockDim.x >> 5)) ? s_tmp[lane] : 0.f;
  t = warp_sum(t);
  return t;  // every thread holds the total
}

}  // namespace

__global__ void __launch_bounds__(kRejThreads) accept_rejection_kernel(const AcceptParams p) {
  __shared__ int s_parent[kMaxNodes];
  __shared__ int s_tok[kMaxNodes];
  __shared__ int s_kids[kMaxNodes];
  __shared__ float s_tmp[32];
  __shared__ double s_dtmp[32];
  __shared__ int s_nk, s_accept, s_owner;
  __shared__ int s_found;
  __shared__ float s_mgflag;
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (p.bad[b] || (p.map_bad && *p.map_bad)) {
    zero_outputs(p, b, tid, blockDim.x);
    return;
  }
  const int n = p.n_nodes[b];
  const size_t rb = (size_t)b * p.N;
  const int V = p.V;
  for (int c = tid; c < n; c += blockDim.x) {
    s_parent[c] = p.parent[rb + c];
    s_tok[c] = p.tokens[rb + c];
  }
  float* Rb[2] = {p.rbuf + (size_t)b * 2 * V, p.rbuf + (size_t)b * 2 * V + V};
  int cur = 0;           // Rb[cur] holds the unnormalised residual when !lazy
  bool lazy = true;      // R is T_e = softmax(z_e / tau), computed on the fly from logits
  float S = 1.f;         // sum of Rb[cur]
  int e = 0, dep = 0, margins = 0;
  __syncthreads();

  auto draft_at = [&](int node, int v) -> float {
    const float* row = p.draft + (rb + node) * (size_t)p.Vd;
    if (p.inv_map) {
      const int j = p.inv_map[v];
      return j >= 0 ? row[j] : 0.f;
    }
    return row[v];
  };

  while (true) {
    if (tid == 0) {
      int k = 0;
      for (int c = e + 1; c < n; ++c)
        if (s_parent[c] == e) s_kids[k++] = c;
      s_nk = k;
    }
    __syncthreads();
    const int nk = s_nk;
    const size_t erow = rb + e;
    const float* lg = p.logits + erow * (size_t)V;
    const float lse_e = p.rlse[erow];
    bool moved = false;
    for (int k = 0; k < nk; ++k) {
      const int c = s_kids[k];
      if (tid == 0) {
        const int x = s_tok[c];
        const float u = accept_uniform(p.seed, (uint32_t)b, (uint32_t)c, 0u);
        const float Dx = draft_at(e, x);
        const float Rx = lazy ? expf(lg[x] * p.inv_tau - lse_e) : Rb[cur][x] / S;
        const float a = (Dx > 0.f) ? fminf(1.f, Rx / Dx) : (Rx > 0.f ? 1.f : 0.f);
        if (fabsf(u - a) < kMargin) ++margins;
        s_accept = (u * Dx < Rx) ? 1 : 0;
      }
      __syncthreads();
      if (s_accept) {
        e = c;
        ++dep;
        lazy = true;
        S = 1.f;
        moved = true;
        break;
      }
      // residual pass: Rnext = relu(R - D_e), S' = sum Rnext
      float* Rn = Rb[cur ^ 1];
      const float* Rc = Rb[cur];
      const float invS = 1.f / S;
      float part = 0.f;
      for (int v = tid; v < V; v += blockDim.x) {
        const float r = lazy ? expf(lg[v] * p.inv_tau - lse_e) : Rc[v] * invS;
        const float nv = fmaxf(r - draft_at(e, v), 0.f);
        Rn[v] = nv;
        part += nv;
      }
      const float Snew = block_sum_f(part, s_tmp);
      if (Snew > 0.f) {
        cur ^= 1;
        S = Snew;
        lazy = false;
      }
      __syncthreads();
    }
    if (!moved) break;
    __syncthreads();
  }

  if (dep + 1 > p.path_cap) {
    if (tid == 0) set_status(p.dev_status, SPEC_ERR_CAPACITY);
    __syncthreads();
    zero_outputs(p, b, tid, blockDim.x);
    return;
  }

  // ---- bonus token: inverse CDF of R at u' = U(seed, b, e, 1) ----
  const size_t erow = rb + e;
  const float* lg = p.logits + erow * (size_t)V;
  const float lse_e = p.rlse[erow];
  const float* Rc = Rb[cur];
  auto rval = [&](int v) -> float { return lazy ? expf(lg[v] * p.inv_tau - lse_e) : Rc[v]; };
  const int CH = (V + kRejThreads - 1) / kRejThreads;
  const int v0 = tid * CH, v1 = min(V, v0 + CH);
  float csum = 0.f;
  for (int v = v0; v < v1; ++v) csum += rval(v);
  // block-wide inclusive scan of the chunk sums in double
  double incl = (double)csum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_dtmp[warp] = incl;
  if (tid == 0) { s_owner = -1; s_found = -1; s_mgflag = 0.f; }
  __syncthreads();
  double wpre = 0.0;
  for (int w = 0; w < warp; ++w) wpre += s_dtmp[w];
  const double excl = wpre + incl - (double)csum;
  double total = 0.0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) total += s_dtmp[w];
  const float u2 = accept_uniform(p.seed, (uint32_t)b, (uint32_t)e, 1u);
  const double target = (double)u2 * total;
  // owner: the last chunk with mass that starts at or below the target
  if (csum > 0.f && excl <= target) atomicMax(&s_owner, tid);
  __syncthreads();
  if (tid == s_owner) {
    double acc = excl, prev = excl;
    int found = -1, last_nz = -1;
    for (int v = v0; v < v1; ++v) {
      const float r = rval(v);
      if (r > 0.f) last_nz = v;
      prev = acc;
      acc += (double)r;
      if (acc > target) { found = v; break; }
    }
    if (found < 0) { found = last_nz; prev = acc; }
    const double band = (double)kMargin * total;
    const bool near = (target - prev < band) || (acc - target < band);
    s_found = found;
    s_mgflag = near ? 1.f : 0.f;
  }
  __syncthreads();
  int bonus = s_found;
  if (bonus < 0) bonus = V - 1;  // no mass at all (cannot happen for a softmax row)
  // any boundary within the band also counts when the crossing sits at a chunk edge
  if (tid == 0) {
    write_path(p, b, e, dep, s_parent, 0, 1);  // single-thread write of root..e
    p.accept_len[b] = dep;
    p.bonus[b] = bonus;
    if (p.margin_count) p.margin_count[b] = margins;
    if (p.bonus_margin) p.bonus_margin[b] = (s_mgflag > 0.f || target < (double)kMargin * total) ? 1 : 0;
  }
  for (int j = tid; j < p.path_cap; j += blockDim.x)
    if (j > dep) p.path[(size_t)b * p.path_cap + j] = -1;
}

// ---- draft map inversion --------------------------------------------------------------------

__global__ void __launch_bounds__(256) inverse_map_kernel(const int32_t* __restrict__ map, int Vd, int V,
                                                          int32_t* __restrict__ inv, int32_t* map_bad,
                                                          int32_t* dev_status) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= Vd) return;
  const int x = map[j];
  if (x < 0 || x >= V || atomicCAS(&inv[x], -1, j) != -1) {
    atomicExch(map_bad, 1);
    set_status(dev_status, SPEC_ERR_BAD_TOKEN);
  }
}

void launch_build_inverse_map(const int32_t* map, int Vd, int V, int32_t* inv, int32_t* map_bad,
                              int32_t* dev_status, cudaStream_t stream) {
  cudaMemsetAsync(inv, 0xFF, (size_t)V * sizeof(int32_t), stream);
  cudaMemsetAsync(map_bad, 0, sizeof(int32_t), stream);
  inverse_map_kernel<<<(Vd + 255) / 256, 256, 0, stream>>>(map, Vd, V, inv, map_bad, dev_status);
}

void launch_accept(const AcceptParams& p, cudaStream_t stream) {
  if (p.rule == SPEC_RULE_REJECTION)
    accept_rejection_kernel<<<p.B, kRejThreads, 0, stream>>>(p);
  else
    accept_tree_kernel<<<p.B, 256, 0, stream>>>(p);
}

}  // namespace spectree

// K2r: per-row statistics and child logits.  K3: per-node acceptance, longest accepted root path
// and the bonus token.
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
// Row finalisation: one CTA per tree row merges the row's LM-head statistics records, computes
// the row's child logit z[parent][token] (typical acceptance) and publishes the row; the CTA
// that completes a request (an atomic arrival counter, nothing waits) then decides the whole
// request for greedy / typical acceptance: every node's decision is independent, reachability
// and depth come from pointer jumping over the parent array (8 rounds for 255 nodes), and the
// deepest reachable node with the lowest index wins.
// Rejection: the walk is sequential over siblings; each rejected sibling costs one pass over the
// vocabulary (R <- relu(R - D_e) and its sum) by all 1024 threads of the request's CTA, and the
// bonus token is an inverse-CDF search (per-thread chunk sums, a block scan, then one chunk).

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

// Loads request b's parent array (and tokens) into shared memory and validates the tree:
// 1 <= n <= N, parent[0] = -1, 0 <= parent[c] < c, 0 <= token[c] < V.  Every thread of the block
// calls it; returns 0 or a status code (the same in every thread).
__device__ int load_and_validate(const AcceptParams& p, int b, int* s_par, int* s_tok) {
  const int n = p.n_nodes[b];
  const bool n_ok = n >= 1 && n <= p.N;
  int bad_tree = !n_ok, bad_tok = 0;
  if (n_ok) {
    for (int c = threadIdx.x; c < n; c += blockDim.x) {
      const int par = p.parent[(size_t)b * p.N + c];
      const int tok = p.tokens[(size_t)b * p.N + c];
      s_par[c] = par;
      if (s_tok) s_tok[c] = tok;
      if (c == 0 ? par != -1 : (par < 0 || par >= c)) bad_tree = 1;
      if (c > 0 && (tok < 0 || tok >= p.V)) bad_tok = 1;
    }
  }
  bad_tree = __syncthreads_or(bad_tree);
  bad_tok = __syncthreads_or(bad_tok);
  return bad_tree ? SPEC_ERR_BAD_TREE : (bad_tok ? SPEC_ERR_BAD_TOKEN : 0);
}

// Writes path = root .. e (depth(e) + 1 entries), -1 beyond.
__device__ void write_path(const AcceptParams& p, int b, int e, int dep, const int* s_par) {
  int32_t* out = p.path + (size_t)b * p.path_cap;
  for (int j = threadIdx.x; j < p.path_cap; j += blockDim.x)
    if (j > dep) out[j] = -1;
  if (threadIdx.x == 0) {
    int node = e;
    for (int j = dep; j >= 0; --j) {
      out[j] = node;
      node = (node > 0) ? s_par[node] : -1;
    }
  }
}

// Greedy / typical acceptance of request b by one CTA of >= 256 threads (one node per thread).
// Row statistics are read with L1-bypassing loads: other CTAs published them.
__device__ void accept_tree_block(const AcceptParams& p, int b) {
  __shared__ int s_par[kMaxNodes];
  __shared__ int s_jump[kMaxNodes];
  __shared__ int s_dep[kMaxNodes];
  __shared__ unsigned char s_ok[kMaxNodes];
  __shared__ unsigned char s_mg[kMaxNodes];
  __shared__ int s_red[32];
  __shared__ int s_red2[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
  const int err = load_and_validate(p, b, s_par, nullptr);
  if (err) {
    if (tid == 0) set_status(p.dev_status, err);
    zero_outputs(p, b, tid, blockDim.x);
    return;
  }
  const int n = p.n_nodes[b];
  const size_t rb = (size_t)b * p.N;
  int par = -1;
  if (tid < n) {
    par = s_par[tid];
    unsigned char acc = 1, mg = 0;
    if (tid > 0) {
      const size_t pr = rb + par;
      if (p.rule == SPEC_RULE_GREEDY) {
        acc = p.tokens[rb + tid] == __ldcg(p.rarg + pr);
        mg = __ldcg(p.rgap + pr) < kMargin;
      } else {
        const float lp = __ldcg(p.clog + rb + tid) * p.inv_tau - __ldcg(p.rlse + pr);
        const float lthr = fminf(p.log_eps, p.log_delta - __ldcg(p.rent + pr));
        acc = lp >= lthr;
        mg = (lthr > -INFINITY) && fabsf(lp - lthr) < kMargin;
      }
    }
    s_ok[tid] = acc;
    s_mg[tid] = mg;
    s_dep[tid] = tid > 0 ? 1 : 0;
    s_jump[tid] = tid > 0 ? par : 0;
  }
  __syncthreads();
  // Pointer jumping: s_ok[c] = AND of the decisions from c up to (not including) s_jump[c],
  // s_dep[c] = number of edges to s_jump[c]; done when every jump reaches the root.
  for (int round = 0; round < 8; ++round) {
    int j = 0, nj = 0, nd = 0;
    unsigned char nok = 0;
    if (tid < n) {
      j = s_jump[tid];
      if (j != 0) {
        nj = s_jump[j];
        nd = s_dep[tid] + s_dep[j];
        nok = s_ok[tid] & s_ok[j];
      }
    }
    __syncthreads();
    if (tid < n && j != 0) {
      s_jump[tid] = nj;
      s_dep[tid] = nd;
      s_ok[tid] = nok;
    }
    __syncthreads();
  }
  int key = -1, mcount = 0;
  if (tid < n) {
    if (s_ok[tid]) key = (s_dep[tid] << 16) | (0xFFFF - tid);
    if (tid > 0 && s_ok[par] && s_mg[tid]) mcount = 1;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    key = max(key, __shfl_xor_sync(0xffffffffu, key, o));
    mcount += __shfl_xor_sync(0xffffffffu, mcount, o);
  }
  if (lane == 0) {
    s_red[warp] = key;
    s_red2[warp] = mcount;
  }
  __syncthreads();
  key = -1;
  mcount = 0;
  for (int w = 0; w < nw; ++w) {
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
  write_path(p, b, e, dep, s_par);
  if (tid == 0) {
    p.accept_len[b] = dep;
    p.bonus[b] = __ldcg(p.rarg + rb + e);
    if (p.margin_count) p.margin_count[b] = mcount;
    if (p.bonus_margin) p.bonus_margin[b] = __ldcg(p.rgap + rb + e) < kMargin;
  }
}

__device__ __forceinline__ RowPart shfl_rowpart(const RowPart& a, int o) {
  RowPart r;
  r.m = __shfl_xor_sync(0xffffffffu, a.m, o);
  r.s = __shfl_xor_sync(0xffffffffu, a.s, o);
  r.t = __shfl_xor_sync(0xffffffffu, a.t, o);
  r.y2 = __shfl_xor_sync(0xffffffffu, a.y2, o);
  r.idx = __shfl_xor_sync(0xffffffffu, a.idx, o);
  return r;
}

__device__ __forceinline__ float block_sum_f(float v, float* s_tmp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) s_tmp[warp] = v;
  __syncthreads();
  float t = (lane < (int)(blockDim.x >> 5)) ? s_tmp[lane] : 0.f;
  return warp_sum(t);  // every thread holds the total
}

}  // namespace

// ---- K2r: row finalisation (+ fused greedy / typical acceptance) ------------------------------

constexpr int kFinThreads = 256;

__global__ void __launch_bounds__(kFinThreads) row_finalize_kernel(const FinalizeParams p) {
  __shared__ float4 s_part[kFinThreads / 32];
  __shared__ int s_pidx[kFinThreads / 32];
  __shared__ float s_tmp[32];
  __shared__ int s_last;
  const int n = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = n / p.N, i = n % p.N;
  const int nb = p.acc.n_nodes[b];
  const bool real = i < nb && nb <= p.N;
  RowPart acc = rowpart_empty();
  if (real) {
    for (int s = tid; s < p.n_parts; s += kFinThreads) {
      const float4 f = p.part[(size_t)s * p.R + n];
      RowPart o;
      o.m = f.x; o.s = f.y; o.t = f.z; o.y2 = f.w; o.idx = p.part_idx[(size_t)s * p.R + n];
      acc = rowpart_merge(acc, o);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc = rowpart_merge(acc, shfl_rowpart(acc, o));
    if (lane == 0) {
      s_part[warp] = make_float4(acc.m, acc.s, acc.t, acc.y2);
      s_pidx[warp] = acc.idx;
    }
  }
  // child logit z[parent(i)][token(i)] (typical acceptance reads it; rejection reads the logits)
  float clog = 0.f;
  if (real && i > 0 && p.acc.rule == SPEC_RULE_TYPICAL) {
    const int pn = p.acc.parent[n];
    const int x = p.acc.tokens[n];
    if (pn >= 0 && pn < i && x >= 0 && x < p.V) {  // invalid trees are reported by the acceptance
      const size_t prow = (size_t)b * p.N + pn;
      float d = 0.f;
      if (p.logits) {
        d = (tid == 0) ? p.logits[prow * p.V + x] : 0.f;
      } else if (p.is_bf16) {
        const __nv_bfloat16* hw = static_cast<const __nv_bfloat16*>(p.hidden) + prow * p.Hd;
        const __nv_bfloat16* ww = static_cast<const __nv_bfloat16*>(p.weight) + (size_t)x * p.Hd;
        for (int k = tid * 8; k < p.Hd; k += kFinThreads * 8) {
          const uint4 hv = *reinterpret_cast<const uint4*>(hw + k);
          const uint4 wv = *reinterpret_cast<const uint4*>(ww + k);
          const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&hv);
          const __nv_bfloat162* w2 = reinterpret_cast<const __nv_bfloat162*>(&wv);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 hf = __bfloat1622float2(h2[e]);
            const float2 wf = __bfloat1622float2(w2[e]);
            d = fmaf(hf.x, wf.x, d);
            d = fmaf(hf.y, wf.y, d);
          }
        }
      } else {
        const float* hw = static_cast<const float*>(p.hidden) + prow * p.Hd;
        const float* ww = static_cast<const float*>(p.weight) + (size_t)x * p.Hd;
        for (int k = tid; k < p.Hd; k += kFinThreads) d = fmaf(hw[k], ww[k], d);
      }
      clog = block_sum_f(d, s_tmp);
    }
  }
  __syncthreads();
  if (tid == 0) {
    float mx = 0.f, lse = 0.f, ent = 0.f, gap = 0.f;
    int am = -1;
    if (real) {
      acc = rowpart_empty();
      for (int w = 0; w < kFinThreads / 32; ++w) {
        RowPart o;
        o.m = s_part[w].x; o.s = s_part[w].y; o.t = s_part[w].z; o.y2 = s_part[w].w; o.idx = s_pidx[w];
        acc = rowpart_merge(acc, o);
      }
      mx = acc.m;
      lse = acc.m + logf(acc.s);
      ent = lse - acc.t / acc.s;
      am = acc.idx;
      gap = (acc.y2 == -INFINITY) ? INFINITY : (acc.m - acc.y2) / p.acc.inv_tau;
    }
    p.rmax[n] = mx; p.rlse[n] = lse; p.rent[n] = ent; p.rgap[n] = gap; p.rarg[n] = am; p.clog[n] = clog;
    if (p.hook_max) p.hook_max[n] = mx;
    if (p.hook_lse) p.hook_lse[n] = lse;
    if (p.hook_ent) p.hook_ent[n] = ent;
    if (p.hook_arg) p.hook_arg[n] = am;
    s_last = 0;
    if (p.fuse_accept) {
      __threadfence();  // publish this row before arriving
      s_last = atomicAdd(&p.counters[b], 1) == p.N - 1;
    }
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();  // every row of request b is visible from here on
  accept_tree_block(p.acc, b);
}

void launch_row_finalize(const FinalizeParams& p, cudaStream_t stream) {
  row_finalize_kernel<<<p.R, kFinThreads, 0, stream>>>(p);
}

// ---- rejection sampling ---------------------------------------------------------------------

namespace {
constexpr int kRejThreads = 1024;
}

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
  const int err = load_and_validate(p, b, s_parent, s_tok);
  if (err || (p.map_bad && *p.map_bad)) {
    if (tid == 0 && err) set_status(p.dev_status, err);
    zero_outputs(p, b, tid, blockDim.x);
    return;
  }
  const int n = p.n_nodes[b];
  const size_t rb = (size_t)b * p.N;
  const int V = p.V;
  float* Rb[2] = {p.rbuf + (size_t)b * 2 * V, p.rbuf + (size_t)b * 2 * V + V};
  int cur = 0;           // Rb[cur] holds the unnormalised residual when !lazy
  bool lazy = true;      // R is T_e = softmax(z_e / tau), computed on the fly from logits
  float S = 1.f;         // sum of Rb[cur]
  int e = 0, dep = 0, margins = 0;

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
  write_path(p, b, e, dep, s_parent);
  if (tid == 0) {
    p.accept_len[b] = dep;
    p.bonus[b] = bonus;
    if (p.margin_count) p.margin_count[b] = margins;
    if (p.bonus_margin) p.bonus_margin[b] = (s_mgflag > 0.f || target < (double)kMargin * total) ? 1 : 0;
  }
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
  accept_rejection_kernel<<<p.B, kRejThreads, 0, stream>>>(p);
}

}  // namespace spectree

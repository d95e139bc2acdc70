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
// vocabulary (R <- relu(R - D_e) and its sum).  A request runs on a thread-block cluster of up
// to 8 CTAs that split the vocabulary: each thread keeps its slice of R in registers and of D_e
// in shared memory, so a rejected sibling costs one on-chip pass and one cluster barrier (the
// partial sums are exchanged through distributed shared memory).  The bonus token is an
// inverse-CDF search: per-warp segment sums, a prefix over CTAs, then one warp scans its segment.
// Vocabularies above 8 x 32768 entries use a single CTA per request with R in global memory.

#include <cooperative_groups.h>

#include <climits>
#include <mutex>

#include "common.cuh"
#include "compact.cuh"
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
      if (c > 0 && p.draft_rows && par >= 0 && par < c) {  // a parent's draft row must exist
        const int dr = p.draft_rows[(size_t)b * p.N + par];
        if (dr < 0 || dr >= p.n_draft_rows) bad_tok = 1;
      }
    }
  }
  bad_tree = __syncthreads_or(bad_tree);
  bad_tok = __syncthreads_or(bad_tok);
  return bad_tree ? SPEC_ERR_BAD_TREE : (bad_tok ? SPEC_ERR_BAD_TOKEN : 0);
}

// ln sum_v exp(z_v / tau) of tree row `row` (rejection), merged by one warp from the LM head's
// per-slice records {max, sum of exp(z / tau - max)}: every lane a strided share, then a shuffle
// merge -- the same order in every CTA, so every CTA of a cluster gets the same value.
__device__ __forceinline__ float row_lse_warp(const AcceptParams& p, size_t row, int lane) {
  float m = -INFINITY, s = 0.f;
  for (int k = lane; k < p.n_parts; k += 32) {
    const float4 f = p.part[(size_t)k * p.R + row];
    const float mm = fmaxf(m, f.x);
    if (mm > -INFINITY)
      s = (s > 0.f ? s * expf(m - mm) : 0.f) + (f.y > 0.f ? f.y * expf(f.x - mm) : 0.f);
    m = mm;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float om = __shfl_xor_sync(0xffffffffu, m, o), os = __shfl_xor_sync(0xffffffffu, s, o);
    const float mm = fmaxf(m, om);
    if (mm > -INFINITY)
      s = (s > 0.f ? s * expf(m - mm) : 0.f) + (os > 0.f ? os * expf(om - mm) : 0.f);
    m = mm;
  }
  return m + logf(s);
}

// Node e's draft distribution (rejection): row b * N + e, or the compact row draft_rows[b][e].
// Called only for nodes with children, whose rows load_and_validate has checked.
__device__ __forceinline__ const float* draft_row(const AcceptParams& p, int b, int e) {
  const size_t r = p.draft_rows ? (size_t)p.draft_rows[(size_t)b * p.N + e] : (size_t)b * p.N + e;
  return p.draft + r * (size_t)p.Vd;
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

// Compacts request b's accepted K/V (the path and length this call just wrote) on KV heads g0,
// g0 + gstep, ..., with the block's dynamic shared memory as staging.
__device__ __forceinline__ void fused_compact_tail(const AcceptParams& p, int b, int g0, int gstep) {
  extern __shared__ uint4 s_cbuf[];
  __syncthreads();
  const int len = p.accept_len[b];
  compact_request(p.cp, p.path + (size_t)b * p.path_cap, len, b, g0, gstep, s_cbuf,
                  reinterpret_cast<int*>(s_cbuf + kCompactBufChunks));
}


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
  if (p.acc.fuse_compact) fused_compact_tail(p.acc, b, 0, 1);
}

constexpr int kFusedCompactSmem = kCompactBufChunks * 16 + kCompactBufChunks / 8 * 4;

void launch_row_finalize(const FinalizeParams& p, cudaStream_t stream) {
  row_finalize_kernel<<<p.R, kFinThreads, p.acc.fuse_compact ? kFusedCompactSmem : 0, stream>>>(p);
}

// ---- rejection sampling ---------------------------------------------------------------------

namespace {
constexpr int kRejThreads = 1024;
}

__device__ void rejection_block_walk(const AcceptParams& p) {
  __shared__ int s_parent[kMaxNodes];
  __shared__ int s_tok[kMaxNodes];
  __shared__ int s_kids[kMaxNodes];
  __shared__ float s_tmp[32];
  __shared__ double s_dtmp[32];
  __shared__ int s_nk, s_accept, s_owner;
  __shared__ int s_found;
  __shared__ float s_mgflag;
  __shared__ float s_lse;
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

  auto draft_at = [&](const float* row, int v) -> float {
    if (p.inv_map) {
      const int j = p.inv_map[v];
      return j >= 0 ? row[j] : 0.f;
    }
    return row[v];
  };

  while (true) {
    if (warp == 0) {
      const float l = row_lse_warp(p, rb + e, lane);
      if (lane == 0) {
        int k = 0;
        for (int c = e + 1; c < n; ++c)
          if (s_parent[c] == e) s_kids[k++] = c;
        s_nk = k;
        s_lse = l;
      }
    }
    __syncthreads();
    const int nk = s_nk;
    const size_t erow = rb + e;
    const float* lg = p.logits + erow * (size_t)V;
    const float lse_e = s_lse;
    const float* de = nk > 0 ? draft_row(p, b, e) : nullptr;
    bool moved = false;
    for (int k = 0; k < nk; ++k) {
      const int c = s_kids[k];
      if (tid == 0) {
        const int x = s_tok[c];
        const float u = accept_uniform(p.seed, (uint32_t)b, (uint32_t)c, 0u);
        const float Dx = draft_at(de, x);
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
        const float nv = fmaxf(r - draft_at(de, v), 0.f);
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
  const float lse_e = s_lse;  // node e's, from its arrival
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

__global__ void __launch_bounds__(kRejThreads) accept_rejection_block_kernel(const AcceptParams p) {
  rejection_block_walk(p);
  if (p.fuse_compact) fused_compact_tail(p, blockIdx.x, 0, 1);
}

// ---- rejection sampling on a thread-block cluster ---------------------------------------------

namespace {

constexpr int kRcThreads = 512;    // threads per CTA
constexpr int kRcEpt = 64;         // vocabulary entries per thread (registers)
constexpr int kRcMaxCluster = 8;   // CTAs per request at most (portable cluster size)
constexpr int kRcSlice = kRcThreads * kRcEpt;  // vocabulary entries per CTA at most
constexpr int kRcSmem = kRcSlice * (int)sizeof(float);

// T(v) = softmax(z / tau)[v], and one residual step relu(R / S - D): written with explicit fused
// operations so that every CTA of a cluster evaluates them bit for bit alike.  T uses the fast
// exponential (__expf: a few ulp, relative error near 1e-6 over these arguments), far inside the
// 1e-4 band of the decisions it feeds.
__device__ __forceinline__ float target_prob(float z, float inv_tau, float lse) {
  return __expf(fmaf(z, inv_tau, -lse));
}
__device__ __forceinline__ float residual_step(float r, float inv_s, float d) {
  return fmaxf(fmaf(r, inv_s, -d), 0.f);
}

__device__ __forceinline__ void cp_async_4(float* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;\n" ::: "memory"); }

// Next child of `node` after child `after` (-1: the first child), from the children bitmask.
__device__ __forceinline__ int next_child(const uint32_t (*kids)[kAncWords], int node, int after) {
  const int from = after + 1;
  for (int w = from >> 5; w < kAncWords; ++w) {
    uint32_t m = kids[node][w];
    if (w == (from >> 5)) m &= ~0u << (from & 31);
    if (m) return w * 32 + __ffs(m) - 1;
  }
  return -1;
}

}  // namespace

// One request per cluster of kc CTAs; CTA `rank` holds vocabulary entries [rank*C, rank*C + C),
// C = ceil(V / kc), entry base + j*512 + tid in register r[j] of thread tid and its draft
// probability in s_D[j*512 + tid].  Every control decision (accept, adopt a residual, which CTA
// owns the bonus) is taken by every CTA from the same shared values in the same order, so all
// CTAs pass the same sequence of cluster barriers.  Exchanged values (partial sums, the next
// sibling's R and D entries) are double-buffered by barrier parity: a slot is rewritten only two
// barriers after it was read.
__device__ void rejection_cluster_walk(const AcceptParams& p) {
  namespace cg = cooperative_groups;
  cg::cluster_group cl = cg::this_cluster();
  extern __shared__ float4 s_dyn4[];
  float* s_D = reinterpret_cast<float*>(s_dyn4);  // D_e of this slice; R of the slice at the end
  __shared__ int s_parent[kMaxNodes];
  __shared__ int s_tok[kMaxNodes];
  __shared__ uint32_t s_kids[kMaxNodes][kAncWords];  // children of each node, as bits
  __shared__ float s_slot[2][3];                     // next sibling's R before / after, and D
  __shared__ float s_part[2][kRcMaxCluster];         // per-CTA residual sums
  __shared__ double s_tot[kRcMaxCluster];            // per-CTA mass of the final distribution
  __shared__ float s_red[kRcThreads / 32];
  __shared__ double s_dred[kRcThreads / 32];         // bonus: mass of the warps before each warp
  __shared__ double s_bonus[3];                      // bonus: total, this CTA's start, target
  __shared__ int s_owner, s_owner_cta;
  __shared__ float s_lse[2];                         // the visited row's LSE, by visit parity

  const int kc = (int)cl.num_blocks(), rank = (int)cl.block_rank();
  const int b = blockIdx.x / kc;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  cl.sync();  // every CTA of the cluster is running before any remote shared-memory access

  const int err = load_and_validate(p, b, s_parent, s_tok);
  if (err || (p.map_bad && *p.map_bad)) {
    if (rank == 0) {
      if (tid == 0 && err) set_status(p.dev_status, err);
      zero_outputs(p, b, tid, blockDim.x);
    }
    return;
  }
  const int n = p.n_nodes[b];
  for (int i = tid; i < n * kAncWords; i += kRcThreads) (&s_kids[0][0])[i] = 0u;
  __syncthreads();
  for (int c = 1 + tid; c < n; c += kRcThreads) atomicOr(&s_kids[s_parent[c]][c >> 5], 1u << (c & 31));
  __syncthreads();

  const int V = p.V;
  const int C = (V + kc - 1) / kc;
  const int base = rank * C;
  const int Lc = max(0, min(C, V - base));
  const size_t rb = (size_t)b * p.N;
  float r[kRcEpt];
  float S = 1.f;  // sum of the residual held in r (1 while r holds T_e itself)
  int e = 0, dep = 0, margins = 0, sp = 0, lp = 0;
  bool moved = true;

  while (moved) {
    // ---- arrive at node e: r <- T_e, s_D <- D_e (this slice; a leaf has no D_e) ----
    const int c_first = next_child(s_kids, e, -1);
    float lse_e;
    {
      const size_t erow = rb + e;
      const float* lg = p.logits + erow * (size_t)V + base;
      const float* drow = c_first >= 0 ? draft_row(p, b, e) : nullptr;
      if (warp == 0) {
        const float l = row_lse_warp(p, erow, lane);
        if (lane == 0) s_lse[lp] = l;
      }
      // The copies into s_D touch no registers of r: rolled loops leave the register file to r.
      // A mapped draft vocabulary: the slice's inverse map first, the logits while it lands,
      // then the gather of the draft entries it names.
      if (drow && p.inv_map) {
#pragma unroll 4
        for (int li = tid; li < Lc; li += kRcThreads) cp_async_4(s_D + li, p.inv_map + base + li);
        asm volatile("cp.async.commit_group;\n" ::: "memory");
      } else if (drow) {  // draft row in target order: this slice, asynchronously
#pragma unroll 4
        for (int li = tid; li < Lc; li += kRcThreads) cp_async_4(s_D + li, drow + base + li);
        asm volatile("cp.async.commit_group;\n" ::: "memory");
      }
#pragma unroll
      for (int j = 0; j < kRcEpt; ++j) {
        const int li = j * kRcThreads + tid;
        r[j] = (li < Lc) ? __ldg(lg + li) : 0.f;
      }
      if (drow && p.inv_map) {
        cp_async_wait_all();
#pragma unroll 4
        for (int li = tid; li < Lc; li += kRcThreads) {
          const int m = __float_as_int(s_D[li]);
          if (m >= 0)
            cp_async_4(s_D + li, drow + m);
          else
            s_D[li] = 0.f;
        }
        asm volatile("cp.async.commit_group;\n" ::: "memory");
      }
      // s_lse[lp] now holds this row's LSE; warp 0 writes this buffer again two visits on, after
      // every thread has passed the next visit's barrier (and so has read it)
      __syncthreads();
      lse_e = s_lse[lp];
      lp ^= 1;
#pragma unroll
      for (int j = 0; j < kRcEpt; ++j) {
        const int li = j * kRcThreads + tid;
        r[j] = (li < Lc) ? target_prob(r[j], p.inv_tau, lse_e) : 0.f;
      }
      S = 1.f;
      cp_async_wait_all();  // each thread reads back only the entries it copied
    }
    moved = false;
    int c = c_first;
    if (c < 0) break;  // a leaf: the bonus is drawn from T_e
    // the first child sees R = T_e: every CTA evaluates R[x] and D[x] itself
    const size_t erow = rb + e;
    {
      const int x = s_tok[c];
      const float* drow = draft_row(p, b, e);
      float rx = target_prob(__ldg(p.logits + erow * (size_t)V + x), p.inv_tau, lse_e);
      float dx;
      if (p.inv_map) {
        const int m = __ldg(p.inv_map + x);
        dx = m >= 0 ? __ldg(drow + m) : 0.f;
      } else {
        dx = __ldg(drow + x);
      }
      float pend_inv = 0.f;  // > 0: the residual step with this 1/S is still to be applied to r
      while (true) {
        const float u = accept_uniform(p.seed, (uint32_t)b, (uint32_t)c, 0u);
        const float Rx = rx / S;
        const float a = (dx > 0.f) ? fminf(1.f, Rx / dx) : (Rx > 0.f ? 1.f : 0.f);
        if (fabsf(u - a) < kMargin) ++margins;
        if (u * dx < Rx) {
          e = c;
          ++dep;
          moved = true;
          break;
        }
        // rejected: apply a pending residual step, then this slice's sum of relu(R / S - D)
        const int nc = next_child(s_kids, e, c);
        const float inv_s = 1.f / S;
        float part = 0.f;
        if (pend_inv > 0.f) {
#pragma unroll
          for (int j = 0; j < kRcEpt; ++j) {
            const int li = j * kRcThreads + tid;
            if (li < Lc) {
              const float d = s_D[li];
              r[j] = residual_step(r[j], pend_inv, d);
              part += residual_step(r[j], inv_s, d);
            }
          }
        } else {
#pragma unroll
          for (int j = 0; j < kRcEpt; ++j) {
            const int li = j * kRcThreads + tid;
            if (li < Lc) part += residual_step(r[j], inv_s, s_D[li]);
          }
        }
        part = warp_sum(part);
        if (lane == 0) s_red[warp] = part;
        if (nc >= 0) {  // the owner of the next sibling's token publishes R[x] before and after
          const int xo = s_tok[nc];
          const int owner = xo / C, li = xo - owner * C;
          if (owner == rank && li % kRcThreads == tid) {
            const int jj = li / kRcThreads;
            float ro = 0.f;
#pragma unroll
            for (int j = 0; j < kRcEpt; ++j)
              if (j == jj) ro = r[j];
            const float dd = s_D[li];
            const float rn = residual_step(ro, inv_s, dd);
            for (int q = 0; q < kc; ++q) {
              float* dst = cl.map_shared_rank(&s_slot[sp][0], q);
              dst[0] = ro;
              dst[1] = rn;
              dst[2] = dd;
            }
          }
        }
        __syncthreads();
        if (tid == 0) {
          float cta = 0.f;
          for (int w = 0; w < kRcThreads / 32; ++w) cta += s_red[w];
          for (int q = 0; q < kc; ++q) cl.map_shared_rank(&s_part[sp][0], q)[rank] = cta;
        }
        cl.sync();
        float s_new = 0.f;
        for (int q = 0; q < kc; ++q) s_new += s_part[sp][q];
        const bool adopt = s_new > 0.f;  // otherwise R stays as it is
        pend_inv = adopt ? inv_s : 0.f;
        if (adopt) S = s_new;
        if (nc >= 0) {
          rx = adopt ? s_slot[sp][1] : s_slot[sp][0];
          dx = s_slot[sp][2];
        }
        sp ^= 1;
        if (nc < 0) break;
        c = nc;
      }
      if (!moved && pend_inv > 0.f) {
#pragma unroll
        for (int j = 0; j < kRcEpt; ++j) {
          const int li = j * kRcThreads + tid;
          if (li < Lc) r[j] = residual_step(r[j], pend_inv, s_D[li]);
        }
      }
    }
  }

  if (dep + 1 > p.path_cap) {
    if (rank == 0) {
      if (tid == 0) set_status(p.dev_status, SPEC_ERR_CAPACITY);
      zero_outputs(p, b, tid, blockDim.x);
    }
    return;
  }

  // ---- bonus token: inverse CDF of R at u' = U(seed, b, e, 1) ----
  // R (unnormalised; T_e when no residual was adopted at e) goes to shared memory in vocabulary
  // order; thread t owns the contiguous chunk [t*CH, t*CH + CH) with CH odd, so that a warp's
  // chunk reads fall in distinct banks.
  __syncthreads();
#pragma unroll
  for (int j = 0; j < kRcEpt; ++j) {
    const int li = j * kRcThreads + tid;
    if (li < Lc) s_D[li] = r[j];
  }
  __syncthreads();
  const int CH = ((Lc + kRcThreads - 1) / kRcThreads) | 1;
  const int v0 = min(Lc, tid * CH), v1 = min(Lc, v0 + CH);
  float csum = 0.f;
  for (int v = v0; v < v1; ++v) csum += s_D[v];
  // Prefix masses: the chunk sums and their scan within a warp in float (their rounding, about
  // 1e-7 of the mass, is far inside the 1e-4 band that flags a near-boundary draw); the sums
  // over warps and over the cluster's CTAs in double, each formed once by one thread (FP64
  // issue is scarce) and read by all.
  float incl = csum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_red[warp] = incl;
  if (tid == 0) s_owner = -1;
  __syncthreads();
  if (tid == 0) {
    double run = 0.0;
    for (int w = 0; w < kRcThreads / 32; ++w) {
      s_dred[w] = run;
      run += (double)s_red[w];
    }
    for (int q = 0; q < kc; ++q) cl.map_shared_rank(&s_tot[0], q)[rank] = run;
  }
  cl.sync();
  if (tid == 0) {
    const float u2 = accept_uniform(p.seed, (uint32_t)b, (uint32_t)e, 1u);
    double total = 0.0, pre = 0.0;
    for (int q = 0; q < kc; ++q) {
      if (q == rank) pre = total;
      total += s_tot[q];
    }
    const double target = (double)u2 * total;
    int oc = -1;
    double run = 0.0;
    for (int q = 0; q < kc; ++q) {  // last CTA with mass that starts at or below the target
      if (s_tot[q] > 0.0 && run <= target) oc = q;
      run += s_tot[q];
    }
    s_bonus[0] = total;
    s_bonus[1] = pre;
    s_bonus[2] = target;
    s_owner_cta = oc;
  }
  __syncthreads();
  const double total = s_bonus[0], pre = s_bonus[1], target = s_bonus[2];
  const double band = (double)kMargin * total;
  const int owner_cta = s_owner_cta;
  const double excl = s_dred[warp] + (double)(incl - csum);  // mass of this slice before the chunk
  if (owner_cta == rank) {
    // owner: the last chunk with mass that starts at or below the target
    if (csum > 0.f && pre + excl <= target) atomicMax(&s_owner, tid);
    __syncthreads();
    if (tid == s_owner) {  // the chunk's scan in float, from the target's offset into the chunk
      const float rem = (float)(target - (pre + excl)), bandf = (float)band;
      float acc = 0.f, prev = 0.f;
      int found = -1, last_nz = -1;
      for (int v = v0; v < v1; ++v) {
        const float rv = s_D[v];
        if (rv > 0.f) last_nz = v;
        prev = acc;
        acc += rv;
        if (acc > rem) { found = v; break; }
      }
      if (found < 0) {
        found = last_nz;
        prev = acc;
      }
      const bool near = (rem - prev < bandf) || (acc - rem < bandf) || (target < band);
      p.bonus[b] = found >= 0 ? base + found : V - 1;
      if (p.bonus_margin) p.bonus_margin[b] = near ? 1 : 0;
    }
  }
  if (rank == 0) {
    write_path(p, b, e, dep, s_parent);
    if (tid == 0) {
      p.accept_len[b] = dep;
      if (owner_cta < 0) {  // no mass at all (cannot happen for a softmax row)
        p.bonus[b] = V - 1;
        if (p.bonus_margin) p.bonus_margin[b] = 0;
      }
      if (p.margin_count) p.margin_count[b] = margins;
    }
  }
}

__global__ void __launch_bounds__(kRcThreads, 1)
    accept_rejection_cluster_kernel(const AcceptParams p) {
  namespace cg = cooperative_groups;
  rejection_cluster_walk(p);
  if (p.fuse_compact) {
    cg::cluster_group cl = cg::this_cluster();
    cl.sync();  // rank 0's path and length are visible to the whole cluster; no remote access follows
    const int kc = (int)cl.num_blocks();
    fused_compact_tail(p, blockIdx.x / kc, (int)cl.block_rank(), kc);
  }
}

bool rejection_uses_cluster(int V) { return V >= 1 && V <= kRcMaxCluster * kRcSlice; }

namespace {

// Largest number of co-resident clusters of 1, 2, 4 and 8 CTAs, per device, measured once.
struct ClusterOccupancy {
  bool ready = false;
  bool ok = false;
  int max_clusters[4] = {0, 0, 0, 0};
};
std::mutex g_rc_mutex;
ClusterOccupancy g_rc_occ[64];

const ClusterOccupancy& cluster_occupancy() {
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(g_rc_mutex);
  ClusterOccupancy& o = g_rc_occ[dev & 63];
  if (o.ready) return o;
  o.ready = true;
  if (cudaFuncSetAttribute(accept_rejection_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kRcSmem) != cudaSuccess)
    return o;
  o.ok = true;
  for (int i = 0; i < 4; ++i) {
    const int kc = 1 << i;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kc, 1, 1);
    cfg.blockDim = dim3(kRcThreads, 1, 1);
    cfg.dynamicSmemBytes = kRcSmem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = kc;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int m = 0;
    if (cudaOccupancyMaxActiveClusters(&m, (void*)accept_rejection_cluster_kernel, &cfg) != cudaSuccess) m = 0;
    o.max_clusters[i] = m;
  }
  cudaGetLastError();
  return o;
}

}  // namespace

void prepare_rejection_launch() { cluster_occupancy(); }

// Cluster size: the smallest that fits the vocabulary in registers, widened (up to 8) while
// every request still gets a co-resident cluster and each CTA keeps >= 1024 entries.
int rejection_cluster_size(int B, int V, const int* max_clusters) {
  int i0 = 0;
  while (i0 < 3 && (V + (1 << i0) - 1) / (1 << i0) > kRcSlice) ++i0;
  int best = i0;
  for (int i = i0 + 1; i < 4; ++i)
    if (B <= max_clusters[i] && V >= (1 << i) * 1024) best = i;
  return 1 << best;
}

cudaError_t launch_accept(const AcceptParams& p, cudaStream_t stream) {
  if (!rejection_uses_cluster(p.V)) {
    accept_rejection_block_kernel<<<p.B, kRejThreads, p.fuse_compact ? kFusedCompactSmem : 0, stream>>>(p);
    return cudaGetLastError();
  }
  const ClusterOccupancy& occ = cluster_occupancy();
  if (!occ.ok) return cudaErrorInvalidConfiguration;
  const int kc = rejection_cluster_size(p.B, p.V, occ.max_clusters);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.B * kc), 1, 1);
  cfg.blockDim = dim3(kRcThreads, 1, 1);
  cfg.dynamicSmemBytes = kRcSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = kc;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, accept_rejection_cluster_kernel, p);
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


}  // namespace spectree

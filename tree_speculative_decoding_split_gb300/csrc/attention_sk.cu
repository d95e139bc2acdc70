// K1s (bf16, long prefixes): persistent, stream-K tree attention on tcgen05 tensor cores.
//
// Parallel verification scores every candidate in one forward pass over the KV cache (qiita
// "EAGLE-3とMedusaで実装するSpeculative Decoding実践ガイド", section "並列検証"); each tree node
// attends only to its ancestors and itself (tech-tldr "多トークン予測（Medusa・EAGLE）", section
// "ツリー検証"; qiita, section "Tree Attention").
//
// The layer's work is a set of segments: (request b, KV head g, block rg of 256 (node, GQA head)
// rows) over the request's keys [0, L_b + n_b) in 64-key tiles.  The CTAs (one per SM) form one
// lane per row block; in its lane's index space, the segments (b, g) of that row block laid end
// to end, every CTA takes an equal contiguous range, so that all SMs finish together whatever the
// prefix lengths and however few segments there are.  CTA i of every lane covers the same
// (b, g, key tiles) at the same time, so the row blocks of a KV head share its K/V through L2.
// A CTA walks its range as pieces (the tiles of one segment inside the range).  A piece that
// covers its whole segment writes the final bf16 rows and LSE; one that covers part of it writes
// a normalised fp32 partial (o, running max, sum) to the workspace and counts itself on the
// segment's arrival counter, and the last of the segment's pieces to arrive merges them.  No CTA
// waits for another.
//
// Inside a CTA the roles are those of the single-launch kernel (attention_tc.cu): a TMA producer
// (each piece's Q, then 64-key K and V tiles into a 4-stage ring shared by both row groups), one
// MMA issuer per 128-row group (S = Q K^T into TMEM, O += P V with P read from TMEM), and four
// softmax warps per group (one row per thread: tree mask from ancestor bits, online softmax in the
// log2 domain, P into one of two TMEM buffers).  Across pieces the producer runs ahead: the next
// piece's first K/V tiles load while the current one drains, its Q is prefetched into L2 at the
// start of the current piece and loaded as soon as the group's last Q K^T of the current piece has
// completed.  The softmax warps validate the request's tree and build their own row's ancestor
// bits by walking the parent chain at the start of each piece, and write the piece's output.

#include "common.cuh"
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace spectree {

namespace {

constexpr int kKT = 64;         // keys per tile
constexpr int kStages = 4;      // K/V ring depth
constexpr int kGR = 128;        // rows per group (MMA M)
constexpr int kNG = 2;          // groups per CTA
constexpr int kSegRows = kGR * kNG;
constexpr float kRescaleLog2 = 8.f;

template <int D>
struct SkCfg {
  // producer warp, MMA warp of group 0, 4 softmax warps per group, MMA warp of group 1
  static constexpr int kThreads = 64 + 128 * kNG + 32;
  static constexpr int kQ = kGR * D * 2;       // Q bytes per group
  static constexpr int kTile = kKT * D * 2;    // K (or V) tile bytes
  static constexpr int kBars = 2 * kStages + 9 * kNG + 1;
  static constexpr int kSmem = 1024 + kNG * kQ + 2 * kStages * kTile + kSegRows * kAncWords * 4 + kBars * 8;
  static constexpr int kColS = 0, kColO = kNG * kKT, kColP = kNG * (kKT + D);
  static constexpr uint32_t kTmemCols = (kNG * (2 * kKT + D) <= 256) ? 256 : 512;
};

// OR of `pred` over the `count` threads that meet at named barrier `id` (a barrier for all).
__device__ __forceinline__ bool bar_red_or(int id, int count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(count)
      : "memory");
  return r != 0;
}

// A lane's tile index space: request b's segments (one per KV head) have T_b tiles each and
// start at pt[b] * HR (HR = Hkv); lane CTA c owns tiles [c * total / grid, (c + 1) * total /
// grid) (grid = the lane's CTAs).  The host keeps the index space below 2^31 tiles.
struct SkSched {
  const int* pt;
  int B, HR, total, grid;
  __device__ int begin(int c) const { return (int)((long long)c * total / grid); }
  __device__ int cta_of(int t) const { return (int)(((long long)(t + 1) * grid - 1) / total); }
};

struct SkPiece {
  int b, j, T, t_lo, t_hi;  // request, segment within the request, tiles of the segment, piece tiles
  int seg_off;              // first tile of the segment in the index space
};

__device__ __forceinline__ void sk_piece(const SkSched& s, int t, int E, SkPiece& pc) {
  int lo = 0, hi = s.B - 1;
  while (lo < hi) {  // the request whose segments hold tile t
    const int mid = (lo + hi + 1) >> 1;
    if (s.pt[mid] * s.HR <= t) lo = mid; else hi = mid - 1;
  }
  const int T = s.pt[lo + 1] - s.pt[lo];
  const int base = s.pt[lo] * s.HR;
  const int j = (t - base) / T;
  pc.b = lo;
  pc.j = j;
  pc.T = T;
  pc.seg_off = base + j * T;
  pc.t_lo = t - pc.seg_off;
  const int hi_t = pc.t_lo + (E - t);
  pc.t_hi = hi_t < T ? hi_t : T;
}

// Tiles of request b's segments: its keys in 64-key tiles, or 1 for a request whose sizes are
// invalid (that piece only writes zeros).
__device__ __forceinline__ int sk_tiles(const AttnParams& p, int b) {
  const long long L = p.prefix_len[b];
  const int n = p.n_nodes[b];
  const bool ok = n >= 1 && n <= p.N && L >= 0 && L + n <= p.L_cap;
  return ok ? (int)((L + n + kKT - 1) / kKT) : 1;
}

}  // namespace

template <int D>
__global__ void __launch_bounds__(SkCfg<D>::kThreads, 1)
    attn_sk_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using C = SkCfg<D>;
  constexpr int kThr = C::kThreads;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;                              // [group][128 rows][D], K-major swizzled
  uint8_t* sK = sQ + kNG * C::kQ;
  uint8_t* sV = sK + kStages * C::kTile;
  uint32_t* sAnc = reinterpret_cast<uint32_t*>(sV + kStages * C::kTile);  // [256 rows][8 words]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sAnc + kSegRows * kAncWords);
  uint64_t* full = bars;                  // [stage] K/V landed
  uint64_t* empty = full + kStages;       // [stage] K/V consumed by both groups
  uint64_t* sfull = empty + kStages;      // [group] S computed
  uint64_t* sfree = sfull + kNG;          // [group] S read by the softmax
  uint64_t* pfull = sfree + kNG;          // [group][P buffer] P written
  uint64_t* ofull = pfull + 2 * kNG;      // [group][P buffer] P V done
  uint64_t* qfull = ofull + 2 * kNG;      // [group] the piece's Q landed
  uint64_t* qfree = qfull + kNG;          // [group] the piece's last Q K^T completed
  uint64_t* drained = qfree + kNG;        // [group] every MMA of the issuer completed
  __shared__ int s_pt[kSkMaxBatch + 1];
  __shared__ int s_par[kNG][kMaxNodes];
  __shared__ int s_last[kNG];
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_issued, s_consumed;
  __shared__ int s_qissued[kNG], s_qdone[kNG];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- the schedule: tiles per request, prefix sums (every CTA computes the same) ----
  for (int b = tid; b < p.B; b += kThr) s_pt[b + 1] = sk_tiles(p, b);
  if (tid == 0) s_pt[0] = 0;
  __syncthreads();
  if (warp == 0) {
    const int per = (p.B + 31) / 32;
    int sum = 0;
    for (int k = 0; k < per; ++k) {
      const int b = lane * per + k;
      if (b < p.B) sum += s_pt[b + 1];
    }
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    int run = inc - sum;
    for (int k = 0; k < per; ++k) {
      const int b = lane * per + k;
      if (b < p.B) {
        run += s_pt[b + 1];
        s_pt[b + 1] = run;
      }
    }
  }
  __syncthreads();
  SkSched sc;
  sc.pt = s_pt;
  sc.B = p.B;
  // lanes: CTA x works on row block x % n_rg as the lane's CTA x / n_rg
  const int lane_rg = (int)blockIdx.x % p.n_rg;
  const int per_lane = (int)gridDim.x / p.n_rg;
  sc.HR = p.Hkv;
  sc.total = s_pt[p.B] * sc.HR;
  // with fewer tiles than CTAs only the first `total` CTAs of a lane work, one tile or more each,
  // so that every CTA between a segment's first and last owner holds a piece of it
  sc.grid = per_lane < sc.total ? per_lane : sc.total;
  const int cta = (int)blockIdx.x / p.n_rg;  // index within the lane
  if (cta >= sc.grid) return;  // uniform exit (also the CTAs beyond n_rg * per_lane)
  const int A = sc.begin(cta), E = sc.begin(cta + 1);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kNG);  // one P V commit per group's issuer
    }
    for (int a = 0; a < kNG; ++a) {
      mbar_init(&sfull[a], 1);
      mbar_init(&sfree[a], 4);
      mbar_init(&pfull[2 * a], 4);
      mbar_init(&pfull[2 * a + 1], 4);
      mbar_init(&ofull[2 * a], 1);
      mbar_init(&ofull[2 * a + 1], 1);
      mbar_init(&qfull[a], 1);
      mbar_init(&qfree[a], 1);
      mbar_init(&drained[a], 1);
      s_qissued[a] = 0;
      s_qdone[a] = 0;
    }
    s_abort = 0;
    s_issued = 0;
    s_consumed = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&s_tmem, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const int rows_total = p.N * p.G;
  const int npg = kGR / p.G;  // nodes per 128-row group

  if (warp == 0) {
    if (lane == 0) {
      // ---- TMA producer ----
      int t = A, rt = 0, k = 0;
      bool ok = true;
      auto issue_kv = [&](const SkPiece& pc, int g, int i) -> bool {
        const int st = rt % kStages;
        if (rt >= kStages && !mbar_wait_bounded(&empty[st], (uint32_t)(((rt / kStages) & 1) ^ 1), &s_abort))
          return false;
        const int key = (pc.t_lo + i) * kKT;
        const int zi = pc.b * p.Hkv + g;
        mbar_arrive_expect_tx(&full[st], 2 * C::kTile);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          tma_load_3d(sK + st * C::kTile + c * kKT * 128, &tmK, &full[st], c * 64, key, zi);
          tma_load_3d(sV + st * C::kTile + c * kKT * 128, &tmV, &full[st], c * 64, key, zi);
        }
        ++rt;
        s_issued = rt;
        return true;
      };
      while (t < E && ok) {
        SkPiece pc;
        sk_piece(sc, t, E, pc);
        const int n = pc.t_hi - pc.t_lo;
        const int g = pc.j, rg = lane_rg;
        if (t + n < E) {  // the next piece's Q into L2 while this piece runs
          SkPiece nx;
          sk_piece(sc, t + n, E, nx);
          const int ng = nx.j, nrg = lane_rg;
          for (int a = 0; a < kNG; ++a)
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
              tma_prefetch_4d(&tmQ, c * 64, ng * p.G, nrg * (kSegRows / p.G) + a * npg, nx.b);
        }
        // The first K/V tiles of this piece only need ring slots the previous piece has released
        // before its last Q K^T completed; then Q (its buffer frees with that last Q K^T).
        const int pre = k == 0 ? 0 : (n < 2 ? n : 2);
        for (int i = 0; i < pre && ok; ++i) ok = issue_kv(pc, g, i);
        for (int a = 0; a < kNG && ok; ++a) {
          if (k > 0 && !mbar_wait_bounded(&qfree[a], (uint32_t)((k - 1) & 1), &s_abort)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&qfull[a], C::kQ);
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_4d(sQ + a * C::kQ + c * kGR * 128, &tmQ, &qfull[a], c * 64, g * p.G,
                        rg * (kSegRows / p.G) + a * npg, pc.b);
          s_qissued[a] = k + 1;
        }
        for (int i = pre; i < n && ok; ++i) ok = issue_kv(pc, g, i);
        t += n;
        ++k;
      }
      if (!ok) {
        if (atomicExch(&s_abort, 1) == 0) set_status(p.dev_status, SPEC_ERR_TIMEOUT);
      }
    }
  } else if (warp == 1 || warp == 2 + 4 * kNG) {
    // ---- MMA issuers: group 0 on warp 1, group 1 on warp 10 ----
    const int ga = (warp == 1) ? 0 : 1;
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kGR, kKT, 0);
      constexpr uint32_t idP = idesc_bf16_f32(kGR, D, 1);
      bool ok = true;
      auto issue_s = [&](int u) -> bool {
        const int st = u % kStages;
        if (!mbar_wait_bounded(&full[st], (uint32_t)((u / kStages) & 1), &s_abort)) return false;
        if (ga == 0) s_consumed = u + 1;
        if (u > 0 && !mbar_wait_bounded(&sfree[ga], (uint32_t)((u - 1) & 1), &s_abort)) return false;
        tc_fence_after();
        const uint32_t qa = smem_u32(sQ + ga * C::kQ), ka = smem_u32(sK + st * C::kTile);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(qa + (kk >> 2) * (kGR * 128) + (kk & 3) * 32, 0, 1024);
          const uint64_t bd = sdesc_sw128(ka + (kk >> 2) * (kKT * 128) + (kk & 3) * 32, 0, 1024);
          umma_bf16(tmem + C::kColS + ga * kKT, ad, bd, idS, kk > 0);
        }
        umma_commit(&sfull[ga]);
        return true;
      };
      auto issue_pv = [&](int u, bool first) -> bool {
        if (!mbar_wait_bounded(&pfull[2 * ga + (u & 1)], (uint32_t)((u >> 1) & 1), &s_abort)) return false;
        tc_fence_after();
        const uint32_t pt = tmem + C::kColP + (2 * ga + (u & 1)) * (kKT / 2);
        const uint32_t va = smem_u32(sV + (u % kStages) * C::kTile);
#pragma unroll
        for (int kk = 0; kk < kKT / 16; ++kk) {
          const uint64_t bd = sdesc_sw128(va + kk * 16 * 128, kKT * 128, 1024);
          umma_bf16_tmem_a(tmem + C::kColO + ga * D, pt + kk * 8, bd, idP, (!first || kk > 0) ? 1u : 0u);
        }
        umma_commit(&ofull[2 * ga + (u & 1)]);
        return true;
      };
      int t = A, ct = 0, k = 0;
      while (t < E && ok) {
        SkPiece pc;
        sk_piece(sc, t, E, pc);
        const int n = pc.t_hi - pc.t_lo;
        ok = mbar_wait_bounded(&qfull[ga], (uint32_t)(k & 1), &s_abort);
        if (!ok) break;
        s_qdone[ga] = k + 1;
        // Per tile: the next tile's Q K^T as soon as the softmax has read this tile's S, then
        // this tile's P V; at the end of the piece the P V goes first (the next piece's Q K^T
        // waits for its Q).
        ok = issue_s(ct);
        if (ok && n == 1) umma_commit(&qfree[ga]);
        for (int i = 0; i < n && ok; ++i) {
          const int u = ct + i;
          if (i + 1 < n) {
            ok = issue_s(u + 1);
            if (!ok) break;
            if (i + 2 == n) umma_commit(&qfree[ga]);  // the piece's last Q K^T is issued
          }
          ok = issue_pv(u, i == 0);
          if (!ok) break;
          umma_commit(&empty[u % kStages]);  // this group is done with K/V tile u
        }
        ct += n;
        t += n;
        ++k;
      }
      if (!ok) {
        if (atomicExch(&s_abort, 1) == 0) set_status(p.dev_status, SPEC_ERR_TIMEOUT);
      }
      umma_commit(&drained[ga]);
      mbar_wait_bounded(&drained[ga], 0, nullptr);
    }
  } else {
    // ---- softmax warps 2..9: group a, TMEM lane quarter q4 ----
    const int a = (warp - 2) >> 2, q4 = warp & 3;
    const int rl = q4 * 32 + lane;        // row within the group (TMEM lane)
    const int rr = a * kGR + rl;          // row within the segment's 256-row block
    const int bar_id = 2 + a;             // named barrier of the group's 128 softmax threads
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const uint32_t tS = tmem + C::kColS + a * kKT + lane_off;
    const uint32_t tO = tmem + C::kColO + a * D + lane_off;
    const uint32_t tP = tmem + C::kColP + 2 * a * (kKT / 2) + lane_off;
    uint32_t* anc = sAnc + rr * kAncWords;
    int t = A, ct = 0;
    bool ok = true;
    while (t < E) {
      SkPiece pc;
      sk_piece(sc, t, E, pc);
      const int n = pc.t_hi - pc.t_lo;
      const int b = pc.b, g = pc.j, rg = lane_rg;
      const int L = p.prefix_len[b];
      const int nn = p.n_nodes[b];
      const int row = rg * kSegRows + rr;
      const bool valid = row < rows_total;
      const int node = row / p.G;

      // ---- piece prologue: tree checks and this row's ancestor bits ----
      named_bar_sync(bar_id, 128);  // every reader of the previous piece's parents is done
      bool cap_bad = !(nn >= 1 && nn <= p.N && L >= 0 && (long long)L + nn <= p.L_cap);
      bool tree_bad = cap_bad ? (nn < 1 || nn > p.N) : false;
      if (!tree_bad) {
        for (int c = rl; c < nn; c += kGR) {
          const int par = p.parent[(size_t)b * p.N + c];
          s_par[a][c] = par;
          if (c == 0 ? par != -1 : (par < 0 || par >= c)) tree_bad = true;
        }
      }
      tree_bad = bar_red_or(bar_id, 128, tree_bad);
      const bool bad = tree_bad || cap_bad;
      {
        uint32_t w[kAncWords];
#pragma unroll
        for (int q = 0; q < kAncWords; ++q) w[q] = 0u;
        if (!bad && valid && node < nn) {
          // the parent chain up to the root (valid tree: strictly decreasing, at most nn steps)
          for (int x = node; x >= 0; x = (x > 0) ? s_par[a][x] : -1) {
#pragma unroll
            for (int q = 0; q < kAncWords; ++q)
              if ((x >> 5) == q) w[q] |= 1u << (x & 31);
          }
        }
#pragma unroll
        for (int q = 0; q < kAncWords; ++q) anc[q] = w[q];
      }

      // ---- tiles of the piece ----
      float m_run = -INFINITY, l_run = 0.f;
      for (int i = 0; i < n; ++i) {
        const int u = ct + i;
        // waits are made warp-uniform: the TMEM loads and stores below are warp-collective
        const bool got = __all_sync(0xffffffffu, ok && mbar_wait_bounded(&sfull[a], (uint32_t)(u & 1), &s_abort));
        if (!got) {
          ok = false;
          continue;  // keep walking the pieces: every named barrier of the group is still met
        }
        tc_fence_after();
        uint32_t s0[32], s1[32];
        tmem_ld_x32(tS, s0);
        tmem_ld_x32(tS + 32, s1);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sfree[a]);
        float v[kKT];  // raw scores; the softmax scale (log2 units) is applied in the exponent
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          v[j] = __uint_as_float(s0[j]);
          v[j + 32] = __uint_as_float(s1[j]);
        }
        const int kbase = (pc.t_lo + i) * kKT;
        if (kbase + kKT > L) {
          // key j of the tile is tree node kbase - L + j when that is >= 0, else a prefix key; the
          // window of ancestor bits is read from shared memory; nodes past n have no bit
          const int off = kbase - L;   // >= -63
          const int lo = off >> 5;
          const int r = off - (lo << 5);
          const uint32_t w0 = (lo >= 0 && lo < kAncWords) ? anc[lo] : 0u;
          const uint32_t w1 = (lo + 1 >= 0 && lo + 1 < kAncWords) ? anc[lo + 1] : 0u;
          const uint32_t w2 = (lo + 2 >= 0 && lo + 2 < kAncWords) ? anc[lo + 2] : 0u;
          const unsigned long long win = ((unsigned long long)w1 << 32) | w0;
          unsigned long long mask = (win >> r) | (r ? ((unsigned long long)w2 << (64 - r)) : 0ull);
          if (off < 0) mask |= (1ull << -off) - 1ull;  // the tile's first -off keys are prefix keys
#pragma unroll
          for (int j = 0; j < kKT; ++j)
            if (!((mask >> j) & 1ull)) v[j] = -INFINITY;
        }
        float mx[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
        for (int j = 4; j < kKT; ++j) mx[j & 3] = fmaxf(mx[j & 3], v[j]);
        const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * p.scale_log2;
        const float m_new = fmaxf(m_run, tmax);
        const bool need = m_new > m_run + kRescaleLog2;  // includes the first finite maximum
        if (__any_sync(0xffffffffu, need)) {
          const float f = need ? exp2f(m_run - m_new) : 1.f;  // 0 when m_run is -inf
          if (i > 0) {
            // P V(u - 1) must have landed in O before O is rescaled (the piece's first P V
            // overwrites O, so its first tile needs no rescale)
            if (!__all_sync(0xffffffffu,
                            mbar_wait_bounded(&ofull[2 * a + ((u - 1) & 1)], (uint32_t)(((u - 1) >> 1) & 1), &s_abort))) {
              ok = false;
              continue;
            }
            tc_fence_after();
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t o[32];
              tmem_ld_x32(tO + c * 32, o);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * f);
              tmem_st_x32(tO + c * 32, o);
            }
            tmem_st_wait();
          }
          if (need) {
            l_run *= f;
            m_run = m_new;
          }
        }
        const float mu = (m_run == -INFINITY) ? 0.f : m_run;
        const float2 sc2 = make_float2(p.scale_log2, p.scale_log2), nmu2 = make_float2(-mu, -mu);
        float2 ps2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        uint32_t pk[kKT / 2];
#pragma unroll
        for (int j = 0; j < kKT; j += 2) {
          const float2 x = __ffma2_rn(make_float2(v[j], v[j + 1]), sc2, nmu2);
          const float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
          ps2[(j >> 1) & 1] = __fadd2_rn(ps2[(j >> 1) & 1], make_float2(p0, p1));
          pk[j / 2] = pack_bf16x2(p0, p1);
        }
        l_run += (ps2[0].x + ps2[1].x) + (ps2[0].y + ps2[1].y);
        // P buffer u & 1 was last read by P V(u - 2), issued before S(u) by this group's issuer;
        // the commit that completed S(u) tracks it.
        tmem_st_x32(tP + (u & 1) * (kKT / 2), pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&pfull[2 * a + (u & 1)]);
      }

      // ---- piece epilogue ----
      const int ul = ct + n - 1;
      const bool fin = __all_sync(0xffffffffu, ok && mbar_wait_bounded(&ofull[2 * a + (ul & 1)],
                                                                         (uint32_t)((ul >> 1) & 1), &s_abort));
      if (!fin) ok = false;
      const bool whole = pc.t_lo == 0 && pc.t_hi == pc.T;
      const bool live = valid && !bad && node < nn;
      size_t orow = 0;
      if (valid) orow = ((size_t)b * p.N + node) * p.Hq + g * p.G + row % p.G;
      if (fin) tc_fence_after();
      if (whole) {
        const float inv = (live && l_run > 0.f) ? 1.f / l_run : 0.f;
        if (valid && p.lse) p.lse[orow] = (live && l_run > 0.f) ? (m_run + log2f(l_run)) * 0.69314718055994531f : 0.f;
        __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + orow * D;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          if (fin) {  // warp-collective: every lane loads; rows past the last node are dropped below
            tmem_ld_x32(tO + c * 32, o);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = 0u;
          }
          if (valid)
#pragma unroll
            for (int j = 0; j < 32; j += 8)
              *reinterpret_cast<uint4*>(out + c * 32 + j) =
                  make_uint4(pack_bf16x2(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv),
                             pack_bf16x2(__uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv),
                             pack_bf16x2(__uint_as_float(o[j + 4]) * inv, __uint_as_float(o[j + 5]) * inv),
                             pack_bf16x2(__uint_as_float(o[j + 6]) * inv, __uint_as_float(o[j + 7]) * inv));
        }
        if (bad && g == 0 && rg == 0 && rr == 0)
          set_status(p.dev_status, tree_bad ? SPEC_ERR_BAD_TREE : SPEC_ERR_CAPACITY);
      } else {
        // partial: normalised o and (running max, sum) into this CTA's slot for the piece
        const int slot = (sc.begin(cta) >= pc.seg_off) ? 0 : 1;
        const size_t pr = ((size_t)blockIdx.x * 2 + slot) * kSegRows + rr;
        if (fin) {
          const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
          float* dst = p.sk_o + pr * D;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld_x32(tO + c * 32, o);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(dst + c * 32 + j) =
                  make_float4(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv,
                              __uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv);
          }
          p.sk_ml[pr] = make_float2(m_run, l_run);
        }
        __threadfence();
        named_bar_sync(bar_id, 128);
        const int segid = (b * p.Hkv + g) * p.n_rg + rg;
        const int c_first = sc.cta_of(pc.seg_off), c_last = sc.cta_of(pc.seg_off + pc.T - 1);
        if (rl == 0) {
          int last = 0;
          if (ok) last = atomicAdd(&p.sk_cnt[segid * kNG + a], 1) == (c_last - c_first);
          s_last[a] = last;
        }
        named_bar_sync(bar_id, 128);
        if (s_last[a]) {
          __threadfence();
          // Merge every piece of the segment for this thread's row.  This CTA's own piece is still
          // in TMEM (O unnormalised, with m_run / l_run); the other pieces' partials (lane CTA c is
          // block c * n_rg + rg) are read from L2 with several loads in flight at once -- under a
          // saturated memory system a round trip costs about a microsecond.
          constexpr int kBatch = 2;  // other pieces whose rows are in flight together
          auto rec_of = [&](int c) -> size_t {
            const int sl = (sc.begin(c) >= pc.seg_off) ? 0 : 1;
            return (((size_t)c * p.n_rg + rg) * 2 + sl) * kSegRows + rr;
          };
          float M = (fin && l_run > 0.f) ? m_run : -INFINITY;
          for (int c0 = c_first; c0 <= c_last; c0 += 4) {  // records, four at a time
            float2 ml[4];
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2)
              ml[k2] = (c0 + k2 <= c_last && c0 + k2 != cta) ? __ldcg(p.sk_ml + rec_of(c0 + k2))
                                                             : make_float2(-INFINITY, 0.f);
#pragma unroll
            for (int k2 = 0; k2 < 4; ++k2)
              if (ml[k2].y > 0.f) M = fmaxf(M, ml[k2].x);
          }
          const float own = (fin && l_run > 0.f) ? exp2f(m_run - M) : 0.f;
          float wsum = l_run * own;
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + orow * D;
#pragma unroll 1
          for (int ch = 0; ch < D / 32; ++ch) {
            float acc[32];
            uint32_t o[32];
            if (fin) {  // warp-collective
              tmem_ld_x32(tO + ch * 32, o);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) o[j] = 0u;
            }
#pragma unroll
            for (int j = 0; j < 32; ++j) acc[j] = own * __uint_as_float(o[j]);
#pragma unroll 1
            for (int c0 = c_first; c0 <= c_last; c0 += kBatch) {
              float2 ml[kBatch];
              size_t q[kBatch];
              float4 x[kBatch][8];
#pragma unroll
              for (int k2 = 0; k2 < kBatch; ++k2) {
                const bool use = c0 + k2 <= c_last && c0 + k2 != cta;
                q[k2] = use ? rec_of(c0 + k2) : 0;
                ml[k2] = use ? __ldcg(p.sk_ml + q[k2]) : make_float2(-INFINITY, 0.f);
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  x[k2][j] = use ? __ldcg(reinterpret_cast<const float4*>(p.sk_o + q[k2] * D + ch * 32) + j)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
              }
#pragma unroll
              for (int k2 = 0; k2 < kBatch; ++k2) {
                const float w = (ml[k2].y > 0.f) ? ml[k2].y * exp2f(ml[k2].x - M) : 0.f;
                if (ch == 0) wsum += w;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  acc[4 * j] = fmaf(w, x[k2][j].x, acc[4 * j]);
                  acc[4 * j + 1] = fmaf(w, x[k2][j].y, acc[4 * j + 1]);
                  acc[4 * j + 2] = fmaf(w, x[k2][j].z, acc[4 * j + 2]);
                  acc[4 * j + 3] = fmaf(w, x[k2][j].w, acc[4 * j + 3]);
                }
              }
            }
            if (valid) {
              // partials are normalised o; the own piece is unnormalised O: both weighted to units
              // of 2^M above, so dividing by the total weight gives the row
              const float inv = (live && wsum > 0.f) ? 1.f / wsum : 0.f;
#pragma unroll
              for (int j = 0; j < 32; j += 8)
                *reinterpret_cast<uint4*>(out + ch * 32 + j) =
                    make_uint4(pack_bf16x2(acc[j] * inv, acc[j + 1] * inv), pack_bf16x2(acc[j + 2] * inv, acc[j + 3] * inv),
                               pack_bf16x2(acc[j + 4] * inv, acc[j + 5] * inv), pack_bf16x2(acc[j + 6] * inv, acc[j + 7] * inv));
            }
          }
          if (valid && p.lse) p.lse[orow] = (live && wsum > 0.f) ? (M + log2f(wsum)) * 0.69314718055994531f : 0.f;
          if (bad && g == 0 && rg == 0 && rr == 0)
            set_status(p.dev_status, tree_bad ? SPEC_ERR_BAD_TREE : SPEC_ERR_CAPACITY);
        }
      }
      ct += n;
      t += n;
    }
    if (!ok && lane == 0) {
      if (atomicExch(&s_abort, 1) == 0) set_status(p.dev_status, SPEC_ERR_TIMEOUT);
    }
  }

  __syncthreads();
  if (tid == 0 && s_abort) {
    // let the copies still in flight land before shared memory is released
    for (int u = s_consumed; u < s_issued; ++u)
      mbar_wait_bounded(&full[u % kStages], (uint32_t)((u / kStages) & 1), nullptr);
    for (int a = 0; a < kNG; ++a)
      if (s_qissued[a] > s_qdone[a]) mbar_wait_bounded(&qfull[a], (uint32_t)(s_qdone[a] & 1), nullptr);
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

template <int D>
static cudaError_t launch_sk(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                             const AttnParams& p, int grid, cudaStream_t stream) {
  using C = SkCfg<D>;
  cudaError_t err = cudaFuncSetAttribute(attn_sk_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (err != cudaSuccess) return err;
  attn_sk_kernel<D><<<grid, C::kThreads, C::kSmem, stream>>>(*tmQ, *tmK, *tmV, p);
  return cudaGetLastError();
}

cudaError_t launch_attention_sk(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                                const AttnParams& p, int grid, cudaStream_t stream) {
  return p.d == 128 ? launch_sk<128>(tmQ, tmK, tmV, p, grid, stream) : launch_sk<64>(tmQ, tmK, tmV, p, grid, stream);
}

}  // namespace spectree

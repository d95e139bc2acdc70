// K1 (bf16): split-KV tree attention on tcgen05 tensor cores.
//
// Parallel verification scores every candidate in one forward pass over the KV cache (qiita
// "EAGLE-3とMedusaで実装するSpeculative Decoding実践ガイド", section "並列検証"); each tree node
// attends only to its ancestors and itself (tech-tldr "多トークン予測（Medusa・EAGLE）", section
// "ツリー検証"; qiita, section "Tree Attention").
//
// One CTA owns (request b, KV head g, key split, NG x 128 rows); a row is a (tree node i, GQA head
// j) pair r = i * G + j, so every K/V tile is read once for all query heads sharing KV head g and
// all tree nodes.  With NG = 2 the two 128-row groups (the M of one MMA each) run in ping-pong:
// while one group's softmax works on its scores, the tensor core computes the other group's P V
// and next Q K^T; small problems use NG = 1 for more, shorter CTAs.  Roles:
//   warp 0     TMA producer: the CTA's Q rows (when G divides 128), then 64-key K and V tiles
//              (128-byte swizzle) into a 4-stage ring;
//   warp 1 (+ one more warp per extra group)  MMA issuer of one group: S = Q K^T into the
//              group's TMEM score buffer as soon as the softmax has read the previous S, and
//              O += P V into the group's TMEM accumulator as soon as P is written, with P read
//              from tensor memory and V consumed MN-major straight from its TMA tiles;
//   softmax    four warps per group: the thread owning TMEM lane r of a group owns that row --
//              it loads its S row, applies the tree mask (ancestor bits, tree tiles only) and
//              the online softmax in the log2 domain, and writes the bf16 P row into one of the
//              group's two P buffers in tensor memory (so P(t) waits only for P V(t - 2)).  O is
//              rescaled in TMEM only when a row's running maximum grows by more than 2^8
//              (exact: P and the running sum use the same stale maximum).
// Every CTA validates the tree; the CTAs of the split that holds the tree keys (the prefix split
// containing slot L, which then also covers [L, L + n)) build the ancestor bits by pointer
// jumping.  Each split writes a normalised partial (bf16 o, running max, sum), merged by the merge
// kernel.

#include "common.cuh"
#include "kernels.cuh"
#include "tc_ptx.cuh"

namespace spectree {

namespace {

constexpr int kKT = 64;          // keys per tile (MMA N of S, K of P V)
constexpr int kStages = 4;       // K/V ring depth
constexpr int kGR = 128;         // rows per group (MMA M)
constexpr float kRescaleLog2 = 8.f;
constexpr int kMaxBlkCta = 1040;  // paged KV: block-table entries a CTA stages in shared memory

template <int D, int NG>
struct AttnTcCfg {
  static constexpr int kGroups = NG;            // 128-row groups per CTA
  static constexpr int kRowsCta = kGR * NG;
  // producer warp, MMA warp (group 0), 4 softmax warps per group, and with two groups a second
  // MMA warp that issues group 1's MMAs, so that neither group's issue waits on the other's
  static constexpr int kThreads = 64 + 128 * NG + (NG > 1 ? 32 * (NG - 1) : 0);
  static constexpr int kQ = kGR * D * 2;        // Q bytes per group
  static constexpr int kTile = kKT * D * 2;     // K (or V) tile bytes
  static constexpr int kSmem =
      1024 + NG * kQ + 2 * kStages * kTile + kRowsCta * kAncWords * 4 + 32 * 8;
  // TMEM columns per group: S (kKT fp32), O (D fp32), and two P buffers (kKT bf16 = kKT / 2
  // columns each)
  static constexpr int kColS = 0, kColO = NG * kKT, kColP = NG * (kKT + D);
  static constexpr uint32_t kTmemCols = (NG * (2 * kKT + D) <= 256) ? 256 : 512;
  // epilogue: the normalised O rows staged in shared memory (fp32, rows padded by 16 bytes so
  // that the quarter-warps' 16-byte stores of consecutive rows hit distinct banks), reusing the
  // Q / K / V / P region once every MMA of the CTA has completed
  static constexpr int kORow = D * 4 + 16;
  static_assert(kRowsCta * kORow <= NG * kQ + 2 * kStages * kTile, "O staging does not fit");
};

__device__ __forceinline__ uint32_t sw128_off(int r, int ch, int rows) {
  return (uint32_t)((ch >> 3) * rows * 128 + r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

// One row of the output partial (fp32) from shared memory to global memory by the bulk-copy
// engine; the row stays readable in shared memory until the matching wait below.
__device__ __forceinline__ void bulk_store_row(void* gdst, const void* ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(smem_u32(ssrc)),
               "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

}  // namespace

template <int D, int NG>
__global__ void __launch_bounds__(AttnTcCfg<D, NG>::kThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const AttnParams p) {
  using C = AttnTcCfg<D, NG>;
  constexpr int kGroups = C::kGroups;
  constexpr int kRowsCta = C::kRowsCta;
  constexpr int kTcThreads = C::kThreads;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = base;                                  // [group][128 rows][D], K-major swizzled
  uint8_t* sK = sQ + kGroups * C::kQ;
  uint8_t* sV = sK + kStages * C::kTile;
  uint32_t* sAnc = reinterpret_cast<uint32_t*>(sV + kStages * C::kTile);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sAnc + kRowsCta * kAncWords);
  uint64_t* full = bars;                 // [stage] K/V landed
  uint64_t* empty = full + kStages;      // [stage] K/V consumed by every group
  uint64_t* sfull = empty + kStages;     // [group] S computed
  uint64_t* sfree = sfull + kGroups;     // [group] S read by the softmax
  uint64_t* pfull = sfree + kGroups;     // [group][P buffer] P written
  uint64_t* ofull = pfull + 2 * kGroups; // [group][P buffer] P V done (O updated, buffer free)
  uint64_t* drained = ofull + 2 * kGroups;
  uint64_t* qfull = drained + kGroups;   // Q of every group landed (TMA path)
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  __shared__ int s_issued, s_consumed;
  __shared__ int s_par[kMaxNodes];
  __shared__ int s_jmp[kMaxNodes];
  __shared__ uint32_t s_nanc[kMaxNodes][kAncWords];
  __shared__ int s_blk[kMaxBlkCta];

  const int rg = blockIdx.x, split = blockIdx.y, bg = blockIdx.z;
  const int b = bg / p.Hkv, g = bg % p.Hkv;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long L = p.prefix_len[b];
  const int n = p.n_nodes[b];
  const int rows_total = p.N * p.G;
  const int row0 = rg * kRowsCta;

  // Split s covers keys [s * chunk, (s + 1) * chunk); the split holding key L (the first tree
  // slot) also takes every tree key, [L, L + n), and the splits after it have none.  (A request
  // that fails the checks below gets a range too; its CTAs only wait for their loads and leave.)
  const int n_keys = (n < 1 || n > p.N) ? 0 : n;
  const int s_tree = (int)(L / p.chunk) < p.n_split - 1 ? (int)(L / p.chunk) : p.n_split - 1;
  const bool tail = (split == s_tree);   // this CTA's keys include the tree
  const long long kb = (long long)split * p.chunk;
  const long long ke = split < s_tree ? kb + p.chunk : (tail ? L + n_keys : kb);
  // Paged KV: tiles start on 64-key boundaries of the logical slots (so that a tile never
  // straddles a block of >= 64 slots, and a block of fewer slots fills whole 16-row groups of
  // the swizzled tile); keys below kb are masked.  Contiguous: tiles start at kb.
  const bool paged = p.table != nullptr;
  const long long t0 = paged ? (kb & ~(long long)(kKT - 1)) : kb;
  const int T = ke > kb ? (int)((ke - t0 + kKT - 1) / kKT) : 0;
  // paged: this CTA's block-table entries (-1 beyond the table), staged for the producer below
  const int blk0 = paged ? (int)(t0 >> p.bs_shift) : 0;
  const int nblk = paged ? (int)(((t0 + (long long)T * kKT - 1) >> p.bs_shift) - blk0 + 1) : 0;
  const bool tbl_staged = nblk <= kMaxBlkCta;

  // K/V tile t of this split -> ring stage t % kStages (the caller has made that stage free and
  // armed the stage's barrier for 2 * kTile bytes): the loads that lane `ln` of `nl` cooperating
  // lanes issues -- a d-chunk of a contiguous tile, or a box of a paged one with its block-table
  // lookup (one thread issuing a paged tile's 16 copies and 4 lookups in turn was the slowest step
  // of the loop with blocks of 16 slots; one lane per copy was no faster than one per box)
  auto tile_loads = [&](int t, int ln, int nl) {
    const int st = t % kStages;
    const long long key = t0 + (long long)t * kKT;
    if (!paged) {
      for (int c = ln; c < D / 64; c += nl) {
        tma_load_3d(sK + st * C::kTile + c * kKT * 128, &tmK, &full[st], c * 64, (int)key, bg);
        tma_load_3d(sV + st * C::kTile + c * kKT * 128, &tmV, &full[st], c * 64, (int)key, bg);
      }
    } else {
      // boxes of min(bs, 64) rows; a slot beyond the table, or an entry out of range, reads
      // from outside the pool map (zero fill)
      const int rows = p.bs < kKT ? p.bs : kKT;
      const long long zlim = (long long)p.num_blocks * p.Hkv;
      for (int i = ln; i < kKT / rows; i += nl) {
        const long long pos = key + (long long)i * rows;
        int y = 0, z = (int)zlim;
        if (pos < p.L_cap) {
          const int lb = (int)(pos >> p.bs_shift);
          const int blk = tbl_staged ? s_blk[lb - blk0] : p.table[(size_t)b * p.max_blocks + lb];
          const long long zz = (long long)blk * p.Hkv + g;
          if (blk >= 0 && zz < zlim) {
            y = (int)(pos & (p.bs - 1));
            z = (int)zz;
          }
        }
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_3d(sK + st * C::kTile + c * kKT * 128 + i * rows * 128, &tmK, &full[st], c * 64, y, z);
        if (p.v_rows < kKT) {  // both halves of the block's V rows in one box: [half][rows][128 B]
          tma_load_4d(sV + st * C::kTile + i * (D / 64) * rows * 128, &tmV, &full[st], 0, y, 0, z);
        } else {
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(sV + st * C::kTile + c * kKT * 128 + i * rows * 128, &tmV, &full[st], c * 64, y, z);
        }
      }
    }
  };
  // one thread: arm the stage's barrier, then every load of the tile
  auto issue_tile = [&](int t) {
    mbar_arrive_expect_tx(&full[t % kStages], 2 * C::kTile);
    tile_loads(t, 0, 1);
  };
  // Q (TMA path) and the first kStages K/V tiles (every stage starts free).  Contiguous caches
  // send them before the tree checks and the ancestor bits, which then overlap the loads; paged
  // pools send them once the block-table entries are staged.
  const int pre = T < kStages ? T : kStages;
  auto issue_first = [&]() {
    if (T == 0) return;
    if (p.q_tma) {
      // box (64 dims, G heads, 128 / G nodes) = 128 rows (node, head) in row order, swizzled
      // like the MMA's A operand; rows past the last node read as zeros
      mbar_arrive_expect_tx(qfull, kGroups * C::kQ);
      const int npg = kGR / p.G;  // nodes per group
#pragma unroll
      for (int a = 0; a < kGroups; ++a)
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
          tma_load_4d(sQ + a * C::kQ + c * kGR * 128, &tmQ, qfull, c * 64, g * p.G, (row0 / p.G) + a * npg, b);
    }
    for (int t = 0; t < pre; ++t) issue_tile(t);
    s_issued = pre;
  };
  const bool early = !paged;
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kGroups);  // one P V commit per group's issuer
    }
    for (int a = 0; a < kGroups; ++a) {
      mbar_init(&sfull[a], 1);
      mbar_init(&sfree[a], 4);
      mbar_init(&pfull[2 * a], 4);
      mbar_init(&pfull[2 * a + 1], 4);
      mbar_init(&ofull[2 * a], 1);
      mbar_init(&ofull[2 * a + 1], 1);
    }
    for (int a = 0; a < kGroups; ++a) mbar_init(&drained[a], 1);
    mbar_init(qfull, 1);
    s_abort = 0;
    s_issued = 0;
    s_consumed = 0;
    fence_mbar_init();
    if (early) issue_first();
  }
  // a CTA that leaves before its tile loop lets its early loads land first (tid 0 issued them)
  auto drain_first = [&]() {
    if (tid != 0 || !early || T == 0) return;
    for (int u = 0; u < s_issued; ++u) mbar_wait_bounded(&full[u], 0, nullptr);
    if (p.q_tma) mbar_wait_bounded(qfull, 0, nullptr);
  };

  // ---- tree checks, done by every CTA of the request (same verdict everywhere) ----
  int bad_tree = (n < 1 || n > p.N) ? 1 : 0, bad_cap = 0;
  if (!bad_tree) {
    bad_cap = (L < 0 || L + n > p.L_cap) ? 1 : 0;
    for (int c = tid; c < n; c += kTcThreads) {
      const int par = p.parent[(size_t)b * p.N + c];
      s_par[c] = par;
      if (c == 0 ? par != -1 : (par < 0 || par >= c)) bad_tree = 1;
    }
  }
  bad_tree = __syncthreads_or(bad_tree);
  bad_cap = __syncthreads_or(bad_cap);
  // With a single split the kernel writes the final rows itself (no merge); rows it does not
  // compute (bad request, padded node) are zeroed here as the merge would.
  auto zero_rows = [&]() {
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out);
    for (int c = tid; c < kRowsCta * (D / 8); c += kTcThreads) {
      const int rr = c / (D / 8), row = row0 + rr;
      if (row >= rows_total) continue;
      const size_t orow = ((size_t)b * p.N + row / p.G) * p.Hq + g * p.G + row % p.G;
      *reinterpret_cast<uint4*>(out + orow * D + (c % (D / 8)) * 8) = make_uint4(0, 0, 0, 0);
      if (p.lse && c % (D / 8) == 0) p.lse[orow] = 0.f;
    }
  };
  const int err = bad_tree ? SPEC_ERR_BAD_TREE : (bad_cap ? SPEC_ERR_CAPACITY : 0);
  if (tid == 0 && split == 0 && rg == 0 && g == 0) p.tree_bad[b] = err ? 1 : 0;  // for the merge
  if (err) {  // the merge kernel (or, with one split, this CTA) zeroes this request's outputs
    if (tid == 0 && rg == 0 && split == 0 && g == 0) set_status(p.dev_status, err);
    if (p.direct) zero_rows();
    drain_first();
    return;
  }
  if (paged && tail) {  // every tree-split CTA of the request checks its whole table (same verdict)
    const long long used = (L + n + p.bs - 1) >> p.bs_shift;
    int badt = 0;
    for (long long j = tid; j < used; j += kTcThreads) {
      const int blk = p.table[(size_t)b * p.max_blocks + j];
      if (blk < 0 || blk >= p.num_blocks) badt = 1;
    }
    badt = __syncthreads_or(badt);
    if (tid == 0) {
      p.req_bad[b] = badt;
      if (badt && rg == 0 && g == 0) set_status(p.dev_status, SPEC_ERR_CAPACITY);
    }
    if (badt && p.direct) {
      zero_rows();
      return;
    }
  }
  if (T == 0) {  // no keys here: the merge skips this split
    if (p.direct) {
      zero_rows();
      return;
    }
    for (int rr = tid; rr < kRowsCta; rr += kTcThreads) {
      if (row0 + rr >= rows_total) break;
      const int row = row0 + rr, i = row / p.G, h = g * p.G + row % p.G;
      const size_t orow = ((size_t)b * p.N + i) * p.Hq + h;
      p.part_ml[orow * p.n_split + split] = make_float2(-INFINITY, 0.f);
    }
    return;
  }

  // ---- ancestor bits of this CTA's rows (tree split) ----
  if (tail) {
    // pointer jumping: s_nanc[c] = nodes from c up to, not including, s_jmp[c]
    for (int c = tid; c < n; c += kTcThreads) {
#pragma unroll
      for (int w = 0; w < kAncWords; ++w) s_nanc[c][w] = 0u;
      s_nanc[c][c >> 5] = 1u << (c & 31);
      s_jmp[c] = (c == 0) ? -1 : s_par[c];
    }
    __syncthreads();
    for (int round = 0; round < 8; ++round) {  // 2^8 >= 255 levels; up to two nodes per thread
      int jj[2] = {-1, -1}, nj[2] = {-1, -1};
      uint32_t up[2][kAncWords];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int c = tid + k * kTcThreads;
        if (c < n) {
          jj[k] = s_jmp[c];
          if (jj[k] >= 0) {
            nj[k] = s_jmp[jj[k]];
#pragma unroll
            for (int w = 0; w < kAncWords; ++w) up[k][w] = s_nanc[jj[k]][w];
          }
        }
      }
      __syncthreads();
      int more = 0;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int c = tid + k * kTcThreads;
        if (c < n && jj[k] >= 0) {
#pragma unroll
          for (int w = 0; w < kAncWords; ++w) s_nanc[c][w] |= up[k][w];
          s_jmp[c] = nj[k];
          more |= nj[k] >= 0;
        }
      }
      if (!__syncthreads_or(more)) break;  // every node's set reaches the root
    }
    for (int c = tid; c < kRowsCta * kAncWords; c += kTcThreads) {
      const int r = c / kAncWords, w = c % kAncWords, row = row0 + r;
      uint32_t word = 0;
      if (row < rows_total) {
        const int i = row / p.G;
        if (i < n) word = s_nanc[i][w];
      }
      sAnc[c] = word;
    }
  }
  if (paged && tbl_staged)
    for (int j = tid; j < nblk; j += kTcThreads) {
      const int lb = blk0 + j;
      s_blk[j] = lb < p.max_blocks ? p.table[(size_t)b * p.max_blocks + lb] : -1;
    }
  if (warp == 1) {
    tmem_alloc(&s_tmem, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();  // barriers initialised, block-table entries staged
  tc_fence_after();

  if (!early && warp == 0 && lane == 0) issue_first();

  if (!p.q_tma) {
    // ---- Q rows -> shared memory in the K-major 128-byte-swizzle layout of the MMA A operand ----
    // Every load of a thread is issued before its first store, so the loads overlap.
    constexpr int NCH = D / 8;
    constexpr int kQPer = (kRowsCta * NCH + kTcThreads - 1) / kTcThreads;
    const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(p.q);
    uint4 qv[kQPer];
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int c = tid + k * kTcThreads;
      const int rr = c / NCH, ch = c % NCH, row = row0 + rr;
      qv[k] = make_uint4(0, 0, 0, 0);
      if (c < kRowsCta * NCH && row < rows_total) {
        const int i = row / p.G, j = row % p.G;
        qv[k] = *reinterpret_cast<const uint4*>(q + (((size_t)b * p.N + i) * p.Hq + g * p.G + j) * D + ch * 8);
      }
    }
#pragma unroll
    for (int k = 0; k < kQPer; ++k) {
      const int c = tid + k * kTcThreads;
      if (c < kRowsCta * NCH) {
        const int rr = c / NCH, ch = c % NCH;
        *reinterpret_cast<uint4*>(sQ + (rr / kGR) * C::kQ + sw128_off(rr % kGR, ch, kGR)) = qv[k];
      }
    }
    fence_proxy_async_smem();  // Q (generic stores) becomes visible to the tensor cores
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
  }
  const uint32_t tmem = s_tmem;

  if (warp == 0) {
    // ---- TMA producer (tiles pre .. T-1): lane 0 waits for the stage and arms its barrier, then
    // the warp's lanes issue the tile's loads side by side ----
    bool ok = true;
    for (int t = pre; t < T; ++t) {
      const int st = t % kStages;
      const bool got = lane == 0 ? mbar_wait_bounded(&empty[st], ((t / kStages) & 1) ^ 1, &s_abort) : true;
      if (!__shfl_sync(0xffffffffu, got, 0)) {
        ok = false;
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(&full[st], 2 * C::kTile);
      __syncwarp();
      tile_loads(t, lane, 32);
      __syncwarp();
      if (lane == 0) s_issued = t + 1;
    }
    if (!ok && lane == 0) {
      s_abort = 1;
      set_status(p.dev_status, SPEC_ERR_TIMEOUT);
    }
  } else if (warp == 1 || warp >= 2 + 4 * kGroups) {
    // ---- MMA issuers: group 0 on warp 1, group g > 0 on warp 1 + 4 * kGroups + g ----
    const int ga = (warp == 1) ? 0 : warp - (1 + 4 * kGroups);
    if (lane == 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kGR, kKT, 0);
      constexpr uint32_t idP = idesc_bf16_f32(kGR, D, 1);
      const int vr = p.v_rows;  // rows per V box group (the tile's layout): 16, 32 or 64
      const int vr_shift = 31 - __clz(vr);
      bool ok = true;
      // Issue order for the group: S(0), then per tile t: S(t + 1) as soon as the softmax has
      // read S(t) (early in its work on tile t, so the next scores are ready when it finishes),
      // then P V(t) as soon as P(t) is written.  K/V stage t is released once every group's
      // issuer has committed its P V(t).  Waits suspend in the barrier.
      auto issue_s = [&](int t) -> bool {
        const int st = t % kStages;
        if (!mbar_wait_bounded(&full[st], (t / kStages) & 1, &s_abort)) return false;
        if (t > 0 && !mbar_wait_bounded(&sfree[ga], (t - 1) & 1, &s_abort)) return false;
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
      auto issue_pv = [&](int t) -> bool {
        // one barrier per P buffer: the softmax may finish tile t + 1 before this wait for tile t
        // begins, but never tile t + 2 (it needs S(t + 2), issued after this P V)
        if (!mbar_wait_bounded(&pfull[2 * ga + (t & 1)], (t >> 1) & 1, &s_abort)) return false;
        tc_fence_after();
        const uint32_t pt = tmem + C::kColP + (2 * ga + (t & 1)) * (kKT / 2);  // P(t) in TMEM
        const uint32_t va = smem_u32(sV + (t % kStages) * C::kTile);
#pragma unroll
        for (int kk = 0; kk < kKT / 16; ++kk) {
          // keys 16 kk .. 16 kk + 15 of the tile: in V block (16 kk) / v_rows, at row (16 kk) % v_rows;
          // the two 64-column halves of d lie v_rows * 128 bytes apart
          const int kr = kk * 16;
          const uint32_t voff = (uint32_t)(((kr >> vr_shift) * (D / 64) << vr_shift) * 128 + (kr & (vr - 1)) * 128);
          const uint64_t bd = sdesc_sw128(va + voff, (uint32_t)vr * 128, 1024);
          umma_bf16_tmem_a(tmem + C::kColO + ga * D, pt + kk * 8, bd, idP, (t > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&ofull[2 * ga + (t & 1)]);
        return true;
      };
      ok = !p.q_tma || mbar_wait_bounded(qfull, 0, &s_abort);
      ok = ok && issue_s(0);
      for (int t = 0; t < T && ok; ++t) {
        if (t + 1 < T) ok = issue_s(t + 1);
        ok = ok && issue_pv(t);
        if (!ok) break;
        umma_commit(&empty[t % kStages]);  // this group is done with K/V tile t
        if (ga == 0) s_consumed = t + 1;
      }
      if (!ok) {
        s_abort = 1;
        set_status(p.dev_status, SPEC_ERR_TIMEOUT);
      }
      // every MMA this thread issued has finished once drained[ga] completes
      umma_commit(&drained[ga]);
      mbar_wait_bounded(&drained[ga], 0, nullptr);
    }
  } else {
    // ---- softmax: warps 2..9; group a = (warp - 2) / 4, TMEM lane quarter q4 = warp % 4 ----
    const int a = (warp - 2) >> 2, q4 = warp & 3;
    const int rl = q4 * 32 + lane;            // row within the group (TMEM lane)
    const int rr = a * kGR + rl;              // row within the CTA
    const int row = row0 + rr;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const uint32_t tS = tmem + C::kColS + a * kKT + lane_off;
    const uint32_t tO = tmem + C::kColO + a * D + lane_off;
    const uint32_t tP = tmem + C::kColP + 2 * a * (kKT / 2) + lane_off;  // + (t & 1) * kKT / 2
    float m_run = -INFINITY, l_run = 0.f;
    const uint32_t* anc = sAnc + rr * kAncWords;  // this row's ancestor words (tree split)
    bool ok = true;
    for (int t = 0; t < T; ++t) {
      if (!mbar_wait_bounded(&sfull[a], t & 1, &s_abort)) {
        ok = false;
        break;
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
      const long long kbase = t0 + (long long)t * kKT;
      if (tail && kbase + kKT > L) {
        // key j of the tile is tree node kbase - L + j when that is >= 0, else a prefix key; the
        // ancestor bits come from a 64-bit window of the row's ancestor words in shared memory
        // (held in registers, the words would need a runtime index, which puts them in local
        // memory); nodes outside [0, n) have no bit
        const int off = (int)(kbase - L);   // >= -63
        const int lo = off >> 5;            // floor division (off may be negative)
        const int r = off - (lo << 5);      // 0..31
        const uint32_t w0 = (lo >= 0 && lo < kAncWords) ? anc[lo] : 0u;
        const uint32_t w1 = (lo + 1 >= 0 && lo + 1 < kAncWords) ? anc[lo + 1] : 0u;
        const uint32_t w2 = (lo + 2 >= 0 && lo + 2 < kAncWords) ? anc[lo + 2] : 0u;
        const unsigned long long win = ((unsigned long long)w1 << 32) | w0;
        unsigned long long mask = (win >> r) | (r ? ((unsigned long long)w2 << (64 - r)) : 0ull);
        if (off < 0) mask |= (1ull << -off) - 1ull;  // the tile's first -off keys are prefix keys
        if (kbase < kb) mask &= ~((1ull << (kb - kbase)) - 1ull);  // paged: keys before the split
#pragma unroll
        for (int j = 0; j < kKT; ++j)
          if (!((mask >> j) & 1ull)) v[j] = -INFINITY;
      } else if (kbase + kKT > ke || kbase < kb) {
#pragma unroll
        for (int j = 0; j < kKT; ++j) {
          const long long kidx = kbase + j;
          if (!(kidx >= kb && kidx < ke)) v[j] = -INFINITY;
        }
      }
      float mx[4] = {v[0], v[1], v[2], v[3]};
#pragma unroll
      for (int j = 4; j < kKT; ++j) mx[j & 3] = fmaxf(mx[j & 3], v[j]);
      const float tmax = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * p.scale_log2;
      const float m_new = fmaxf(m_run, tmax);
      const bool need = m_new > m_run + kRescaleLog2;  // includes the first finite maximum
      if (__any_sync(0xffffffffu, need)) {
        const float f = need ? exp2f(m_run - m_new) : 1.f;  // 0 when m_run is -inf
        if (t > 0) {
          // P V(t - 1) must have landed in O before O is rescaled
          if (!mbar_wait_bounded(&ofull[2 * a + ((t - 1) & 1)], ((t - 1) >> 1) & 1, &s_abort)) {
            ok = false;
            break;
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
      // exponents two at a time (packed fp32 pairs: one FFMA2 per pair, one FADD2 per pair into
      // two running pair sums)
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
      // P buffer t & 1 was last read by P V(t - 2).  This group's issuer issued that MMA before
      // S(t), and the commit that completed sfull for S(t) tracks every earlier MMA of that
      // thread, so the buffer is already free.
      tmem_st_x32(tP + (t & 1) * (kKT / 2), pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pfull[2 * a + (t & 1)]);
    }
    // the TMEM loads below are warp-collective: the warp takes one branch
    const bool fin = __all_sync(0xffffffffu, ok && mbar_wait_bounded(&ofull[2 * a + ((T - 1) & 1)], ((T - 1) >> 1) & 1, &s_abort));
    // Once every group's last P V has completed, no MMA or copy reads or writes the Q / K / V / P
    // region any more: the O rows are staged there and leave through the bulk-copy engine.
    named_bar_sync(1, 128 * kGroups);
    const bool valid = row < rows_total;
    const int i_node = row / p.G;
    size_t orow = 0;
    if (valid) orow = ((size_t)b * p.N + i_node) * p.Hq + g * p.G + row % p.G;
    uint8_t* srow = base + rr * C::kORow;
    if (p.direct) {
      // one split: the final bf16 row and its natural-log LSE (zeros for padded nodes and after a
      // failed wait)
      const bool live = fin && i_node < n;
      if (fin) tc_fence_after();
      const float inv = (live && l_run > 0.f) ? 1.f / l_run : 0.f;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        if (fin) {
          tmem_ld_x32(tO + c * 32, o);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) o[j] = 0u;
        }
#pragma unroll
        for (int j = 0; j < 32; j += 8)
          *reinterpret_cast<uint4*>(srow + (c * 32 + j) * 2) =
              make_uint4(pack_bf16x2(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv),
                         pack_bf16x2(__uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv),
                         pack_bf16x2(__uint_as_float(o[j + 4]) * inv, __uint_as_float(o[j + 5]) * inv),
                         pack_bf16x2(__uint_as_float(o[j + 6]) * inv, __uint_as_float(o[j + 7]) * inv));
      }
      if (valid) {
        if (p.lse) p.lse[orow] = (live && l_run > 0.f) ? (m_run + log2f(l_run)) * 0.69314718055994531f : 0.f;
        fence_proxy_async_smem();
        bulk_store_row(static_cast<__nv_bfloat16*>(p.out) + orow * D, srow, D * 2);
        bulk_wait_read();
      }
      if (!fin && lane == 0) {
        s_abort = 1;
        set_status(p.dev_status, SPEC_ERR_TIMEOUT);
      }
    } else if (fin) {
      tc_fence_after();
      if (valid) p.part_ml[orow * p.n_split + split] = make_float2(m_run, l_run);
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      // the normalised partial row in bf16: its rounding (2^-9 relative) is far inside the output
      // tolerance, and it halves what the merge reads
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld_x32(tO + c * 32, o);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; j += 8)
          *reinterpret_cast<uint4*>(srow + (c * 32 + j) * 2) =
              make_uint4(pack_bf16x2(__uint_as_float(o[j]) * inv, __uint_as_float(o[j + 1]) * inv),
                         pack_bf16x2(__uint_as_float(o[j + 2]) * inv, __uint_as_float(o[j + 3]) * inv),
                         pack_bf16x2(__uint_as_float(o[j + 4]) * inv, __uint_as_float(o[j + 5]) * inv),
                         pack_bf16x2(__uint_as_float(o[j + 6]) * inv, __uint_as_float(o[j + 7]) * inv));
      }
      if (valid) {
        fence_proxy_async_smem();  // the staged row (generic stores) becomes visible to the copy
        bulk_store_row(p.part_o + (orow * p.n_split + split) * D, srow, D * 2);
        bulk_wait_read();
      }
    } else {
      if (lane == 0) {
        s_abort = 1;
        set_status(p.dev_status, SPEC_ERR_TIMEOUT);
      }
      if (valid) p.part_ml[orow * p.n_split + split] = make_float2(-INFINITY, 0.f);  // the merge skips this split
    }
  }

  __syncthreads();
  if (tid == 0 && s_abort) {
    // let the copies still in flight land before shared memory is released
    for (int u = s_consumed; u < s_issued; ++u)
      mbar_wait_bounded(&full[u % kStages], (uint32_t)((u / kStages) & 1), nullptr);
    if (p.q_tma) mbar_wait_bounded(qfull, 0, nullptr);
  }
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, C::kTmemCols);
}

int attention_tc_rows_per_cta(int groups) { return kGR * groups; }

template <int D, int NG>
static cudaError_t launch_tc(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV, const AttnParams& p,
                             cudaStream_t stream) {
  using C = AttnTcCfg<D, NG>;
  const dim3 grid(p.n_rg, p.n_split, p.B * p.Hkv);
  cudaError_t err = cudaFuncSetAttribute(attn_tc_kernel<D, NG>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (err != cudaSuccess) return err;
  attn_tc_kernel<D, NG><<<grid, C::kThreads, C::kSmem, stream>>>(*tmQ, *tmK, *tmV, p);
  return cudaGetLastError();
}

cudaError_t launch_attention_tc(const CUtensorMap* tmQ, const CUtensorMap* tmK, const CUtensorMap* tmV,
                                const AttnParams& p, cudaStream_t stream) {
  if (p.d == 128)
    return p.groups == 2 ? launch_tc<128, 2>(tmQ, tmK, tmV, p, stream) : launch_tc<128, 1>(tmQ, tmK, tmV, p, stream);
  return p.groups == 2 ? launch_tc<64, 2>(tmQ, tmK, tmV, p, stream) : launch_tc<64, 1>(tmQ, tmK, tmV, p, stream);
}

}  // namespace spectree

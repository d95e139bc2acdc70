// K4: KV compaction after acceptance.
//
// Candidates after a rejection are discarded and the accepted prefix is kept (qiita
// "EAGLE-3とMedusaで実装するSpeculative Decoding実践ガイド", section "棄却サンプリング").  The
// accepted path's K/V rows are gathered from their tree slots L + path[j] to L + j, in place.
// Paged caches map each logical slot through the request's block table (the moves are the
// same, between physical rows).
// One CTA per (request, KV head); rows are copied in batches of up to 64 that are read whole
// into shared memory before any of them is written, batches in increasing j.  That order is
// hazard-free: path[j] >= j for a root path in topological order, so a row's source slot
// L + path[j'] can only be the destination L + j of a row j >= j', i.e. of a row in the same
// batch (written after the whole batch was read) or in a later batch.

#include "common.cuh"
#include "kernels.cuh"

namespace spectree {

constexpr int kCompactBufChunks = 2048;  // 32 KB of staged rows (64 bf16 rows of d = 128, K and V)

__global__ void __launch_bounds__(128) compact_kv_kernel(
    uint8_t* __restrict__ k, uint8_t* __restrict__ v, int row_bytes, const int32_t* __restrict__ prefix_len,
    const int32_t* __restrict__ path, const int32_t* __restrict__ accept_len, int Hkv, long long L_cap,
    int path_cap, int32_t* __restrict__ src_slot, int32_t* __restrict__ new_len, int32_t* dev_status,
    const PagedKV pg) {
  const int b = blockIdx.x / Hkv, g = blockIdx.x % Hkv, tid = threadIdx.x;
  const long long L = prefix_len[b];
  const int len = accept_len[b];
  const int32_t* pth = path + (size_t)b * path_cap;
  __shared__ uint4 s_buf[kCompactBufChunks];
  __shared__ int s_pth[kCompactBufChunks / 8];
  // path checks, spread over the threads (every branch below depends on block-uniform values)
  int err = 0;
  if (len < 0 || len >= path_cap || L < 0) {
    err = (len >= path_cap) ? SPEC_ERR_CAPACITY : SPEC_ERR_BAD_TREE;
  } else {
    int bad = 0;
    for (int j = tid; j <= len; j += blockDim.x) {
      const int pj = pth[j];
      if (j == 0 ? pj != 0 : pj <= pth[j - 1]) bad = 1;
    }
    if (__syncthreads_or(bad)) {
      err = SPEC_ERR_BAD_TREE;
    } else {
      const long long last = L + pth[len];
      if (last >= L_cap) {
        err = SPEC_ERR_CAPACITY;
      } else if (pg.table) {  // every block the moves touch: slots [L, L + path[len]]
        int badb = 0;
        for (long long lb = (L >> pg.bs_shift) + tid; lb <= (last >> pg.bs_shift); lb += blockDim.x) {
          const int blk = pg.table[(size_t)b * pg.max_blocks + lb];
          if (blk < 0 || blk >= pg.num_blocks) badb = 1;
        }
        if (__syncthreads_or(badb)) err = SPEC_ERR_CAPACITY;
      }
    }
  }
  if (err) {
    if (g == 0) {
      if (tid == 0) {
        set_status(dev_status, err);
        if (new_len) new_len[b] = (int)L;
      }
      if (src_slot)
        for (int j = tid; j < path_cap; j += blockDim.x) src_slot[(size_t)b * path_cap + j] = -1;
    }
    return;
  }
  const int chunks = row_bytes / 16;       // 16-byte pieces of one K (or V) row
  const int per_row = 2 * chunks;            // K and V
  const int batch = kCompactBufChunks / per_row;
  const size_t head_off = ((size_t)b * Hkv + g) * (size_t)L_cap;
  // row index of logical slot s of this (request, KV head) in the cache, or in the paged pool
  auto phys = [&](long long s) -> size_t {
    if (!pg.table) return head_off + (size_t)s;
    const int blk = pg.table[(size_t)b * pg.max_blocks + (s >> pg.bs_shift)];
    return ((size_t)blk * Hkv + g) * (size_t)pg.bs + (size_t)(s & (pg.bs - 1));
  };
  for (int j0 = 1; j0 <= len; j0 += batch) {
    const int nb = min(batch, len + 1 - j0);
    if (tid < nb) s_pth[tid] = pth[j0 + tid];
    __syncthreads();
    for (int i = tid; i < nb * per_row; i += blockDim.x) {
      const int jj = i / per_row, c = i - jj * per_row;
      const uint8_t* base = (c < chunks) ? k : v;
      const int cc = (c < chunks) ? c : c - chunks;
      const size_t src = phys(L + s_pth[jj]);
      s_buf[i] = *reinterpret_cast<const uint4*>(base + src * row_bytes + cc * 16);
    }
    __syncthreads();
    for (int i = tid; i < nb * per_row; i += blockDim.x) {
      const int jj = i / per_row, c = i - jj * per_row;
      if (s_pth[jj] == j0 + jj) continue;  // already in place
      uint8_t* base = (c < chunks) ? k : v;
      const int cc = (c < chunks) ? c : c - chunks;
      const size_t dst = phys(L + j0 + jj);
      *reinterpret_cast<uint4*>(base + dst * row_bytes + cc * 16) = s_buf[i];
    }
    __syncthreads();
  }
  if (g == 0) {
    if (src_slot)
      for (int j = tid; j < path_cap; j += blockDim.x)
        src_slot[(size_t)b * path_cap + j] = (j <= len) ? (int)(L + pth[j]) : -1;
    if (tid == 0 && new_len) new_len[b] = (int)(L + 1 + len);
  }
}

void launch_compact_kv(void* k, void* v, int elem_bytes, const int32_t* prefix_len,
                       const int32_t* path, const int32_t* accept_len, int B, int Hkv, int d,
                       long long L_cap, int path_cap, int32_t* src_slot, int32_t* new_len,
                       int32_t* dev_status, const PagedKV& pg, cudaStream_t stream) {
  compact_kv_kernel<<<B * Hkv, 128, 0, stream>>>(static_cast<uint8_t*>(k), static_cast<uint8_t*>(v),
                                                d * elem_bytes, prefix_len, path, accept_len, Hkv,
                                                L_cap, path_cap, src_slot, new_len, dev_status, pg);
}

}  // namespace spectree

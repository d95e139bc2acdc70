// Device side of KV compaction (K4), shared by the compaction kernel and the acceptance kernels
// that fold compaction into their tail.
//
// Candidates after a rejection are discarded and the accepted prefix is kept (qiita
// "EAGLE-3とMedusaで実装するSpeculative Decoding実践ガイド", section "棄却サンプリング"): the accepted
// path's K/V rows move from their tree slots L + path[j] to L + j, in place.  Rows are copied in
// batches of up to 64 that are read whole into shared memory before any of them is written,
// batches in increasing j.  That order is hazard-free: path[j] >= j for a root path in
// topological order, so a row's source slot L + path[j'] can only be the destination L + j of a
// row j >= j', i.e. of a row in the same batch (written after the whole batch was read) or in a
// later batch.
#pragma once

#include "common.cuh"
#include "kernels.cuh"

namespace spectree {

// Compacts request b on KV heads g = g0, g0 + gstep, ... < Hkv.  Every thread of the block calls
// it (block-wide barriers inside, block-uniform arguments); s_buf holds kCompactBufChunks 16-byte
// chunks, s_pth kCompactBufChunks / 8 ints.  Writes src_slot / new_len when it handles head 0.
// `pth` (global or shared memory) holds request b's accepted path and `len` its length.
__device__ __forceinline__ void compact_request(const CompactParams& c, const int32_t* pth, int len, int b, int g0,
                                                int gstep, uint4* s_buf, int* s_pth) {
  const int tid = threadIdx.x;
  const long long L = c.prefix_len[b];
  // path checks, spread over the threads (every branch below depends on block-uniform values)
  int err = 0;
  if (len < 0 || len >= c.path_cap || L < 0) {
    err = (len >= c.path_cap) ? SPEC_ERR_CAPACITY : SPEC_ERR_BAD_TREE;
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
      if (last >= c.L_cap) {
        err = SPEC_ERR_CAPACITY;
      } else if (c.pg.table) {  // every block the moves touch: slots [L, L + path[len]]
        int badb = 0;
        for (long long lb = (L >> c.pg.bs_shift) + tid; lb <= (last >> c.pg.bs_shift); lb += blockDim.x) {
          const int blk = c.pg.table[(size_t)b * c.pg.max_blocks + lb];
          if (blk < 0 || blk >= c.pg.num_blocks) badb = 1;
        }
        if (__syncthreads_or(badb)) err = SPEC_ERR_CAPACITY;
      }
    }
  }
  if (err) {
    if (g0 == 0) {
      if (tid == 0) {
        set_status(c.dev_status, err);
        if (c.new_len) c.new_len[b] = (int)L;
      }
      if (c.src_slot)
        for (int j = tid; j < c.path_cap; j += blockDim.x) c.src_slot[(size_t)b * c.path_cap + j] = -1;
    }
    return;
  }
  const int chunks = c.row_bytes / 16;       // 16-byte pieces of one K (or V) row
  const int per_row = 2 * chunks;            // K and V
  const int batch = kCompactBufChunks / per_row;
  for (int g = g0; g < c.Hkv; g += gstep) {
    const size_t head_off = ((size_t)b * c.Hkv + g) * (size_t)c.L_cap;
    // row index of logical slot s of this (request, KV head) in the cache, or in the paged pool
    auto phys = [&](long long s) -> size_t {
      if (!c.pg.table) return head_off + (size_t)s;
      const int blk = c.pg.table[(size_t)b * c.pg.max_blocks + (s >> c.pg.bs_shift)];
      return ((size_t)blk * c.Hkv + g) * (size_t)c.pg.bs + (size_t)(s & (c.pg.bs - 1));
    };
    for (int j0 = 1; j0 <= len; j0 += batch) {
      const int nb = min(batch, len + 1 - j0);
      if (tid < nb) s_pth[tid] = pth[j0 + tid];
      __syncthreads();
      for (int i = tid; i < nb * per_row; i += blockDim.x) {
        const int jj = i / per_row, cc0 = i - jj * per_row;
        const uint8_t* base = (cc0 < chunks) ? c.k : c.v;
        const int cc = (cc0 < chunks) ? cc0 : cc0 - chunks;
        const size_t src = phys(L + s_pth[jj]);
        s_buf[i] = *reinterpret_cast<const uint4*>(base + src * c.row_bytes + cc * 16);
      }
      __syncthreads();
      for (int i = tid; i < nb * per_row; i += blockDim.x) {
        const int jj = i / per_row, cc0 = i - jj * per_row;
        if (s_pth[jj] == j0 + jj) continue;  // already in place
        uint8_t* base = (cc0 < chunks) ? c.k : c.v;
        const int cc = (cc0 < chunks) ? cc0 : cc0 - chunks;
        const size_t dst = phys(L + j0 + jj);
        *reinterpret_cast<uint4*>(base + dst * c.row_bytes + cc * 16) = s_buf[i];
      }
      __syncthreads();
    }
  }
  if (g0 == 0) {
    if (c.src_slot)
      for (int j = tid; j < c.path_cap; j += blockDim.x)
        c.src_slot[(size_t)b * c.path_cap + j] = (j <= len) ? (int)(L + pth[j]) : -1;
    if (tid == 0 && c.new_len) c.new_len[b] = (int)(L + 1 + len);
  }
}

}  // namespace spectree
